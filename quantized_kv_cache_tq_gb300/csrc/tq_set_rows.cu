// SET_ROWS: quantise-on-write of K/V rows into the packed TurboQuant cache.
//
// [TQ#36] "shuffle WHT": per 128-element block -- block norm, sign-randomised
// Walsh-Hadamard rotation (butterfly stages h = 1..64), nearest-centroid codes.
// The page moved the stages h < 32 from shared memory to warp shuffles and kept
// barriers for h = 32, 64 because its kernel holds one element per thread.  Here
// one warp owns a whole block (4 elements per lane, loaded with one 16-byte
// load), so stages h = 1, 2 stay inside a lane, h = 4..64 are lane shuffles and
// the kernel needs no shared memory and no barrier at all.
#include "tq_common.cuh"

namespace tq {
namespace {

template <int SRC>
__device__ __forceinline__ void load4(const void *base, int64_t off, int valid, float v[4]) {
  if (SRC == TQ_F32) {
    const float *p = static_cast<const float *>(base) + off;
    if (valid >= 4) {
      const float4 x = *reinterpret_cast<const float4 *>(p);
      v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else {
#pragma unroll
      for (int r = 0; r < 4; ++r) v[r] = (r < valid) ? p[r] : 0.f;
    }
  } else {
    const uint16_t *p = static_cast<const uint16_t *>(base) + off;
    uint16_t h[4] = {0, 0, 0, 0};
    if (valid >= 4) {
      const uint2 x = *reinterpret_cast<const uint2 *>(p);
      h[0] = x.x & 0xffff; h[1] = x.x >> 16; h[2] = x.y & 0xffff; h[3] = x.y >> 16;
    } else {
#pragma unroll
      for (int r = 0; r < 4; ++r) h[r] = (r < valid) ? p[r] : 0;
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if (SRC == TQ_F16) v[r] = __half2float(__ushort_as_half(h[r]));
      else v[r] = __bfloat162float(__ushort_as_bfloat16(h[r]));
    }
    if (valid <= 0) v[0] = v[1] = v[2] = v[3] = 0.f;
  }
}

// bit position of element (16w + i') inside qs word w, i' = 4a + r of lane a
__device__ __forceinline__ int qs2_bit(int ip) { return ip < 8 ? 4 * ip : 4 * (ip - 8) + 2; }
// bit position of element 32u + rr inside signs word u
__device__ __forceinline__ int sg_bit(int rr) {
  return rr < 16 ? 4 * (rr & 7) + 2 + (rr >> 3) : 4 * ((rr - 16) & 7) + ((rr - 16) >> 3);
}

template <int TYPE, int SRC>
__global__ void __launch_bounds__(256) set_rows_kernel(const SetRowsArgs a) {
  constexpr int NC = TypeTraits<TYPE>::NC;
  constexpr int QSB = TypeTraits<TYPE>::QSB;
  constexpr int HALF = NC / 2;
  const int lane = threadIdx.x & 31;
  const int64_t total = a.n_rows * a.n_kv_heads * a.n_blocks;
  const int64_t wid = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (wid >= total) return;

  // midpoints between neighbouring centroids (exact in fp32 for binary16 centroids)
  float thr[NC - 1];
#pragma unroll
  for (int k = 0; k < NC - 1; ++k) thr[k] = 0.5f * (a.cb.c[k] + a.cb.c[k + 1]);

  const int b = static_cast<int>(wid % a.n_blocks);
  const int64_t rh = wid / a.n_blocks;
  const int h = static_cast<int>(rh % a.n_kv_heads);
  const int64_t row = rh / a.n_kv_heads;
  const int64_t cell = a.cell_ids[row];
  if (cell < 0 || cell >= a.n_cells) {
    if (lane == 0) set_status(a.dev_status, TQ_ERR_DEVICE_CHECK);
    return;
  }

  const int e0 = b * QK + 4 * lane;
  const int valid = a.head_dim - e0;
  float v[4];
  load4<SRC>(a.src, (row * a.n_kv_heads + h) * a.head_dim + e0, valid, v);

  const float ss = warp_sum(v[0] * v[0] + v[1] * v[1] + v[2] * v[2] + v[3] * v[3]);
  const float scale = ss > 0.f ? rsqrtf(ss * 128.f) : 0.f;   // 1 / (|x| sqrt(128))
  apply_signs(v, a.cb, lane);
  wht128_warp(v, lane);

  int code[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const float y = v[r] * scale;
    int i = 0;
#pragma unroll
    for (int k = 0; k < NC - 1; ++k) i += (y >= thr[k]) ? 1 : 0;
    code[r] = (i >= HALF) ? i : (HALF - 1 - i);
  }

  const int64_t blk = (static_cast<int64_t>(h) * a.n_cells + cell) * a.n_blocks + b;
  if (lane == 0) a.norms[blk] = __half_as_ushort(__float2half_rn(sqrtf(ss)));

  uint32_t *qs = reinterpret_cast<uint32_t *>(a.qs + blk * QSB);
  if (TYPE == 4) {
    // word w <- lanes 2w, 2w+1; element 8w + 4a + r at bits 4(4a + r)
    const int aa = lane & 1;
    uint32_t x = 0;
#pragma unroll
    for (int r = 0; r < 4; ++r) x |= static_cast<uint32_t>(code[r]) << (4 * (4 * aa + r));
    x = warp_or(x, 2);
    if (aa == 0) qs[lane >> 1] = x;
  } else {
    // word w <- lanes 4w..4w+3; element 16w + i' (i' = 4a + r)
    const int aa = lane & 3;
    uint32_t x = 0;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint32_t f = (TYPE == 3) ? (code[r] & 3) : code[r];
      x |= f << qs2_bit(4 * aa + r);
    }
    x = warp_or(x, 4);
    if (aa == 0) qs[lane >> 2] = x;
    if (TYPE == 3) {
      // signs word u <- lanes 8u..8u+7; element 32u + rr (rr = 4a + r)
      const int a8 = lane & 7;
      uint32_t s = 0;
#pragma unroll
      for (int r = 0; r < 4; ++r) s |= static_cast<uint32_t>(code[r] >> 2) << sg_bit(4 * a8 + r);
      s = warp_or(s, 8);
      if (a8 == 0) reinterpret_cast<uint32_t *>(a.signs + blk * 16)[lane >> 3] = s;
    }
  }
}

template <int TYPE>
cudaError_t launch_type(int src_type, const SetRowsArgs &a, cudaStream_t s) {
  const int64_t warps = a.n_rows * a.n_kv_heads * a.n_blocks;
  const int64_t grid = (warps + 7) / 8;
  switch (src_type) {
    case TQ_F32: set_rows_kernel<TYPE, TQ_F32><<<(unsigned)grid, 256, 0, s>>>(a); break;
    case TQ_F16: set_rows_kernel<TYPE, TQ_F16><<<(unsigned)grid, 256, 0, s>>>(a); break;
    default: set_rows_kernel<TYPE, TQ_BF16><<<(unsigned)grid, 256, 0, s>>>(a); break;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_set_rows(int type, int src_type, const SetRowsArgs &a, cudaStream_t s) {
  switch (type) {
    case TQ_TURBO2: return launch_type<2>(src_type, a, s);
    case TQ_TURBO3: return launch_type<3>(src_type, a, s);
    default: return launch_type<4>(src_type, a, s);
  }
}

}  // namespace tq

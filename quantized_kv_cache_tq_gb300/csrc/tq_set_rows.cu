// SET_ROWS: quantise-on-write of K/V rows into the packed TurboQuant cache.
//
// [TQ#36] "shuffle WHT": per 128-element block -- block norm, sign-randomised
// Walsh-Hadamard rotation (butterfly stages h = 1..64), nearest-centroid codes.
// The page's kernel holds one element per thread, so it needs shuffles for
// h = 1..16 and barriers for h = 32, 64.  Here four lanes own a block, 32
// elements each (lane l4 holds elements 4*l4 + 16*i + r, i = 0..7, r = 0..3, read
// as eight coalesced 16-byte loads), so five of the seven stages (h = 1, 2, 16,
// 32, 64) stay inside a lane and only h = 4, 8 are lane shuffles -- no shared
// memory, no barrier, and ~11 warp shuffles per block (one warp owns 8 blocks)
// instead of ~33 with one block per warp.
//
// The normalisation by the block norm is folded into the decision thresholds:
// with y = v / (|x| sqrt(128)) (v the unnormalised transform), y >= t becomes
// v >= t |x| sqrt(128), one multiply per threshold and block instead of one per
// element.  Codes are sign-magnitude: s = (y >= 0), j = #{positive thresholds
// <= |y|}.
#include "tq_common.cuh"

namespace tq {
namespace {

template <int SRC>
__device__ __forceinline__ void load4(const void *base, int64_t off, int valid, float v[4]) {
  if (SRC == TQ_F32) {
    const float *p = static_cast<const float *>(base) + off;
    if (valid >= 4) {
      const float4 x = __ldcs(reinterpret_cast<const float4 *>(p));
      v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else {
#pragma unroll
      for (int r = 0; r < 4; ++r) v[r] = (r < valid) ? p[r] : 0.f;
    }
  } else {
    const uint16_t *p = static_cast<const uint16_t *>(base) + off;
    uint16_t h[4] = {0, 0, 0, 0};
    if (valid >= 4) {
      const uint2 x = __ldcs(reinterpret_cast<const uint2 *>(p));
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
  }
}

__device__ __forceinline__ uint32_t pick4(uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3, int i) {
  return i == 0 ? x0 : i == 1 ? x1 : i == 2 ? x2 : x3;
}

// bit position of element 16w + ip inside qs word w (turbo2/3)
__device__ __forceinline__ int qs2_bit(int ip) { return ip < 8 ? 4 * ip : 4 * (ip - 8) + 2; }
// bit position of element 32u + rr inside signs word u (turbo3)
__device__ __forceinline__ int sg_bit(int rr) {
  return rr < 16 ? 4 * (rr & 7) + 2 + (rr >> 3) : 4 * ((rr - 16) & 7) + ((rr - 16) >> 3);
}

template <int TYPE, int SRC>
__global__ void __launch_bounds__(256) set_rows_kernel(const SetRowsArgs a) {
  constexpr int NC = TypeTraits<TYPE>::NC;
  constexpr int QSB = TypeTraits<TYPE>::QSB;
  constexpr int HALF = NC / 2;
  const int lane = threadIdx.x & 31;
  const int l4 = lane & 3;                     // position inside the block's 4 lanes
  const int64_t total = a.n_rows * a.n_kv_heads * a.n_blocks;
  const int64_t blk_id = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 2;
  const bool active = blk_id < total;          // whole 4-lane groups are active or not

  // per-lane +-1 multipliers of its 32 elements (bit 16i + 4*l4 + r of sign word i/2)
  float sgn[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const uint32_t w = a.cb.sign_bits[i >> 1];
      sgn[i][r] = ((w >> (16 * (i & 1) + 4 * l4 + r)) & 1u) ? -1.f : 1.f;
    }

  int b = 0, h = 0;
  int64_t row = 0, cell = 0;
  bool ok = false;
  float v[8][4];
  if (active) {
    b = static_cast<int>(blk_id % a.n_blocks);
    const int64_t rh = blk_id / a.n_blocks;
    h = static_cast<int>(rh % a.n_kv_heads);
    row = rh / a.n_kv_heads;
    cell = a.cell_ids[row];
    ok = cell >= 0 && cell < a.n_cells;
    if (!ok && l4 == 0) set_status(a.dev_status, TQ_ERR_DEVICE_CHECK);
  }
  const int64_t base = (row * a.n_kv_heads + h) * a.head_dim + b * QK;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e0 = 4 * l4 + 16 * i;
    if (ok) load4<SRC>(a.src, base + e0, a.head_dim - b * QK - e0, v[i]);
    else v[i][0] = v[i][1] = v[i][2] = v[i][3] = 0.f;
  }

  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      ss = fmaf(v[i][r], v[i][r], ss);
      v[i][r] *= sgn[i][r];
    }
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  ss += __shfl_xor_sync(0xffffffffu, ss, 2);

  // butterflies inside the lane: h = 1, 2 (r bits) and h = 16, 32, 64 (i bits)
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float a0 = v[i][0] + v[i][1], a1 = v[i][0] - v[i][1];
    const float a2 = v[i][2] + v[i][3], a3 = v[i][2] - v[i][3];
    v[i][0] = a0 + a2; v[i][2] = a0 - a2; v[i][1] = a1 + a3; v[i][3] = a1 - a3;
  }
#pragma unroll
  for (int hb = 1; hb < 8; hb <<= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (!(i & hb))
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float x = v[i][r], y = v[i | hb][r];
          v[i][r] = x + y;
          v[i | hb][r] = x - y;
        }
  // across the 4 lanes: h = 4 (lane ^ 1), h = 8 (lane ^ 2); element j takes
  // o = x[j ^ h] and becomes (j & h) ? o - x[j] : x[j] + o
#pragma unroll
  for (int m = 1; m < 4; m <<= 1) {
    const float sg = (l4 & m) ? -1.f : 1.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float o = __shfl_xor_sync(0xffffffffu, v[i][r], m);
        v[i][r] = fmaf(sg, v[i][r], o);
      }
  }

  // thresholds between positive centroids, scaled to the unnormalised domain
  const float nrm_scale = sqrtf(ss * 128.f);
  float thr[HALF - 1];
#pragma unroll
  for (int k = 0; k < HALF - 1; ++k)
    thr[k] = ss > 0.f ? 0.5f * (a.cb.c[HALF + k] + a.cb.c[HALF + k + 1]) * nrm_scale : INFINITY;

  uint32_t code[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float y = v[i][r], ay = fabsf(y);
      uint32_t j = 0;
#pragma unroll
      for (int k = 0; k < HALF - 1; ++k) j += (ay >= thr[k]) ? 1u : 0u;
      code[i][r] = (y >= 0.f) ? (HALF + j) : j;
    }

  // every lane takes part in the packing shuffles below; only valid blocks store
  const int64_t blk = (static_cast<int64_t>(h) * a.n_cells + cell) * a.n_blocks + b;
  if (ok && l4 == 0) a.norms[blk] = __half_as_ushort(__float2half_rn(sqrtf(ss)));
  uint32_t *qs = reinterpret_cast<uint32_t *>(a.qs + blk * QSB);
  if (TYPE == 4) {
    // word w = 2i + l4/2, element nibble 4*(l4 & 1) + r; lanes l4 and l4^1 share a word
    uint32_t wv[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t x = 0;
#pragma unroll
      for (int r = 0; r < 4; ++r) x |= code[i][r] << (4 * (4 * (l4 & 1) + r));
      wv[i] = x | __shfl_xor_sync(0xffffffffu, x, 1);
    }
    if (ok && (l4 & 1) == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) qs[2 * i + (l4 >> 1)] = wv[i];
    }
  } else {
    // qs word i holds elements 16i .. 16i+15; this lane's are 16i + 4*l4 + r
    uint32_t wq[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t x = 0;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t f = (TYPE == 3) ? (code[i][r] & 3u) : code[i][r];
        x |= f << qs2_bit(4 * l4 + r);
      }
      x |= __shfl_xor_sync(0xffffffffu, x, 1);
      x |= __shfl_xor_sync(0xffffffffu, x, 2);
      wq[i] = x;
    }
    if (ok)
      reinterpret_cast<uint2 *>(qs)[l4] = make_uint2(pick4(wq[0], wq[2], wq[4], wq[6], l4),
                                                     pick4(wq[1], wq[3], wq[5], wq[7], l4));
    if (TYPE == 3) {
      uint32_t ws[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        uint32_t x = 0;
#pragma unroll
        for (int ih = 0; ih < 2; ++ih)
#pragma unroll
          for (int r = 0; r < 4; ++r)
            x |= (code[2 * u + ih][r] >> 2) << sg_bit(16 * ih + 4 * l4 + r);
        x |= __shfl_xor_sync(0xffffffffu, x, 1);
        x |= __shfl_xor_sync(0xffffffffu, x, 2);
        ws[u] = x;
      }
      if (ok) reinterpret_cast<uint32_t *>(a.signs + blk * 16)[l4] = pick4(ws[0], ws[1], ws[2], ws[3], l4);
    }
  }
}

template <int TYPE>
cudaError_t launch_type(int src_type, const SetRowsArgs &a, cudaStream_t s) {
  const int64_t blocks = a.n_rows * a.n_kv_heads * a.n_blocks;
  const int64_t grid = (blocks * 4 + 255) / 256;
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

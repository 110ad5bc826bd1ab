// Prompt attention over an int8 KV cache with one binary16 scale per row,
// rows scattered over the cells ([QSA#1821] "What", "Change"):
//   k_t = k_int[cell_of_pos[t]] * scale_k,  v_t = v_int[...] * scale_v,
//   out[i][h] = softmax_{t <= p_i}(scale * q[i][h] . k_t) v_t.
//
// The page's sm_75 kernel gathers each 32-cell chunk's rows into registers
// during the previous chunk and shares one shared buffer between K and V to fit
// two blocks per SM.  On GB300 the gather is asynchronous instead: warp 0
// issues one 128-byte cp.async.bulk per scattered K or V row into a 2-deep ring,
// completion counted on an mbarrier, so the next tile's rows stream in while the
// tensor cores work on the current one.  The tile math is tcgen05:
//   S = Q K_int^T (M = 128 rows, N = 64 keys, K = 128), fp16 operands -- int8
//   values and the fp16 queries are exact in binary16, so S is exact up to fp32
//   accumulation; the row scales and the softmax scale are applied in fp32;
//   O += P' V_int with P' = p * scale_v split into fp16 hi + lo parts.
// int8 -> binary16 in registers: a byte b becomes the half 0x64xx with
// xx = b ^ 0x80 (value 1024 + b + 128) by one byte permute, then one packed
// subtraction of 1152 gives b exactly.
#include <math.h>

#include "tq_common.cuh"
#include "tq_tc.cuh"

namespace tq {

struct Int8Args {
  const int8_t *k;
  const uint16_t *k_scale;
  const int8_t *v;
  const uint16_t *v_scale;
  const int32_t *cell_of_pos;
  const uint16_t *q;
  float *out;
  int32_t *status;
  int64_t n_cells;
  int64_t ctx;
  int32_t nq, n_q_heads, n_kv_heads, group, causal;
  float scale_log2;
};

namespace i8 {

constexpr int BM = 128, BN = 64, D = 128, NT = 256;
constexpr uint32_t SQ = 0;                      // Q      [d/8][row/8]      32 KB
constexpr uint32_t SK = SQ + 32768;             // K'     [key/8][d/8]      16 KB
constexpr uint32_t SV = SK + 16384;             // V'     [key/8][d/8]      16 KB
constexpr uint32_t SP = SV + 16384;             // P' hi, lo [key/8][row/8] 2 x 16 KB
constexpr uint32_t SSTG = SP + 32768;           // raw rows: 2 stages x (K 8 KB + V 8 KB)
constexpr uint32_t STAGE = 2 * BN * D;
constexpr uint32_t SCELL = SSTG + 2 * STAGE;    // int32 cells [2][BN]
constexpr uint32_t SSCL = SCELL + 2 * BN * 4;   // float scales [BN][2] (k, v) of the current tile
constexpr uint32_t TOTAL = SSCL + BN * 2 * 4;
constexpr int TMEM_COLS = 256;                  // O: 128 columns, S: 64 columns

__device__ __forceinline__ long long i64min(long long x, long long y) { return x < y ? x : y; }
__device__ __forceinline__ long long i64max(long long x, long long y) { return x > y ? x : y; }

// 4 int8 values (one 32-bit word) -> 2 half2 (exact)
__device__ __forceinline__ void i8x4_to_h(uint32_t w, uint32_t &h01, uint32_t &h23) {
  const uint32_t u = w ^ 0x80808080u;
  const uint32_t a = prmt_b32(u, 0x64646464u, 0x5150u);    // (b0^0x80, 0x64, b1^0x80, 0x64)
  const uint32_t b = prmt_b32(u, 0x64646464u, 0x5352u);
  const __half2 off = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));   // 1152
  const __half2 ha = __hsub2(*reinterpret_cast<const __half2 *>(&a), off);
  const __half2 hb = __hsub2(*reinterpret_cast<const __half2 *>(&b), off);
  h01 = *reinterpret_cast<const uint32_t *>(&ha);
  h23 = *reinterpret_cast<const uint32_t *>(&hb);
}

__global__ void __launch_bounds__(NT, 1) int8_attn_kernel(const Int8Args a) {
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[2];
  __shared__ __align__(8) uint64_t bar_s, bar_pv;
  __shared__ uint32_t tmem_slot;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hk = blockIdx.y, G = a.group;
  const int q0 = blockIdx.x * (BM / G);
  const int q_last = min(a.nq, q0 + BM / G) - 1;
  const int64_t pos0 = a.ctx - a.nq;
  const int64_t kv_hi = a.causal ? i64min(a.ctx, pos0 + q_last + 1) : a.ctx;
  const int n_tiles = static_cast<int>((kv_hi + BN - 1) / BN);
  const int64_t row_stride = static_cast<int64_t>(a.n_kv_heads) * D;      // bytes per cell
  int32_t *cells = reinterpret_cast<int32_t *>(smem + SCELL);

  // warp 0: gather the tile's scattered rows (one bulk copy per row)
  auto issue = [&](int tile) {
    const int st = tile & 1;
    unsigned char *kst = smem + SSTG + st * STAGE, *vst = kst + BN * D;
    int cl[2];
    bool ok[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int key = lane + 32 * h;
      const int64_t t = static_cast<int64_t>(tile) * BN + key;
      int c = -1;
      if (t < kv_hi) c = a.cell_of_pos[t];
      ok[h] = t < kv_hi && c >= 0 && c < a.n_cells;
      if (t < kv_hi && !ok[h]) set_status(a.status, TQ_ERR_DEVICE_CHECK);
      cl[h] = ok[h] ? c : -1;
      cells[st * BN + key] = cl[h];
      if (!ok[h]) {                       // out-of-range cell: a zero row; beyond kv_hi: unused
        for (int i = 0; i < D; i += 16) {
          *reinterpret_cast<uint4 *>(kst + key * D + i) = make_uint4(0, 0, 0, 0);
          *reinterpret_cast<uint4 *>(vst + key * D + i) = make_uint4(0, 0, 0, 0);
        }
      }
    }
    const uint32_t n_ok = __popc(__ballot_sync(0xffffffffu, ok[0])) + __popc(__ballot_sync(0xffffffffu, ok[1]));
    if (lane == 0) tc::mbar_expect_tx(&full[st], n_ok * 2 * D);
    __syncwarp();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (ok[h]) {
        const int key = lane + 32 * h;
        const int64_t off = static_cast<int64_t>(cl[h]) * row_stride + hk * D;
        tc::bulk_g2s(kst + key * D, a.k + off, D, &full[st]);
        tc::bulk_g2s(vst + key * D, a.v + off, D, &full[st]);
      }
    }
  };

  if (warp == 0) tc::tmem_alloc<TMEM_COLS>(&tmem_slot);
  if (tid == 0) {
    tc::mbar_init(&full[0], 1);
    tc::mbar_init(&full[1], 1);
    tc::mbar_init(&bar_s, 1);
    tc::mbar_init(&bar_pv, 1);
    tc::mbar_init_fence();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  if (warp == 0)
    for (int i = 0; i < 2 && i < n_tiles; ++i) issue(i);

  // Q tile (binary16 as given): row r = query q0 + r/G, head hk*G + r%G
  for (int it = tid; it < BM * (D / 8); it += NT) {
    const int r = it / (D / 8), dc = it % (D / 8);
    const int qi = q0 + r / G, h = hk * G + r % G;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (qi < a.nq) val = *reinterpret_cast<const uint4 *>(a.q + (static_cast<size_t>(qi) * a.n_q_heads + h) * D + dc * 8);
    *reinterpret_cast<uint4 *>(smem + SQ + (dc * 16 + (r >> 3)) * 128 + (r & 7) * 16) = val;
  }

  constexpr uint32_t ID_S = tc::idesc_f16(BM, BN, false, false);
  constexpr uint32_t ID_PV = tc::idesc_f16(BM, D, false, true);
  const uint32_t sbase = tc::smem_u32(smem);
  float *scl = reinterpret_cast<float *>(smem + SSCL);

  const int row = tid;
  const int row_q = q0 + row / G;
  const bool row_ok = tid < BM && row_q < a.nq;
  const int64_t row_end = a.causal ? (pos0 + row_q + 1) : a.ctx;
  float m_used = -INFINITY, l_sum = 0.f;
  bool failed = false;

  for (int tile = 0; tile < n_tiles; ++tile) {
    const int st = tile & 1;
    bool ok = tc::mbar_wait(&full[st], (tile >> 1) & 1);
    if (__syncthreads_or(!ok)) { failed = true; break; }

    // ---- int8 rows -> binary16 K' / V' tiles; row scales as floats
    const unsigned char *kst = smem + SSTG + st * STAGE, *vst = kst + BN * D;
    for (int it = tid; it < 2 * BN * (D / 8); it += NT) {
      const bool is_v = it >= BN * (D / 8);
      const int rem = is_v ? it - BN * (D / 8) : it;
      const int dc = rem / BN, key = rem % BN;
      const uint2 w = *reinterpret_cast<const uint2 *>((is_v ? vst : kst) + key * D + dc * 8);
      uint4 o;
      i8x4_to_h(w.x, o.x, o.y);
      i8x4_to_h(w.y, o.z, o.w);
      *reinterpret_cast<uint4 *>(smem + (is_v ? SV : SK) + ((key >> 3) * 16 + dc) * 128 + (key & 7) * 16) = o;
    }
    if (tid < BN) {
      const int c = cells[st * BN + tid];
      float ks = 0.f, vs = 0.f;
      if (c >= 0) {
        ks = __half2float(__ushort_as_half(a.k_scale[static_cast<int64_t>(c) * a.n_kv_heads + hk]));
        vs = __half2float(__ushort_as_half(a.v_scale[static_cast<int64_t>(c) * a.n_kv_heads + hk]));
      }
      scl[2 * tid] = ks;
      scl[2 * tid + 1] = vs;
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    if (warp == 0 && tile + 2 < n_tiles) issue(tile + 2);
    if (tid == 0) {
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const uint64_t ad = tc::sdesc(sbase + SQ + ks * 4096, 2048, 128);
        const uint64_t bd = tc::sdesc(sbase + SK + ks * 256, 128, 2048);
        tc::mma_f16(tmem + 128, ad, bd, ID_S, ks > 0);
      }
      tc::mma_commit(&bar_s);
    }
    ok = tc::mbar_wait(&bar_s, tile & 1);
    if (__syncthreads_or(!ok)) { failed = true; break; }
    tc::fence_after_sync();

    if (warp < 4) {
      const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
      float s[BN];
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t r0[32];
        tc::tmem_ld32(tmem + lane_off + 128 + c0, r0);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c0 + i] = __uint_as_float(r0[i]) * scl[2 * (c0 + i)] * a.scale_log2;
      }
      const int64_t key0 = static_cast<int64_t>(tile) * BN;
      const int nvis = row_ok ? static_cast<int>(i64max(0, i64min(BN, row_end - key0))) : 0;
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < BN; ++i)
        if (i < nvis) mt = fmaxf(mt, s[i]);
      const bool raise = mt > m_used + 8.f || (m_used == -INFINITY && mt > -INFINITY);
      const float fct = (raise && m_used != -INFINITY) ? exp2f(m_used - mt) : 1.f;
      if (raise) m_used = mt;
      if (__any_sync(0xffffffffu, fct != 1.f)) {
        l_sum *= fct;
#pragma unroll
        for (int c = 0; c < D; c += 32) {
          uint32_t r[32];
          tc::tmem_ld32(tmem + lane_off + c, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * fct);
          tc::tmem_st32(tmem + lane_off + c, r);
        }
        tc::tmem_wait_st();
      }
      float psum = 0.f;
#pragma unroll
      for (int i = 0; i < BN; ++i) {
        s[i] = (i < nvis) ? tc::ex2(s[i] - m_used) : 0.f;
        psum += s[i];
      }
      l_sum += psum;
#pragma unroll
      for (int kc = 0; kc < BN / 8; ++kc) {
        uint32_t wh[4], wl[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int k0 = kc * 8 + 2 * j;
          const float x0 = s[k0] > 0.f ? s[k0] * scl[2 * k0 + 1] : 0.f;
          const float x1 = s[k0 + 1] > 0.f ? s[k0 + 1] * scl[2 * (k0 + 1) + 1] : 0.f;
          const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
          wh[j] = __half_as_ushort(h0) | (static_cast<uint32_t>(__half_as_ushort(h1)) << 16);
          wl[j] = __half_as_ushort(__float2half_rn(x0 - __half2float(h0))) |
                  (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(x1 - __half2float(h1)))) << 16);
        }
        const uint32_t off = (kc * 16 + (row >> 3)) * 128 + (row & 7) * 16;
        *reinterpret_cast<uint4 *>(smem + SP + off) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        *reinterpret_cast<uint4 *>(smem + SP + 16384 + off) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    if (tid == 0) {
#pragma unroll
      for (int part = 0; part < 2; ++part)
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
          const uint64_t ad = tc::sdesc(sbase + SP + part * 16384 + ks * 4096, 2048, 128);
          const uint64_t bd = tc::sdesc(sbase + SV + ks * 4096, 2048, 128);
          tc::mma_f16(tmem, ad, bd, ID_PV, tile > 0 || part > 0 || ks > 0);
        }
      tc::mma_commit(&bar_pv);
    }
    ok = tc::mbar_wait(&bar_pv, tile & 1);
    if (__syncthreads_or(!ok)) { failed = true; break; }
    tc::fence_after_sync();
  }

  if (failed) {
    if (tid == 0) set_status(a.status, TQ_ERR_TIMEOUT);
  } else if (warp < 4) {
    const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
    const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
    const int h = hk * G + row % G;
    float *orow = a.out + (static_cast<size_t>(row_ok ? row_q : 0) * a.n_q_heads + h) * D;
#pragma unroll
    for (int c = 0; c < D; c += 32) {
      uint32_t r[32];
      tc::tmem_ld32(tmem + lane_off + c, r);
      tc::tmem_wait_ld();
      if (row_ok) {
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4 *>(orow + c + i) =
              make_float4(__uint_as_float(r[i]) * inv, __uint_as_float(r[i + 1]) * inv,
                          __uint_as_float(r[i + 2]) * inv, __uint_as_float(r[i + 3]) * inv);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc<TMEM_COLS>(tmem);
}

}  // namespace i8

cudaError_t launch_int8_attn(const Int8Args &a, cudaStream_t s) {
  static_assert(i8::TOTAL <= 227 * 1024, "shared memory");
  cudaError_t e = cudaFuncSetAttribute(i8::int8_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)i8::TOTAL);
  if (e != cudaSuccess) return e;
  const int rows = a.nq * a.group;
  dim3 grid((rows + i8::BM - 1) / i8::BM, a.n_kv_heads);
  i8::int8_attn_kernel<<<grid, i8::NT, i8::TOTAL, s>>>(a);
  return cudaGetLastError();
}

}  // namespace tq

using namespace tq;

extern "C" size_t tq_int8_prompt_attn_workspace(int nq, int n_q_heads, int n_kv_heads, int head_dim, int64_t ctx) {
  if (nq < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads || head_dim != 128 || ctx < 0) return 0;
  return 256;    // the status word
}

extern "C" tq_status tq_int8_prompt_attn(const int8_t *k, const uint16_t *k_scale, const int8_t *v,
                                         const uint16_t *v_scale, int64_t n_cells, const int32_t *cell_of_pos,
                                         int64_t ctx, const uint16_t *q, int nq, int n_q_heads, int n_kv_heads,
                                         int head_dim, float scale, int causal, float *out, void *workspace,
                                         size_t workspace_bytes, tq_stream stream) {
  auto al = [](const void *p, uintptr_t m) { return (reinterpret_cast<uintptr_t>(p) & (m - 1)) == 0; };
  if (n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return TQ_ERR_INVALID_ARG;
  const int group = n_q_heads / n_kv_heads;
  if ((group & (group - 1)) != 0 || group > 128) return TQ_ERR_UNSUPPORTED;
  if (head_dim != 128) return TQ_ERR_UNSUPPORTED;
  if (nq < 0 || ctx < 0 || n_cells <= 0 || (causal && nq > ctx) || !isfinite(scale)) return TQ_ERR_INVALID_ARG;
  if (nq == 0) return TQ_OK;
  if (!out || !al(out, 16) || !q || !al(q, 16)) return TQ_ERR_INVALID_ARG;
  if (!workspace || !al(workspace, 256) || workspace_bytes < 256) return TQ_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (ctx == 0) return cudaMemsetAsync(out, 0, sizeof(float) * nq * n_q_heads * head_dim, s) == cudaSuccess
                           ? TQ_OK : TQ_ERR_CUDA;
  if (!k || !v || !al(k, 16) || !al(v, 16) || !k_scale || !v_scale || !al(k_scale, 2) || !al(v_scale, 2) ||
      !cell_of_pos || !al(cell_of_pos, 4))
    return TQ_ERR_INVALID_ARG;
  if (static_cast<int64_t>(nq) * group > 0x7fffffffLL) return TQ_ERR_INVALID_ARG;
  Int8Args a;
  a.k = k;
  a.k_scale = k_scale;
  a.v = v;
  a.v_scale = v_scale;
  a.cell_of_pos = cell_of_pos;
  a.q = q;
  a.out = out;
  a.status = static_cast<int32_t *>(workspace);
  a.n_cells = n_cells;
  a.ctx = ctx;
  a.nq = nq;
  a.n_q_heads = n_q_heads;
  a.n_kv_heads = n_kv_heads;
  a.group = group;
  a.causal = causal ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  return launch_int8_attn(a, s) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

// Multi-query (prefill / verify) attention over the packed TurboQuant cache on
// the tcgen05 tensor cores, with the K/V tiles dequantised inline
// ([HIP#28] "2. Inline-dequant TILE prefill": expand the packed cache while it
// is loaded into on-chip tiles, never write an f16 copy of the cache).
//
// One CTA = one KV head x 128 query rows (128/G queries x the G query heads of
// the GQA group, row r = query (r / G), head (r % G)), looping over key tiles of
// BN = 64 keys (32 when a 256-dim head leaves too little shared memory):
//   1. cp.async.bulk brings the tile's packed K/V planes into a 2-deep ring;
//   2. all threads expand them with byte permutes into binary16 centroid tiles
//      (exact values; block norms are kept aside as floats);
//   3. one thread issues S_b = Q'_b K'_b^T per 128-dim block b (M=128, N=BN,
//      K=128) into tensor memory;
//   4. one thread per row reads S, forms s = sum_b |k_b| S_b, applies the causal
//      mask, the online softmax (log2 domain, running max raised only when it
//      grows by more than 2^8, then O is rescaled in tensor memory), and writes
//      P'_b = p * |v_b| as binary16;
//   5. one thread issues O_b += P'_b V'_b (M=128, N=128, K=BN) into tensor memory.
// Precision: Q' and P' are each split into binary16 hi + lo parts (x = hi + lo
// with lo = fp16(x - hi)) and both halves go through the tensor cores, so S and
// O carry ~22 significant bits; K' and V' are binary16-exact centroids.  One
// fp16 rounding of Q' or P' alone moves outputs by up to ~1e-2 on these
// workloads, beyond the 2e-3 absolute tolerance.
// The epilogue divides by the softmax sum, rotates each 128-dim block back
// (o = S H o' / sqrt(128), in registers) and stores fp32 rows.
//
// Q is rotated into the K codebook's domain on load (q' = H S q / sqrt(128),
// softmax scale and log2(e) folded in); S = q'.k' = q.k because the rotation is
// orthogonal, and O accumulates in the V codebook's rotated domain.
//
// Shared-memory operand tiles (SWIZZLE_NONE core matrices of 8 rows x 16 B):
//   Q'_b  A, K-major   [d/8][row/8]  LBO 2048 (along d)   SBO 128 (along rows)
//   K'_b  B, K-major   [key/8][d/8]  LBO 128  (along d)   SBO 2048 (along keys)
//   V'_b  B, MN-major  [key/8][d/8]  LBO 2048 (along keys) SBO 128 (along d)
//   P'_b  A, K-major   [key/8][row/8] LBO 2048 (along keys) SBO 128 (along rows)
// (hi and lo copies of Q' and P' side by side).
// K' and V' share one physical layout: a core matrix is 8 keys x 8 dims.
#pragma once

#include "tq_common.cuh"
#include "tq_tc.cuh"

namespace tq {
namespace pf {

constexpr int BM = 128;     // query rows per CTA (TMEM lanes)
constexpr int NT = 256;     // threads
constexpr float kLazyRescale = 8.f;   // log2 units

template <int T, int NBK, int NBV>
struct Smem {
  static constexpr int BN = (NBK == 2) ? 32 : 64;                    // keys per tile
  static constexpr int QSB = TypeTraits<T>::QSB, SGB = TypeTraits<T>::SGB;
  static constexpr uint32_t QBLK = 32768;                            // 128 rows x 128 dims fp16
  static constexpr uint32_t KBLK = BN * 256;                         // BN keys x 128 dims fp16
  static constexpr uint32_t PBLK = BN * 256;                         // 128 rows x BN keys fp16
  static constexpr uint32_t Q = 0;                                   // hi [NBK], lo [NBK]
  static constexpr uint32_t K = Q + 2 * NBK * QBLK;
  static constexpr uint32_t V = K + NBK * KBLK;
  static constexpr uint32_t P = V + NBV * KBLK;                      // hi [NBV], lo [NBV]
  // packed staging ring: per stage K qs, K signs, K norms, V qs, V signs, V norms
  static constexpr uint32_t S_KQS = 0;
  static constexpr uint32_t S_KSG = S_KQS + BN * NBK * QSB;
  static constexpr uint32_t S_KN = S_KSG + BN * NBK * SGB;
  static constexpr uint32_t S_VQS = S_KN + BN * NBK * 2;
  static constexpr uint32_t S_VSG = S_VQS + BN * NBV * QSB;
  static constexpr uint32_t S_VN = S_VSG + BN * NBV * SGB;
  static constexpr uint32_t STAGE = (S_VN + BN * NBV * 2 + 127) / 128 * 128;
  static constexpr uint32_t STG = P + 2 * NBV * PBLK;                // 2 stages
  static constexpr uint32_t NRM = STG + 2 * STAGE;                   // floats [BN][NBK + NBV]
  static constexpr uint32_t TOTAL = NRM + BN * (NBK + NBV) * 4;
  static constexpr uint32_t TX = BN * (NBK + NBV) * (QSB + SGB + 2);  // bytes per stage copy
  // tensor memory: O_b at columns 128 b, S_b at S_COL + BN b
  static constexpr uint32_t S_COL = NBV * 128;
  static constexpr int TMEM_COLS = (NBV * 128 + NBK * BN <= 256) ? 256 : 512;
};

__device__ __forceinline__ long long i64min(long long x, long long y) { return x < y ? x : y; }
__device__ __forceinline__ long long i64max(long long x, long long y) { return x > y ? x : y; }

template <int T, int NBK, int NBV>
__global__ void __launch_bounds__(NT, 1) prefill_kernel(const PrefillArgs a) {
  using SM = Smem<T, NBK, NBV>;
  constexpr int QSB = SM::QSB, SGB = SM::SGB, BN = SM::BN;
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[2];
  __shared__ __align__(8) uint64_t bar_s, bar_pv;
  __shared__ uint32_t tmem_slot;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hk = blockIdx.y;
  const int G = a.group;
  const int q0 = blockIdx.x * (BM / G);                       // first query of this CTA
  const int q_last = min(a.nq, q0 + BM / G) - 1;
  const int64_t pos0 = a.kv_len - a.nq;                        // position of query 0 (causal)
  const int64_t kv_hi = a.causal ? i64min(a.kv_len, pos0 + q_last + 1) : a.kv_len;
  const int n_tiles = static_cast<int>((kv_hi + BN - 1) / BN);

  const uint8_t *kqs = a.kqs + static_cast<size_t>(hk) * a.n_cells * NBK * QSB;
  const uint8_t *ksg = SGB ? a.ksg + static_cast<size_t>(hk) * a.n_cells * NBK * SGB : nullptr;
  const uint16_t *kn = a.kn + static_cast<size_t>(hk) * a.n_cells * NBK;
  const uint8_t *vqs = a.vqs + static_cast<size_t>(hk) * a.n_cells * NBV * QSB;
  const uint8_t *vsg = SGB ? a.vsg + static_cast<size_t>(hk) * a.n_cells * NBV * SGB : nullptr;
  const uint16_t *vn = a.vn + static_cast<size_t>(hk) * a.n_cells * NBV;

  auto issue = [&](int tile) {
    unsigned char *st = smem + SM::STG + (tile & 1) * SM::STAGE;
    uint64_t *bar = &full[tile & 1];
    const int64_t key0 = static_cast<int64_t>(tile) * BN;
    tc::mbar_expect_tx(bar, SM::TX);
    tc::bulk_g2s(st + SM::S_KQS, kqs + key0 * NBK * QSB, BN * NBK * QSB, bar);
    if (SGB) tc::bulk_g2s(st + SM::S_KSG, ksg + key0 * NBK * SGB, BN * NBK * SGB, bar);
    tc::bulk_g2s(st + SM::S_KN, kn + key0 * NBK, BN * NBK * 2, bar);
    tc::bulk_g2s(st + SM::S_VQS, vqs + key0 * NBV * QSB, BN * NBV * QSB, bar);
    if (SGB) tc::bulk_g2s(st + SM::S_VSG, vsg + key0 * NBV * SGB, BN * NBV * SGB, bar);
    tc::bulk_g2s(st + SM::S_VN, vn + key0 * NBV, BN * NBV * 2, bar);
  };

  if (warp == 0) tc::tmem_alloc<SM::TMEM_COLS>(&tmem_slot);
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
  if (tid == 0)
    for (int i = 0; i < 2 && i < n_tiles; ++i) issue(i);

  // ---- Q' = fp16(q rotated per block, scale * log2(e) / sqrt(128) folded in)
  {
    const float f = a.scale_log2 * kInvSqrtQK;
    for (int pr = warp; pr < BM * NBK; pr += NT / 32) {
      const int r = pr % BM, b = pr / BM;
      const int qi = q0 + r / G, h = hk * G + r % G;
      float v[4] = {0.f, 0.f, 0.f, 0.f};
      if (qi < a.nq) {
        const size_t base = (static_cast<size_t>(qi) * a.n_q_heads + h) * a.dk;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int d = b * QK + 4 * lane + k;
          if (d < a.dk) {
            if (a.q_type == TQ_BF16)
              v[k] = __bfloat162float(__ushort_as_bfloat16(static_cast<const uint16_t *>(a.q)[base + d]));
            else if (a.q_type == TQ_F16)
              v[k] = __half2float(__ushort_as_half(static_cast<const uint16_t *>(a.q)[base + d]));
            else
              v[k] = static_cast<const float *>(a.q)[base + d];
          }
        }
      }
      apply_signs(v, a.cbk, lane);
      wht128_warp(v, lane);
      const int d0 = 4 * lane;
      uint16_t hb[4], lb[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float x = v[k] * f;
        const __half h = __float2half_rn(x);
        hb[k] = __half_as_ushort(h);
        lb[k] = __half_as_ushort(__float2half_rn(x - __half2float(h)));
      }
      const uint32_t off = b * SM::QBLK + ((d0 >> 3) * 16 + (r >> 3)) * 128 + (r & 7) * 16 + (d0 & 7) * 2;
      *reinterpret_cast<uint2 *>(smem + SM::Q + off) =
          make_uint2(hb[0] | (static_cast<uint32_t>(hb[1]) << 16), hb[2] | (static_cast<uint32_t>(hb[3]) << 16));
      *reinterpret_cast<uint2 *>(smem + SM::Q + NBK * SM::QBLK + off) =
          make_uint2(lb[0] | (static_cast<uint32_t>(lb[1]) << 16), lb[2] | (static_cast<uint32_t>(lb[3]) << 16));
    }
  }

  const Tab tab_k = make_tab<T>(a.cbk);
  const Tab tab_v = make_tab<T>(a.cbv);
  constexpr uint32_t ID_S = tc::idesc_f16(BM, SM::BN, false, false);
  constexpr uint32_t ID_PV = tc::idesc_f16(BM, 128, false, true);
  const uint32_t sbase = tc::smem_u32(smem);

  // softmax state of row `tid` (threads 0..127)
  const int row = tid;
  const int row_q = q0 + row / G;
  const bool row_ok = tid < BM && row_q < a.nq;
  const int64_t row_end = a.causal ? (pos0 + row_q + 1) : a.kv_len;      // keys < row_end visible
  float m_used = -INFINITY, l_sum = 0.f;
  float *nrm = reinterpret_cast<float *>(smem + SM::NRM);                 // [BN][NBK + NBV]
  bool failed = false;

  for (int tile = 0; tile < n_tiles && !failed; ++tile) {
    const unsigned char *st = smem + SM::STG + (tile & 1) * SM::STAGE;
    bool ok = tc::mbar_wait(&full[tile & 1], (tile >> 1) & 1);
    if (__syncthreads_or(!ok)) { failed = true; break; }

    // ---- expand the packed tile into binary16 K' / V' tiles
    for (int it = tid; it < (NBK + NBV) * BN * 16; it += NT) {
      const int bb = it / (BN * 16), rem = it % (BN * 16);
      const int dc = rem / BN, key = rem % BN;
      const bool is_v = bb >= NBK;
      const int b = is_v ? bb - NBK : bb;
      const int nb = is_v ? NBV : NBK;
      const uint8_t *qrow = st + (is_v ? SM::S_VQS : SM::S_KQS) + (key * nb + b) * QSB;
      uint32_t sel;
      if (T == 4) {
        sel = reinterpret_cast<const uint32_t *>(qrow)[dc];
      } else {
        const uint32_t w = reinterpret_cast<const uint32_t *>(qrow)[dc >> 1];
        uint32_t sg = 0;
        if (T == 3) sg = reinterpret_cast<const uint32_t *>(st + (is_v ? SM::S_VSG : SM::S_KSG) + (key * nb + b) * SGB)[dc >> 2];
        uint32_t s0, s1;
        sel_words<T>(w, sg, ((dc >> 1) & 1) != 0, s0, s1);
        sel = (dc & 1) ? s1 : s0;
      }
      const Tab &tb = is_v ? tab_v : tab_k;
      uint4 o;
      dq4<T>(sel & 0xffffu, tb, o.x, o.y);
      dq4<T>(sel >> 16, tb, o.z, o.w);
      *reinterpret_cast<uint4 *>(smem + (is_v ? SM::V : SM::K) + b * SM::KBLK + ((key >> 3) * 16 + dc) * 128 +
                                 (key & 7) * 16) = o;
    }
    for (int i = tid; i < BN * (NBK + NBV); i += NT) {
      const int key = i / (NBK + NBV), j = i % (NBK + NBV);
      const uint16_t *np = reinterpret_cast<const uint16_t *>(st + (j < NBK ? SM::S_KN : SM::S_VN));
      const float n = (j < NBK) ? __half2float(__ushort_as_half(np[key * NBK + j]))
                                : __half2float(__ushort_as_half(np[key * NBV + (j - NBK)]));
      nrm[key * (NBK + NBV) + j] = n;
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    if (tid == 0) {
      if (tile + 2 < n_tiles) issue(tile + 2);              // staging stage is free again
#pragma unroll
      for (int b = 0; b < NBK; ++b)
#pragma unroll
        for (int part = 0; part < 2; ++part)                     // q'_hi, then q'_lo
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t ad =
                tc::sdesc(sbase + SM::Q + (part * NBK + b) * SM::QBLK + ks * 4096, 2048, 128);
            const uint64_t bd = tc::sdesc(sbase + SM::K + b * SM::KBLK + ks * 256, 128, 2048);
            tc::mma_f16(tmem + SM::S_COL + b * BN, ad, bd, ID_S, part > 0 || ks > 0);
          }
      tc::mma_commit(&bar_s);
    }
    ok = tc::mbar_wait(&bar_s, tile & 1);
    if (__syncthreads_or(!ok)) { failed = true; break; }
    tc::fence_after_sync();

    // ---- softmax: one thread per row (warps 0..3 own TMEM lanes 0..127)
    if (warp < 4) {
      const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
      float s[BN];
#pragma unroll
      for (int i = 0; i < BN; ++i) s[i] = 0.f;
#pragma unroll
      for (int b = 0; b < NBK; ++b)
#pragma unroll
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t r0[32];
          tc::tmem_ld32(tmem + lane_off + SM::S_COL + b * BN + c0, r0);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            s[c0 + i] = fmaf(nrm[(c0 + i) * (NBK + NBV) + b], __uint_as_float(r0[i]), s[c0 + i]);
        }
      const int64_t key0 = static_cast<int64_t>(tile) * BN;
      const int nvis = row_ok ? static_cast<int>(i64max(0, i64min(BN, row_end - key0))) : 0;
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < BN; ++i)
        if (i < nvis) mt = fmaxf(mt, s[i]);
      // raise the reference maximum only when the row max grew by more than 2^8;
      // the tensor-memory rescale is warp-collective, so lanes that need none use 1
      const bool raise = mt > m_used + kLazyRescale || (m_used == -INFINITY && mt > -INFINITY);
      const float fct = (raise && m_used != -INFINITY) ? exp2f(m_used - mt) : 1.f;
      if (raise) m_used = mt;
      if (__any_sync(0xffffffffu, fct != 1.f)) {
        l_sum *= fct;
#pragma unroll
        for (int c = 0; c < NBV * 128; c += 32) {
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
        s[i] = (i < nvis) ? exp2f(s[i] - m_used) : 0.f;
        psum += s[i];
      }
      l_sum += psum;
#pragma unroll
      for (int b = 0; b < NBV; ++b)
#pragma unroll
        for (int kc = 0; kc < BN / 8; ++kc) {
          uint32_t wh[4], wl[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const int k0 = kc * 8 + 2 * j;
            // masked keys may carry garbage norms: select, never multiply, a zero
            const float x0 = s[k0] > 0.f ? s[k0] * nrm[k0 * (NBK + NBV) + NBK + b] : 0.f;
            const float x1 = s[k0 + 1] > 0.f ? s[k0 + 1] * nrm[(k0 + 1) * (NBK + NBV) + NBK + b] : 0.f;
            const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
            wh[j] = __half_as_ushort(h0) | (static_cast<uint32_t>(__half_as_ushort(h1)) << 16);
            wl[j] = __half_as_ushort(__float2half_rn(x0 - __half2float(h0))) |
                    (static_cast<uint32_t>(__half_as_ushort(__float2half_rn(x1 - __half2float(h1)))) << 16);
          }
          const uint32_t off = b * SM::PBLK + (kc * 16 + (row >> 3)) * 128 + (row & 7) * 16;
          *reinterpret_cast<uint4 *>(smem + SM::P + off) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
          *reinterpret_cast<uint4 *>(smem + SM::P + NBV * SM::PBLK + off) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
        }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    if (tid == 0) {
#pragma unroll
      for (int b = 0; b < NBV; ++b)
#pragma unroll
        for (int part = 0; part < 2; ++part)                     // P'_hi, then P'_lo
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks) {
            const uint64_t ad = tc::sdesc(sbase + SM::P + (part * NBV + b) * SM::PBLK + ks * 4096, 2048, 128);
            const uint64_t bd = tc::sdesc(sbase + SM::V + b * SM::KBLK + ks * 4096, 2048, 128);
            tc::mma_f16(tmem + b * 128, ad, bd, ID_PV, tile > 0 || part > 0 || ks > 0);
          }
      tc::mma_commit(&bar_pv);
    }
    ok = tc::mbar_wait(&bar_pv, tile & 1);
    if (__syncthreads_or(!ok)) { failed = true; break; }
    tc::fence_after_sync();
  }

  if (failed) {
    if (tid == 0) set_status(a.status, TQ_ERR_TIMEOUT);
  } else if (warp < 4) {                 // warp-uniform: tensor-memory loads are collective
    // ---- epilogue: o = S H (O / l) / sqrt(128) per 128-dim block, fp32 rows
    const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
    const float inv = (l_sum > 0.f ? 1.f / l_sum : 0.f) * kInvSqrtQK;
    const int h = hk * G + row % G;
    float *orow = a.out + (static_cast<size_t>(row_ok ? row_q : 0) * a.n_q_heads + h) * a.dv;
#pragma unroll 1
    for (int b = 0; b < NBV; ++b) {
      float o[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tc::tmem_ld32(tmem + lane_off + b * 128 + 32 * c, r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) o[32 * c + i] = __uint_as_float(r[i]);
      }
#pragma unroll
      for (int hb = 1; hb < 128; hb <<= 1)
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (!(i & hb)) {
            const float x = o[i], y = o[i | hb];
            o[i] = x + y;
            o[i | hb] = x - y;
          }
      const int dmax = a.dv - b * 128;
#pragma unroll
      for (int i = 0; i < 128; i += 4) {
        float4 w;
        w.x = ((a.cbv.sign_bits[i >> 5] >> ((i + 0) & 31)) & 1u) ? -o[i] * inv : o[i] * inv;
        w.y = ((a.cbv.sign_bits[i >> 5] >> ((i + 1) & 31)) & 1u) ? -o[i + 1] * inv : o[i + 1] * inv;
        w.z = ((a.cbv.sign_bits[i >> 5] >> ((i + 2) & 31)) & 1u) ? -o[i + 2] * inv : o[i + 2] * inv;
        w.w = ((a.cbv.sign_bits[i >> 5] >> ((i + 3) & 31)) & 1u) ? -o[i + 3] * inv : o[i + 3] * inv;
        if (row_ok && i + 4 <= dmax) *reinterpret_cast<float4 *>(orow + b * 128 + i) = w;
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc<SM::TMEM_COLS>(tmem);
}

template <int T, int NBK, int NBV>
cudaError_t launch_one(const PrefillArgs &a, cudaStream_t s) {
  using SM = Smem<T, NBK, NBV>;
  static_assert(SM::TOTAL <= 227 * 1024, "shared memory");
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<T, NBK, NBV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)SM::TOTAL);
  if (e != cudaSuccess) return e;
  const int rows = a.nq * a.group;
  dim3 grid((rows + BM - 1) / BM, a.n_kv_heads);
  static_assert(SM::BN % 16 == 0 && SM::BN <= 64, "key tile");
  prefill_kernel<T, NBK, NBV><<<grid, NT, SM::TOTAL, s>>>(a);
  return cudaGetLastError();
}

template <int T>
cudaError_t launch_type(const PrefillArgs &a, cudaStream_t s) {
  if (a.nbk == 1 && a.nbv == 1) return launch_one<T, 1, 1>(a, s);
  if (a.nbk == 2 && a.nbv == 2) return launch_one<T, 2, 2>(a, s);
  if (a.nbk == 2 && a.nbv == 1) return launch_one<T, 2, 1>(a, s);
  return cudaErrorNotSupported;
}

}  // namespace pf
}  // namespace tq

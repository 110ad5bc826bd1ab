// Multi-query (prefill / verify) attention over the packed TurboQuant cache on
// the tcgen05 tensor cores, with the K/V tiles dequantised inline
// ([HIP#28] "2. Inline-dequant TILE prefill": expand the packed cache while it
// is loaded into on-chip tiles, never write an f16 copy of the cache).
//
// One CTA = one KV head x 128 query rows (128/G queries x the G query heads of
// the GQA group, row r = query (r / G), head (r % G)) x one range of key tiles
// (BN = 64 keys, 32 for 256-dim heads).  Warp roles, connected by mbarriers
// only (no CTA barrier inside the key loop):
//   control warp (one thread): cp.async.bulk of the packed K/V planes into a
//     3-stage ring; issues S_j = Q'K'_j^T into tensor memory, then
//     O += P'_{j-1} V'_{j-1} -- the tensor cores compute S_j while the softmax
//     warps work on tile j-1;
//   4 dequant warps: expand tile j into binary16 K'/V' tiles (exact centroid
//     values; double buffered; one key-block row per thread);
//   4 softmax warps (one query row per thread, TMEM lanes 0..127): read S_j,
//     form s = sum_b |k_b| S_b, apply the causal mask and the online softmax
//     (log2 domain; the reference maximum is raised only when the row maximum
//     grows by more than 2^8, then O is rescaled in tensor memory), and write
//     P'_b = p |v_b| as binary16 hi + lo straight into tensor memory over S_j,
//     where the PV mma reads it as its A operand.
// Precision: Q' and P' are split into binary16 hi + lo parts and both go
// through the tensor cores; K'/V' are exact; accumulation is fp32.
// Few query tiles (short prompts, verify batches) split the key range over
// several CTAs; the last CTA to finish a query tile merges the partial
// (max, sum, O) rows (4 + 128 nbv floats each) with log-sum-exp weights.
// Epilogue: o = S H (O / l) / sqrt(128) per 128-dim block (V codebook), fp32.
//
// Shared-memory operands (SWIZZLE_NONE core matrices of 8 rows x 16 B):
//   Q'_b (hi, lo)  A, K-major   [d/8][row/8]   LBO 2048 (along d)    SBO 128
//   K'_b           B, K-major   [key/8][d/8]   LBO 128 (along d)     SBO 2048
//   V'_b           B, MN-major  [key/8][d/8]   LBO 2048 (along keys) SBO 128
// Tensor memory (fp32 columns): O_b at 128 b; per buffer S_b at BN b, aliased by
// P'_(b, part) at (2b + part) BN/2 (fp16 pairs, row = lane).
#pragma once

#include "tq_common.cuh"
#include "tq_tc.cuh"

namespace tq {
namespace pf {

constexpr int BM = 128;          // query rows per CTA (TMEM lanes)
constexpr int NWARP = 9;         // 0-3 softmax, 4-7 dequant, 8 control
constexpr int NT = NWARP * 32;
constexpr int STAGES = 3;
constexpr float kLazyRescale = 8.f;   // log2 units

template <int T, int NBK, int NBV>
struct Cfg {
  static constexpr int BN = (NBK == 2) ? 32 : 64;
  static constexpr int QSB = TypeTraits<T>::QSB, SGB = TypeTraits<T>::SGB;
  static constexpr uint32_t QBLK = 32768;                  // 128 rows x 128 dims fp16
  static constexpr uint32_t TBLK = BN * 256;               // BN keys x 128 dims fp16
  static constexpr uint32_t KVBUF = (NBK + NBV) * TBLK;    // one K'/V' buffer
  static constexpr uint32_t Q = 0;                         // [part][NBK] blocks
  static constexpr uint32_t KV = Q + 2 * NBK * QBLK;       // 2 buffers: K'_b then V'_b
  // packed staging ring: K qs, K signs, K norms, V qs, V signs, V norms
  static constexpr uint32_t S_KQS = 0;
  static constexpr uint32_t S_KSG = S_KQS + BN * NBK * QSB;
  static constexpr uint32_t S_KN = S_KSG + BN * NBK * SGB;
  static constexpr uint32_t S_VQS = S_KN + BN * NBK * 2;
  static constexpr uint32_t S_VSG = S_VQS + BN * NBV * QSB;
  static constexpr uint32_t S_VN = S_VSG + BN * NBV * SGB;
  static constexpr uint32_t STAGE = (S_VN + BN * NBV * 2 + 127) / 128 * 128;
  static constexpr uint32_t STG = KV + 2 * KVBUF;
  static constexpr uint32_t NRM = STG + STAGES * STAGE;    // floats [2][BN][NBK + NBV]
  static constexpr uint32_t TOTAL = NRM + 2 * BN * (NBK + NBV) * 4;
  static constexpr uint32_t TX = BN * (NBK + NBV) * (QSB + SGB + 2);
  // tensor memory
  static constexpr uint32_t SPW = (NBK > NBV ? NBK : NBV) * BN;   // columns per S/P' buffer
  static constexpr uint32_t SP0 = NBV * 128;
  static constexpr uint32_t COLS_NEEDED = NBV * 128 + 2 * SPW;
  static constexpr int TMEM_COLS = COLS_NEEDED <= 256 ? 256 : 512;
  static constexpr int DVP = 128 * NBV;
};

__device__ __forceinline__ long long i64min(long long x, long long y) { return x < y ? x : y; }
__device__ __forceinline__ long long i64max(long long x, long long y) { return x > y ? x : y; }

// tcgen05.mma with the A operand in tensor memory
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(static_cast<uint32_t>(acc)));
}

template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const uint32_t *r);
template <>
__device__ __forceinline__ void tmem_st<16>(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
template <>
__device__ __forceinline__ void tmem_st<32>(uint32_t taddr, const uint32_t *r) {
  tc::tmem_st32(taddr, r);
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

struct Bars {
  uint64_t full[STAGES];   // packed tile staged (tx)
  uint64_t dq[2];          // K'/V' tile expanded (4 dequant warps)
  uint64_t sf[2];          // S_j computed (mma commit)
  uint64_t pf[2];          // P'_j written (4 softmax warps)
  uint64_t pv[2];          // PV_j computed (mma commit)
};

// o = S H o' / sqrt(128) of one 128-dim block held by one thread, stored as fp32
__device__ __forceinline__ void rotate_store_block(float o[128], float scale, const DevCodebook &cbv, float *dst,
                                                   int dmax, bool store) {
#pragma unroll
  for (int hb = 1; hb < 128; hb <<= 1)
#pragma unroll
    for (int i = 0; i < 128; ++i)
      if (!(i & hb)) {
        const float x = o[i], y = o[i | hb];
        o[i] = x + y;
        o[i | hb] = x - y;
      }
#pragma unroll
  for (int i = 0; i < 128; i += 4) {
    float4 w;
    w.x = ((cbv.sign_bits[i >> 5] >> ((i + 0) & 31)) & 1u) ? -o[i] * scale : o[i] * scale;
    w.y = ((cbv.sign_bits[i >> 5] >> ((i + 1) & 31)) & 1u) ? -o[i + 1] * scale : o[i + 1] * scale;
    w.z = ((cbv.sign_bits[i >> 5] >> ((i + 2) & 31)) & 1u) ? -o[i + 2] * scale : o[i + 2] * scale;
    w.w = ((cbv.sign_bits[i >> 5] >> ((i + 3) & 31)) & 1u) ? -o[i + 3] * scale : o[i + 3] * scale;
    if (store && i + 4 <= dmax) *reinterpret_cast<float4 *>(dst + i) = w;
  }
}

template <int T, int NBK, int NBV>
__global__ void __launch_bounds__(NT, 1) prefill_kernel(const PrefillArgs a) {
  using C = Cfg<T, NBK, NBV>;
  constexpr int BN = C::BN, QSB = C::QSB, SGB = C::SGB, DVP = C::DVP;
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ __align__(8) Bars bars;
  __shared__ uint32_t tmem_slot;
  __shared__ int s_fail;
  __shared__ int s_last;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hk = blockIdx.y, split = blockIdx.z, n_split = gridDim.z;
  const int G = a.group;
  const int q0 = blockIdx.x * (BM / G);
  const int q_last = min(a.nq, q0 + BM / G) - 1;
  const int64_t pos0 = a.kv_len - a.nq;
  const int64_t kv_hi = a.causal ? i64min(a.kv_len, pos0 + q_last + 1) : a.kv_len;
  const int tiles_all = static_cast<int>((kv_hi + BN - 1) / BN);
  const int t_lo = static_cast<int>(static_cast<long long>(tiles_all) * split / n_split);
  const int t_hi = static_cast<int>(static_cast<long long>(tiles_all) * (split + 1) / n_split);
  const int n_tiles = t_hi - t_lo;

  const uint8_t *kqs = a.kqs + static_cast<size_t>(hk) * a.n_cells * NBK * QSB;
  const uint8_t *ksg = SGB ? a.ksg + static_cast<size_t>(hk) * a.n_cells * NBK * SGB : nullptr;
  const uint16_t *kn = a.kn + static_cast<size_t>(hk) * a.n_cells * NBK;
  const uint8_t *vqs = a.vqs + static_cast<size_t>(hk) * a.n_cells * NBV * QSB;
  const uint8_t *vsg = SGB ? a.vsg + static_cast<size_t>(hk) * a.n_cells * NBV * SGB : nullptr;
  const uint16_t *vn = a.vn + static_cast<size_t>(hk) * a.n_cells * NBV;

  auto issue = [&](int j) {       // local tile j -> stage j % STAGES
    unsigned char *st = smem + C::STG + (j % STAGES) * C::STAGE;
    uint64_t *bar = &bars.full[j % STAGES];
    const int64_t key0 = static_cast<int64_t>(t_lo + j) * BN;
    tc::mbar_expect_tx(bar, C::TX);
    tc::bulk_g2s(st + C::S_KQS, kqs + key0 * NBK * QSB, BN * NBK * QSB, bar);
    if (SGB) tc::bulk_g2s(st + C::S_KSG, ksg + key0 * NBK * SGB, BN * NBK * SGB, bar);
    tc::bulk_g2s(st + C::S_KN, kn + key0 * NBK, BN * NBK * 2, bar);
    tc::bulk_g2s(st + C::S_VQS, vqs + key0 * NBV * QSB, BN * NBV * QSB, bar);
    if (SGB) tc::bulk_g2s(st + C::S_VSG, vsg + key0 * NBV * SGB, BN * NBV * SGB, bar);
    tc::bulk_g2s(st + C::S_VN, vn + key0 * NBV, BN * NBV * 2, bar);
  };

  if (warp == 0) tc::tmem_alloc<C::TMEM_COLS>(&tmem_slot);
  if (tid == NT - 32) {
    s_fail = 0;
    for (int s = 0; s < STAGES; ++s) tc::mbar_init(&bars.full[s], 1);
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&bars.dq[b], 4);
      tc::mbar_init(&bars.sf[b], 1);
      tc::mbar_init(&bars.pf[b], 4);
      tc::mbar_init(&bars.pv[b], 1);
    }
    tc::mbar_init_fence();
    tc::fence_async_smem();
    for (int i = 0; i < STAGES && i < n_tiles; ++i) issue(i);
  }

  // ---- Q' = q rotated per block (scale * log2(e) / sqrt(128) folded in), binary16 hi + lo
  {
    const float f = a.scale_log2 * kInvSqrtQK;
    for (int pr = warp; pr < BM * NBK; pr += NWARP) {
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
        const __half hh = __float2half_rn(x);
        hb[k] = __half_as_ushort(hh);
        lb[k] = __half_as_ushort(__float2half_rn(x - __half2float(hh)));
      }
      const uint32_t off = b * C::QBLK + ((d0 >> 3) * 16 + (r >> 3)) * 128 + (r & 7) * 16 + (d0 & 7) * 2;
      *reinterpret_cast<uint2 *>(smem + C::Q + off) =
          make_uint2(hb[0] | (static_cast<uint32_t>(hb[1]) << 16), hb[2] | (static_cast<uint32_t>(hb[3]) << 16));
      *reinterpret_cast<uint2 *>(smem + C::Q + NBK * C::QBLK + off) =
          make_uint2(lb[0] | (static_cast<uint32_t>(lb[1]) << 16), lb[2] | (static_cast<uint32_t>(lb[3]) << 16));
    }
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  const uint32_t sbase = tc::smem_u32(smem);
  float *nrm = reinterpret_cast<float *>(smem + C::NRM);

  // softmax state (warps 0..3: row = tid)
  const int row = tid & (BM - 1);
  const int row_q = q0 + row / G;
  const bool row_ok = warp < 4 && row_q < a.nq;
  const int64_t row_end = a.causal ? (pos0 + row_q + 1) : a.kv_len;
  float m_used = -INFINITY, l_sum = 0.f;

  if (warp == 8) {
    // ===================== control: copies and mma issue =====================
    if (lane == 0) {
      constexpr uint32_t ID_S = tc::idesc_f16(BM, BN, false, false);
      constexpr uint32_t ID_PV = tc::idesc_f16(BM, 128, false, true);
      // Descriptors: the start-address field holds addr >> 4 in 14 bits and no
      // operand crosses 256 KB, so an operand at base + off has the descriptor
      // desc(base) + (off >> 4) -- one add per mma instead of a rebuild.
      const uint64_t q_desc = tc::sdesc(sbase + C::Q, 2048, 128);
      const uint64_t k_desc = tc::sdesc(sbase + C::KV, 128, 2048);
      const uint64_t v_desc = tc::sdesc(sbase + C::KV + NBK * C::TBLK, 2048, 128);
      auto issue_pv = [&](int j) {
        const uint32_t pbuf = tmem + C::SP0 + (j & 1) * C::SPW;
        const uint64_t vb = v_desc + (((j & 1) * C::KVBUF) >> 4);
#pragma unroll
        for (int b = 0; b < NBV; ++b)
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int ks = 0; ks < BN / 16; ++ks) {
              const uint64_t bd = vb + ((b * C::TBLK + ks * 4096) >> 4);
              mma_f16_ta(tmem + b * 128, pbuf + (2 * b + part) * (BN / 2) + ks * 8, bd, ID_PV,
                         j > 0 || part > 0 || ks > 0);
            }
        tc::mma_commit(&bars.pv[j & 1]);
      };
      bool ok = true;
      for (int j = 0; j < n_tiles && ok; ++j) {
        ok = tc::mbar_wait(&bars.dq[j & 1], (j >> 1) & 1);
        if (ok && j >= 2) ok = tc::mbar_wait(&bars.pv[j & 1], ((j - 2) >> 1) & 1);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t sbuf = tmem + C::SP0 + (j & 1) * C::SPW;
        const uint64_t kb = k_desc + (((j & 1) * C::KVBUF) >> 4);
#pragma unroll
        for (int b = 0; b < NBK; ++b)
#pragma unroll
          for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
              const uint64_t ad = q_desc + (((part * NBK + b) * C::QBLK + ks * 4096) >> 4);
              const uint64_t bd = kb + ((b * C::TBLK + ks * 256) >> 4);
              tc::mma_f16(sbuf + b * BN, ad, bd, ID_S, part > 0 || ks > 0);
            }
        tc::mma_commit(&bars.sf[j & 1]);
        if (j >= 1) {
          ok = tc::mbar_wait(&bars.pf[(j - 1) & 1], ((j - 1) >> 1) & 1);
          if (!ok) break;
          tc::fence_after_sync();
          issue_pv(j - 1);
        }
      }
      if (ok && n_tiles > 0) {
        const int j = n_tiles - 1;
        ok = tc::mbar_wait(&bars.pf[j & 1], (j >> 1) & 1);
        if (ok) {
          tc::fence_after_sync();
          issue_pv(j);
        }
      }
      if (!ok) s_fail = 1;
    }
  } else if (warp >= 4) {
    // ===================== dequant: one key-block row per thread =====================
    const int dt = tid - 128;                                  // 0..127
    const Tab tab_k{a.tabk[0], a.tabk[1], a.tabk[2], a.tabk[3]};
    const Tab tab_v{a.tabv[0], a.tabv[1], a.tabv[2], a.tabv[3]};
    for (int j = 0; j < n_tiles; ++j) {
      bool ok = tc::mbar_wait(&bars.full[j % STAGES], (j / STAGES) & 1);
      if (ok && j >= 2) ok = tc::mbar_wait(&bars.pv[j & 1], ((j - 2) >> 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) { s_fail = 1; break; }
      tc::fence_after_sync();
      const unsigned char *st = smem + C::STG + (j % STAGES) * C::STAGE;
      unsigned char *buf = smem + C::KV + (j & 1) * C::KVBUF;
      for (int r = dt; r < (NBK + NBV) * BN; r += 128) {
        const bool is_v = r >= NBK * BN;
        const int rr = is_v ? r - NBK * BN : r;
        const int b = rr / BN, key = rr % BN;
        const int nb = is_v ? NBV : NBK;
        const Tab &tb = is_v ? tab_v : tab_k;
        const uint8_t *qrow = st + (is_v ? C::S_VQS : C::S_KQS) + (key * nb + b) * QSB;
        unsigned char *dst = buf + (is_v ? NBK + b : b) * C::TBLK + (key >> 3) * 2048 + (key & 7) * 16;
        if (T == 4) {
#pragma unroll
          for (int w4 = 0; w4 < 4; ++w4) {
            const uint4 w = reinterpret_cast<const uint4 *>(qrow)[w4];
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 o;
              dq4<4>(ws[i], tb, o.x, o.y);
              dq4<4>(ws[i] >> 16, tb, o.z, o.w);
              *reinterpret_cast<uint4 *>(dst + (4 * w4 + i) * 128) = o;
            }
          }
        } else {
          uint32_t sgw[4] = {0u, 0u, 0u, 0u};
          if (T == 3) {
            const uint4 sg4 =
                *reinterpret_cast<const uint4 *>(st + (is_v ? C::S_VSG : C::S_KSG) + (key * nb + b) * SGB);
            sgw[0] = sg4.x; sgw[1] = sg4.y; sgw[2] = sg4.z; sgw[3] = sg4.w;
          }
#pragma unroll
          for (int hq = 0; hq < 2; ++hq) {
            const uint4 w = reinterpret_cast<const uint4 *>(qrow)[hq];
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int wi = 4 * hq + i;                       // qs word: elements 16 wi ..
              uint32_t s0, s1;
              sel_words<T>(ws[i], sgw[wi >> 1], (wi & 1) != 0, s0, s1);
              uint4 o0, o1;
              dq4<T>(s0, tb, o0.x, o0.y);
              dq4<T>(s0 >> 16, tb, o0.z, o0.w);
              dq4<T>(s1, tb, o1.x, o1.y);
              dq4<T>(s1 >> 16, tb, o1.z, o1.w);
              *reinterpret_cast<uint4 *>(dst + (2 * wi) * 128) = o0;
              *reinterpret_cast<uint4 *>(dst + (2 * wi + 1) * 128) = o1;
            }
          }
        }
        const uint16_t *np = reinterpret_cast<const uint16_t *>(st + (is_v ? C::S_VN : C::S_KN));
        nrm[(j & 1) * BN * (NBK + NBV) + key * (NBK + NBV) + (is_v ? NBK + b : b)] =
            __half2float(__ushort_as_half(np[key * nb + b]));
      }
      tc::fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.dq[j & 1]);
      // the stage of tile j is free once all four dequant warps are done with it:
      // one of them refills it (the control thread only issues mma)
      if (warp == 4 && lane == 0 && j + STAGES < n_tiles) {
        if (tc::mbar_wait(&bars.dq[j & 1], (j >> 1) & 1)) issue(j + STAGES);
        else s_fail = 1;
      }
    }
  } else {
    // ===================== softmax: one query row per thread =====================
    const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      ok = tc::mbar_wait(&bars.sf[j & 1], (j >> 1) & 1);
      if (ok) ok = tc::mbar_wait(&bars.dq[j & 1], (j >> 1) & 1);     // norms of tile j are written
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc::fence_after_sync();
      const uint32_t sbuf = tmem + lane_off + C::SP0 + (j & 1) * C::SPW;
      const float *nr = nrm + (j & 1) * BN * (NBK + NBV);
      float s[BN];
#pragma unroll
      for (int i = 0; i < BN; ++i) s[i] = 0.f;
      {
        uint32_t r0[NBK * BN];                                 // all S columns, one wait
#pragma unroll
        for (int c0 = 0; c0 < NBK * BN; c0 += 32) tc::tmem_ld32(sbuf + c0, r0 + c0);
        tc::tmem_wait_ld();
#pragma unroll
        for (int b = 0; b < NBK; ++b)
#pragma unroll
          for (int i = 0; i < BN; ++i) s[i] = fmaf(nr[i * (NBK + NBV) + b], __uint_as_float(r0[b * BN + i]), s[i]);
      }
      const int64_t key0 = static_cast<int64_t>(t_lo + j) * BN;
      const int nvis = row_ok ? static_cast<int>(i64max(0, i64min(BN, row_end - key0))) : 0;
      float mt = -INFINITY;
#pragma unroll
      for (int i = 0; i < BN; ++i)
        if (i < nvis) mt = fmaxf(mt, s[i]);
      const bool raise = mt > m_used + kLazyRescale || (m_used == -INFINITY && mt > -INFINITY);
      const float fct = (raise && m_used != -INFINITY) ? exp2f(m_used - mt) : 1.f;
      if (raise) m_used = mt;
      if (__any_sync(0xffffffffu, fct != 1.f)) {
        // O must be stable: wait for the PV mma of the previous tile
        bool okp = (j == 0) || tc::mbar_wait(&bars.pv[(j - 1) & 1], ((j - 1) >> 1) & 1);
        if (!__all_sync(0xffffffffu, okp)) { ok = false; break; }
        tc::fence_after_sync();
        l_sum *= fct;
#pragma unroll
        for (int c = 0; c < DVP; c += 32) {
          uint32_t r[32];
          tc::tmem_ld32(tmem + lane_off + c, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * fct);
          tc::tmem_st32(tmem + lane_off + c, r);
        }
      }
      float psum = 0.f;
#pragma unroll
      for (int i = 0; i < BN; ++i) {
        s[i] = (i < nvis) ? tc::ex2(s[i] - m_used) : 0.f;
        psum += s[i];
      }
      l_sum += psum;
      // P'_(b, hi/lo) into tensor memory over S_j: row = lane, fp16 pairs of keys
#pragma unroll
      for (int b = 0; b < NBV; ++b) {
        uint32_t ph[BN / 2], pl[BN / 2];
#pragma unroll
        for (int i = 0; i < BN / 2; ++i) {
          const int k0 = 2 * i;
          // masked keys may carry garbage norms: select, never multiply, a zero
          const float x0 = s[k0] > 0.f ? s[k0] * nr[k0 * (NBK + NBV) + NBK + b] : 0.f;
          const float x1 = s[k0 + 1] > 0.f ? s[k0 + 1] * nr[(k0 + 1) * (NBK + NBV) + NBK + b] : 0.f;
          const __half2 h = __floats2half2_rn(x0, x1);
          const float2 hf = __half22float2(h);
          const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
          ph[i] = *reinterpret_cast<const uint32_t *>(&h);
          pl[i] = *reinterpret_cast<const uint32_t *>(&l);
        }
        tmem_st<BN / 2>(sbuf + (2 * b) * (BN / 2), ph);
        tmem_st<BN / 2>(sbuf + (2 * b + 1) * (BN / 2), pl);
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.pf[j & 1]);
    }
    // the last PV must be complete before O is read
    if (ok && n_tiles > 0) {
      const int j = n_tiles - 1;
      ok = tc::mbar_wait(&bars.pv[j & 1], (j >> 1) & 1);
      ok = __all_sync(0xffffffffu, ok);
      tc::fence_after_sync();
    }
    if (!ok) s_fail = 1;
  }

  // ===================== epilogue =====================
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const bool failed = s_fail != 0;
  if (failed && tid == 0) set_status(a.status, TQ_ERR_TIMEOUT);
  const int h_row = hk * G + row % G;
  float *orow = a.out + (static_cast<size_t>(row_ok ? row_q : 0) * a.n_q_heads + h_row) * a.dv;

  if (n_split == 1) {
    if (warp < 4 && !failed) {
      const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
      const float inv = (l_sum > 0.f ? 1.f / l_sum : 0.f) * kInvSqrtQK;
#pragma unroll 1
      for (int b = 0; b < NBV; ++b) {
        float o[128];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tc::tmem_ld32(tmem + lane_off + b * 128 + 32 * c, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[32 * c + i] = n_tiles > 0 ? __uint_as_float(r[i]) : 0.f;
        }
        rotate_store_block(o, inv, a.cbv, orow + b * 128, a.dv - b * 128, row_ok);
      }
    }
  } else {
    // split key range: store (m, l, O) of every row; the last CTA of this query tile merges
    const size_t tile_id = static_cast<size_t>(blockIdx.x) * a.n_kv_heads + hk;
    const size_t stride = 4 + DVP;             // m, l, 2 pad floats: O rows stay 16-byte aligned
    float *part = a.part + (tile_id * n_split + split) * BM * stride;
    if (warp < 4) {
      const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
      float *pr = part + static_cast<size_t>(row) * stride;
      const bool has = !failed && n_tiles > 0;
      pr[0] = has ? m_used : -INFINITY;
      pr[1] = has ? l_sum : 0.f;
#pragma unroll 1
      for (int c = 0; c < DVP; c += 32) {
        uint32_t r[32];
        tc::tmem_ld32(tmem + lane_off + c, r);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          *reinterpret_cast<float4 *>(pr + 4 + c + i) =
              has ? make_float4(__uint_as_float(r[i]), __uint_as_float(r[i + 1]), __uint_as_float(r[i + 2]),
                                __uint_as_float(r[i + 3]))
                  : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = (atomicAdd(&a.counters[tile_id], 1) == n_split - 1);
    __syncthreads();
    if (s_last) {
      __threadfence();
      const float *base = a.part + tile_id * n_split * BM * stride;
      float *wts = reinterpret_cast<float *>(smem + C::STG);        // [BM][n_split] weights / L
      float *acc = reinterpret_cast<float *>(smem + C::Q);          // [BM][DVP] merged rows
      if (tid < min(BM, (a.nq - q0) * G)) {
        float M = -INFINITY;
        for (int s2 = 0; s2 < n_split; ++s2)
          M = fmaxf(M, __ldcg(base + (static_cast<size_t>(s2) * BM + tid) * stride));
        float L = 0.f;
        for (int s2 = 0; s2 < n_split; ++s2) {
          const float *p = base + (static_cast<size_t>(s2) * BM + tid) * stride;
          const float m = __ldcg(p);
          const float w = (m == -INFINITY) ? 0.f : exp2f(m - M);
          wts[tid * n_split + s2] = w;
          L += w * __ldcg(p + 1);
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        for (int s2 = 0; s2 < n_split; ++s2) wts[tid * n_split + s2] *= inv;
      }
      __syncthreads();
      const int rows_valid = min(BM, (a.nq - q0) * G);          // rows of queries < nq
      for (int i = tid; i < rows_valid * DVP; i += NT) {
        const int r = i / DVP, d = i % DVP;
        float o = 0.f;
        for (int s2 = 0; s2 < n_split; ++s2)
          o += wts[r * n_split + s2] * __ldcg(base + (static_cast<size_t>(s2) * BM + r) * stride + 4 + d);
        acc[i] = o;
      }
      __syncthreads();
      if (warp < 4) {
#pragma unroll 1
        for (int b = 0; b < NBV; ++b) {
          float o[128];
#pragma unroll
          for (int i = 0; i < 128; ++i) o[i] = acc[row * DVP + b * 128 + i];
          rotate_store_block(o, kInvSqrtQK, a.cbv, orow + b * 128, a.dv - b * 128, row_ok);
        }
      }
      if (tid == 0) a.counters[tile_id] = 0;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc<C::TMEM_COLS>(tmem);
}

template <int T, int NBK, int NBV>
cudaError_t launch_one(const PrefillArgs &a, cudaStream_t s) {
  using C = Cfg<T, NBK, NBV>;
  static_assert(C::TOTAL <= 227 * 1024, "shared memory");
  static_assert(C::COLS_NEEDED <= 512, "tensor memory");
  static_assert(C::BN % 16 == 0 && C::BN <= 64, "key tile");
  // the merge reuses the Q region for BM x DVP floats and the staging ring for the weights
  static_assert(2 * NBK * C::QBLK >= BM * C::DVP * 4, "merge buffer");
  static_assert(STAGES * C::STAGE >= BM * 16 * 4, "merge weights");
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel<T, NBK, NBV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)C::TOTAL);
  if (e != cudaSuccess) return e;
  dim3 grid((a.nq * a.group + BM - 1) / BM, a.n_kv_heads, a.n_split);
  prefill_kernel<T, NBK, NBV><<<grid, NT, C::TOTAL, s>>>(a);
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

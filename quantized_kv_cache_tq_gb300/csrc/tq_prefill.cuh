// Multi-query (prefill / verify) attention over the packed TurboQuant cache on
// the tcgen05 tensor cores, with the K/V tiles dequantised inline
// ([HIP#28] "2. Inline-dequant TILE prefill": expand the packed cache while it
// is loaded into on-chip tiles, never write an f16 copy of the cache).
//
// Persistent CTAs (at most one per SM) take work items from an atomic queue: one
// KV head x 128 query rows (128/G queries x the G query heads of the GQA group,
// row r = query (r / G), head (r % G)) x one range of key tiles (BN = 64 keys for
// 256-dim K rows, 128 for 128-dim rows).  Warp roles, connected by mbarriers
// only (no CTA barrier inside the key loop):
//   control warp (one thread): issues S_j = Q'K'_j^T into tensor memory as soon
//     as K'_j is expanded, then O += P'_{j-1} V'_{j-1} once the softmax warps
//     have written P'_{j-1} -- the tensor cores compute S_{j+1} while the
//     softmax warps work on tile j;
//   4 dequant warps: expand the packed K/V tiles (staged by cp.async.bulk in
//     two small rings, K with both tiles' norms, V) into binary16 K'/V' operand
//     tiles (exact centroid values), one key-block row per thread.  K' and V'
//     are single-buffered: K'_{j+1} is written as soon as S_j is done, before
//     V'_j (which waits for PV_{j-1}), so the next S never waits for a V tile;
//   8 softmax warps, two per TMEM lane quarter (one query row, half the tile's
//     keys per thread): read S_j, form s = sum_b |k_b| S_b, apply the causal
//     mask and the online softmax (log2 domain; the row maximum is exchanged
//     between the two halves through shared memory; the reference maximum is
//     raised only when it grows by more than 2^8, then O is rescaled in tensor
//     memory), and write P'_b = p |v_b| as binary16 hi + lo straight into tensor
//     memory over S_j, where the PV mma reads it as its A operand.
// Precision: Q' and P' are split into binary16 hi + lo parts and both go
// through the tensor cores; K'/V' are exact; accumulation is fp32.
// Work items are queued longest first (the causal tiles near the end of the
// prompt attend the most keys).  When the query tiles do not fill the SMs, each
// query tile's key range is split over several items; they store their
// (max, sum, O) rows (4 + 128 nbv floats each) and a second kernel merges them
// with log-sum-exp weights (tq_prefill_merge.cu).
// Epilogue: o = S H (O / l) / sqrt(128) per 128-dim block (V codebook), fp32.
//
// Shared-memory operands (SWIZZLE_NONE core matrices of 8 rows x 16 B):
//   Q'_b (hi, lo)  A, K-major   [d/8][row/8]   LBO 2048 (along d)    SBO 128
//   K'_b           B, K-major   [key/8][d/8]   LBO 128 (along d)     SBO 2048
//   V'_b           B, MN-major  [key/8][d/8]   LBO 2048 (along keys) SBO 128
// Tensor memory (fp32 columns): O_b at 128 b; per buffer S_b at BN b, aliased by
// P'_(b, part) at (2b + part) BN/2 (fp16 pairs of keys, row = lane).
#pragma once

#include "tq_common.cuh"
#include "tq_tc.cuh"

namespace tq {
namespace pf {

constexpr int BM = 128;          // query rows per CTA (TMEM lanes)
constexpr int NSM = 8;           // softmax warps 0..7 (warps w and w + 4 share TMEM lane quarter w)
constexpr int DQ0 = 8;           // dequant warps 8..11
constexpr int CTRL = 12;         // control warp
constexpr int NWARP = 13;
constexpr int NT = NWARP * 32;
constexpr float kLazyRescale = 8.f;   // log2 units

template <int T, int NBK, int NBV>
struct Cfg {
  static constexpr int BN = (NBK == 2) ? 64 : 128;         // keys per tile
  static constexpr int HB = BN / 2;                        // keys per softmax thread
  static constexpr int QSB = TypeTraits<T>::QSB, SGB = TypeTraits<T>::SGB;
  static constexpr uint32_t QBLK = 32768;                  // 128 rows x 128 dims fp16
  static constexpr uint32_t TBLK = BN * 256;               // BN keys x 128 dims fp16
  static constexpr uint32_t Q = 0;                         // [part][NBK] blocks
  static constexpr uint32_t KT = Q + 2 * NBK * QBLK;       // K'_b tiles
  static constexpr uint32_t VT = KT + NBK * TBLK;          // V'_b tiles
  // K staging: K qs, K signs, K norms, V norms; V staging: V qs, V signs
  static constexpr uint32_t K_QS = 0;
  static constexpr uint32_t K_SG = K_QS + BN * NBK * QSB;
  static constexpr uint32_t K_KN = K_SG + BN * NBK * SGB;
  static constexpr uint32_t K_VN = K_KN + BN * NBK * 2;
  static constexpr uint32_t KSTAGE = (K_VN + BN * NBV * 2 + 127) / 128 * 128;
  static constexpr uint32_t V_QS = 0;
  static constexpr uint32_t V_SG = V_QS + BN * NBV * QSB;
  static constexpr uint32_t VSTAGE = (V_SG + BN * NBV * SGB + 127) / 128 * 128;
  static constexpr int KST = 2;
  static constexpr int VST = (T == 4 && NBK == 2) ? 1 : 2;
  static constexpr uint32_t KSTG = VT + NBV * TBLK;
  static constexpr uint32_t VSTG = KSTG + KST * KSTAGE;
  static constexpr uint32_t NRM = VSTG + VST * VSTAGE;     // floats [2][4][BN]: |k_0|, |k_1|, |v_0|, |v_1| of each key
  static constexpr uint32_t TOTAL = NRM + 2 * BN * 4 * 4;
  static constexpr uint32_t KTX = BN * (NBK * (QSB + SGB + 2) + NBV * 2);   // bytes of a full K stage
  static constexpr uint32_t VTX = BN * NBV * (QSB + SGB);                   // bytes of a full V stage
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
  uint64_t kfull[2];       // packed K stage (and both tiles' norms) landed (tx)
  uint64_t vfull[2];       // packed V stage landed (tx)
  uint64_t dqk;            // K'_j expanded (4 dequant warps)
  uint64_t dqv;            // V'_j expanded (4 dequant warps)
  uint64_t nrmf[2];        // norms of tile j in buffer j & 1 (4 dequant warps)
  uint64_t sf[2];          // S_j computed (mma commit)
  uint64_t pf[2];          // P'_j written (8 softmax warps)
  uint64_t pv[2];          // PV_j computed (mma commit)
};

// Output rows of one warp: 32 rows x one 128-dim V block in shared memory (row
// r at stg + r * stride floats, already divided by l and by sqrt(128); with SWZ
// the 16-byte chunk c of row r sits at chunk c ^ (r & 7), so that 32 threads
// writing one row each do not collide on a bank).  Each row is rotated back by
// the whole warp (o = S H o', 4 dims per lane, the page's butterflies with
// shuffles) and stored as 512 contiguous bytes.
template <bool SWZ>
__device__ __forceinline__ void rotate_store_rows(const float *stg, int stride, const PrefillArgs &a, int row0, int q0,
                                                  int hk, int b, int lane) {
  const int G = a.group, g_shift = __ffs(G) - 1;
  const int n_rows = max(0, min(32, (a.nq - q0) * G - row0));       // rows of queries < nq
  const int d = b * QK + 4 * lane;
  for (int r0 = 0; r0 < n_rows; r0 += 4) {                         // four independent rows at a time
    float v[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int r = r0 + u;
      const int chunk = SWZ ? (lane ^ (r & 7)) : lane;
      const float4 x = *reinterpret_cast<const float4 *>(stg + r * stride + 4 * chunk);
      v[u][0] = x.x; v[u][1] = x.y; v[u][2] = x.z; v[u][3] = x.w;
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      wht128_warp(v[u], lane);
      apply_signs(v[u], a.cbv, lane);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int rr = row0 + r0 + u;
      if (r0 + u < n_rows && d + 4 <= a.dv) {
        float *o = a.out + (static_cast<size_t>(q0 + (rr >> g_shift)) * a.n_q_heads + hk * G + (rr & (G - 1))) * a.dv + d;
        *reinterpret_cast<float4 *>(o) = make_float4(v[u][0], v[u][1], v[u][2], v[u][3]);
      }
    }
  }
}

// Half hw (elements 64 hw .. 64 hw + 63) of one key-block row of a packed tile
// (qs row, signs row) -> 64 binary16 values in the core-matrix layout of an
// operand tile (`dst` = the row's first core matrix; the 16 d-octets of the row
// follow at 128-byte steps).
template <int T>
__device__ __forceinline__ void expand_half(const uint8_t *qrow, const uint8_t *srow, const Tab &tb, unsigned char *dst,
                                            int hw) {
  if (T == 4) {
#pragma unroll
    for (int w2 = 0; w2 < 2; ++w2) {
      const int w4 = 2 * hw + w2;
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
    uint32_t sgw[2] = {0u, 0u};
    if (T == 3) {
      const uint2 sg2 = reinterpret_cast<const uint2 *>(srow)[hw];
      sgw[0] = sg2.x; sgw[1] = sg2.y;
    }
    const uint4 w = reinterpret_cast<const uint4 *>(qrow)[hw];
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int wi = 4 * hw + i;                       // qs word: elements 16 wi ..
      uint32_t s0, s1;
      sel_words<T>(ws[i], sgw[i >> 1], (wi & 1) != 0, s0, s1);
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

// Q'_b of the CTA's query rows: q rotated per 128-dim block (the K codebook's
// signs, then the page's butterflies; scale * log2(e) / sqrt(128) folded in),
// stored as binary16 hi + lo in the core-matrix layout of the S mma's A operand.
// This warp takes row-block groups gi = warp + NWARP (u0 + u), u < NG: rows
// 8 (gi % (BM / 8)) .. + 7 of block gi / (BM / 8).  Lane 4 j + l4 holds elements
// 16 i + 4 l4 + k (i < 8, k < 4) of the group's row j, so the butterflies
// h = 1, 2, 16, 32, 64 stay in the lane and h = 4, 8 cross lanes, and one store
// instruction covers 8 rows, which sit in 8 different bank groups (one row per
// warp put all 32 lanes of a store in one 16-byte bank window).  All NG groups'
// loads are issued before any of them is used.
template <int NBK, int NG, bool F32>
__device__ __forceinline__ void prep_q_groups(const PrefillArgs &a, unsigned char *qsm, int u0, int warp, int lane,
                                              int q0, int hk, int g_shift, float f, uint32_t smask) {
  constexpr int NW = F32 ? 4 : 2;
  constexpr int NGRP = BM * NBK / 8;
  constexpr uint32_t QBLK = 32768;
  const int G = a.group, j = lane >> 2, l4 = lane & 3;
  uint32_t raw[NG][8][NW];
#pragma unroll
  for (int u = 0; u < NG; ++u) {
    const int gi = warp + NWARP * (u0 + u);
    const int pr = gi * 8 + j, r = pr % BM, b = pr / BM;
    const int qi = q0 + (r >> g_shift), h = hk * G + (r & (G - 1));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
      for (int k = 0; k < NW; ++k) raw[u][i][k] = 0u;
      const int d = b * QK + 16 * i + 4 * l4;
      if (gi < NGRP && qi < a.nq && d + 4 <= a.dk) {
        const size_t e = (static_cast<size_t>(qi) * a.n_q_heads + h) * a.dk + d;
        if (F32) {
          const uint4 x = *reinterpret_cast<const uint4 *>(static_cast<const float *>(a.q) + e);
          raw[u][i][0] = x.x; raw[u][i][1] = x.y; raw[u][i][2 % NW] = x.z; raw[u][i][3 % NW] = x.w;
        } else {
          const uint2 x = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(a.q) + e);
          raw[u][i][0] = x.x; raw[u][i][1] = x.y;
        }
      }
    }
  }
#pragma unroll
  for (int u = 0; u < NG; ++u) {
    const int gi = warp + NWARP * (u0 + u);
    if (gi >= NGRP) break;                          // warp-uniform
    const int pr = gi * 8 + j, r = pr % BM, b = pr / BM;
    float v[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float x;
        if (F32) {
          x = __uint_as_float(raw[u][i][k % NW]);
        } else {
          const uint16_t bits = static_cast<uint16_t>(raw[u][i][k >> 1] >> (16 * (k & 1)));
          x = a.q_type == TQ_BF16 ? __bfloat162float(__ushort_as_bfloat16(bits)) : __half2float(__ushort_as_half(bits));
        }
        v[i][k] = __uint_as_float(__float_as_uint(x) ^ ((smask << (31 - (4 * i + k))) & 0x80000000u));
      }
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
          for (int k = 0; k < 4; ++k) {
            const float x = v[i][k], y = v[i | hb][k];
            v[i][k] = x + y;
            v[i | hb][k] = x - y;
          }
#pragma unroll
    for (int m = 1; m < 4; m <<= 1) {
      const float sg = (l4 & m) ? -1.f : 1.f;
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float o = __shfl_xor_sync(0xffffffffu, v[i][k], m);
          v[i][k] = fmaf(sg, v[i][k], o);
        }
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint16_t hb[4], lb[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float x = v[i][k] * f;
        const __half hh = __float2half_rn(x);
        hb[k] = __half_as_ushort(hh);
        lb[k] = __half_as_ushort(__float2half_rn(x - __half2float(hh)));
      }
      const int dd = 16 * i + 4 * l4;
      const uint32_t off = b * QBLK + ((dd >> 3) * 16 + (r >> 3)) * 128 + (r & 7) * 16 + (dd & 7) * 2;
      *reinterpret_cast<uint2 *>(qsm + off) =
          make_uint2(hb[0] | (static_cast<uint32_t>(hb[1]) << 16), hb[2] | (static_cast<uint32_t>(hb[3]) << 16));
      *reinterpret_cast<uint2 *>(qsm + NBK * QBLK + off) =
          make_uint2(lb[0] | (static_cast<uint32_t>(lb[1]) << 16), lb[2] | (static_cast<uint32_t>(lb[3]) << 16));
    }
  }
}

template <int T, int NBK, int NBV>
__global__ void __launch_bounds__(NT, 1) prefill_kernel(const PrefillArgs a) {
  using C = Cfg<T, NBK, NBV>;
  constexpr int BN = C::BN, HB = C::HB, QSB = C::QSB, SGB = C::SGB, DVP = C::DVP;
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ __align__(8) Bars bars;
  __shared__ uint32_t tmem_slot;
  __shared__ int s_fail;
  __shared__ int s_item;
  // exchange between the two softmax warps of a row (value per row, flag per warp),
  // double-buffered by the parity of the exchange count
  __shared__ float xv[2][2][BM];
  __shared__ int xf[2][2][4];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.group;
  const int g_shift = __ffs(G) - 1;              // G is a power of two
  const int n_split = a.n_split;
  const int64_t pos0 = a.kv_len - a.nq;
  const uint32_t sbase = tc::smem_u32(smem);
  float *nrm = reinterpret_cast<float *>(smem + C::NRM);
  const int row = 32 * (warp & 3) + lane;        // softmax warps: TMEM lane / query row
  const int half = (warp >> 2) & 1;              // softmax warps: which half of each tile's keys
  const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;

  if (warp == 0) tc::tmem_alloc<C::TMEM_COLS>(&tmem_slot);
  if (tid == CTRL * 32) {
    s_fail = 0;
    for (int s = 0; s < 2; ++s) {
      tc::mbar_init(&bars.kfull[s], 1);
      tc::mbar_init(&bars.vfull[s], 1);
      tc::mbar_init(&bars.nrmf[s], 4);
      tc::mbar_init(&bars.sf[s], 1);
      tc::mbar_init(&bars.pf[s], NSM);
      tc::mbar_init(&bars.pv[s], 1);
    }
    tc::mbar_init(&bars.dqk, 4);
    tc::mbar_init(&bars.dqv, 4);
    tc::mbar_init_fence();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  int xc = 0;                                    // softmax pair exchanges so far
  int g0 = 0;                                    // tiles this CTA processed before the current item
                                                 // (every mbarrier phase follows this running count)

  // Persistent loop over work items (query tile, KV head, key split), the longest
  // query tiles first; each CTA takes the next item when it is done with one.
  for (;;) {
    if (tid == 0) s_item = atomicAdd(&a.sched[0], 1);
    __syncthreads();
    const int item = s_item;
    if (item >= a.n_items || s_fail) break;
    const int per_qt = a.n_kv_heads * n_split;
    const int qt = a.n_qt - 1 - item / per_qt;
    const int hk = (item % per_qt) % a.n_kv_heads;
    const int split = (item % per_qt) / a.n_kv_heads;
    const int q0 = qt * (BM / G);
    const int q_last = min(a.nq, q0 + BM / G) - 1;
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

    // bulk copies of local tile j (keys past n_cells are not read; n_cells is a
    // multiple of 64, so every copy stays a multiple of 16 bytes); ring slots and
    // phases follow the running tile count g0 + j
    auto tile_keys = [&](int j) -> int {
      const int64_t key0 = static_cast<int64_t>(t_lo + j) * BN;
      return static_cast<int>(i64min(BN, a.n_cells - key0));
    };
    auto issue_k = [&](int j) {
      const int g = g0 + j;
      unsigned char *st = smem + C::KSTG + (g % C::KST) * C::KSTAGE;
      uint64_t *bar = &bars.kfull[g % C::KST];
      const int64_t key0 = static_cast<int64_t>(t_lo + j) * BN;
      const int nk = tile_keys(j);
      tc::mbar_expect_tx(bar, nk * (NBK * (QSB + SGB + 2) + NBV * 2));
      tc::bulk_g2s(st + C::K_QS, kqs + key0 * NBK * QSB, nk * NBK * QSB, bar);
      if (SGB) tc::bulk_g2s(st + C::K_SG, ksg + key0 * NBK * SGB, nk * NBK * SGB, bar);
      tc::bulk_g2s(st + C::K_KN, kn + key0 * NBK, nk * NBK * 2, bar);
      tc::bulk_g2s(st + C::K_VN, vn + key0 * NBV, nk * NBV * 2, bar);
    };
    auto issue_v = [&](int j) {
      const int g = g0 + j;
      unsigned char *st = smem + C::VSTG + (g % C::VST) * C::VSTAGE;
      uint64_t *bar = &bars.vfull[g % C::VST];
      const int64_t key0 = static_cast<int64_t>(t_lo + j) * BN;
      const int nk = tile_keys(j);
      tc::mbar_expect_tx(bar, nk * NBV * (QSB + SGB));
      tc::bulk_g2s(st + C::V_QS, vqs + key0 * NBV * QSB, nk * NBV * QSB, bar);
      if (SGB) tc::bulk_g2s(st + C::V_SG, vsg + key0 * NBV * SGB, nk * NBV * SGB, bar);
    };
    if (tid == CTRL * 32) {
      tc::fence_async_smem();
      for (int i = 0; i < C::KST && i < n_tiles; ++i) issue_k(i);
      for (int i = 0; i < C::VST && i < n_tiles; ++i) issue_v(i);
    }

    // ---- Q' = q rotated per block, binary16 hi + lo
    {
      constexpr int GPW = (BM * NBK / 8 + NWARP - 1) / NWARP;      // row-block groups per warp
      const float f = a.scale_log2 * kInvSqrtQK;
      const int l4 = lane & 3;
      uint32_t smask = 0;                                           // K-codebook signs of this lane's elements
#pragma unroll
      for (int i = 0; i < 8; ++i) smask |= ((a.cbk.sign_bits[i >> 1] >> (16 * (i & 1) + 4 * l4)) & 0xFu) << (4 * i);
      if (a.q_type == TQ_F32) {
        prep_q_groups<NBK, (GPW + 1) / 2, true>(a, smem + C::Q, 0, warp, lane, q0, hk, g_shift, f, smask);
        if (GPW / 2 > 0)
          prep_q_groups<NBK, (GPW / 2 > 0 ? GPW / 2 : 1), true>(a, smem + C::Q, (GPW + 1) / 2, warp, lane, q0, hk,
                                                                g_shift, f, smask);
      } else {
        prep_q_groups<NBK, GPW, false>(a, smem + C::Q, 0, warp, lane, q0, hk, g_shift, f, smask);
      }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();

    // softmax state (warps 0..7)
    const int row_q = q0 + (row >> g_shift);
    const bool row_ok = warp < NSM && row_q < a.nq;
    const int64_t row_end = a.causal ? (pos0 + row_q + 1) : a.kv_len;
    float m_used = -INFINITY, l_sum = 0.f;

    if (warp == CTRL) {
      // ===================== control: mma issue =====================
      if (lane == 0) {
        constexpr uint32_t ID_S = tc::idesc_f16(BM, BN, false, false);
        constexpr uint32_t ID_PV = tc::idesc_f16(BM, 128, false, true);
        // Descriptors: the start-address field holds addr >> 4 in 14 bits and no
        // operand crosses 256 KB, so an operand at base + off has the descriptor
        // desc(base) + (off >> 4) -- one add per mma instead of a rebuild.
        const uint64_t q_desc = tc::sdesc(sbase + C::Q, 2048, 128);
        const uint64_t k_desc = tc::sdesc(sbase + C::KT, 128, 2048);
        const uint64_t v_desc = tc::sdesc(sbase + C::VT, 2048, 128);
        auto issue_pv = [&](int j) {
          const int g = g0 + j;
          const uint32_t pbuf = tmem + C::SP0 + (g & 1) * C::SPW;
#pragma unroll
          for (int b = 0; b < NBV; ++b)
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
              for (int ks = 0; ks < BN / 16; ++ks) {
                const uint64_t bd = v_desc + ((b * C::TBLK + ks * 4096) >> 4);
                mma_f16_ta(tmem + b * 128, pbuf + (2 * b + part) * (BN / 2) + ks * 8, bd, ID_PV,
                           j > 0 || part > 0 || ks > 0);
              }
          tc::mma_commit(&bars.pv[g & 1]);
        };
        bool ok = true;
        for (int j = 0; j < n_tiles && ok; ++j) {
          const int g = g0 + j;
          ok = tc::mbar_wait(&bars.dqk, g & 1);                       // K'_j expanded
          if (!ok) break;
          tc::fence_after_sync();
          const uint32_t sbuf = tmem + C::SP0 + (g & 1) * C::SPW;
#pragma unroll
          for (int b = 0; b < NBK; ++b)
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
              for (int ks = 0; ks < 8; ++ks) {
                const uint64_t ad = q_desc + (((part * NBK + b) * C::QBLK + ks * 4096) >> 4);
                const uint64_t bd = k_desc + ((b * C::TBLK + ks * 256) >> 4);
                tc::mma_f16(sbuf + b * BN, ad, bd, ID_S, part > 0 || ks > 0);
              }
          tc::mma_commit(&bars.sf[g & 1]);
          if (j >= 1) {
            ok = tc::mbar_wait(&bars.pf[(g - 1) & 1], ((g - 1) >> 1) & 1) && tc::mbar_wait(&bars.dqv, (g - 1) & 1);
            if (!ok) break;
            tc::fence_after_sync();
            issue_pv(j - 1);
          }
        }
        if (ok && n_tiles > 0) {
          const int j = n_tiles - 1, g = g0 + j;
          ok = tc::mbar_wait(&bars.pf[g & 1], (g >> 1) & 1) && tc::mbar_wait(&bars.dqv, g & 1);
          if (ok) {
            tc::fence_after_sync();
            issue_pv(j);
          }
        }
        if (!ok) s_fail = 1;
      }
    } else if (warp >= DQ0) {
      // ===================== dequant: one key-block row per thread =====================
      // program order K'_0, then K'_{j+1} before V'_j: S_{j+1} never waits for a V tile
      const int dt = tid - DQ0 * 32;                             // 0..127
      const Tab tab_k{a.tabk[0], a.tabk[1], a.tabk[2], a.tabk[3]};
      const Tab tab_v{a.tabv[0], a.tabv[1], a.tabv[2], a.tabv[3]};
      unsigned char *kt = smem + C::KT;
      unsigned char *vt = smem + C::VT;
      auto k_phase = [&](int j) -> bool {
        const int g = g0 + j;
        bool ok = tc::mbar_wait(&bars.kfull[g % C::KST], (g / C::KST) & 1);
        if (ok && j >= 2) ok = tc::mbar_wait(&bars.pf[(g - 2) & 1], ((g - 2) >> 1) & 1);    // norm buffer free
        if (!__all_sync(0xffffffffu, ok)) return false;
        tc::fence_after_sync();
        const unsigned char *st = smem + C::KSTG + (g % C::KST) * C::KSTAGE;
        if (dt < BN) {
          // norms of the tile's keys; keys past the last one any row of this
          // item attends (or past the cells) read as 0, so that a masked key's
          // weight p = 0 gives p |v| = 0 whatever its bytes
          const uint16_t *knp = reinterpret_cast<const uint16_t *>(st + C::K_KN) + dt * NBK;
          const uint16_t *vnp = reinterpret_cast<const uint16_t *>(st + C::K_VN) + dt * NBV;
          const bool live = static_cast<int64_t>(t_lo + j) * BN + dt < kv_hi;
          float *nb = nrm + (g & 1) * 4 * BN + dt;
          nb[0] = live ? __half2float(__ushort_as_half(knp[0])) : 0.f;
          nb[BN] = (live && NBK > 1) ? __half2float(__ushort_as_half(knp[NBK > 1 ? 1 : 0])) : 0.f;
          nb[2 * BN] = live ? __half2float(__ushort_as_half(vnp[0])) : 0.f;
          nb[3 * BN] = (live && NBV > 1) ? __half2float(__ushort_as_half(vnp[NBV > 1 ? 1 : 0])) : 0.f;
        }
        // K' (two threads per key row, half a row each) once S_{j-1} is done with it
        ok = (j == 0) || tc::mbar_wait(&bars.sf[(g - 1) & 1], ((g - 1) >> 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) return false;
        tc::fence_after_sync();
        for (int r = dt; r < 2 * NBK * BN; r += 128) {
          const int b = r / (2 * BN), key = (r >> 1) % BN, hw = r & 1;
          expand_half<T>(st + C::K_QS + (key * NBK + b) * QSB, st + C::K_SG + (key * NBK + b) * SGB, tab_k,
                         kt + b * C::TBLK + (key >> 3) * 2048 + (key & 7) * 16, hw);
        }
        tc::fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&bars.nrmf[g & 1]);
          mbar_arrive(&bars.dqk);
        }
        // the K stage of tile j is free once all four dequant warps are done with it
        if (warp == DQ0 && lane == 0 && j + C::KST < n_tiles) {
          if (tc::mbar_wait(&bars.dqk, g & 1)) issue_k(j + C::KST);
          else s_fail = 1;
        }
        return true;
      };
      auto v_phase = [&](int j) -> bool {
        const int g = g0 + j;
        bool ok = tc::mbar_wait(&bars.vfull[g % C::VST], (g / C::VST) & 1);
        if (ok && j >= 1) ok = tc::mbar_wait(&bars.pv[(g - 1) & 1], ((g - 1) >> 1) & 1);    // V' tile free
        if (!__all_sync(0xffffffffu, ok)) return false;
        tc::fence_after_sync();
        const unsigned char *st = smem + C::VSTG + (g % C::VST) * C::VSTAGE;
        for (int r = dt; r < 2 * NBV * BN; r += 128) {
          const int b = r / (2 * BN), key = (r >> 1) % BN, hw = r & 1;
          expand_half<T>(st + C::V_QS + (key * NBV + b) * QSB, st + C::V_SG + (key * NBV + b) * SGB, tab_v,
                         vt + b * C::TBLK + (key >> 3) * 2048 + (key & 7) * 16, hw);
        }
        tc::fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.dqv);
        if (warp == DQ0 && lane == 0 && j + C::VST < n_tiles) {
          if (tc::mbar_wait(&bars.dqv, g & 1)) issue_v(j + C::VST);
          else s_fail = 1;
        }
        return true;
      };
      bool ok = n_tiles == 0 || k_phase(0);
      for (int j = 0; j < n_tiles && ok; ++j) {
        if (j + 1 < n_tiles) ok = k_phase(j + 1);
        if (ok) ok = v_phase(j);
      }
      if (!ok) s_fail = 1;
    } else {
      // ===================== softmax: one query row, half the keys per thread =====================
      const int bar_id = 1 + (warp & 3);                     // named barrier of the warp pair
      // swap a value (per row) and a warp-uniform flag with the partner warp; both
      // warps of a pair make the same sequence of calls, so a failed wait ends both
      // loops at the same point and no named barrier is left waiting
      auto exchange = [&](float v, bool f, float &pv, bool &pflag) {
        const int p = xc & 1;
        ++xc;
        xv[p][half][row] = v;
        if (lane == 0) xf[p][half][warp & 3] = f ? 1 : 0;
        tc::named_sync(bar_id, 64);
        pv = xv[p][half ^ 1][row];
        pflag = xf[p][half ^ 1][warp & 3] != 0;
      };
      bool ok = true;
      for (int j = 0; j < n_tiles; ++j) {
        const int g = g0 + j;
        bool okw = tc::mbar_wait(&bars.sf[g & 1], (g >> 1) & 1);
        if (okw) okw = tc::mbar_wait(&bars.nrmf[g & 1], (g >> 1) & 1);
        okw = __all_sync(0xffffffffu, okw);
        tc::fence_after_sync();
        const uint32_t sbuf = tmem + lane_off + C::SP0 + (g & 1) * C::SPW;
        const float *nr = nrm + (g & 1) * 4 * BN + half * HB;
        const int64_t key0 = static_cast<int64_t>(t_lo + j) * BN + half * HB;
        const int nvis = row_ok ? static_cast<int>(i64max(0, i64min(HB, i64min(row_end, kv_hi) - key0))) : 0;
        float s[HB];
        float mt = -INFINITY;
        if (okw) {
          uint32_t r0[NBK * HB];                               // this thread's S columns, one wait
#pragma unroll
          for (int b = 0; b < NBK; ++b)
#pragma unroll
            for (int c0 = 0; c0 < HB; c0 += 32) tc::tmem_ld32(sbuf + b * BN + half * HB + c0, r0 + b * HB + c0);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i4 = 0; i4 < HB; i4 += 4) {
            const float4 k0 = *reinterpret_cast<const float4 *>(nr + i4);
            const float4 k1 = *reinterpret_cast<const float4 *>(nr + BN + i4);
            const float n0[4] = {k0.x, k0.y, k0.z, k0.w}, n1[4] = {k1.x, k1.y, k1.z, k1.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int i = i4 + e;
              float x = n0[e] * __uint_as_float(r0[i]);
              if (NBK > 1) x = fmaf(n1[e], __uint_as_float(r0[(NBK > 1 ? HB : 0) + i]), x);
              s[i] = (i < nvis) ? x : -INFINITY;
              mt = fmaxf(mt, s[i]);
            }
          }
        }
        // row maximum over both halves of the tile
        float pmt;
        bool pok;
        exchange(mt, okw, pmt, pok);
        if (!(okw && pok)) { ok = false; break; }
        mt = fmaxf(mt, pmt);
        const bool raise = mt > m_used + kLazyRescale || (m_used == -INFINITY && mt > -INFINITY);
        const float fct = (raise && m_used != -INFINITY) ? exp2f(m_used - mt) : 1.f;
        if (raise) m_used = mt;
        if (__any_sync(0xffffffffu, fct != 1.f)) {           // the same decision in both warps of the pair
          // O must be stable: wait for the PV mma of the previous tile; each half
          // rescales its half of the O columns
          bool okp = (j == 0) || tc::mbar_wait(&bars.pv[(g - 1) & 1], ((g - 1) >> 1) & 1);
          okp = __all_sync(0xffffffffu, okp);
          float unused;
          bool pokp;
          exchange(0.f, okp, unused, pokp);
          if (!(okp && pokp)) { ok = false; break; }
          tc::fence_after_sync();
#pragma unroll
          for (int c = half * (DVP / 2); c < (half + 1) * (DVP / 2); c += 32) {
            uint32_t r[32];
            tc::tmem_ld32(tmem + lane_off + c, r);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * fct);
            tc::tmem_st32(tmem + lane_off + c, r);
          }
        }
        l_sum *= fct;
        // m_used is finite once any key was visible; a row with no visible key so
        // far keeps -inf and every weight 0
        const float msub = m_used == -INFINITY ? 0.f : m_used;
        float psum = 0.f;
#pragma unroll
        for (int i = 0; i < HB; ++i) {
          s[i] = tc::ex2(s[i] - msub);                       // -inf -> 0
          psum += s[i];
        }
        l_sum += psum;
        // P'_(b, hi/lo) into tensor memory over S_j: row = lane, fp16 pairs of keys;
        // this half's keys are columns half * HB/2 .. of each (b, part) region
#pragma unroll
        for (int b = 0; b < NBV; ++b)
#pragma unroll
          for (int c16 = 0; c16 < HB / 2; c16 += 16) {        // 16 columns (32 keys) at a time
            uint32_t ph[16], pl[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int k0 = 2 * (c16 + i);
              const float2 vv = *reinterpret_cast<const float2 *>(nr + (2 + b) * BN + k0);
              const float x0 = s[k0] * vv.x;
              const float x1 = s[k0 + 1] * vv.y;
              const __half2 h = __floats2half2_rn(x0, x1);
              const float2 hf = __half22float2(h);
              const __half2 l = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
              ph[i] = *reinterpret_cast<const uint32_t *>(&h);
              pl[i] = *reinterpret_cast<const uint32_t *>(&l);
            }
            tmem_st<16>(sbuf + (2 * b) * (BN / 2) + half * (HB / 2) + c16, ph);
            tmem_st<16>(sbuf + (2 * b + 1) * (BN / 2) + half * (HB / 2) + c16, pl);
          }
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.pf[g & 1]);
      }
      // the last PV must be complete before O is read
      if (ok && n_tiles > 0) {
        const int g = g0 + n_tiles - 1;
        ok = tc::mbar_wait(&bars.pv[g & 1], (g >> 1) & 1);
        ok = __all_sync(0xffffffffu, ok);
        tc::fence_after_sync();
      }
      if (!ok) s_fail = 1;
    }

    // ===================== epilogue of the item =====================
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    // row sums of the two halves
    if (warp < NSM) xv[0][half][row] = l_sum;
    __syncthreads();
    const float l_row = (warp < NSM) ? xv[0][0][row] + xv[0][1][row] : 0.f;
    const bool failed = s_fail != 0;
    if (failed && tid == 0) set_status(a.status, TQ_ERR_TIMEOUT);

    float *stg = reinterpret_cast<float *>(smem + C::Q) + (warp & 7) * 32 * 128;   // [32][128] per softmax warp
    if (n_split == 1) {
      // half b stages V block b of its row (divided by l and sqrt(128)), then its
      // warp rotates the 32 rows back and stores them
      if (warp < NSM && half < NBV && !failed) {
        const float inv = (l_row > 0.f ? 1.f / l_row : 0.f) * kInvSqrtQK;
        const int b = half;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t r[32];
          tc::tmem_ld32(tmem + lane_off + b * 128 + 32 * c, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4 *>(stg + lane * 128 + 4 * ((8 * c + i / 4) ^ (lane & 7))) =
                n_tiles > 0 ? make_float4(__uint_as_float(r[i]) * inv, __uint_as_float(r[i + 1]) * inv,
                                          __uint_as_float(r[i + 2]) * inv, __uint_as_float(r[i + 3]) * inv)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncwarp();
        rotate_store_rows<true>(stg, 128, a, 32 * (warp & 3), q0, hk, b, lane);
      }
    } else {
      // split key range: store (m, l, O) of every row; a second kernel merges the splits
      // of every query tile once this launch is done (tq_prefill_merge.cu)
      const size_t tile_id = static_cast<size_t>(qt) * a.n_kv_heads + hk;
      const size_t stride = 4 + DVP;             // m, l, 2 pad floats: O rows stay 16-byte aligned
      float *part = a.part + (tile_id * n_split + split) * BM * stride;
      if (warp < NSM) {
        float *pr = part + static_cast<size_t>(row) * stride;
        const bool has = !failed && n_tiles > 0;
        if (half == 0) {
          pr[0] = has ? m_used : -INFINITY;
          pr[1] = has ? l_row : 0.f;
        }
#pragma unroll 1
        for (int c = half * (DVP / 2); c < (half + 1) * (DVP / 2); c += 32) {
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
    }
    g0 += n_tiles;
    tc::fence_before_sync();
    __syncthreads();                             // shared memory and tensor memory free for the next item
    tc::fence_after_sync();
  }

  // the last CTA out resets the work counters for the next launch
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&a.sched[1], 1) == static_cast<int>(gridDim.x) - 1) {
      a.sched[0] = 0;
      a.sched[1] = 0;
      __threadfence();
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc<C::TMEM_COLS>(tmem);
}

template <int T, int NBK, int NBV>
cudaError_t launch_one(const PrefillArgs &a, cudaStream_t s) {
  using C = Cfg<T, NBK, NBV>;
  static_assert(C::TOTAL + 4 * 2 * 2 * BM + 512 <= 227 * 1024, "shared memory (dynamic + static)");
  static_assert(C::COLS_NEEDED <= 512, "tensor memory");
  static_assert(C::BN % 64 == 0 && C::HB % 32 == 0, "key tile");
  cudaError_t e = set_dynamic_smem(reinterpret_cast<const void *>(prefill_kernel<T, NBK, NBV>), (int)C::TOTAL);
  if (e != cudaSuccess) return e;
  // persistent: at most one CTA per SM (each CTA holds most of an SM's shared memory)
  const int grid = min(a.n_items, sm_count());
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

// Single-query decode on the tensor cores with register dequantisation.
//
// Why not the page's LUT ([TQ#36] "Q x centroid LUT") on GB300: with a GQA
// group of 4 every K element costs 4 shared-memory table reads, i.e. ~16 B of
// shared-memory traffic per 0.39 B of HBM traffic, and the SMs' shared-memory
// bandwidth is only ~5x HBM -- the LUT kernel is bound by shared memory at
// several times the HBM time.  Here the packed codes go from HBM to shared
// memory once (cp.async.bulk into a per-warp mbarrier ring; each warp streams
// its own contiguous key range, so the main loop has no CTA barrier) and each
// thread turns them
// into fp16 mma.sync operand fragments with byte permutes: a code nibble is the
// prmt selector into a 4-register table holding the low / high bytes of the
// binary16 centroid values, so a centroid costs ~1.5 integer ops and feeds all
// query heads of the group at once.
//
//   scores  S^T[key][n] = K'[key][d] . B[d][n]      m16n8k16, A = K' (16 keys),
//           B = [q'_hi(heads) | q'_lo(heads) | 0]    n = 8 columns
//   values  O'^T[d][n] += V'^T[d][key] . P'^T[key][n]   A = V' (16 rotated dims),
//           P' = p * |v_key| split into fp16 hi + lo columns
// The spare columns of the n = 8 tile carry the low halves of q' and P', so the
// fp16 operands reach fp32 accuracy at no extra tensor-core cost; centroids are
// binary16-exact, so K' and V' are exact.
//
// Layout of the d index inside a block (the contraction index can be permuted
// freely as long as both operands agree):
//   K side: thread column c = lane % 4 owns rotated dims 32c .. 32c+31 (qs words
//           2c, 2c+1); k-step kk uses dims 32c + 4kk + {0,1} (k = 2c, 2c+1) and
//           32c + 4kk + {2,3} (k = 2c+8, 2c+9).
//   V side: thread row g = lane / 4 owns dims 16g .. 16g+15 (one qs word);
//           m-tile mt, row g   <-> dim 16g + 2mt,  row g+8 <-> dim 16g + 2mt + 1.
#pragma once

#include "tq_decode_common.cuh"
#include "tq_quant.cuh"
#include "tq_tc.cuh"

namespace tq {
namespace mmadec {

constexpr int WK = 32;               // keys per warp per iteration (two mma key groups)

__device__ __forceinline__ void mma16816(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// K side: the 32 rotated dims 32c .. 32c+31 of one key block -> h[p] = half2 of
// dims (32c + 2p, 32c + 2p + 1), p = 0..15.
template <int T>
__device__ __forceinline__ void dq_chunk32(const uint8_t *qs_row, const uint8_t *sg_row, int c, const Tab &t,
                                           uint32_t h[16]) {
  if (T == 4) {
    const uint4 w = *reinterpret_cast<const uint4 *>(qs_row + 16 * c);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      dq4<4>(ws[i], t, h[4 * i + 0], h[4 * i + 1]);
      dq4<4>(ws[i] >> 16, t, h[4 * i + 2], h[4 * i + 3]);
    }
  } else {
    const uint2 w = *reinterpret_cast<const uint2 *>(qs_row + 8 * c);
    const uint32_t sg = (T == 3) ? *reinterpret_cast<const uint32_t *>(sg_row + 4 * c) : 0u;
    const uint32_t ws[2] = {w.x, w.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      uint32_t s0, s1;
      sel_words<T>(ws[i], sg, i == 1, s0, s1);
      dq4<T>(s0, t, h[8 * i + 0], h[8 * i + 1]);
      dq4<T>(s0 >> 16, t, h[8 * i + 2], h[8 * i + 3]);
      dq4<T>(s1, t, h[8 * i + 4], h[8 * i + 5]);
      dq4<T>(s1 >> 16, t, h[8 * i + 6], h[8 * i + 7]);
    }
  }
}

// V side: 16 dims (16g .. 16g+15) of two keys (k0, k1) -> a[el/2... ] pairs:
// out[e] = half2(V[k0][16g + e], V[k1][16g + e]), e = 0..15.
// `sel*` are the selector words of each key (elements 0..7 and 8..15).
template <int T>
__device__ __forceinline__ void dq_pair16(uint32_t a0, uint32_t a1, uint32_t b0, uint32_t b1, const Tab &t,
                                          uint32_t out[16]) {
  // a0/a1: key k0 elements 0..7 / 8..15; b0/b1: key k1
  const uint32_t sa[2] = {a0, a1}, sb[2] = {b0, b1};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    // even elements of both keys interleaved, then odd elements
    const uint32_t ev = (sa[i] & 0x0F0F0F0Fu) | ((sb[i] & 0x0F0F0F0Fu) << 4);
    const uint32_t od = ((sa[i] >> 4) & 0x0F0F0F0Fu) | (sb[i] & 0xF0F0F0F0u);
    // ev nibbles: (k0 e0, k1 e0, k0 e2, k1 e2 | k0 e4, k1 e4, k0 e6, k1 e6)
    dq4<T>(ev, t, out[8 * i + 0], out[8 * i + 2]);
    dq4<T>(ev >> 16, t, out[8 * i + 4], out[8 * i + 6]);
    dq4<T>(od, t, out[8 * i + 1], out[8 * i + 3]);
    dq4<T>(od >> 16, t, out[8 * i + 5], out[8 * i + 7]);
  }
}

// selector words (elements 0..7, 8..15 of the 16-dim group g) of one V key block.
// turbo3: the group's sign bits sit in signs word g/2 at the positions sel_words
// expects for an even (odd) qs word rotated left by rl0 = 0 (2) and right by
// rr1 = 1 (31) -- rotations rather than shifts, so that g's parity is two
// per-thread constants instead of selects (the wrapped bits fall outside the
// 0x44444444 mask).
template <int T>
__device__ __forceinline__ void v_sel(const uint8_t *qs_row, const uint8_t *sg_row, int g, int rl0, int rr1,
                                      uint32_t &s0, uint32_t &s1) {
  if (T == 4) {
    const uint2 w = *reinterpret_cast<const uint2 *>(qs_row + 8 * g);
    s0 = w.x;
    s1 = w.y;
  } else {
    const uint32_t w = reinterpret_cast<const uint32_t *>(qs_row)[g];
    s0 = w & 0x33333333u;
    s1 = (w >> 2) & 0x33333333u;
    if (T == 3) {
      const uint32_t sg = reinterpret_cast<const uint32_t *>(sg_row)[g >> 1];
      s0 |= __funnelshift_l(sg, sg, rl0) & 0x44444444u;
      s1 |= __funnelshift_r(sg, sg, rr1) & 0x44444444u;
    }
  }
}

// Per-warp staging ring: every warp streams its own contiguous key range
// (32 keys per iteration) through STAGES bulk-copy buffers, so the main loop
// has no CTA-wide barrier at all.
template <int T, int NBK, int NBV>
struct WarpStage {
  static constexpr uint32_t QSB = TypeTraits<T>::QSB, SGB = TypeTraits<T>::SGB;
  static constexpr uint32_t KEYB = (NBK + NBV) * (QSB + SGB + 2);      // packed bytes per key (K and V)
  static constexpr uint32_t BYTES0 = (WK * KEYB + 127) / 128 * 128;
  // warps per CTA (one CTA per SM): 16 when three 32-key stages of every warp fit, else 8
  static constexpr int NW = (16 * 3 * BYTES0 <= 200 * 1024) ? 16 : 8;
  static constexpr int NT = NW * 32;
  // P tiles, rotated q and the B columns (sized for a group of 4) beside the rings
  // P' tile per warp and V block: 8 columns x PSTR words (16 key pairs, padded so
  // that neither the pair stores nor the fragment loads conflict on a bank)
  static constexpr int PSTR = 20;
  static constexpr uint32_t PTW = NBV * 8 * PSTR * 4;                 // bytes per warp
  static constexpr uint32_t EXTRA = NW * PTW + 4 * 128 * NBK * 4 + 8 * 128 * NBK * 2;
  static constexpr uint32_t BUDGET = 222 * 1024;
  // A stage holds SUB groups of 32 keys (fewer, larger bulk copies: the copy count,
  // not the bytes, limits how fast the copies are issued).  Two 64-key stages per
  // warp where they fit, else 32-key stages, as many as fit (up to 4).
  static constexpr uint32_t bytes_of(int keys) { return (keys * KEYB + 127) / 128 * 128; }
  static constexpr int SUB = (NW * 2 * bytes_of(2 * WK) + EXTRA <= BUDGET) ? 2 : 1;
  static constexpr int SK = SUB * WK;                                   // keys per stage
  static constexpr uint32_t KQS = 0;
  static constexpr uint32_t KSG = KQS + SK * NBK * QSB;
  static constexpr uint32_t KN = KSG + SK * NBK * SGB;
  static constexpr uint32_t VQS = KN + SK * NBK * 2;
  static constexpr uint32_t VSG = VQS + SK * NBV * QSB;
  static constexpr uint32_t VN = VSG + SK * NBV * SGB;
  static constexpr uint32_t BYTES = bytes_of(SK);
  static constexpr int STAGES = (SUB == 2) ? 2
                                : (NW * 4 * BYTES + EXTRA <= BUDGET) ? 4
                                : (NW * 3 * BYTES + EXTRA <= BUDGET) ? 3 : 2;
  static constexpr uint32_t RING = STAGES * BYTES;                    // per warp
  static constexpr uint32_t PT = NW * RING;                           // P' tiles [NW][NBV][8][PSTR] u32
  static constexpr uint32_t QR = PT + NW * PTW;                       // rotated q (floats)
};

template <int T, int G, int NBK, int NBV>
struct WarpStageQ {
  static constexpr uint32_t QC = WarpStage<T, NBK, NBV>::QR + G * 128 * NBK * 4;   // B columns fp16 [8][128 NBK]
  static constexpr uint32_t TOTAL = QC + 8 * 128 * NBK * 2;
};

template <int T, int G, int NBK, int NBV>
__host__ __device__ constexpr uint32_t smem_bytes() {
  return WarpStageQ<T, G, NBK, NBV>::TOTAL;
}

__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Split merge inside a cluster (one cluster of n_splits CTAs per KV head): each
// CTA's partial m[G], l[G], o'[G][128 NBV] sits at `cpart` in its own shared
// memory.  Output block (head g, V block b) is merged by CTA rank (g NBV + b)
// mod n_splits: thread t reads the n_splits partials of dim t over distributed
// shared memory (one round trip), forms o' = sum_s o'_s 2^(m_s - M) / L,
// then a warp rotates the block back (o = S H o' / sqrt(128)) and stores it.
// `scratch` holds 128 floats of this CTA's shared memory.  The second cluster
// barrier keeps every CTA's partial alive until all reads are done.
template <int G, int NBV, int NT>
__device__ void cluster_merge(const DecodeArgs &a, int hk, const float *cpart, float *scratch) {
  constexpr int DVP = 128 * NBV, MAXS = 16;
  const uint32_t rank = tc::cluster_rank();
  const int ns = a.n_splits;                          // == cluster size, <= MAXS
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t base = tc::smem_u32(cpart);
  tc::cluster_sync();
  for (int wb = static_cast<int>(rank); wb < G * NBV; wb += ns) {
    const int g = wb / NBV, b = wb % NBV;
    const int t = threadIdx.x;
    if (t < 128) {
      float m[MAXS], l[MAXS], o[MAXS];
#pragma unroll
      for (int s = 0; s < MAXS; ++s) {
        m[s] = -INFINITY;
        l[s] = 0.f;
        o[s] = 0.f;
        if (s < ns) {
          const uint32_t r = tc::dsmem_addr(base, static_cast<uint32_t>(s));
          m[s] = tc::dsmem_ld(r + 4u * g);
          l[s] = tc::dsmem_ld(r + 4u * (G + g));
          o[s] = tc::dsmem_ld(r + 4u * (2 * G + g * DVP + b * 128 + t));
        }
      }
      float M = -INFINITY;
#pragma unroll
      for (int s = 0; s < MAXS; ++s) M = fmaxf(M, m[s]);
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int s = 0; s < MAXS; ++s) {
        const float w = (m[s] == -INFINITY) ? 0.f : fast_exp2(m[s] - M);
        L = fmaf(w, l[s], L);
        O = fmaf(w, o[s], O);
      }
      scratch[t] = (L > 0.f) ? O / L : 0.f;
    }
    __syncthreads();
    if (warp == 0) {
      float v[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) v[r] = scratch[4 * lane + r];
      wht128_warp(v, lane);
#pragma unroll
      for (int r = 0; r < 4; ++r) v[r] *= kInvSqrtQK;
      apply_signs(v, a.cbv, lane);
      float *out = a.out + static_cast<size_t>(hk * G + g) * a.dv;
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const int d = b * 128 + 4 * lane + r;
        if (d < a.dv) out[d] = v[r];
      }
    }
    __syncthreads();
  }
  tc::cluster_sync();
}

template <int T, int G, int NBK, int NBV, bool SV>
__global__ void __launch_bounds__(WarpStage<T, NBK, NBV>::NT, 1) decode_mma_kernel(const DecodeArgs a) {
  static_assert(G == 1 || G == 2 || G == 4, "GQA group must be 1, 2 or 4");
  using WS = WarpStage<T, NBK, NBV>;
  constexpr int NW = WS::NW, NT = WS::NT;
  using WQ = WarpStageQ<T, G, NBK, NBV>;
  constexpr int QSB = TypeTraits<T>::QSB, SGB = TypeTraits<T>::SGB;
  constexpr int STAGES = WS::STAGES;
  constexpr int DVP = 128 * NBV;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ __align__(8) uint64_t full[NW][STAGES];
  __shared__ __align__(8) uint64_t first_b[NW];      // group 1 of stage 0 (64-key stages)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  // launch head hk serves query heads hk G .. hk G + G - 1 of KV head hk_cache
  // (kv_rep launch heads per KV head when the GQA group is larger than G); in a
  // batched decode sequence hk / hkv, whose cells start at seq_cell0.  q, out and
  // the split bookkeeping are indexed by the launch head.
  const int hk = blockIdx.y, split = blockIdx.x;
  const bool batched = a.n_seq > 0;
  const int hk_cache = (batched ? hk % a.hkv : hk) / a.kv_rep;
  const int64_t cell0 = batched ? a.seq_cell0[hk / a.hkv] : 0;
  const int64_t len = batched ? a.seq_len[hk / a.hkv] : a.kv_len;
  const int64_t t0 = static_cast<int64_t>(split) * a.chunk;
  const int64_t t1 = min(len, t0 + a.chunk);
  // this warp's key range [w0, w1): the CTA's groups of WK keys dealt out evenly
  // (warps differ by at most one group).  The warps with an extra group are the
  // first ones, so that they fall on different SM sub-partitions (warp w runs on
  // sub-partition w % 4): the main loop is bound by each sub-partition's issue
  // and integer-pipe throughput, so the CTA takes as long as its busiest one.
  const int n_grp = (t1 > t0) ? static_cast<int>((t1 - t0 + WK - 1) / WK) : 0;
  const int gbase = n_grp / NW, gextra = n_grp % NW;
  const int gb = warp * gbase + min(warp, gextra), ge = gb + gbase + (warp < gextra ? 1 : 0);
  const int64_t w0 = t0 + static_cast<int64_t>(gb) * WK;
  const int64_t w1 = min(t1, t0 + static_cast<int64_t>(ge) * WK);
  const int n_it = ge - gb;

  unsigned char *ring = smem + warp * WS::RING;
  uint32_t *pw32 = reinterpret_cast<uint32_t *>(smem + WS::PT + warp * WS::PTW);   // P' pairs [NBV][8][PSTR]
  float *qrot = reinterpret_cast<float *>(smem + WS::QR);

  const size_t cbase = static_cast<size_t>(hk_cache) * a.n_cells + cell0;     // first cell of this head's keys
  const uint8_t *kqs = a.kqs + cbase * NBK * QSB;
  const uint8_t *ksg = SGB ? a.ksg + cbase * NBK * SGB : nullptr;
  const uint16_t *kn = a.kn + cbase * NBK;
  const uint8_t *vqs = a.vqs + cbase * NBV * QSB;
  const uint8_t *vsg = SGB ? a.vsg + cbase * NBV * SGB : nullptr;
  const uint16_t *vn = a.vn + cbase * NBV;

  // lane 0 of the warp: bring groups [jg, jg + ng) of stage si (groups SUB si .. of
  // this warp, keys w0 + SK si + 32 jg ..) into ring slot si % STAGES, completing
  // on `bar`; a last stage may hold fewer groups
  const int n_st = (n_it + WS::SUB - 1) / WS::SUB;
  auto issue_part = [&](int si, int jg, int ng, uint64_t *bar) {
    const int64_t key0 = w0 + static_cast<int64_t>(si) * WS::SK + jg * WK;   // multiple of 32
    const int nk = ng * WK;                                                   // key0 + nk <= n_cells
    unsigned char *st = ring + (si % STAGES) * WS::BYTES;
    const int r0 = jg * WK;
    tc::mbar_expect_tx(bar, nk * WS::KEYB);
    tc::bulk_g2s(st + WS::KQS + r0 * NBK * QSB, kqs + key0 * NBK * QSB, nk * NBK * QSB, bar);
    if (SGB) tc::bulk_g2s(st + WS::KSG + r0 * NBK * SGB, ksg + key0 * NBK * SGB, nk * NBK * SGB, bar);
    tc::bulk_g2s(st + WS::KN + r0 * NBK * 2, kn + key0 * NBK, nk * NBK * 2, bar);
    tc::bulk_g2s(st + WS::VQS + r0 * NBV * QSB, vqs + key0 * NBV * QSB, nk * NBV * QSB, bar);
    if (SGB) tc::bulk_g2s(st + WS::VSG + r0 * NBV * SGB, vsg + key0 * NBV * SGB, nk * NBV * SGB, bar);
    tc::bulk_g2s(st + WS::VN + r0 * NBV * 2, vn + key0 * NBV, nk * NBV * 2, bar);
  };
  auto issue = [&](int si) {
    issue_part(si, 0, min(WS::SUB, n_it - si * WS::SUB), &full[warp][si % STAGES]);
  };

  // The query loads go out before any bulk copy: issued after them they would
  // queue behind the key/value traffic.  One query block per warp (NW >= G * NBK).
  static_assert(NW >= G * NBK, "one query block per warp");
  // Programmatic dependent launch: the next launch on the stream may be
  // scheduled onto SMs that this grid's CTAs leave (it is launched with the
  // programmatic-serialisation attribute), and every CTA waits for the previous
  // grid to complete, its writes visible, before its first global access, so
  // only the launch and the set-up above overlap the previous launch's merge.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float qv[4] = {0.f, 0.f, 0.f, 0.f};
  if (warp < G * NBK) load_query_block(a, hk, warp, lane, qv);

  // ---- append ([TQ#36] SET_ROWS of the new token, fused): the CTA whose key
  // range holds the cell (split 0 when the cell lies beyond kv_len) quantises the
  // token's K and V row blocks of KV head hk_cache with warp QWARP (4 lanes per block: K
  // blocks first, then V), writes them to the cache and keeps a copy in `patch`;
  // the warp that attends the cell copies it over its staged bytes once
  // `patch_bar` has completed.  Warp QWARP quantises after the prologue, while its
  // first tiles are in flight, and no other warp waits for it there: the last
  // warp holds the fewest key groups, on the sub-partition with the fewest.
  constexpr int PQ = 0, PS = PQ + (NBK + NBV) * QSB, PN = PS + (NBK + NBV) * (SGB ? SGB : 4);
  __shared__ __align__(16) uint8_t patch[PN + 2 * (NBK + NBV)];
  __shared__ __align__(8) uint64_t patch_bar;
  constexpr int QWARP = NW - 1;
  // A CTA barrier waits for every load issued before it: the cell id and the
  // epoch go out with the query loads, then each warp's first bulk copy, then
  // the first barrier (one lane per CTA reads the cell id: the same 8 bytes read
  // by every warp of the grid queue up at one L2 line for about a microsecond).
  // The CTA that owns the cell stages the token's rows in `rowbuf` with cp.async
  // after the first barrier (the later barriers do not wait for those copies),
  // or, for rows that are not 16-byte aligned per head, loads them into registers.
  const bool append = a.cell_id != nullptr;
  __shared__ int64_t s_cell;
  __shared__ uint32_t s_epoch;
  __shared__ __align__(16) unsigned char rowbuf[(NBK + NBV) * QK * 4];
  uint32_t e_ld = 0;
  int64_t c_ld = -1;
  if (warp == QWARP && lane == 0) {
    e_ld = load_epoch(a, hk);
    if (append) c_ld = __ldg(a.cell_id);
  }
  // Each warp's barriers and ring are its own, so lane 0 sets them up and sends
  // the first copy before the first CTA barrier.  The first group alone goes
  // first: every CTA's first 32 keys are in the first wave of HBM traffic, so
  // the compute starts as early as it can.  With 64-key stages the second group
  // follows after the prologue on its own barrier; the other stages once the
  // first has landed.
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) tc::mbar_init(&full[warp][s], 1);
    tc::mbar_init(&first_b[warp], 1);
    if (warp == QWARP) tc::mbar_init(&patch_bar, 1);
    tc::mbar_init_fence();
    tc::fence_async_smem();
    if (n_st > 0) {
      if (WS::SUB == 2) issue_part(0, 0, 1, &full[warp][0]);
      else issue(0);
    }
  }
  if (warp == QWARP && lane == 0) {
    s_cell = c_ld;
    s_epoch = e_ld;
  }
  __syncthreads();
  const int64_t cell = s_cell;
  const bool cell_ok = cell >= 0 && cell < a.n_cells;
  const bool owner = append && cell_ok && ((cell >= t0 && cell < t1) || (cell >= a.kv_len && split == 0));
  if (append && !cell_ok && split == 0 && tid == 0) set_status(a.status, TQ_ERR_DEVICE_CHECK);
  const int gq = lane >> 2, l4 = lane & 3;                  // block of the quantising warp's lane group
  const bool qblk = gq < NBK + NBV;
  float nv[8][4];
  if (owner && warp == QWARP) {
    if (a.row_async) {
      const int es = (a.src_type == TQ_F32) ? 4 : 2;
#pragma unroll
      for (int blk = 0; blk < NBK + NBV; ++blk) {
        const bool isk = blk < NBK;
        const int b = isk ? blk : blk - NBK;
        const int dim = isk ? a.dk : a.dv;
        const int nbytes = max(0, min(QK, dim - b * QK)) * es;
        const unsigned char *s0 =
            static_cast<const unsigned char *>(isk ? a.k_src : a.v_src) + (static_cast<int64_t>(hk_cache) * dim + b * QK) * es;
        for (int off = lane * 16; off < QK * es; off += 32 * 16) {
          const int n = min(max(nbytes - off, 0), 16);
          tc::cp_async16(rowbuf + blk * QK * 4 + off, n > 0 ? s0 + off : s0, n);
        }
      }
      tc::cp_async_commit();
    } else {
      const bool isk = gq < NBK;
      const int b = isk ? gq : gq - NBK;
      const int dim = isk ? a.dk : a.dv;
      const void *src = isk ? a.k_src : a.v_src;
      const int64_t base = static_cast<int64_t>(hk_cache) * dim + b * QK;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int e0 = 4 * l4 + 16 * i;
        if (qblk) quant_load4_rt(a.src_type, src, base + e0, dim - b * QK - e0, nv[i]);
        else nv[i][0] = nv[i][1] = nv[i][2] = nv[i][3] = 0.f;
      }
    }
  }

  // rotated queries (scale and log2(e) folded in) while the first tiles land, then
  // the score mma's B columns as binary16: n = 2h q'_hi, n = 2h + 1 q'_lo of head h,
  // zero for h >= G
  if (warp < G * NBK) rotate_query_block(a, warp, lane, qv, qrot);
  for (int i = lane; i < NBV * 8 * WS::PSTR; i += 32) pw32[i] = 0;
  __shared__ int s_mref[4];                 // largest score published per query head (sparse V)
  if (SV && tid < 4) s_mref[tid] = ordered_int(-INFINITY);
  __syncthreads();
  uint16_t *qcol = reinterpret_cast<uint16_t *>(smem + WQ::QC);              // [8][128*NBK]
  for (int i = tid; i < 8 * 128 * NBK; i += NT) {
    const int n = i / (128 * NBK), d = i % (128 * NBK);
    float x = 0.f;
    if (n < 2 * G) {                      // column 2h: q'_hi of head h, 2h + 1: q'_lo
      const float q = qrot[(n >> 1) * 128 * NBK + d];
      const __half hi = __float2half_rn(q);
      x = (n & 1) ? (q - __half2float(hi)) : __half2float(hi);
    }
    qcol[i] = __half_as_ushort(__float2half_rn(x));
  }
  __syncthreads();
  if (WS::SUB == 2 && lane == 0 && n_it > 1) issue_part(0, 1, 1, &first_b[warp]);
  if (owner && warp == QWARP) {
    const bool isk = gq < NBK;
    const int b = isk ? gq : gq - NBK, nb = isk ? NBK : NBV;
    if (a.row_async) {
      tc::cp_async_wait_all();
      __syncwarp();
      const int es = (a.src_type == TQ_F32) ? 4 : 2;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (qblk) quant_unpack4_rt(a.src_type, rowbuf + gq * QK * 4 + (4 * l4 + 16 * i) * es, nv[i]);
        else nv[i][0] = nv[i][1] = nv[i][2] = nv[i][3] = 0.f;
      }
    }
    PackedShare<T> pb;
    quantise_block4<T>(isk ? a.cbk : a.cbv, l4, nv, pb);
    if (qblk) {
      // every launch head of the KV head quantises the row for its own copy; the
      // first one writes it to the cache
      if (hk % a.kv_rep == 0) {
        const int64_t blk = (static_cast<int64_t>(hk_cache) * a.n_cells + cell) * nb + b;
        uint16_t *gn = const_cast<uint16_t *>(isk ? a.kn : a.vn) + blk;
        uint8_t *gqs = const_cast<uint8_t *>(isk ? a.kqs : a.vqs) + blk * QSB;
        uint8_t *gsg = SGB ? const_cast<uint8_t *>(isk ? a.ksg : a.vsg) + blk * SGB : nullptr;
        store_block4<T>(pb, l4, gn, gqs, gsg);
      }
      store_block4<T>(pb, l4, reinterpret_cast<uint16_t *>(patch + PN) + gq, patch + PQ + gq * QSB,
                      SGB ? patch + PS + gq * SGB : nullptr);
    }
    __syncwarp();
    if (lane == 0) tc::mbar_arrive(&patch_bar);
  }

  const Tab tab_k{a.tabk[0], a.tabk[1], a.tabk[2], a.tabk[3]};
  const Tab tab_v{a.tabv[0], a.tabv[1], a.tabv[2], a.tabv[3]};

  // B fragments: k-step kk of block b uses dims 32c + 4kk + {0,1} (b0) and + {2,3} (b1)
  uint32_t qb[NBK][8][2];
#pragma unroll
  for (int b = 0; b < NBK; ++b)
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint2 v = *reinterpret_cast<const uint2 *>(qcol + g * 128 * NBK + b * QK + 32 * c + 4 * kk);
      qb[b][kk][0] = v.x;
      qb[b][kk][1] = v.y;
    }

  float oacc[NBV][8][4];
#pragma unroll
  for (int b = 0; b < NBV; ++b)
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) oacc[b][mt][i] = 0.f;
  // Thread (g, c) owns query head c (if c < G): its score columns 2c, 2c + 1
  // (hi, lo) and output columns 2c, 2c + 1 are in the thread's own fragments.
  const bool has_head = c < G;
  const int rl0 = (g & 1) ? 2 : 0, rr1 = (g & 1) ? 31 : 1;   // v_sel's sign-word rotations
  float m_run = -INFINITY, l_run = 0.f;
  bool timed_out = false;

  // the group of this warp that holds the appended cell, if any
  const int patch_it = (owner && cell >= w0 && cell < w1) ? static_cast<int>((cell - w0) / WK) : -1;
  for (int it = 0; it < n_it; ++it) {
    const int si = it / WS::SUB, j = it % WS::SUB;             // stage, 32-key group inside it
    if (j == 0 || (WS::SUB == 2 && it == 1)) {
      const bool ok = (it == 1 && WS::SUB == 2) ? tc::mbar_wait_warp(&first_b[warp], 0)
                                                : tc::mbar_wait_warp(&full[warp][si % STAGES], (si / STAGES) & 1);
      if (!ok) { timed_out = true; break; }
      // the other stages only once the first has landed: issued earlier, every
      // CTA's later stages compete with the other CTAs' first stages for HBM
      if (it == 0) {
        if (lane == 0)
          for (int i = 1; i < STAGES && i < n_st; ++i) issue(i);
        __syncwarp();
      }
    }
    const unsigned char *st = ring + (si % STAGES) * WS::BYTES;
    const int64_t key0 = w0 + static_cast<int64_t>(it) * WK;
    if (it == patch_it) {
      // the appended cell is in this group (landed): its freshly quantised bytes
      // replace whatever the bulk copy read
      if (!tc::mbar_wait_warp(&patch_bar, 0)) { timed_out = true; break; }
      const int row = static_cast<int>(cell - key0) + j * WK;                 // row inside the stage
      unsigned char *sw = ring + (si % STAGES) * WS::BYTES;
      constexpr int QW = QSB / 4, SW = SGB / 4;
      for (int i = lane; i < (NBK + NBV) * (QW + SW + 1); i += 32) {
        const int blk = i / (QW + SW + 1), e = i % (QW + SW + 1);
        const bool isk = blk < NBK;
        const int b = isk ? blk : blk - NBK, nb = isk ? NBK : NBV;
        const uint32_t qso = isk ? WS::KQS : WS::VQS, sgo = isk ? WS::KSG : WS::VSG, no = isk ? WS::KN : WS::VN;
        if (e < QW) {
          reinterpret_cast<uint32_t *>(sw + qso + (row * nb + b) * QSB)[e] =
              reinterpret_cast<const uint32_t *>(patch + PQ + blk * QSB)[e];
        } else if (e < QW + SW) {
          reinterpret_cast<uint32_t *>(sw + sgo + (row * nb + b) * SGB)[e - QW] =
              reinterpret_cast<const uint32_t *>(patch + PS + blk * SGB)[e - QW];
        } else {
          reinterpret_cast<uint16_t *>(sw + no)[row * nb + b] = reinterpret_cast<const uint16_t *>(patch + PN)[blk];
        }
      }
      __syncwarp();
    }
    const unsigned char *skq = st + WS::KQS + j * WK * NBK * QSB, *sks = st + WS::KSG + j * WK * NBK * SGB;
    const unsigned char *svq = st + WS::VQS + j * WK * NBV * QSB, *svs = st + WS::VSG + j * WK * NBV * SGB;
    const uint16_t *knr = reinterpret_cast<const uint16_t *>(st + WS::KN) + j * WK * NBK;
    const uint16_t *vnr = reinterpret_cast<const uint16_t *>(st + WS::VN) + j * WK * NBV;

    // keys of this group that are in the warp's range (rows >= rem are masked)
    const int rem = static_cast<int>(min(w1 - key0, static_cast<int64_t>(WK)));

    // ---- scores S^T[key][n] for two groups of 16 keys (rows grp*16 + g, + 8):
    // sc[grp][0] = row grp*16 + g, sc[grp][1] = row grp*16 + g + 8, head c
    float sc[2][2];
#pragma unroll
    for (int grp = 0; grp < 2; ++grp) {
      const int r0 = grp * 16 + g, r1 = r0 + 8;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int b = 0; b < NBK; ++b) {
        uint32_t ka0[16], ka1[16];
        dq_chunk32<T>(skq + (r0 * NBK + b) * QSB, sks + (r0 * NBK + b) * SGB, c, tab_k, ka0);
        dq_chunk32<T>(skq + (r1 * NBK + b) * QSB, sks + (r1 * NBK + b) * SGB, c, tab_k, ka1);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma16816(acc, ka0[2 * kk], ka1[2 * kk], ka0[2 * kk + 1], ka1[2 * kk + 1], qb[b][kk][0], qb[b][kk][1]);
        const float n0 = __half2float(__ushort_as_half(knr[r0 * NBK + b]));
        const float n1 = __half2float(__ushort_as_half(knr[r1 * NBK + b]));
        s0 = fmaf(n0, acc[0] + acc[1], s0);         // hi + lo columns of head c
        s1 = fmaf(n1, acc[2] + acc[3], s1);
      }
      sc[grp][0] = (r0 < rem) ? s0 : -INFINITY;
      sc[grp][1] = (r1 < rem) ? s1 : -INFINITY;
    }

    // ---- online softmax of head c (log2 domain); the reference maximum is raised
    // only when the running maximum grows by more than 2^8 (then O and l rescale)
    bool vkeep[2] = {true, true};
    {
      float tm = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
      tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 4));
      tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 8));
      tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 16));
      // sparse V ([TQ#36] "VEC tuning"): a group of 16 keys whose weights,
      // relative to the largest score known so far, are below the threshold for
      // every query head of the warp adds nothing to O' (its weights still count
      // in l).  The largest known score is this group's or one that a warp of
      // the CTA published (`s_mref`), never above the final maximum, so every
      // key left out is below the threshold relative to the final maximum too.
      if (SV) {
        if (g == 0 && has_head) atomicMax(&s_mref[c], ordered_int(tm));
        const float mref = has_head ? fmaxf(tm, ordered_float(*reinterpret_cast<volatile int *>(&s_mref[c & 3])))
                                    : tm;
        const float cut = mref + a.v_log2_thresh;
#pragma unroll
        for (int grp = 0; grp < 2; ++grp)
          vkeep[grp] = __any_sync(0xffffffffu, has_head && (sc[grp][0] >= cut || sc[grp][1] >= cut));
      }
      if (tm > m_run + 8.f) {
        const float fct = (m_run == -INFINITY) ? 0.f : fast_ex2(m_run - tm);
        l_run *= fct;
#pragma unroll
        for (int b = 0; b < NBV; ++b)
#pragma unroll
          for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int i = 0; i < 4; ++i) oacc[b][mt][i] *= fct;
        m_run = tm;
      }
#pragma unroll
      for (int grp = 0; grp < 2; ++grp)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          sc[grp][r] = fast_ex2(sc[grp][r] - m_run);             // -inf -> 0
          l_run += sc[grp][r];
        }
    }

    // ---- P' = p * |v| (per V block) as binary16 (hi, lo) key pairs: column 2c (hi)
    // and 2c + 1 (lo), pair g of group grp = keys (grp*16 + g, grp*16 + g + 8)
#pragma unroll
    for (int b = 0; b < NBV; ++b) {
#pragma unroll
      for (int grp = 0; grp < 2; ++grp) {
        if (SV && !vkeep[grp]) continue;
        const int r0 = grp * 16 + g, r1 = r0 + 8;
        const float v0 = __half2float(__ushort_as_half(vnr[r0 * NBV + b]));
        const float v1 = __half2float(__ushort_as_half(vnr[r1 * NBV + b]));
        // masked keys have p = 0 and may carry garbage norms: select the zero
        const float x0 = sc[grp][0] > 0.f ? sc[grp][0] * v0 : 0.f;
        const float x1 = sc[grp][1] > 0.f ? sc[grp][1] * v1 : 0.f;
        const __half2 hi = __floats2half2_rn(x0, x1);
        const float2 hf = __half22float2(hi);
        const __half2 lo = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
        if (has_head) {
          pw32[(b * 8 + 2 * c) * WS::PSTR + grp * 8 + g] = *reinterpret_cast<const uint32_t *>(&hi);
          pw32[(b * 8 + 2 * c + 1) * WS::PSTR + grp * 8 + g] = *reinterpret_cast<const uint32_t *>(&lo);
        }
      }
    }
    __syncwarp();

    // ---- O'^T[d][n] += V'^T[d][key] P'^T[key][n], contraction order: k-slots
    // (2c, 2c + 1) <-> keys (c, c + 8), (2c + 8, 2c + 9) <-> keys (c + 4, c + 12)
#pragma unroll
    for (int b = 0; b < NBV; ++b) {
#pragma unroll
      for (int grp = 0; grp < 2; ++grp) {
        if (SV && !vkeep[grp]) continue;
        const uint32_t pb0 = pw32[(b * 8 + g) * WS::PSTR + grp * 8 + c];
        const uint32_t pb1 = pw32[(b * 8 + g) * WS::PSTR + grp * 8 + c + 4];
        const int kr = grp * 16;
        uint32_t s00, s01, s10, s11, s20, s21, s30, s31;
        const uint8_t *vq = svq, *vs = svs;
        v_sel<T>(vq + ((kr + c) * NBV + b) * QSB, vs + ((kr + c) * NBV + b) * SGB, g, rl0, rr1, s00, s01);
        v_sel<T>(vq + ((kr + c + 8) * NBV + b) * QSB, vs + ((kr + c + 8) * NBV + b) * SGB, g, rl0, rr1, s10, s11);
        v_sel<T>(vq + ((kr + c + 4) * NBV + b) * QSB, vs + ((kr + c + 4) * NBV + b) * SGB, g, rl0, rr1, s20, s21);
        v_sel<T>(vq + ((kr + c + 12) * NBV + b) * QSB, vs + ((kr + c + 12) * NBV + b) * SGB, g, rl0, rr1, s30, s31);
        uint32_t lo[16], hi[16];
        dq_pair16<T>(s00, s01, s10, s11, tab_v, lo);     // keys c, c + 8
        dq_pair16<T>(s20, s21, s30, s31, tab_v, hi);     // keys c + 4, c + 12
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
          mma16816(oacc[b][mt], lo[2 * mt], lo[2 * mt + 1], hi[2 * mt], hi[2 * mt + 1], pb0, pb1);
      }
    }
    __syncwarp();
    // the stage is free again after its last group
    if ((j == WS::SUB - 1 || it == n_it - 1) && si + STAGES < n_st) {     // warp-uniform
      if (lane == 0) issue(si + STAGES);
      __syncwarp();
    }
  }

  // ---- per-warp results -> this warp's ring (all its copies have landed), CTA merge
  if (timed_out && lane == 0) set_status(a.status, TQ_ERR_TIMEOUT);
  // m[G], l[G], o[G][WHS]: output dim d of head h at 2G + h WHS + d + (d >> 5), so that
  // the fragment stores below (dims 16g + 2mt of head c) fall on 32 different banks.
  // With the plain layout (h 128 + d) every lane with the same parity of g hit one
  // bank, a 16-way conflict when the warps leave their loops together (1.9 us of a
  // 32K call).  The CTA merge reads 32 consecutive d, which share d >> 5.
  constexpr int WHS = DVP + 36;
  float *wbuf = reinterpret_cast<float *>(ring);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 4);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 8);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 16);
  if (has_head) {
    const int h = c;
    if (g == 0) {
      wbuf[h] = timed_out ? -INFINITY : m_run;
      wbuf[G + h] = timed_out ? 0.f : l_run;
    }
#pragma unroll
    for (int b = 0; b < NBV; ++b)
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        // columns 2c (hi part of P') and 2c + 1 (lo part) of dims 16g + 2mt, + 1
        float *o = wbuf + 2 * G + h * WHS + b * 128 + 16 * g + 2 * mt + 4 * b + (g >> 1);
        o[0] = timed_out ? 0.f : oacc[b][mt][0] + oacc[b][mt][1];
        o[1] = timed_out ? 0.f : oacc[b][mt][2] + oacc[b][mt][3];
      }
  }
  __syncthreads();
  // CTA partial over the warps.  Launched as one cluster per KV head (cluster
  // size == n_splits) the partial stays in this CTA's shared memory for the
  // cluster merge; otherwise it goes to the workspace, tagged, for the
  // cooperative merge (every CTA resident: each output block merged by one CTA
  // of the head) or, for a grid larger than the GPU holds, the last-CTA merge.
  // There the CTA arrives at its head's counter first, so that the atomic's
  // round trip overlaps the CTA merge and the stores.
  const bool in_cluster = tc::cluster_size() == static_cast<uint32_t>(a.n_splits);
  int prev = 0;
  if (!in_cluster && !a.coop && tid == 0) prev = split_arrive(a, hk);
  const uint32_t epoch = s_epoch, tag = split_tag(epoch, hk);
  float *cpart = reinterpret_cast<float *>(smem + WS::PT);      // m[G], l[G], o'[G][DVP]
  for (int i = tid; i < G * DVP; i += NT) {
    const int h = i / DVP, d = i % DVP;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, reinterpret_cast<const float *>(smem + w * WS::RING)[h]);
    float o = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float *wb = reinterpret_cast<const float *>(smem + w * WS::RING);
      const float f = (wb[h] == -INFINITY) ? 0.f : fast_exp2(wb[h] - M);
      o += f * wb[2 * G + h * WHS + d + (d >> 5)];
      l += f * wb[G + h];
    }
    if (in_cluster) {
      cpart[2 * G + i] = o;
      if (d == 0) {
        cpart[h] = M;
        cpart[G + h] = l;
      }
    } else {
      store_partial_o(a, hk * G + h, split, d, o, tag);
      if (d == 0) store_partial_ml(a, hk * G + h, split, M, l, tag);
    }
  }
  if (in_cluster) {
    cluster_merge<G, NBV, NT>(a, hk, cpart, qrot);
  } else if (a.coop) {
    // every CTA is resident: the head's output blocks are merged by its first
    // CTAs, one block each, as soon as all partials are there
    if (tid < 128) coop_merge(a, hk, split, epoch, qrot);
  } else {
    __shared__ int s_last;
    if (tid == 0) s_last = (prev == a.n_splits - 1);
    __syncthreads();
    if (s_last) decode_merge<NT>(a, hk, epoch, reinterpret_cast<float *>(smem));
  }
}

template <int T, int G, int NBK, int NBV, bool SV>
cudaError_t launch_one(const DecodeArgs &a, cudaStream_t s) {
  constexpr uint32_t bytes = smem_bytes<T, G, NBK, NBV>();
  static_assert(bytes <= 227 * 1024, "shared memory");
  // the epilogue: each warp's ring holds its results; the split merge reuses the front
  static_assert(WarpStage<T, NBK, NBV>::RING >= 4 * (2 * G + G * (128 * NBV + 36)), "ring too small for the epilogue");
  static_assert(WarpStage<T, NBK, NBV>::NW * WarpStage<T, NBK, NBV>::RING >= 4 * (G * 128 * NBV + 2 * G * 256),
                "merge region");
  static_assert(WarpStage<T, NBK, NBV>::QR - WarpStage<T, NBK, NBV>::PT >= 4 * (2 * G + G * 128 * NBV),
                "P-tile region too small for the CTA partial");
  auto kern = decode_mma_kernel<T, G, NBK, NBV, SV>;
  cudaError_t e = set_dynamic_smem(reinterpret_cast<const void *>(kern), (int)bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_splits, a.n_kv_heads);
  cfg.blockDim = dim3(WarpStage<T, NBK, NBV>::NT);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  // one cluster per KV head, all resident together; else, when the whole grid
  // fits on the GPU at once, a cooperative launch (every CTA merges a share);
  // else the last-CTA merge
  const int want = min(a.n_kv_heads, max(1, sm_count() / a.n_splits));
  DecodeArgs b = a;
  if (a.n_splits > 1 && cluster_merge_ok(reinterpret_cast<const void *>(kern), a.n_splits,
                                         WarpStage<T, NBK, NBV>::NT, bytes, want)) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = a.n_splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    b.coop = 0;
  } else if (a.coop) {
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  // the kernel's first global access waits for the previous grid (see above)
  attr[cfg.numAttrs].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[cfg.numAttrs].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs += 1;
  e = cudaLaunchKernelEx(&cfg, kern, b);
  if (e == cudaErrorCooperativeLaunchTooLarge) {          // fewer SMs available than the device has
    cudaGetLastError();
    b.coop = 0;
    attr[0] = attr[cfg.numAttrs - 1];
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, b);
  }
  return e == cudaSuccess ? cudaGetLastError() : e;
}

template <int T>
cudaError_t launch_type(const DecodeArgs &a, cudaStream_t s) {
#define TQ_DEC_CASE(GG, BK, BV) \
  if (a.group == GG && a.nbk == BK && a.nbv == BV)                      \
    return a.v_thresh > 0.f ? launch_one<T, GG, BK, BV, true>(a, s) : launch_one<T, GG, BK, BV, false>(a, s);
  TQ_DEC_CASE(4, 1, 1)
  TQ_DEC_CASE(2, 1, 1)
  TQ_DEC_CASE(1, 1, 1)
  TQ_DEC_CASE(4, 2, 2)
  TQ_DEC_CASE(2, 2, 2)
  TQ_DEC_CASE(1, 2, 2)
  TQ_DEC_CASE(1, 2, 1)
  TQ_DEC_CASE(2, 2, 1)
  TQ_DEC_CASE(4, 2, 1)
#undef TQ_DEC_CASE
  return cudaErrorNotSupported;
}

}  // namespace mmadec
}  // namespace tq

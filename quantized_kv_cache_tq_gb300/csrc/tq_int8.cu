// Prompt attention over an int8 KV cache with one binary16 scale per row,
// rows scattered over the cells ([QSA#1821] "What", "Change"):
//   k_t = k_int[cell_of_pos[t]] * scale_k,  v_t = v_int[...] * scale_v,
//   out[i][h] = softmax_{t <= p_i}(scale * q[i][h] . k_t) v_t.
//
// The page's sm_75 kernel gathers each 32-cell chunk's rows into registers
// during the previous chunk and shares one shared buffer between K and V to fit
// two blocks per SM.  On GB300 the gather is asynchronous and spread over four
// warps: every gather thread owns one K or V row of the key tile and streams it
// with 16-byte cp.async copies into its own slots of a 4-deep ring (its cell id
// one tile ahead of the copy, its scale one tile ahead of the use), so it only
// ever waits for its own copies.  The math runs on tcgen05 in the same
// warp-specialised pipeline as the turbo prefill:
//   control warp (one thread): S_j = Q K'_j^T into tensor memory, then
//     O += P'_{j-1} V'_{j-1} while the softmax works on tile j;
//   4 gather warps: int8 rows -> exact binary16 K' / V' tiles (a byte b becomes
//     the half 0x64xx, xx = b ^ 0x80, i.e. 1024 + b + 128, by one byte permute;
//     one packed subtraction of 1152 gives b), row scales as floats;
//   4 softmax warps (one query row per thread, TMEM lanes 0..127): read S_j,
//     apply scale_k * scale * log2(e) and the causal mask by logical position,
//     the online softmax (lazy rescale of O in tensor memory), and write
//     P' = p * scale_v as binary16 hi + lo over S_j, where the PV mma reads it.
// Q is binary16 as given, so S is exact up to fp32 accumulation.
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
  int32_t f16;            // rows are binary16 (k, v hold uint16), no scales
  float scale_log2;
  int32_t n_split;        // key-range splits per query tile (merged by the last CTA of the tile)
  int32_t qt_fastest;     // grid order: query tiles fastest (else KV heads fastest)
  int32_t *counters;      // [q tile][kv head] arrivals, self-resetting
  float *part;            // split partials [q tile][kv head][split][128 rows][4 + 128]
};

namespace i8 {

constexpr int BM = 128, BN = 64, D = 128;
constexpr int NWARP = 9;                        // 0-3 softmax, 4-7 gather, 8 control
constexpr int NT = NWARP * 32;
constexpr int RING = 4;                         // raw-row ring depth (tiles)
constexpr int LOOK = RING - 1;                  // copies run this many tiles ahead
constexpr uint32_t SQ = 0;                      // Q       [d/8][row/8]            32 KB
constexpr uint32_t RSTAGE = 2 * BN * D;
// Shared-memory layout per cache mode.  int8 rows pass through the raw ring
// (RING x 16 KB) and keep three K'/V' buffers; binary16 rows go straight to the
// operand tiles, so that space holds two more buffers and the copies run four
// tiles ahead instead of two.
template <bool F16>
struct Lay {
  static constexpr int NB = F16 ? 5 : 3;        // K'/V' tiles, scales and S / P' buffers in flight
  static constexpr uint32_t SK = SQ + 32768;    // K'      NB x [key/8][d/8]      NB x 16 KB
  static constexpr uint32_t SV = SK + NB * 16384;   // V'  NB x [key/8][d/8]      NB x 16 KB
  static constexpr uint32_t SR = SV + NB * 16384;   // raw RING x [K|V][key][128 B] (int8 only)
  static constexpr uint32_t SSC = SR + (F16 ? 0 : RING * RSTAGE);   // scales  NB x ([BN] k, [BN] v) floats
  static constexpr uint32_t TOTAL = SSC + NB * BN * 2 * 4;
};
constexpr int TMEM_COLS = 512;                  // O: 128 columns, S / P': NB x 64 columns (NB <= 6)
constexpr uint32_t SP0 = 128;

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

// 16-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(tc::smem_u32(dst)), "l"(src),
               "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(tc::smem_u32(bar)) : "memory");
}

// tcgen05.mma with the A operand in tensor memory
__device__ __forceinline__ void mma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(static_cast<uint32_t>(acc)));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t *r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t *r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

template <int NB>
struct Bars {               // buffer j % NB, phase (j / NB) & 1
  uint64_t cv[NB];         // K'/V' tile and its scales written (4 gather warps)
  uint64_t sf[NB];         // S_j computed (mma commit)
  uint64_t pf[NB];         // P'_j written (4 softmax warps)
  uint64_t pv[NB];         // PV_j computed (mma commit)
};

// F16 = false: int8 rows with binary16 scales; true: binary16 rows, no scales
// (the second cache mode of the same prompt attention).
template <bool F16>
__global__ void __launch_bounds__(NT, 1) prompt_attn_kernel(const Int8Args a) {
  using L = Lay<F16>;
  constexpr int NB = L::NB;
  constexpr uint32_t SK = L::SK, SV = L::SV, SR = L::SR, SSC = L::SSC;
  static_assert(SP0 + NB * BN <= TMEM_COLS, "tensor memory");
  extern __shared__ __align__(1024) unsigned char smem[];
  __shared__ __align__(8) Bars<NB> bars;
  __shared__ uint32_t tmem_slot;
  __shared__ int s_fail;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // grid (KV head, split, query tile): the query tiles at the end of the prompt
  // (the longest under the causal mask) are launched first
  // launch order (longest query tiles first either way): query tiles fastest when their
  // key counts are about equal, so that the CTAs in flight share (KV head, key range)
  // and its rows stay in L2; else KV heads fastest, so that the shortest query tiles
  // of every head are the last wave
  const int hk = a.qt_fastest ? blockIdx.y : blockIdx.x;
  const int split = a.qt_fastest ? blockIdx.z : blockIdx.y, n_split = a.n_split, G = a.group;
  const int qt = a.qt_fastest ? gridDim.x - 1 - blockIdx.x : gridDim.z - 1 - blockIdx.z;
  const int q0 = qt * (BM / G);
  const int q_last = min(a.nq, q0 + BM / G) - 1;
  const int64_t pos0 = a.ctx - a.nq;
  const int64_t kv_hi = a.causal ? i64min(a.ctx, pos0 + q_last + 1) : a.ctx;
  const int tiles_all = static_cast<int>((kv_hi + BN - 1) / BN);
  // this CTA's key tiles t_lo .. t_hi - 1 (local tile j is key tile t_lo + j)
  const int t_lo = static_cast<int>(static_cast<long long>(tiles_all) * split / n_split);
  const int n_tiles = static_cast<int>(static_cast<long long>(tiles_all) * (split + 1) / n_split) - t_lo;
  const int64_t kbase = static_cast<int64_t>(t_lo) * BN;
  float *scl = reinterpret_cast<float *>(smem + SSC);

  if (warp == 0) tc::tmem_alloc<TMEM_COLS>(&tmem_slot);
  if (tid == NT - 32) {
    s_fail = 0;
    for (int b = 0; b < NB; ++b) {
      tc::mbar_init(&bars.cv[b], 4);
      tc::mbar_init(&bars.sf[b], 1);
      tc::mbar_init(&bars.pf[b], 4);
      tc::mbar_init(&bars.pv[b], 1);
    }
    tc::mbar_init_fence();
  }
  // Q tile (binary16 as given): row r = query q0 + r/G, head hk*G + r%G
  for (int it = tid; it < BM * (D / 8); it += NT) {
    const int r = it / (D / 8), dc = it % (D / 8);
    const int qi = q0 + r / G, h = hk * G + r % G;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (qi < a.nq) val = *reinterpret_cast<const uint4 *>(a.q + (static_cast<size_t>(qi) * a.n_q_heads + h) * D + dc * 8);
    *reinterpret_cast<uint4 *>(smem + SQ + (dc * 16 + (r >> 3)) * 128 + (r & 7) * 16) = val;
  }
  tc::fence_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_slot;
  const uint32_t sbase = tc::smem_u32(smem);

  const int row = tid & (BM - 1);
  const int row_q = q0 + row / G;
  const bool row_ok = warp < 4 && row_q < a.nq;
  const int64_t row_end = a.causal ? (pos0 + row_q + 1) : a.ctx;
  float m_used = -INFINITY, l_sum = 0.f;

  if (warp == 8) {
    // ===================== control: mma issue =====================
    if (lane == 0) {
      constexpr uint32_t ID_S = tc::idesc_f16(BM, BN, false, false);
      constexpr uint32_t ID_PV = tc::idesc_f16(BM, D, false, true);
      // descriptor of base + off = descriptor of base + (off >> 4) (14-bit address field, < 256 KB)
      const uint64_t q_desc = tc::sdesc(sbase + SQ, 2048, 128);
      const uint64_t k_desc = tc::sdesc(sbase + SK, 128, 2048);
      const uint64_t v_desc = tc::sdesc(sbase + SV, 2048, 128);
      auto issue_pv = [&](int j) {
        const uint32_t pbuf = tmem + SP0 + (j % NB) * BN;
        const uint64_t vb = v_desc + (((j % NB) * 16384) >> 4);
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks)
            mma_f16_ta(tmem, pbuf + part * (BN / 2) + ks * 8, vb + ((ks * 4096) >> 4), ID_PV,
                       j > 0 || part > 0 || ks > 0);
        tc::mma_commit(&bars.pv[j % NB]);
      };
      bool ok = true;
      for (int j = 0; j < n_tiles && ok; ++j) {
        ok = tc::mbar_wait(&bars.cv[j % NB], (j / NB) & 1);
        if (ok && j >= NB) ok = tc::mbar_wait(&bars.pv[j % NB], ((j - NB) / NB) & 1);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t sbuf = tmem + SP0 + (j % NB) * BN;
        const uint64_t kb = k_desc + (((j % NB) * 16384) >> 4);
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks)
          tc::mma_f16(sbuf, q_desc + ((ks * 4096) >> 4), kb + ((ks * 256) >> 4), ID_S, ks > 0);
        tc::mma_commit(&bars.sf[j % NB]);
        if (j >= 1) {
          ok = tc::mbar_wait(&bars.pf[(j - 1) % NB], ((j - 1) / NB) & 1);
          if (!ok) break;
          tc::fence_after_sync();
          issue_pv(j - 1);
        }
      }
      if (ok && n_tiles > 0) {
        const int j = n_tiles - 1;
        ok = tc::mbar_wait(&bars.pf[j % NB], (j / NB) & 1);
        if (ok) {
          tc::fence_after_sync();
          issue_pv(j);
        }
      }
      if (!ok) s_fail = 1;
    }
  } else if (warp >= 4) {
    // ===================== gather: one K or V row of the tile per thread =====================
    const int gt = tid - 128;                     // 0..127
    const bool is_v = gt >= BN;
    const int key = gt & (BN - 1);
    if constexpr (F16) {
      // binary16 rows are operand-ready: each 16-byte chunk (8 dims) is copied
      // straight to its core-matrix slot of the K'/V' tile, LOOK16 tiles ahead,
      // once that tile's buffer is free (PV of the tile NB before it is done)
      constexpr int LOOK16 = NB - 1;
      constexpr int RING16 = LOOK16 + 2;          // cell ids: loaded two tiles before their copies
      const uint8_t *src = reinterpret_cast<const uint8_t *>(is_v ? a.v : a.k) + static_cast<int64_t>(hk) * D * 2;
      const int64_t row_stride = static_cast<int64_t>(a.n_kv_heads) * D * 2;
      auto cell_load = [&](int j) -> int64_t {
        const int64_t t = kbase + static_cast<int64_t>(j) * BN + key;
        return (j < n_tiles && t < kv_hi) ? static_cast<int64_t>(__ldg(a.cell_of_pos + t)) : -1;
      };
      auto fetch = [&](int j, int64_t c) {
        const int64_t t = kbase + static_cast<int64_t>(j) * BN + key;
        const bool okc = c >= 0 && c < a.n_cells;
        if (!okc && t < kv_hi && !is_v) set_status(a.status, TQ_ERR_DEVICE_CHECK);   // a zero row
        unsigned char *dst = smem + (is_v ? SV : SK) + (j % NB) * 16384 + (key >> 3) * 2048 + (key & 7) * 16;
        const uint8_t *p = okc ? src + c * row_stride : src;
        const uint32_t nb = okc ? 16u : 0u;
#pragma unroll
        for (int i = 0; i < D / 8; ++i) cp_async16(dst + i * 128, p + 16 * i, nb);
      };
      // constant scales: k * scale * log2(e), v * 1, for every buffer
      for (int i = gt; i < NB * BN; i += 128) {
        scl[(i / BN) * 2 * BN + i % BN] = a.scale_log2;
        scl[(i / BN) * 2 * BN + BN + i % BN] = 1.f;
      }
      int64_t cb[RING16];                         // cb[t % RING16]: cell of tile t
#pragma unroll
      for (int k = 0; k < RING16; ++k) cb[k] = cell_load(k);
#pragma unroll
      for (int k = 0; k < LOOK16; ++k) {
        if (k < n_tiles) fetch(k, cb[k]);
        cp_async_commit();
      }
      bool ok = true;
      for (int j0 = 0; j0 < n_tiles && ok; j0 += RING16) {
#pragma unroll
        for (int u = 0; u < RING16; ++u) {
          const int j = j0 + u;
          if (j >= n_tiles) break;
          // tile j first: the control thread issues PV_{j-1} only after S_j, so
          // tile j must be published before this thread waits for PV_{j-1}
          cp_async_wait<LOOK16 - 1>();              // this thread's row of tile j has landed
          tc::fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.cv[j % NB]);
          const int jn = j + LOOK16;                // its buffer was used by tile jn - NB = j - 1
          if (jn < n_tiles) {
            if (jn >= NB) ok = tc::mbar_wait(&bars.pv[(jn - NB) % NB], ((jn - NB) / NB) & 1);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; s_fail = 1; break; }
            tc::fence_after_sync();
            fetch(jn, cb[(u + LOOK16) % RING16]);
          }
          cp_async_commit();
          cb[u] = cell_load(j + RING16);
        }
      }
    } else {
      const int8_t *src = (is_v ? a.v : a.k) + static_cast<int64_t>(hk) * D;
      const uint16_t *ssrc = (is_v ? a.v_scale : a.k_scale) + hk;
      const int64_t row_stride = static_cast<int64_t>(a.n_kv_heads) * D;
      // Loaded values are only read one or more tiles after their load (the loop is
      // unrolled by RING, so the per-tile registers rotate by renaming, not by moves
      // that would wait for the load): a thread never stalls on a global load.
      static_assert(RING == 4 && LOOK == 3, "register rotation below assumes a 4-deep ring");
      auto cell_load = [&](int j) -> int64_t {       // raw cell id of this thread's key in tile j, or -1
        const int64_t t = kbase + static_cast<int64_t>(j) * BN + key;
        return (j < n_tiles && t < kv_hi) ? static_cast<int64_t>(__ldg(a.cell_of_pos + t)) : -1;
      };
      auto cell_ok = [&](int64_t c) { return c >= 0 && c < a.n_cells; };
      auto fetch = [&](int j, int64_t c) {          // this thread's row of tile j -> ring slot j % RING
        const int64_t t = kbase + static_cast<int64_t>(j) * BN + key;
        const bool ok = cell_ok(c);
        if (!ok && t < kv_hi && !is_v) set_status(a.status, TQ_ERR_DEVICE_CHECK);   // a zero row
        unsigned char *dst = smem + SR + (j % RING) * RSTAGE + (is_v ? BN * D : 0) + key * D;
        const int8_t *p = ok ? src + c * row_stride : src;
        const uint32_t nb = ok ? 16u : 0u;
        // 16-byte chunk i of the row sits in slot i ^ (key & 7): the lanes of a warp
        // (consecutive keys, rows 128 bytes apart) then hit different banks
  #pragma unroll
        for (int i = 0; i < D / 16; ++i) cp_async16(dst + 16 * (i ^ (key & 7)), p + 16 * i, nb);
      };
      auto scale_load = [&](int64_t c) -> float {
        return cell_ok(c) ? __half2float(__ushort_as_half(__ldg(ssrc + c * a.n_kv_heads))) : 0.f;
      };
      int64_t cb[RING];                             // cb[t % RING]: cell of tile t (t = j .. j + LOOK)
      float sb[RING];                               // sb[t % RING]: scale of tile t (t = j, j + 1)
  #pragma unroll
      for (int k = 0; k < RING; ++k) cb[k] = cell_load(k);
  #pragma unroll
      for (int k = 0; k < LOOK; ++k) {
        fetch(k, cb[k]);
        cp_async_commit();
      }
      sb[0] = scale_load(cb[0]);
      bool ok = true;
      for (int j0 = 0; j0 < n_tiles && ok; j0 += RING) {
  #pragma unroll
        for (int u = 0; u < RING; ++u) {
          const int j = j0 + u;
          if (j >= n_tiles) break;
          // tile j + LOOK's copies (its cell was loaded a tile ago), tile j + 1's scale,
          // then tile j + RING's cell into the slot tile j no longer needs
          if (j + LOOK < n_tiles) fetch(j + LOOK, cb[(u + LOOK) % RING]);
          cp_async_commit();
          sb[(u + 1) % RING] = scale_load(cb[(u + 1) % RING]);
          const float sc_j = sb[u];
          cb[u] = cell_load(j + RING);
          cp_async_wait<LOOK>();                      // this thread's row of tile j has landed
          // K'/V' buffer j % NB is free once PV_{j-NB} is done
          if (j >= NB) ok = tc::mbar_wait(&bars.pv[j % NB], ((j - NB) / NB) & 1);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; s_fail = 1; break; }
          tc::fence_after_sync();
          const unsigned char *rw = smem + SR + (j % RING) * RSTAGE + (is_v ? BN * D : 0) + key * D;
          unsigned char *dst = smem + (is_v ? SV : SK) + (j % NB) * 16384 + (key >> 3) * 2048 + (key & 7) * 16;
  #pragma unroll
          for (int i = 0; i < D / 16; ++i) {
            const uint4 w = *reinterpret_cast<const uint4 *>(rw + 16 * (i ^ (key & 7)));
            uint4 o0, o1;
            i8x4_to_h(w.x, o0.x, o0.y);
            i8x4_to_h(w.y, o0.z, o0.w);
            i8x4_to_h(w.z, o1.x, o1.y);
            i8x4_to_h(w.w, o1.z, o1.w);
            *reinterpret_cast<uint4 *>(dst + (2 * i) * 128) = o0;          // dims 16 i .. 16 i + 7
            *reinterpret_cast<uint4 *>(dst + (2 * i + 1) * 128) = o1;      // dims 16 i + 8 .. 16 i + 15
          }
          // k scales pre-multiplied by scale * log2(e): the softmax does one multiply per score
          scl[(j % NB) * 2 * BN + (is_v ? BN : 0) + key] = is_v ? sc_j : sc_j * a.scale_log2;
          tc::fence_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars.cv[j % NB]);
        }
      }
    }
    cp_async_wait<0>();
  } else {
    // ===================== softmax: one query row per thread =====================
    const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      ok = tc::mbar_wait(&bars.sf[j % NB], (j / NB) & 1);
      if (ok) ok = tc::mbar_wait(&bars.cv[j % NB], (j / NB) & 1);      // scales of tile j are written
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc::fence_after_sync();
      const uint32_t sbuf = tmem + lane_off + SP0 + (j % NB) * BN;
      const float *sc = scl + (j % NB) * BN * 2;
      float s[BN];
      {
        uint32_t r0[BN];
        tc::tmem_ld32(sbuf, r0);
        tc::tmem_ld32(sbuf + 32, r0 + 32);
        tc::tmem_wait_ld();
#pragma unroll
        for (int i4 = 0; i4 < BN; i4 += 4) {
          const float4 k4 = *reinterpret_cast<const float4 *>(sc + i4);     // k scales of keys i4 .. i4 + 3
          const float2 a0 = mul2(make_float2(__uint_as_float(r0[i4]), __uint_as_float(r0[i4 + 1])), make_float2(k4.x, k4.y));
          const float2 a1 = mul2(make_float2(__uint_as_float(r0[i4 + 2]), __uint_as_float(r0[i4 + 3])), make_float2(k4.z, k4.w));
          s[i4] = a0.x;
          s[i4 + 1] = a0.y;
          s[i4 + 2] = a1.x;
          s[i4 + 3] = a1.y;
        }
      }
      const int64_t key0 = kbase + static_cast<int64_t>(j) * BN;
      const int nvis = row_ok ? static_cast<int>(i64max(0, i64min(BN, row_end - key0))) : 0;
      const bool full_tile = __all_sync(0xffffffffu, nvis == BN);     // no mask in this warp
      if (!full_tile) {
#pragma unroll
        for (int i = 0; i < BN; ++i)
          if (i >= nvis) s[i] = -INFINITY;
      }
      // four independent chains for the maximum (and the sum below)
      float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < BN; i += 8)
#pragma unroll
        for (int c = 0; c < 4; ++c) mx[c] = max3(mx[c], s[i + c], s[i + c + 4]);
      const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
      const bool raise = mt > m_used + 8.f || (m_used == -INFINITY && mt > -INFINITY);
      const float fct = (raise && m_used != -INFINITY) ? exp2f(m_used - mt) : 1.f;
      if (raise) m_used = mt;
      if (__any_sync(0xffffffffu, fct != 1.f)) {
        // O must be stable: wait for the PV mma of the previous tile
        bool okp = (j == 0) || tc::mbar_wait(&bars.pv[(j - 1) % NB], ((j - 1) / NB) & 1);
        if (!__all_sync(0xffffffffu, okp)) { ok = false; break; }
        tc::fence_after_sync();
        l_sum *= fct;
#pragma unroll 1
        for (int c = 0; c < D; c += 16) {          // 16 columns at a time: s[] is live here
          uint32_t r[16];
          tmem_ld16(tmem + lane_off + c, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * fct);
          tmem_st16(tmem + lane_off + c, r);
        }
      }
      // P' = p * scale_v as binary16 (hi, lo) key pairs over S_j (row = lane), 32 keys
      // at a time.  Every scale of the tile is finite (0 beyond kv_hi and for
      // rejected cells); a row with nothing visible yet has m_used = -inf and p = 0.
      const float m_ref = (m_used == -INFINITY) ? 0.f : m_used;
      const float2 m_ref2 = make_float2(m_ref, m_ref);
      float ps[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ch = 0; ch < BN / 32; ++ch) {
        uint32_t ph[16], pl[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int k0 = 32 * ch + 2 * i;
          const float2 e = sub2(make_float2(s[k0], s[k0 + 1]), m_ref2);
          const float p0 = tc::ex2(e.x), p1 = tc::ex2(e.y);                    // masked: 0
          ps[i & 3] += p0 + p1;
          const float2 v2 = *reinterpret_cast<const float2 *>(sc + BN + k0);    // v scales of keys k0, k0 + 1
          const float2 x = mul2(make_float2(p0, p1), v2);
          const __half2 h = __floats2half2_rn(x.x, x.y);
          const float2 lo = sub2(x, __half22float2(h));
          const __half2 l = __floats2half2_rn(lo.x, lo.y);
          ph[i] = *reinterpret_cast<const uint32_t *>(&h);
          pl[i] = *reinterpret_cast<const uint32_t *>(&l);
        }
        tmem_st16(sbuf + 16 * ch, ph);
        tmem_st16(sbuf + BN / 2 + 16 * ch, pl);
      }
      l_sum += (ps[0] + ps[1]) + (ps[2] + ps[3]);
      tc::tmem_wait_st();
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars.pf[j % NB]);
    }
    // the last PV must be complete before O is read
    if (ok && n_tiles > 0) {
      const int j = n_tiles - 1;
      ok = tc::mbar_wait(&bars.pv[j % NB], (j / NB) & 1);
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
  const int h = hk * G + row % G;
  if (n_split == 1) {
    if (warp < 4 && !failed) {
      const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
      const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
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
                n_tiles > 0 ? make_float4(__uint_as_float(r[i]) * inv, __uint_as_float(r[i + 1]) * inv,
                                          __uint_as_float(r[i + 2]) * inv, __uint_as_float(r[i + 3]) * inv)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
    }
  } else {
    // split key range: store (m, l, O) of every row; the last CTA of this query
    // tile merges them with log-sum-exp weights
    __shared__ int s_last;
    const size_t tile_id = static_cast<size_t>(qt) * a.n_kv_heads + hk;
    const size_t stride = 4 + D;                // m, l, 2 pad floats: O rows stay 16-byte aligned
    if (warp < 4) {
      const uint32_t lane_off = static_cast<uint32_t>(32 * warp) << 16;
      float *pr = a.part + ((tile_id * n_split + split) * BM + row) * stride;
      const bool has = !failed && n_tiles > 0;
      pr[0] = has ? m_used : -INFINITY;
      pr[1] = has ? l_sum : 0.f;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
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
      float *wts = reinterpret_cast<float *>(smem + SQ);            // [BM][n_split] weights / L
      const int rows_valid = min(BM, (a.nq - q0) * G);             // rows of queries < nq
      if (tid < rows_valid) {
        float M = -INFINITY;
        for (int s2 = 0; s2 < n_split; ++s2) M = fmaxf(M, __ldcg(base + (static_cast<size_t>(s2) * BM + tid) * stride));
        float Ls = 0.f;
        for (int s2 = 0; s2 < n_split; ++s2) {
          const float *p = base + (static_cast<size_t>(s2) * BM + tid) * stride;
          const float m = __ldcg(p);
          const float w = (m == -INFINITY) ? 0.f : exp2f(m - M);
          wts[tid * n_split + s2] = w;
          Ls += w * __ldcg(p + 1);
        }
        const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
        for (int s2 = 0; s2 < n_split; ++s2) wts[tid * n_split + s2] *= inv;
      }
      __syncthreads();
      for (int i = tid; i < rows_valid * (D / 4); i += NT) {
        const int r = i / (D / 4), d = 4 * (i % (D / 4));
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s2 = 0; s2 < n_split; ++s2) {
          const float w = wts[r * n_split + s2];
          const float4 x = __ldcg(reinterpret_cast<const float4 *>(base + (static_cast<size_t>(s2) * BM + r) * stride + 4 + d));
          o.x = fmaf(w, x.x, o.x); o.y = fmaf(w, x.y, o.y); o.z = fmaf(w, x.z, o.z); o.w = fmaf(w, x.w, o.w);
        }
        const int qi = q0 + r / G, hh = hk * G + r % G;
        *reinterpret_cast<float4 *>(a.out + (static_cast<size_t>(qi) * a.n_q_heads + hh) * D + d) = o;
      }
      if (tid == 0) a.counters[tile_id] = 0;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc<TMEM_COLS>(tmem);
}

}  // namespace i8

cudaError_t launch_int8_attn(const Int8Args &a, cudaStream_t s) {
  static_assert(i8::Lay<false>::TOTAL <= 227 * 1024 && i8::Lay<true>::TOTAL <= 227 * 1024, "shared memory");
  auto kern = a.f16 ? i8::prompt_attn_kernel<true> : i8::prompt_attn_kernel<false>;
  const uint32_t total = a.f16 ? i8::Lay<true>::TOTAL : i8::Lay<false>::TOTAL;
  cudaError_t e = set_dynamic_smem(reinterpret_cast<const void *>(kern), (int)total);
  if (e != cudaSuccess) return e;
  const int rows = a.nq * a.group;
  const unsigned n_qt = static_cast<unsigned>((rows + i8::BM - 1) / i8::BM);
  const dim3 grid = a.qt_fastest ? dim3(n_qt, a.n_kv_heads, a.n_split) : dim3(a.n_kv_heads, a.n_split, n_qt);
  kern<<<grid, i8::NT, total, s>>>(a);
  return cudaGetLastError();
}

}  // namespace tq

using namespace tq;

namespace tq {
// Key-range splits per query tile: the count (1 .. 8) whose CTAs fill the last
// wave of the GPU best (one CTA per SM), the smallest one within 1% of the best,
// with at least 48 key tiles per split (a split's fixed costs -- Q tile, pipeline
// fill, partial store and merge -- stay small).  Workspace: status word, then
// (with splits) the merge counters [q tile][kv head] and the partials.
struct Int8Layout {
  int n_split;
  size_t counters_off, part_off, total;
};
static Int8Layout int8_layout(int nq, int n_q_heads, int n_kv_heads, int64_t ctx) {
  Int8Layout L;
  const int64_t qt = (static_cast<int64_t>(nq) * (n_q_heads / n_kv_heads) + i8::BM - 1) / i8::BM;
  const int64_t base = qt * n_kv_heads;
  const int64_t tiles = (ctx + i8::BN - 1) / i8::BN;
  const int sms = sm_count();
  double best = 0.0;
  double eff[9] = {0.0};
  for (int sp = 1; sp <= 8; ++sp) {
    if (sp > 1 && tiles / sp < 48) break;
    const double waves = static_cast<double>(base * sp) / sms;
    eff[sp] = waves / ceil(waves);
    if (eff[sp] > best) best = eff[sp];
  }
  L.n_split = 1;
  for (int sp = 1; sp <= 8; ++sp)
    if (eff[sp] >= best - 0.01) { L.n_split = sp; break; }
  L.counters_off = 256;
  L.part_off = L.counters_off + (sizeof(int32_t) * base + 255) / 256 * 256;
  L.total = L.n_split > 1 ? L.part_off + sizeof(float) * base * L.n_split * i8::BM * (4 + i8::D) : 256;
  return L;
}
}  // namespace tq

extern "C" size_t tq_int8_prompt_attn_workspace(int nq, int n_q_heads, int n_kv_heads, int head_dim, int64_t ctx) {
  if (nq < 0 || n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads || head_dim != 128 || ctx < 0) return 0;
  return int8_layout(nq, n_q_heads, n_kv_heads, ctx).total;
}

static tq_status prompt_attn_call(const void *k, const uint16_t *k_scale, const void *v, const uint16_t *v_scale,
                                  bool f16, int64_t n_cells, const int32_t *cell_of_pos, int64_t ctx,
                                  const uint16_t *q, int nq, int n_q_heads, int n_kv_heads, int head_dim, float scale,
                                  int causal, float *out, void *workspace, size_t workspace_bytes, tq_stream stream) {
  auto al = [](const void *p, uintptr_t m) { return (reinterpret_cast<uintptr_t>(p) & (m - 1)) == 0; };
  if (n_q_heads <= 0 || n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return TQ_ERR_INVALID_ARG;
  const int group = n_q_heads / n_kv_heads;
  if ((group & (group - 1)) != 0 || group > 128) return TQ_ERR_UNSUPPORTED;
  if (head_dim != 128) return TQ_ERR_UNSUPPORTED;
  if (nq < 0 || ctx < 0 || n_cells <= 0 || (causal && nq > ctx) || !isfinite(scale)) return TQ_ERR_INVALID_ARG;
  if (nq == 0) return TQ_OK;
  if (!out || !al(out, 16) || !q || !al(q, 16)) return TQ_ERR_INVALID_ARG;
  const Int8Layout WL = int8_layout(nq, n_q_heads, n_kv_heads, ctx);
  if (!workspace || !al(workspace, 256) || workspace_bytes < WL.total) return TQ_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (ctx == 0) {
    if (cudaMemsetAsync(out, 0, sizeof(float) * nq * n_q_heads * head_dim, s) == cudaSuccess) return TQ_OK;
    cudaGetLastError();               // the status reports it; leave no stale error behind
    return TQ_ERR_CUDA;
  }
  if (!k || !v || !al(k, 16) || !al(v, 16) || !cell_of_pos || !al(cell_of_pos, 4)) return TQ_ERR_INVALID_ARG;
  if (!f16 && (!k_scale || !v_scale || !al(k_scale, 2) || !al(v_scale, 2))) return TQ_ERR_INVALID_ARG;
  if (static_cast<int64_t>(nq) * group > 0x7fffffffLL) return TQ_ERR_INVALID_ARG;
  if ((static_cast<int64_t>(nq) * group + i8::BM - 1) / i8::BM > 65535 || n_kv_heads > 65535) return TQ_ERR_UNSUPPORTED;
  Int8Args a;
  a.k = static_cast<const int8_t *>(k);
  a.k_scale = k_scale;
  a.v = static_cast<const int8_t *>(v);
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
  a.f16 = f16 ? 1 : 0;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.n_split = WL.n_split;
  // the shortest causal query tile sees about ctx - nq + its rows of keys, the longest ctx
  a.qt_fastest = !causal || 4 * (ctx - nq + i8::BM / group) >= 3 * ctx;
  a.counters = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + WL.counters_off);
  a.part = reinterpret_cast<float *>(static_cast<char *>(workspace) + WL.part_off);
  if (launch_int8_attn(a, s) == cudaSuccess) return TQ_OK;
  cudaGetLastError();                 // the status reports it; leave no stale error behind
  return TQ_ERR_CUDA;
}

extern "C" tq_status tq_int8_prompt_attn(const int8_t *k, const uint16_t *k_scale, const int8_t *v,
                                         const uint16_t *v_scale, int64_t n_cells, const int32_t *cell_of_pos,
                                         int64_t ctx, const uint16_t *q, int nq, int n_q_heads, int n_kv_heads,
                                         int head_dim, float scale, int causal, float *out, void *workspace,
                                         size_t workspace_bytes, tq_stream stream) {
  return prompt_attn_call(k, k_scale, v, v_scale, false, n_cells, cell_of_pos, ctx, q, nq, n_q_heads, n_kv_heads,
                          head_dim, scale, causal, out, workspace, workspace_bytes, stream);
}

extern "C" tq_status tq_f16_prompt_attn(const uint16_t *k, const uint16_t *v, int64_t n_cells,
                                        const int32_t *cell_of_pos, int64_t ctx, const uint16_t *q, int nq,
                                        int n_q_heads, int n_kv_heads, int head_dim, float scale, int causal,
                                        float *out, void *workspace, size_t workspace_bytes, tq_stream stream) {
  return prompt_attn_call(k, nullptr, v, nullptr, true, n_cells, cell_of_pos, ctx, q, nq, n_q_heads, n_kv_heads,
                          head_dim, scale, causal, out, workspace, workspace_bytes, stream);
}

// Single-query decode on the tensor cores with register dequantisation.
//
// Why not the page's LUT ([TQ#36] "Q x centroid LUT") on GB300: with a GQA
// group of 4 every K element costs 4 shared-memory table reads, i.e. ~16 B of
// shared-memory traffic per 0.39 B of HBM traffic, and the SMs' shared-memory
// bandwidth is only ~5x HBM -- the LUT kernel is bound by shared memory at
// several times the HBM time.  Here the packed codes go from HBM to shared
// memory once (cp.async.bulk, 4-stage mbarrier ring) and each thread turns them
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

namespace tq {
namespace mmadec {

constexpr int NW = 8;                // warps per CTA
constexpr int NT = NW * 32;
constexpr int WKEYS = 16;            // keys per warp per tile
constexpr int CKEYS = NW * WKEYS;    // keys per CTA tile (128)
constexpr int STAGES = 4;
constexpr long long kWaitLimit = 1ll << 22;

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t s) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(s));
  return d;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// bounded wait on phase `parity`; returns false if the limit was hit
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  for (long long it = 0; it < kWaitLimit; ++it) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(a), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

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
      dq4<4>(ws[i] & 0xffffu, t, h[4 * i + 0], h[4 * i + 1]);
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
      dq4<T>(s0 & 0xffffu, t, h[8 * i + 0], h[8 * i + 1]);
      dq4<T>(s0 >> 16, t, h[8 * i + 2], h[8 * i + 3]);
      dq4<T>(s1 & 0xffffu, t, h[8 * i + 4], h[8 * i + 5]);
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
    dq4<T>(ev & 0xffffu, t, out[8 * i + 0], out[8 * i + 2]);
    dq4<T>(ev >> 16, t, out[8 * i + 4], out[8 * i + 6]);
    dq4<T>(od & 0xffffu, t, out[8 * i + 1], out[8 * i + 3]);
    dq4<T>(od >> 16, t, out[8 * i + 5], out[8 * i + 7]);
  }
}

// selector words (elements 0..7, 8..15 of the 16-dim group g) of one V key block
template <int T>
__device__ __forceinline__ void v_sel(const uint8_t *qs_row, const uint8_t *sg_row, int g, uint32_t &s0,
                                      uint32_t &s1) {
  if (T == 4) {
    const uint2 w = *reinterpret_cast<const uint2 *>(qs_row + 8 * g);
    s0 = w.x;
    s1 = w.y;
  } else {
    const uint32_t w = reinterpret_cast<const uint32_t *>(qs_row)[g];
    const uint32_t sg = (T == 3) ? reinterpret_cast<const uint32_t *>(sg_row)[g >> 1] : 0u;
    sel_words<T>(w, sg, (g & 1) != 0, s0, s1);
  }
}

struct StageLayout {
  uint32_t kqs, ksg, kn, vqs, vsg, vn, bytes;
};

template <int T, int NBK, int NBV>
__host__ __device__ constexpr StageLayout stage_layout() {
  constexpr uint32_t QSB = TypeTraits<T>::QSB, SGB = TypeTraits<T>::SGB;
  StageLayout s{};
  uint32_t o = 0;
  s.kqs = o; o += CKEYS * NBK * QSB;
  s.ksg = o; o += CKEYS * NBK * SGB;
  s.kn = o;  o += CKEYS * NBK * 2;
  s.vqs = o; o += CKEYS * NBV * QSB;
  s.vsg = o; o += CKEYS * NBV * SGB;
  s.vn = o;  o += CKEYS * NBV * 2;
  s.bytes = (o + 127) / 128 * 128;
  return s;
}

template <int T, int G, int NBK, int NBV>
__host__ __device__ constexpr uint32_t smem_bytes() {
  // stages + P tiles (per warp, per V block: 8 columns x 16 keys fp16) + rotated q
  return STAGES * stage_layout<T, NBK, NBV>().bytes + NW * NBV * 8 * WKEYS * 2 + G * 128 * NBK * 4 + 64;
}

template <int T, int G, int NBK, int NBV>
__global__ void __launch_bounds__(NT, 2) decode_mma_kernel(const DecodeArgs a) {
  static_assert(G == 1 || G == 2 || G == 4, "GQA group must be 1, 2 or 4");
  constexpr StageLayout SL = stage_layout<T, NBK, NBV>();
  constexpr int QSB = TypeTraits<T>::QSB, SGB = TypeTraits<T>::SGB;
  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char *stages = smem;
  uint16_t *ptile = reinterpret_cast<uint16_t *>(smem + STAGES * SL.bytes);     // [NW][NBV][8][16]
  float *qrot = reinterpret_cast<float *>(smem + STAGES * SL.bytes + NW * NBV * 8 * WKEYS * 2);
  __shared__ __align__(8) uint64_t full[STAGES];
  __shared__ int s_timeout;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, c = lane & 3;
  const int hk = blockIdx.y, split = blockIdx.x;
  const int64_t t0 = static_cast<int64_t>(split) * a.chunk;
  const int64_t t1 = min(a.kv_len, t0 + a.chunk);
  const int n_tiles = static_cast<int>((t1 - t0 + CKEYS - 1) / CKEYS);

  const uint8_t *kqs = a.kqs + static_cast<size_t>(hk) * a.n_cells * NBK * QSB;
  const uint8_t *ksg = SGB ? a.ksg + static_cast<size_t>(hk) * a.n_cells * NBK * SGB : nullptr;
  const uint16_t *kn = a.kn + static_cast<size_t>(hk) * a.n_cells * NBK;
  const uint8_t *vqs = a.vqs + static_cast<size_t>(hk) * a.n_cells * NBV * QSB;
  const uint8_t *vsg = SGB ? a.vsg + static_cast<size_t>(hk) * a.n_cells * NBV * SGB : nullptr;
  const uint16_t *vn = a.vn + static_cast<size_t>(hk) * a.n_cells * NBV;

  auto issue = [&](int tile) {
    const int64_t key0 = t0 + static_cast<int64_t>(tile) * CKEYS;
    const int64_t left = a.n_cells - key0;                    // multiple of 64
    const uint32_t nk = static_cast<uint32_t>(left < CKEYS ? left : CKEYS);
    unsigned char *st = stages + (tile % STAGES) * SL.bytes;
    uint64_t *bar = &full[tile % STAGES];
    const uint32_t bytes = nk * (NBK * (QSB + SGB + 2) + NBV * (QSB + SGB + 2));
    mbar_expect_tx(bar, bytes);
    bulk_g2s(st + SL.kqs, kqs + key0 * NBK * QSB, nk * NBK * QSB, bar);
    if (SGB) bulk_g2s(st + SL.ksg, ksg + key0 * NBK * SGB, nk * NBK * SGB, bar);
    bulk_g2s(st + SL.kn, kn + key0 * NBK, nk * NBK * 2, bar);
    bulk_g2s(st + SL.vqs, vqs + key0 * NBV * QSB, nk * NBV * QSB, bar);
    if (SGB) bulk_g2s(st + SL.vsg, vsg + key0 * NBV * SGB, nk * NBV * SGB, bar);
    bulk_g2s(st + SL.vn, vn + key0 * NBV, nk * NBV * 2, bar);
  };

  if (tid == 0) {
    s_timeout = 0;
#pragma unroll
    for (int s = 0; s < STAGES; ++s) mbar_init(&full[s], 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  if (tid == 0)
    for (int i = 0; i < STAGES && i < n_tiles; ++i) issue(i);

  // rotated queries (scale and log2(e) folded in) while the first tiles land
  rotate_queries<NT>(a, hk, qrot);
  for (int i = tid; i < NW * NBV * 8 * WKEYS; i += NT) ptile[i] = 0;
  __syncthreads();

  const Tab tab_k = make_tab<T>(a.cbk);
  const Tab tab_v = make_tab<T>(a.cbv);

  // B fragments of the score mma: column n = g holds q'_hi (n < G), q'_lo (G <= n < 2G) or 0
  uint32_t qb[NBK][8][2];
#pragma unroll
  for (int b = 0; b < NBK; ++b)
#pragma unroll
    for (int kk = 0; kk < 8; ++kk)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint16_t v[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int d = b * QK + 32 * c + 4 * kk + 2 * h + j;
          float x = 0.f;
          if (g < 2 * G) {
            const float q = qrot[(g % G) * QK * NBK + d];
            const __half hi = __float2half_rn(q);
            x = (g < G) ? __half2float(hi) : (q - __half2float(hi));
          }
          v[j] = __half_as_ushort(__float2half_rn(x));
        }
        qb[b][kk][h] = v[0] | (static_cast<uint32_t>(v[1]) << 16);
      }

  float oacc[NBV][8][4];
#pragma unroll
  for (int b = 0; b < NBV; ++b)
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) oacc[b][mt][i] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

  uint16_t *pw = ptile + warp * NBV * 8 * WKEYS;
  bool timed_out = false;

  for (int tile = 0; tile < n_tiles; ++tile) {
    if (!timed_out && !mbar_wait(&full[tile % STAGES], (tile / STAGES) & 1)) {
      timed_out = true;
      s_timeout = 1;
    }
    const unsigned char *st = stages + (tile % STAGES) * SL.bytes;
    const int64_t key0 = t0 + static_cast<int64_t>(tile) * CKEYS + warp * WKEYS;
    const int r0 = warp * WKEYS + g, r1 = r0 + 8;              // rows of this thread's keys
    const bool ok0 = key0 + g < t1 && !timed_out, ok1 = key0 + g + 8 < t1 && !timed_out;

    if (key0 < t1 && !timed_out) {
      // ---- scores: S^T[key][n], one accumulator per K block (own norm)
      float s[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int b = 0; b < NBK; ++b) {
        uint32_t ka0[16], ka1[16];
        dq_chunk32<T>(st + SL.kqs + (r0 * NBK + b) * QSB, st + SL.ksg + (r0 * NBK + b) * SGB, c, tab_k, ka0);
        dq_chunk32<T>(st + SL.kqs + (r1 * NBK + b) * QSB, st + SL.ksg + (r1 * NBK + b) * SGB, c, tab_k, ka1);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma16816(acc, ka0[2 * kk], ka1[2 * kk], ka0[2 * kk + 1], ka1[2 * kk + 1], qb[b][kk][0], qb[b][kk][1]);
        const uint16_t *knr = reinterpret_cast<const uint16_t *>(st + SL.kn);
        const float n0 = __half2float(__ushort_as_half(knr[r0 * NBK + b]));
        const float n1 = __half2float(__ushort_as_half(knr[r1 * NBK + b]));
        s[0] += n0 * acc[0];
        s[1] += n0 * acc[1];
        s[2] += n1 * acc[2];
        s[3] += n1 * acc[3];
      }
      // hi + lo columns -> full scores; thread then holds heads hA, hA+1 of keys g, g+8
      if (G == 4) {
#pragma unroll
        for (int i = 0; i < 4; ++i) s[i] += __shfl_xor_sync(0xffffffffu, s[i], 2);
      } else if (G == 2) {
#pragma unroll
        for (int i = 0; i < 4; ++i) s[i] += __shfl_xor_sync(0xffffffffu, s[i], 1);
      } else {
        s[0] += s[1];
        s[2] += s[3];
        s[1] = s[0];
        s[3] = s[2];
      }
      if (!ok0) s[0] = s[1] = -INFINITY;
      if (!ok1) s[2] = s[3] = -INFINITY;

      // ---- online softmax per head (log2 domain); l kept per thread, reduced at the end
      float p[4];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float tm = fmaxf(s[j], s[2 + j]);
        tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 4));
        tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 8));
        tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 16));
        const float mnew = fmaxf(m_run[j], tm);
        const float alpha = (mnew == -INFINITY) ? 1.f : exp2f(m_run[j] - mnew);
        p[j] = (mnew == -INFINITY) ? 0.f : exp2f(s[j] - mnew);
        p[2 + j] = (mnew == -INFINITY) ? 0.f : exp2f(s[2 + j] - mnew);
        l_run[j] = l_run[j] * alpha + p[j] + p[2 + j];
        m_run[j] = mnew;
        // rescale the O' columns of this head (column 2c + j)
#pragma unroll
        for (int b = 0; b < NBV; ++b)
#pragma unroll
          for (int mt = 0; mt < 8; ++mt) {
            oacc[b][mt][j] *= alpha;
            oacc[b][mt][2 + j] *= alpha;
          }
      }

      // ---- P' = p * |v| (per V block) as fp16 hi/lo columns of the per-warp tile [n][key]
      const bool writer = (G == 4) ? (c < 2) : (c == 0);
      const int hA = (G == 4) ? 2 * (c & 1) : 0;
      const int nh = (G == 1) ? 1 : 2;
#pragma unroll
      for (int b = 0; b < NBV; ++b) {
        const uint16_t *vnr = reinterpret_cast<const uint16_t *>(st + SL.vn);
        const float v0 = ok0 ? __half2float(__ushort_as_half(vnr[r0 * NBV + b])) : 0.f;
        const float v1 = ok1 ? __half2float(__ushort_as_half(vnr[r1 * NBV + b])) : 0.f;
        if (writer) {
          uint16_t *pt = pw + b * 8 * WKEYS;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (j < nh) {
              const float x0 = p[j] * v0, x1 = p[2 + j] * v1;
              const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
              const int nhi = hA + j, nlo = G + hA + j;
              pt[nhi * WKEYS + g] = __half_as_ushort(h0);
              pt[nhi * WKEYS + g + 8] = __half_as_ushort(h1);
              pt[nlo * WKEYS + g] = __half_as_ushort(__float2half_rn(x0 - __half2float(h0)));
              pt[nlo * WKEYS + g + 8] = __half_as_ushort(__float2half_rn(x1 - __half2float(h1)));
            }
          }
        }
      }
      __syncwarp();

      // ---- O'^T[d][n] += V'^T[d][key] P'^T[key][n]
#pragma unroll
      for (int b = 0; b < NBV; ++b) {
        const uint32_t *pt32 = reinterpret_cast<const uint32_t *>(pw + b * 8 * WKEYS);
        const uint32_t pb0 = pt32[g * (WKEYS / 2) + c], pb1 = pt32[g * (WKEYS / 2) + c + 4];
        const int kr = warp * WKEYS;                 // first key row of this warp in the stage
        uint32_t s00, s01, s10, s11, s20, s21, s30, s31;
        const uint8_t *vq = st + SL.vqs, *vs = st + SL.vsg;
        v_sel<T>(vq + ((kr + 2 * c) * NBV + b) * QSB, vs + ((kr + 2 * c) * NBV + b) * SGB, g, s00, s01);
        v_sel<T>(vq + ((kr + 2 * c + 1) * NBV + b) * QSB, vs + ((kr + 2 * c + 1) * NBV + b) * SGB, g, s10, s11);
        v_sel<T>(vq + ((kr + 2 * c + 8) * NBV + b) * QSB, vs + ((kr + 2 * c + 8) * NBV + b) * SGB, g, s20, s21);
        v_sel<T>(vq + ((kr + 2 * c + 9) * NBV + b) * QSB, vs + ((kr + 2 * c + 9) * NBV + b) * SGB, g, s30, s31);
        uint32_t lo[16], hi[16];
        dq_pair16<T>(s00, s01, s10, s11, tab_v, lo);     // keys 2c, 2c+1
        dq_pair16<T>(s20, s21, s30, s31, tab_v, hi);     // keys 2c+8, 2c+9
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
          mma16816(oacc[b][mt], lo[2 * mt], lo[2 * mt + 1], hi[2 * mt], hi[2 * mt + 1], pb0, pb1);
      }
      __syncwarp();
    }
    __syncthreads();
    if (tid == 0 && tile + STAGES < n_tiles && !s_timeout) issue(tile + STAGES);
  }

  // ---- per-warp results -> shared memory (reusing the stage buffers), CTA merge
  __syncthreads();
  if (s_timeout) {
    // a bounded wait gave up: report it and leave this split empty (weight 0 in the merge)
    if (tid == 0) set_status(a.status, TQ_ERR_TIMEOUT);
    for (int i = tid; i < G * 128 * NBV; i += NT) {
      const int h = i / (128 * NBV), d = i % (128 * NBV);
      float *part = a.part + (static_cast<size_t>(hk * G + h) * a.n_splits + split) * a.part_stride;
      part[2 + d] = 0.f;
      if (d == 0) { part[0] = -INFINITY; part[1] = 0.f; }
    }
    decode_merge<NT>(a, hk, reinterpret_cast<float *>(stages));
    return;
  }
  float *wm = reinterpret_cast<float *>(stages);                 // [NW][G]
  float *wl = wm + NW * 4;                                      // [NW][G]
  float *wo = wl + NW * 4;                                      // [NW][G][128*NBV]
  constexpr int DVP = 128 * NBV;
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    float l = l_run[j];
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    l_run[j] = l;
  }
  // combine hi/lo output columns
#pragma unroll
  for (int b = 0; b < NBV; ++b)
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float v = oacc[b][mt][i];
        if (G == 4) v += __shfl_xor_sync(0xffffffffu, v, 2);
        else if (G == 2) v += __shfl_xor_sync(0xffffffffu, v, 1);
        oacc[b][mt][i] = v;
      }
  {
    const bool writer = (G == 4) ? (c < 2) : (c == 0);
    const int hA = (G == 4) ? 2 * (c & 1) : 0;
    if (writer) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int h = hA + j;
        if (h < G) {
          if (g == 0) {
            wm[warp * 4 + h] = m_run[j];
            wl[warp * 4 + h] = l_run[j];
          }
#pragma unroll
          for (int b = 0; b < NBV; ++b)
#pragma unroll
            for (int mt = 0; mt < 8; ++mt) {
              // G == 1: columns 0 (hi) and 1 (lo) of head 0
              const float top = (G == 1) ? oacc[b][mt][0] + oacc[b][mt][1] : oacc[b][mt][j];
              const float bot = (G == 1) ? oacc[b][mt][2] + oacc[b][mt][3] : oacc[b][mt][2 + j];
              float *o = wo + (warp * G + h) * DVP + b * 128 + 16 * g + 2 * mt;
              o[0] = top;
              o[1] = bot;
            }
        }
      }
    }
  }
  __syncthreads();
  for (int i = tid; i < G * DVP; i += NT) {
    const int h = i / DVP, d = i % DVP;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, wm[w * 4 + h]);
    float o = 0.f, l = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float f = (wm[w * 4 + h] == -INFINITY) ? 0.f : exp2f(wm[w * 4 + h] - M);
      o += f * wo[(w * G + h) * DVP + d];
      l += f * wl[w * 4 + h];
    }
    float *part = a.part + (static_cast<size_t>(hk * G + h) * a.n_splits + split) * a.part_stride;
    part[2 + d] = o;
    if (d == 0) {
      part[0] = M;
      part[1] = l;
    }
  }
  decode_merge<NT>(a, hk, wo + NW * G * DVP);
}

template <int T, int G, int NBK, int NBV>
cudaError_t launch_one(const DecodeArgs &a, cudaStream_t s) {
  constexpr uint32_t bytes = smem_bytes<T, G, NBK, NBV>();
  static_assert(bytes <= 227 * 1024, "shared memory");
  // the epilogue reuses the stage buffers: per-warp results + the split merge (<= 256 splits)
  static_assert(STAGES * stage_layout<T, NBK, NBV>().bytes >=
                    4 * (2 * NW * 4 + NW * G * 128 * NBV + 2 * G * 128 * NBV + 2 * G * 256),
                "stage buffers too small for the epilogue");
  cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<T, G, NBK, NBV>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e != cudaSuccess) return e;
  dim3 grid(a.n_splits, a.n_kv_heads);
  decode_mma_kernel<T, G, NBK, NBV><<<grid, NT, bytes, s>>>(a);
  return cudaGetLastError();
}

template <int T>
cudaError_t launch_type(const DecodeArgs &a, cudaStream_t s) {
#define TQ_DEC_CASE(GG, BK, BV) \
  if (a.group == GG && a.nbk == BK && a.nbv == BV) return launch_one<T, GG, BK, BV>(a, s);
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

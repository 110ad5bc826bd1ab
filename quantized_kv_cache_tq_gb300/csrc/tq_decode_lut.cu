// Single-query decode attention through a per-step Q x centroid shared-memory
// table ([TQ#36] "Q x centroid LUT"): LUT_g[d][c] = q'_g[d] * centroid[c] is
// built once per CTA, so each K element costs one shared-memory read per query
// head; rows of the table are n_centroids + 1 floats apart as on the page.
// Unlike the page (no table for turbo4), GB300's 227 KB of shared memory holds
// the 16-entry turbo4 table too.
//
// Work split: grid (n_splits, n_kv_heads); a CTA scans one contiguous key range
// of one KV head for all query heads of its GQA group, one key per thread per
// 256-key tile, keeps a running max / sum per head (online softmax, log2
// domain), accumulates V in the rotated domain from packed codes staged in
// shared memory, and hands its partial to the split merge.
#include "tq_decode_common.cuh"

namespace tq {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 256;
constexpr int kMaxG = 8;

struct LutSmem {
  // byte offsets into dynamic shared memory
  size_t qrot, lut, sp, vqs, vsg, vnorm, red, acc, vtab, total;
};

template <int KT, int VT>
__host__ __device__ inline LutSmem lut_smem(int group, int nbk, int nbv) {
  constexpr int KNC = TypeTraits<KT>::NC;
  constexpr int VQSB = TypeTraits<VT>::QSB, VSGB = TypeTraits<VT>::SGB;
  LutSmem s;
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o += (bytes + 15) & ~size_t(15); return r; };
  s.qrot = take(sizeof(float) * group * QK * nbk);
  s.lut = take(sizeof(float) * group * QK * nbk * (KNC + 1));
  s.sp = take(sizeof(float) * group * kTile);
  s.vqs = take(size_t(kTile) * nbv * VQSB);
  s.vsg = take(size_t(kTile) * nbv * (VSGB ? VSGB : 16));
  s.vnorm = take(sizeof(uint16_t) * kTile * nbv);
  s.red = take(sizeof(float) * 2 * (kThreads / 32) * kMaxG);
  s.acc = take(sizeof(float) * group * QK * 2);
  s.vtab = take(sizeof(float) * 16);
  s.total = o;
  return s;
}

template <int KT, int VT>
__global__ void __launch_bounds__(kThreads) decode_lut_kernel(const DecodeArgs a) {
  constexpr int KNC = TypeTraits<KT>::NC, KQSB = TypeTraits<KT>::QSB, KSGB = TypeTraits<KT>::SGB;
  constexpr int VNC = TypeTraits<VT>::NC, VQSB = TypeTraits<VT>::QSB, VSGB = TypeTraits<VT>::SGB;
  (void)VNC;
  extern __shared__ __align__(16) unsigned char smem[];
  const LutSmem L = lut_smem<KT, VT>(a.group, a.nbk, a.nbv);
  float *qrot = reinterpret_cast<float *>(smem + L.qrot);
  float *lut = reinterpret_cast<float *>(smem + L.lut);
  float *sp = reinterpret_cast<float *>(smem + L.sp);
  uint8_t *vqs_s = smem + L.vqs;
  uint8_t *vsg_s = smem + L.vsg;
  uint16_t *vn_s = reinterpret_cast<uint16_t *>(smem + L.vnorm);
  float *red = reinterpret_cast<float *>(smem + L.red);
  float *accbuf = reinterpret_cast<float *>(smem + L.acc);
  float *vtab = reinterpret_cast<float *>(smem + L.vtab);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int hk = blockIdx.y, split = blockIdx.x;
  const int G = a.group;
  const int dkp = QK * a.nbk, dvp = QK * a.nbv;
  const int64_t t0 = static_cast<int64_t>(split) * a.chunk;
  const int64_t t1 = min(a.kv_len, t0 + a.chunk);

  // 1. rotated, pre-scaled queries and the Q x centroid table
  __shared__ uint32_t s_epoch;
  __shared__ int s_last;
  if (tid == 0) s_epoch = load_epoch(a, hk);
  rotate_queries<kThreads>(a, hk, qrot);
  if (tid < 16) vtab[tid] = (tid < a.cbv.n) ? code_value(a.cbv.c, a.cbv.n, tid) : 0.f;
  __syncthreads();
  for (int i = tid; i < G * dkp * KNC; i += kThreads) {
    const int k = i % KNC, gd = i / KNC;
    lut[gd * (KNC + 1) + k] = qrot[gd] * code_value(a.cbk.c, KNC, k);
  }
  __syncthreads();

  // V accumulation layout: thread owns rotated coordinate d, key residue kr
  const int n_kr = kThreads / dvp;          // 2 for dv <= 128, 1 for dv <= 256
  const int d = tid % dvp, kr = tid / dvp;
  const int vb = d / QK, ve = d % QK;
  float acc[kMaxG], m_run[kMaxG], l_run[kMaxG];
#pragma unroll
  for (int g = 0; g < kMaxG; ++g) { acc[g] = 0.f; m_run[g] = -INFINITY; l_run[g] = 0.f; }

  const uint16_t *kn = a.kn + static_cast<size_t>(hk) * a.n_cells * a.nbk;
  const uint8_t *kqs = a.kqs + static_cast<size_t>(hk) * a.n_cells * a.nbk * KQSB;
  const uint8_t *ksg = KSGB ? a.ksg + static_cast<size_t>(hk) * a.n_cells * a.nbk * KSGB : nullptr;
  const uint16_t *vn = a.vn + static_cast<size_t>(hk) * a.n_cells * a.nbv;
  const uint8_t *vqs = a.vqs + static_cast<size_t>(hk) * a.n_cells * a.nbv * VQSB;
  const uint8_t *vsg = VSGB ? a.vsg + static_cast<size_t>(hk) * a.n_cells * a.nbv * VSGB : nullptr;

  for (int64_t tt = t0; tt < t1; tt += kTile) {
    const int tile_n = (t1 - tt < kTile) ? static_cast<int>(t1 - tt) : kTile;
    const bool valid = tid < tile_n;

    // 2. scores of this thread's key: s_g = sum_b n_b * sum_e LUT_g[e][code_e]
    float sc[kMaxG];
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) sc[g] = valid ? 0.f : -INFINITY;
    if (valid) {
      const int64_t key = tt + tid;
      for (int b = 0; b < a.nbk; ++b) {
        const int64_t blk = key * a.nbk + b;
        const float nrm = __half2float(__ushort_as_half(kn[blk]));
        uint32_t w[KQSB / 4], s[4];
#pragma unroll
        for (int i = 0; i < KQSB / 16; ++i) {
          const uint4 x = reinterpret_cast<const uint4 *>(kqs + blk * KQSB)[i];
          w[4 * i] = x.x; w[4 * i + 1] = x.y; w[4 * i + 2] = x.z; w[4 * i + 3] = x.w;
        }
        if (KSGB) {
          const uint4 x = *reinterpret_cast<const uint4 *>(ksg + blk * KSGB);
          s[0] = x.x; s[1] = x.y; s[2] = x.z; s[3] = x.w;
        }
        float part[kMaxG];
#pragma unroll
        for (int g = 0; g < kMaxG; ++g) part[g] = 0.f;
        const float *lb = lut + static_cast<size_t>(b) * QK * (KNC + 1);
#pragma unroll
        for (int e = 0; e < QK; ++e) {
          int k;
          if (KT == 4) {
            k = (w[e >> 3] >> (4 * (e & 7))) & 15;
          } else {
            const int r = e & 15;
            k = (w[e >> 4] >> ((r < 8) ? 4 * r : 4 * (r - 8) + 2)) & 3;
            if (KT == 3) {
              const int rr = e & 31;
              const int sb = (rr < 16) ? 4 * (rr & 7) + 2 + (rr >> 3) : 4 * ((rr - 16) & 7) + ((rr - 16) >> 3);
              k |= ((s[e >> 5] >> sb) & 1) << 2;
            }
          }
#pragma unroll
          for (int g = 0; g < kMaxG; ++g)
            if (g < G) part[g] += lb[(static_cast<size_t>(g) * dkp + e) * (KNC + 1) + k];
        }
#pragma unroll
        for (int g = 0; g < kMaxG; ++g) sc[g] += nrm * part[g];
      }
    }

    // 3. stage this tile's packed V rows (contiguous per head) in shared memory
    {
      const size_t qs_bytes = static_cast<size_t>(tile_n) * a.nbv * VQSB;
      const uint4 *src = reinterpret_cast<const uint4 *>(vqs + static_cast<size_t>(tt) * a.nbv * VQSB);
      for (size_t i = tid; i < qs_bytes / 16; i += kThreads) reinterpret_cast<uint4 *>(vqs_s)[i] = src[i];
      if (VSGB) {
        const size_t sg_bytes = static_cast<size_t>(tile_n) * a.nbv * VSGB;
        const uint4 *ss = reinterpret_cast<const uint4 *>(vsg + static_cast<size_t>(tt) * a.nbv * VSGB);
        for (size_t i = tid; i < sg_bytes / 16; i += kThreads) reinterpret_cast<uint4 *>(vsg_s)[i] = ss[i];
      }
      for (int i = tid; i < tile_n * a.nbv; i += kThreads) vn_s[i] = vn[tt * a.nbv + i];
    }

    // 4. online softmax over the tile (block-wide max and sum per head)
    float *red_max = red, *red_sum = red + (kThreads / 32) * kMaxG;
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) {
      const float wm = warp_max(sc[g]);
      if (lane == 0) red_max[warp * kMaxG + g] = wm;
    }
    __syncthreads();
    float alpha[kMaxG];
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) {
      float tm = -INFINITY;
      for (int w = 0; w < kThreads / 32; ++w) tm = fmaxf(tm, red_max[w * kMaxG + g]);
      const float mnew = fmaxf(m_run[g], tm);
      alpha[g] = (g < G) ? exp2f(m_run[g] - mnew) : 0.f;
      m_run[g] = mnew;
      const float p = (valid && g < G) ? exp2f(sc[g] - mnew) : 0.f;
      if (g < G) sp[g * kTile + tid] = p;
      const float ws = warp_sum(p);
      if (lane == 0) red_sum[warp * kMaxG + g] = ws;
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < kMaxG; ++g) {
      float ts = 0.f;
      for (int w = 0; w < kThreads / 32; ++w) ts += red_sum[w * kMaxG + g];
      l_run[g] = l_run[g] * alpha[g] + ts;
      acc[g] *= alpha[g];
    }

    // 5. o'_g[d] += p_g(t) * n_t * c[code_{t,d}]; with sparse V a key whose
    // weights (relative to the running maximum) are all below the threshold
    // adds nothing
    for (int kk = kr; kk < tile_n; kk += n_kr) {
      if (a.v_thresh > 0.f) {
        bool keep = false;
        for (int g = 0; g < G; ++g) keep = keep || sp[g * kTile + kk] >= a.v_thresh;
        if (!keep) continue;
      }
      const int blk = kk * a.nbv + vb;
      const float nrm = __half2float(__ushort_as_half(vn_s[blk]));
      const int code = load_code<VT>(vqs_s + static_cast<size_t>(blk) * VQSB,
                                     vsg_s + static_cast<size_t>(blk) * (VSGB ? VSGB : 16), ve);
      const float val = nrm * vtab[code];
#pragma unroll
      for (int g = 0; g < kMaxG; ++g)
        if (g < G) acc[g] += sp[g * kTile + kk] * val;
    }
    __syncthreads();
  }

  // 6. combine key residues and store this split's partials
  if (n_kr > 1) {
    if (kr == 1)
      for (int g = 0; g < G; ++g) accbuf[g * dvp + d] = acc[g];
    __syncthreads();
    if (kr == 0)
      for (int g = 0; g < G; ++g) acc[g] += accbuf[g * dvp + d];
  }
  int prev = 0;
  if (!a.coop && tid == 0) prev = split_arrive(a, hk);
  const uint32_t epoch = s_epoch, tag = split_tag(epoch, hk);
  if (kr == 0) {
    for (int g = 0; g < G; ++g) {
      store_partial_o(a, hk * G + g, split, d, acc[g], tag);
      if (d == 0) store_partial_ml(a, hk * G + g, split, m_run[g], l_run[g], tag);
    }
  }
  if (a.coop) {
    __syncthreads();                      // the table region becomes the merge buffer
    if (tid < 128) coop_merge(a, hk, split, epoch, lut);
    return;
  }
  if (tid == 0) s_last = (prev == a.n_splits - 1);
  __syncthreads();
  if (s_last) decode_merge<kThreads>(a, hk, epoch, lut);
}

template <int KT, int VT>
cudaError_t launch_kt_vt(const DecodeArgs &a, cudaStream_t s) {
  const LutSmem L = lut_smem<KT, VT>(a.group, a.nbk, a.nbv);
  // the merge reuses the table region: it must hold group * 128 * nbv floats
  size_t bytes = L.total;
  const size_t merge_need = L.lut + sizeof(float) * merge_smem_floats(a.group, a.nbv, a.n_splits);
  if (merge_need > bytes) bytes = merge_need;
  cudaError_t e = set_dynamic_smem(reinterpret_cast<const void *>(decode_lut_kernel<KT, VT>), (int)bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.n_splits, a.n_kv_heads);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (a.coop) {                           // every CTA resident: each merges a share (coop_merge)
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  e = cudaLaunchKernelEx(&cfg, decode_lut_kernel<KT, VT>, a);
  if (e == cudaErrorCooperativeLaunchTooLarge) {          // fewer SMs available than the device has
    cudaGetLastError();
    DecodeArgs b = a;
    b.coop = 0;
    cfg.numAttrs = 0;
    e = cudaLaunchKernelEx(&cfg, decode_lut_kernel<KT, VT>, b);
  }
  return e == cudaSuccess ? cudaGetLastError() : e;
}

template <int KT>
cudaError_t launch_kt(int vtype, const DecodeArgs &a, cudaStream_t s) {
  switch (vtype) {
    case TQ_TURBO2: return launch_kt_vt<KT, 2>(a, s);
    case TQ_TURBO3: return launch_kt_vt<KT, 3>(a, s);
    default: return launch_kt_vt<KT, 4>(a, s);
  }
}

}  // namespace

size_t decode_lut_max_group() { return kMaxG; }

cudaError_t launch_decode_lut(int ktype, int vtype, const DecodeArgs &a, cudaStream_t s) {
  switch (ktype) {
    case TQ_TURBO2: return launch_kt<2>(vtype, a, s);
    case TQ_TURBO3: return launch_kt<3>(vtype, a, s);
    default: return launch_kt<4>(vtype, a, s);
  }
}

}  // namespace tq

// Split-KV bookkeeping shared by the decode kernels: the log-sum-exp merge of
// the per-split partials and the inverse rotation of the merged output.
#pragma once

#include "tq_common.cuh"

namespace tq {

// 2^x for x <= 0 (split weights), approximate to a few ulp.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Floats of shared memory decode_merge needs.
__host__ __device__ inline int merge_smem_floats(int group, int nbv, int n_splits) {
  return group * QK * nbv + 2 * group * n_splits;
}

// Called by every CTA of a decode grid after it stored its partials.  The last
// CTA to arrive for KV head `hk` (counter in the workspace) merges the splits:
//   M = max_s m_s,  L = sum_s l_s 2^(m_s - M),  o' = sum_s o'_s 2^(m_s - M) / L
// (scores are kept in the log2 domain), rotates back with the V codebook,
//   o = S H o' / sqrt(128)   (R^T for R = H S / sqrt(128)),
// writes out[h][0 .. dv) and resets the counter so the next launch (or graph
// replay) finds it at zero.  No CTA ever waits for another one.
// Each warp merges 32 consecutive outputs of one head, 24 splits at a time:
// lane s < 24 holds split s's maximum and sum, every lane loads its output's
// values of the 24 splits at once (one L2 round trip per 24 splits).
// `smem` must hold merge_smem_floats(group, nbv, n_splits) floats.
template <int NT>
__device__ void decode_merge(const DecodeArgs &a, int hk, float *smem) {
  __shared__ int s_last;
  // the CTA's partial stores are ordered before the counter update by the CTA
  // barrier and the release half of thread 0's acq_rel atomic; its acquire half
  // orders the last CTA's loads of the other partials after it
  __syncthreads();
  if (threadIdx.x == 0) {
    int prev;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(prev) : "l"(a.counters + hk) : "memory");
    s_last = (prev == a.n_splits - 1);
  }
  __syncthreads();
  if (!s_last) return;

  const int G = a.group, ns = a.n_splits, dvp = QK * a.nbv;
  const int stride = a.part_stride;
  float *orot = smem;                     // [G][dvp]
  const float *base = a.part + static_cast<size_t>(hk) * G * ns * stride;
  const float *base_ml = a.part_ml + static_cast<size_t>(hk) * G * ns * 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i0 = warp * 32; i0 < G * dvp; i0 += NT) {     // dvp is a multiple of 32: one head per warp pass
    const int i = i0 + lane, g = i / dvp, d = i % dvp;
    const float *p = base + static_cast<size_t>(g) * ns * stride;
    const float *pml = base_ml + static_cast<size_t>(g) * ns * 2;
    float M = -INFINITY, L = 0.f, o = 0.f;
    for (int s0 = 0; s0 < ns; s0 += 24) {
      const int n = min(24, ns - s0);
      const float *ps = p + static_cast<size_t>(s0) * stride;
      float2 ml = make_float2(-INFINITY, 0.f);
      if (lane < n) ml = __ldcg(reinterpret_cast<const float2 *>(pml) + s0 + lane);
      const float ms = ml.x, ls = ml.y;
      float ov[24];
#pragma unroll
      for (int j = 0; j < 24; ++j) ov[j] = (j < n) ? __ldcg(ps + static_cast<size_t>(j) * stride + d) : 0.f;
      const float Mn = fmaxf(M, warp_max(ms));
      const float f = (M == -INFINITY) ? 0.f : fast_exp2(M - Mn);
      const float w = (ms == -INFINITY) ? 0.f : fast_exp2(ms - Mn);
      L = L * f + warp_sum(w * ls);
      o *= f;
#pragma unroll
      for (int j = 0; j < 24; ++j) o = fmaf(__shfl_sync(0xffffffffu, w, j), ov[j], o);
      M = Mn;
    }
    orot[i] = (L > 0.f) ? o / L : 0.f;
  }
  __syncthreads();

  for (int wb = warp; wb < G * a.nbv; wb += NT / 32) {
    const int g = wb / a.nbv, b = wb % a.nbv;
    float v[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) v[r] = orot[g * dvp + b * QK + 4 * lane + r];
    wht128_warp(v, lane);
#pragma unroll
    for (int r = 0; r < 4; ++r) v[r] *= kInvSqrtQK;
    apply_signs(v, a.cbv, lane);
    const int h = hk * G + g;
    float *o = a.out + static_cast<size_t>(h) * a.dv;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int d = b * QK + 4 * lane + r;
      if (d < a.dv) o[d] = v[r];
    }
  }
  if (threadIdx.x == 0) a.counters[hk] = 0;
}

// Query block wb = g * nbk + b (head hk * group + g, dims 128 b ..): lane i
// loads dims 4i .. 4i+3 of the block, zero beyond dk.
__device__ __forceinline__ void load_query_block(const DecodeArgs &a, int hk, int wb, int lane, float v[4]) {
  const int g = wb / a.nbk, b = wb % a.nbk;
  const float *q = a.q + static_cast<size_t>(hk * a.group + g) * a.dk;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int d = b * QK + 4 * lane + r;
    v[r] = (d < a.dk) ? q[d] : 0.f;
  }
}

// Rotate a loaded query block into the K codebook's domain and fold in the
// softmax scale:  q'_g = scale * log2(e) * H S q_g / sqrt(128).
// Writes qrot[g * 128*nbk + d].
__device__ __forceinline__ void rotate_query_block(const DecodeArgs &a, int wb, int lane, float v[4], float *qrot) {
  const int g = wb / a.nbk, b = wb % a.nbk;
  const float f = a.scale_log2 * kInvSqrtQK;
  apply_signs(v, a.cbk, lane);
  wht128_warp(v, lane);
#pragma unroll
  for (int r = 0; r < 4; ++r) qrot[g * QK * a.nbk + b * QK + 4 * lane + r] = v[r] * f;
}

// All query heads of KV head hk, one block per warp at a time.
template <int NT>
__device__ void rotate_queries(const DecodeArgs &a, int hk, float *qrot) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int wb = warp; wb < a.group * a.nbk; wb += NT / 32) {
    float v[4];
    load_query_block(a, hk, wb, lane, v);
    rotate_query_block(a, wb, lane, v, qrot);
  }
}

}  // namespace tq

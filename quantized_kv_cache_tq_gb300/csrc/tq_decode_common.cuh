// Split-KV bookkeeping shared by the decode kernels: the log-sum-exp merge of
// the per-split partials and the inverse rotation of the merged output.
#pragma once

#include "tq_common.cuh"

namespace tq {

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
// The split maxima and sums are staged in shared memory first and the partial
// outputs are read with independent loads, so the merge costs a few L2 round
// trips.  `smem` must hold merge_smem_floats(group, nbv, n_splits) floats.
template <int NT>
__device__ void decode_merge(const DecodeArgs &a, int hk, float *smem) {
  __shared__ int s_last;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(&a.counters[hk], 1);
    s_last = (prev == a.n_splits - 1);
  }
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const int G = a.group, ns = a.n_splits, dvp = QK * a.nbv;
  const int stride = a.part_stride;
  float *orot = smem;                     // [G][dvp]
  float *wt = smem + G * dvp;             // [G][ns]: m_s, then the weights
  float *ls = wt + G * ns;                // [G][ns]
  const float *base = a.part + static_cast<size_t>(hk) * G * ns * stride;
  for (int i = threadIdx.x; i < G * ns; i += NT) {
    wt[i] = __ldcg(base + static_cast<size_t>(i) * stride);
    ls[i] = __ldcg(base + static_cast<size_t>(i) * stride + 1);
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int g = warp; g < G; g += NT / 32) {
    float M = -INFINITY;
    for (int s = lane; s < ns; s += 32) M = fmaxf(M, wt[g * ns + s]);
    M = warp_max(M);
    float L = 0.f;
    for (int s = lane; s < ns; s += 32) {
      const float m = wt[g * ns + s];
      L += (m == -INFINITY) ? 0.f : ls[g * ns + s] * exp2f(m - M);
    }
    L = warp_sum(L);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    __syncwarp();
    for (int s = lane; s < ns; s += 32) {
      const float m = wt[g * ns + s];
      wt[g * ns + s] = (m == -INFINITY) ? 0.f : exp2f(m - M) * inv;
    }
  }
  __syncthreads();
  for (int i = threadIdx.x; i < G * dvp; i += NT) {
    const int g = i / dvp, d = i % dvp;
    const float *p = base + static_cast<size_t>(g) * ns * stride + 2 + d;
    const float *w = wt + g * ns;
    float o = 0.f;
    int s = 0;
    for (; s + 8 <= ns; s += 8) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = __ldcg(p + static_cast<size_t>(s + j) * stride);
#pragma unroll
      for (int j = 0; j < 8; ++j) o += w[s + j] * v[j];
    }
    for (; s < ns; ++s) o += w[s] * __ldcg(p + static_cast<size_t>(s) * stride);
    orot[i] = o;
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

// Rotate the query heads of KV head hk into the K codebook's domain and fold in
// the softmax scale:  q'_g = scale * log2(e) * H S q_g / sqrt(128), per block.
// Zero-pads q beyond dk.  Writes qrot[g * 128*nbk + d].
template <int NT>
__device__ void rotate_queries(const DecodeArgs &a, int hk, float *qrot) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int dkp = QK * a.nbk;
  const float f = a.scale_log2 * kInvSqrtQK;
  for (int wb = warp; wb < a.group * a.nbk; wb += NT / 32) {
    const int g = wb / a.nbk, b = wb % a.nbk;
    const float *q = a.q + static_cast<size_t>(hk * a.group + g) * a.dk;
    float v[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int d = b * QK + 4 * lane + r;
      v[r] = (d < a.dk) ? q[d] : 0.f;
    }
    apply_signs(v, a.cbk, lane);
    wht128_warp(v, lane);
#pragma unroll
    for (int r = 0; r < 4; ++r) qrot[g * dkp + b * QK + 4 * lane + r] = v[r] * f;
  }
}

}  // namespace tq

// Split-KV bookkeeping shared by the decode kernels: the log-sum-exp merge of
// the per-split partials and the inverse rotation of the merged output.
#pragma once

#include "tq_common.cuh"

namespace tq {

// Called by every CTA of a decode grid after it stored its partials.  The last
// CTA to arrive for KV head `hk` (counter in the workspace) merges the splits:
//   M = max_s m_s,  L = sum_s l_s 2^(m_s - M),  o' = sum_s o'_s 2^(m_s - M) / L
// (scores are kept in the log2 domain), rotates back with the V codebook,
//   o = S H o' / sqrt(128)   (R^T for R = H S / sqrt(128)),
// writes out[h][0 .. dv) and resets the counter so the next launch (or graph
// replay) finds it at zero.  No CTA ever waits for another one.
// `smem` must hold group * 128 * nbv floats.
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

  const int dvp = QK * a.nbv;
  const int stride = a.part_stride;
  for (int g = 0; g < a.group; ++g) {
    const int h = hk * a.group + g;
    const float *p = a.part + static_cast<size_t>(h) * a.n_splits * stride;
    float M = -INFINITY;
    for (int s = 0; s < a.n_splits; ++s) M = fmaxf(M, __ldcg(p + static_cast<size_t>(s) * stride));
    float L = 0.f;
    for (int s = 0; s < a.n_splits; ++s) {
      const float *ps = p + static_cast<size_t>(s) * stride;
      L += __ldcg(ps + 1) * exp2f(__ldcg(ps) - M);
    }
    const float invL = 1.f / L;
    for (int d = threadIdx.x; d < dvp; d += NT) {
      float o = 0.f;
      for (int s = 0; s < a.n_splits; ++s) {
        const float *ps = p + static_cast<size_t>(s) * stride;
        o += __ldcg(ps + 2 + d) * exp2f(__ldcg(ps) - M);
      }
      smem[g * dvp + d] = o * invL;
    }
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int wb = warp; wb < a.group * a.nbv; wb += NT / 32) {
    const int g = wb / a.nbv, b = wb % a.nbv;
    float v[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) v[r] = smem[g * dvp + b * QK + 4 * lane + r];
    wht128_warp(v, lane);
#pragma unroll
    for (int r = 0; r < 4; ++r) v[r] *= kInvSqrtQK;
    apply_signs(v, a.cbv, lane);
    const int h = hk * a.group + g;
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

// Merge of the key-range splits of a prefill launch ([HIP#28] "2. Inline-dequant
// TILE prefill"; the splits are this library's way to fill the SMs when few query
// tiles are in flight).  Split s of a query tile left, for each of its 128 rows,
//   (m_s, l_s, O'_s)   running maximum (log2 domain), sum of weights, unnormalised O'
// in the workspace.  Here, after the prefill kernel:
//   M = max_s m_s,  o' = sum_s 2^(m_s - M) O'_s / sum_s 2^(m_s - M) l_s,
// then the inverse rotation of each 128-dim V block (o = S H o' / sqrt(128)) and the
// store of out[query][head].
//
// A block takes 8 rows of one query tile, so that the tiles' partials are read by
// many SMs at once; every thread issues the loads of all splits of its four
// columns before it uses any.
#include "tq_common.cuh"
#include "tq_internal.h"

namespace tq {
namespace pfm {

constexpr int BM = 128;         // rows of a query tile (the prefill kernel's)
constexpr int RB = 8;           // rows per block
constexpr int NT = 128;
constexpr int MAXS = 16;        // at most 16 splits (the prefill layout's bound)

template <int NBV>
__global__ void __launch_bounds__(NT) prefill_merge_kernel(const PrefillArgs a) {
  constexpr int DVP = 128 * NBV, STRIDE = 4 + DVP;     // m, l, 2 pad floats, O' (16-byte aligned rows)
  const int tile_id = blockIdx.x;                       // query tile * n_kv_heads + KV head
  const int qt = tile_id / a.n_kv_heads, hk = tile_id % a.n_kv_heads;
  const int G = a.group, g_shift = __ffs(G) - 1;
  const int q0 = qt * (BM / G);
  const int rows_valid = min(BM, (a.nq - q0) * G);     // rows of queries < nq
  const int r0 = blockIdx.y * RB;
  if (r0 >= rows_valid) return;
  const int ns = a.n_split;
  const float *base = a.part + static_cast<size_t>(tile_id) * ns * BM * STRIDE;
  __shared__ float s_w[RB][MAXS];                        // weights / L / sqrt(128)
  __shared__ __align__(16) float s_o[RB][DVP];
  const int t = threadIdx.x, warp = t >> 5, lane = t & 31;

  if (t < RB) {
    const int r = r0 + t;
    float ms[MAXS], ls[MAXS];
#pragma unroll
    for (int s = 0; s < MAXS; ++s) {
      ms[s] = -INFINITY;
      ls[s] = 0.f;
      if (s < ns) {
        const float2 ml = __ldcg(reinterpret_cast<const float2 *>(base + (static_cast<size_t>(s) * BM + r) * STRIDE));
        ms[s] = ml.x;
        ls[s] = ml.y;
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < MAXS; ++s) M = fmaxf(M, ms[s]);
    float L = 0.f;
#pragma unroll
    for (int s = 0; s < MAXS; ++s) {
      ms[s] = (ms[s] == -INFINITY) ? 0.f : exp2f(ms[s] - M);      // a split with no visible key weighs 0
      L = fmaf(ms[s], ls[s], L);
    }
    const float inv = (L > 0.f ? 1.f / L : 0.f) * kInvSqrtQK;
#pragma unroll
    for (int s = 0; s < MAXS; ++s) s_w[t][s] = ms[s] * inv;
  }
  __syncthreads();

  for (int i = t; i < RB * DVP / 4; i += NT) {
    const int rr = i / (DVP / 4), d = 4 * (i % (DVP / 4));
    const int r = r0 + rr;
    float4 x[MAXS];
#pragma unroll
    for (int s = 0; s < MAXS; ++s)
      if (s < ns) x[s] = __ldcg(reinterpret_cast<const float4 *>(base + (static_cast<size_t>(s) * BM + r) * STRIDE + 4 + d));
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < MAXS; ++s)
      if (s < ns) {
        const float w = s_w[rr][s];
        o.x = fmaf(w, x[s].x, o.x);
        o.y = fmaf(w, x[s].y, o.y);
        o.z = fmaf(w, x[s].z, o.z);
        o.w = fmaf(w, x[s].w, o.w);
      }
    *reinterpret_cast<float4 *>(&s_o[rr][d]) = o;
  }
  __syncthreads();

  // inverse rotation of each (row, V block) by one warp, then the store
  for (int u = warp; u < RB * NBV; u += NT / 32) {
    const int rr = u / NBV, b = u % NBV, r = r0 + rr;
    if (r >= rows_valid) continue;                       // warp-uniform
    float v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = s_o[rr][b * QK + 4 * lane + k];
    wht128_warp(v, lane);
    apply_signs(v, a.cbv, lane);
    const int d = b * QK + 4 * lane;
    if (d + 4 <= a.dv) {
      float *o = a.out + (static_cast<size_t>(q0 + (r >> g_shift)) * a.n_q_heads + hk * G + (r & (G - 1))) * a.dv + d;
      *reinterpret_cast<float4 *>(o) = make_float4(v[0], v[1], v[2], v[3]);
    }
  }
}

}  // namespace pfm

cudaError_t launch_prefill_merge(const PrefillArgs &a, cudaStream_t s) {
  if (a.n_split < 2) return cudaSuccess;
  if (a.n_split > pfm::MAXS) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(a.n_qt) * a.n_kv_heads, pfm::BM / pfm::RB);
  if (a.nbv == 2) pfm::prefill_merge_kernel<2><<<grid, pfm::NT, 0, s>>>(a);
  else pfm::prefill_merge_kernel<1><<<grid, pfm::NT, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace tq

// Device helpers shared by the kernels of the tq library (sm_103a).
//
// Page tags used in comments (page title -- section):
//   [TQ#36]    llama-cpp-turboquant PR #36 -- commits "shuffle WHT",
//              "asymmetric D", "Q x centroid LUT", "VEC tuning"
//   [HIP#28]   atomic-llama-cpp-turboquant PR #28 "HIP/turbo3: graph-safe decode +
//              inline-dequant TILE prefill" -- "1. Graph-safe decode",
//              "2. Inline-dequant TILE prefill", "Correctness"
//   [QSA#1821] "qsa_prompt_attn: int8 K/V prefetched in registers and sharing one
//              buffer" -- "What", "Why", "Change"
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "tq_internal.h"

namespace tq {

constexpr int QK = 128;            // elements per quantisation block
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kInvSqrtQK = 0.08838834764831845f;   // 1/sqrt(128)

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, m));
  return v;
}

__device__ __forceinline__ uint32_t warp_or(uint32_t v, int width) {
  for (int m = 1; m < width; m <<= 1) v |= __shfl_xor_sync(0xffffffffu, v, m);
  return v;
}

// Sign word covering elements 32*(lane/8) .. +31 of a 128-element block.
__device__ __forceinline__ uint32_t sign_word_for_lane(const DevCodebook &cb, int lane) {
  const int w = lane >> 3;
  uint32_t s = cb.sign_bits[0];
  s = (w == 1) ? cb.sign_bits[1] : s;
  s = (w == 2) ? cb.sign_bits[2] : s;
  s = (w == 3) ? cb.sign_bits[3] : s;
  return s;
}

// Multiply the 4 elements a lane holds (elements 4*lane + r) by the +-1 signs.
__device__ __forceinline__ void apply_signs(float v[4], const DevCodebook &cb, int lane) {
  const uint32_t w = sign_word_for_lane(cb, lane) >> ((4 * lane) & 31);
#pragma unroll
  for (int r = 0; r < 4; ++r)
    if ((w >> r) & 1u) v[r] = -v[r];
}

// Unnormalised 128-point Walsh-Hadamard transform of one block spread over a
// warp, 4 consecutive elements per lane (element 4*lane + r in v[r]).
// [TQ#36] "shuffle WHT": for stage h element j takes o = x[j^h] and becomes
// (j & h) ? o - x[j] : x[j] + o.  Stages h = 1, 2 pair elements inside one lane;
// h = 4..64 pair lanes lane^(h/4), exchanged with shuffles -- a 128-element block
// fits one warp, so no stage needs shared memory or a barrier.
__device__ __forceinline__ void wht128_warp(float v[4], int lane) {
  const float a0 = v[0] + v[1], a1 = v[0] - v[1];
  const float a2 = v[2] + v[3], a3 = v[2] - v[3];
  v[0] = a0 + a2;
  v[2] = a0 - a2;
  v[1] = a1 + a3;
  v[3] = a1 - a3;
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const float o = __shfl_xor_sync(0xffffffffu, v[r], m);
      v[r] = (lane & m) ? (o - v[r]) : (v[r] + o);
    }
  }
}

// Value of sign-magnitude code k: (s ? +1 : -1) * c[n/2 + j], k = s*(n/2) + j.
__device__ __forceinline__ float code_value(const float *c, int n, int k) {
  const int half = n >> 1;
  const float mag = c[half + (k & (half - 1))];
  return (k & half) ? mag : -mag;
}

// Code of element e (0..127) of one block from its qs row (and turbo3 signs row).
template <int TYPE>
__device__ __forceinline__ int load_code(const uint8_t *qs, const uint8_t *sg, int e) {
  if (TYPE == 4) {
    const uint32_t w = reinterpret_cast<const uint32_t *>(qs)[e >> 3];
    return (w >> (4 * (e & 7))) & 15u;
  } else {
    const uint32_t w = reinterpret_cast<const uint32_t *>(qs)[e >> 4];
    const int r = e & 15;
    const int bit = (r < 8) ? 4 * r : 4 * (r - 8) + 2;
    int k = (w >> bit) & 3u;
    if (TYPE == 3) {
      const uint32_t s = reinterpret_cast<const uint32_t *>(sg)[e >> 5];
      const int rr = e & 31;
      const int sb = (rr < 16) ? 4 * (rr & 7) + 2 + (rr >> 3) : 4 * ((rr - 16) & 7) + ((rr - 16) >> 3);
      k |= ((s >> sb) & 1u) << 2;
    }
    return k;
  }
}

template <int TYPE> struct TypeTraits;
template <> struct TypeTraits<2> { static constexpr int NC = 4, QSB = 32, SGB = 0; };
template <> struct TypeTraits<3> { static constexpr int NC = 8, QSB = 32, SGB = 16; };
template <> struct TypeTraits<4> { static constexpr int NC = 16, QSB = 64, SGB = 0; };

__device__ __forceinline__ void set_status(int32_t *st, int32_t code) {
  if (st) atomicCAS(st, 0, code);
}

}  // namespace tq

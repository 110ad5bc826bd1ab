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

// Two fp32 values per instruction (the f32x2 forms of add, sub and mul on sm_100 and
// later).  Each half is rounded to nearest exactly as the scalar operation, so a
// packed computation gives the same bits as the scalar one; what it saves is issue
// slots.  No multiply is fused into an add here.
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  float2 r;
  asm("{\n .reg .b64 x, y, z;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n"
      " sub.rn.f32x2 z, x, y;\n mov.b64 {%0, %1}, z;\n}"
      : "=f"(r.x), "=f"(r.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return r;
}
// max of three (one instruction on sm_100 and later; exact, like two fmaxf)
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
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


__device__ __forceinline__ uint32_t prmt_b32(uint32_t a, uint32_t b, uint32_t s) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(s));
  return d;
}

// ---- register dequantisation of packed codes into binary16 values
// A code nibble (3 bits for turbo2/3, 4 bits for turbo4) is used as a prmt
// byte selector into tables holding the low / high bytes of the binary16 code
// values, so four codes become two half2 registers in 4 byte permutes.
// Byte tables of the binary16 code values: l0/l1 low bytes of values 0..3 / 4..7,
// h0/h1 the high bytes.  turbo2/3: value of code k; turbo4: magnitude j (the sign
// is applied separately from bit 3 of the code).
struct Tab {
  uint32_t l0, l1, h0, h1;
};

template <int T>
__device__ __forceinline__ Tab make_tab(const DevCodebook &cb) {
  constexpr int NC = TypeTraits<T>::NC;
  uint32_t v[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    float f = 0.f;
    if (T == 4) f = cb.c[8 + k];
    else if (k < NC) f = code_value(cb.c, NC, k);
    v[k] = __half_as_ushort(__float2half_rn(f));
  }
  Tab t;
  t.l0 = (v[0] & 0xff) | (v[1] & 0xff) << 8 | (v[2] & 0xff) << 16 | (v[3] & 0xff) << 24;
  t.l1 = (v[4] & 0xff) | (v[5] & 0xff) << 8 | (v[6] & 0xff) << 16 | (v[7] & 0xff) << 24;
  t.h0 = (v[0] >> 8) | (v[1] >> 8) << 8 | (v[2] >> 8) << 16 | (v[3] >> 8) << 24;
  t.h1 = (v[4] >> 8) | (v[5] >> 8) << 8 | (v[6] >> 8) << 16 | (v[7] >> 8) << 24;
  return t;
}

// Four codes in the low 16 bits of `sel` (one per nibble) -> two half2 registers
// (code0, code1) and (code2, code3).  prmt reads only bits 15:0 of its selector,
// so the upper half of `sel` may hold anything.
template <int T>
__device__ __forceinline__ void dq4(uint32_t sel, const Tab &t, uint32_t &h01, uint32_t &h23) {
  const uint32_t s = (T == 4) ? (sel & 0x7777u) : sel;      // turbo4: bit 3 is the sign
  const uint32_t lo = prmt_b32(t.l0, t.l1, s);
  uint32_t hi = prmt_b32(t.h0, t.h1, s);
  if (T == 4) hi |= prmt_b32(0x80808080u, 0u, ((sel >> 1) & 0x4444u) | 0x3210u);   // sign bit 3 == 0 -> negative
  h01 = prmt_b32(lo, hi, 0x5140u);
  h23 = prmt_b32(lo, hi, 0x7362u);
}

// turbo2/3 selector words of one 16-element qs word: sel0 = elements 0..7,
// sel1 = elements 8..15, one 3-bit code per nibble.  `sg` is the signs word of
// the 32-element group, `odd` whether the qs word is the second of the group.
template <int T>
__device__ __forceinline__ void sel_words(uint32_t w, uint32_t sg, bool odd, uint32_t &sel0, uint32_t &sel1) {
  sel0 = w & 0x33333333u;
  sel1 = (w >> 2) & 0x33333333u;
  if (T == 3) {
    const uint32_t s0 = odd ? (sg << 2) : sg;
    const uint32_t s1 = odd ? (sg << 1) : (sg >> 1);
    sel0 |= s0 & 0x44444444u;
    sel1 |= s1 & 0x44444444u;
  }
}

}  // namespace tq

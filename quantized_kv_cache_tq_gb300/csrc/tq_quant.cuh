// Quantisation of one 128-element block by four lanes: the SET_ROWS arithmetic
// ([TQ#36] "shuffle WHT": block norm, sign-randomised Walsh-Hadamard rotation
// with butterfly stages h = 1..64, nearest-centroid codes), shared by the
// SET_ROWS kernel and the decode kernel's append path so both write identical
// bytes.
//
// Four lanes own a block, 32 elements each: lane l4 holds elements
// 4*l4 + 16*i + r (i = 0..7, r = 0..3), read as eight coalesced 16-byte loads,
// so five of the seven butterfly stages (h = 1, 2, 16, 32, 64) stay inside a lane
// and only h = 4, 8 are lane shuffles: no shared memory and no barrier.
//
// The normalisation by the block norm is folded into the decision thresholds:
// with y = v / (|x| sqrt(128)) (v the unnormalised transform), y >= t becomes
// v >= t |x| sqrt(128), one multiply per threshold and block instead of one per
// element.  Codes are sign-magnitude: s = (y >= 0), j = #{positive thresholds
// <= |y|}.  An exact tie goes to the higher centroid.
#pragma once

#include "tq_common.cuh"

namespace tq {

// Four source elements at `off` (fewer when `valid` < 4; the rest read as 0).
template <int SRC>
__device__ __forceinline__ void quant_load4(const void *base, int64_t off, int valid, float v[4]) {
  if (SRC == TQ_F32) {
    const float *p = static_cast<const float *>(base) + off;
    if (valid >= 4) {
      const float4 x = __ldcs(reinterpret_cast<const float4 *>(p));
      v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
    } else {
#pragma unroll
      for (int r = 0; r < 4; ++r) v[r] = (r < valid) ? p[r] : 0.f;
    }
  } else {
    const uint16_t *p = static_cast<const uint16_t *>(base) + off;
    uint16_t h[4] = {0, 0, 0, 0};
    if (valid >= 4) {
      const uint2 x = __ldcs(reinterpret_cast<const uint2 *>(p));
      h[0] = x.x & 0xffff; h[1] = x.x >> 16; h[2] = x.y & 0xffff; h[3] = x.y >> 16;
    } else {
#pragma unroll
      for (int r = 0; r < 4; ++r) h[r] = (r < valid) ? p[r] : 0;
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      if (SRC == TQ_F16) v[r] = __half2float(__ushort_as_half(h[r]));
      else v[r] = __bfloat162float(__ushort_as_bfloat16(h[r]));
    }
  }
}

// The same with the source type chosen at run time.
__device__ __forceinline__ void quant_load4_rt(int src_type, const void *base, int64_t off, int valid, float v[4]) {
  if (src_type == TQ_F32) quant_load4<TQ_F32>(base, off, valid, v);
  else if (src_type == TQ_F16) quant_load4<TQ_F16>(base, off, valid, v);
  else quant_load4<TQ_BF16>(base, off, valid, v);
}

// Four source elements staged in shared memory (16-byte aligned for f32, 8 for
// f16 / bf16), source type chosen at run time.
__device__ __forceinline__ void quant_unpack4_rt(int src_type, const unsigned char *p, float v[4]) {
  if (src_type == TQ_F32) {
    const float4 x = *reinterpret_cast<const float4 *>(p);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  } else {
    const uint2 x = *reinterpret_cast<const uint2 *>(p);
    const uint16_t h[4] = {static_cast<uint16_t>(x.x & 0xffff), static_cast<uint16_t>(x.x >> 16),
                           static_cast<uint16_t>(x.y & 0xffff), static_cast<uint16_t>(x.y >> 16)};
#pragma unroll
    for (int r = 0; r < 4; ++r)
      v[r] = (src_type == TQ_F16) ? __half2float(__ushort_as_half(h[r])) : __bfloat162float(__ushort_as_bfloat16(h[r]));
  }
}

__device__ __forceinline__ uint32_t pick4(uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3, int i) {
  return i == 0 ? x0 : i == 1 ? x1 : i == 2 ? x2 : x3;
}

// bit position of element 16w + ip inside qs word w (turbo2/3)
__device__ __forceinline__ int qs2_bit(int ip) { return ip < 8 ? 4 * ip : 4 * (ip - 8) + 2; }
// bit position of element 32u + rr inside signs word u (turbo3)
__device__ __forceinline__ int sg_bit(int rr) {
  return rr < 16 ? 4 * (rr & 7) + 2 + (rr >> 3) : 4 * ((rr - 16) & 7) + ((rr - 16) >> 3);
}

// Decisions of element r of a lane's group of four (the bits of element r at 4 r, as
// immediates): predicates |y| >= t_k and y >= 0, predicate logic, predicated ORs.
// turbo3: bit 0 = odd count of t0, t1, t2 <= |y|, bit 1 = |y| >= t1; sign bit in xs.
template <int R>
__device__ __forceinline__ void decide3(float ay, float y, const float *thr, uint32_t &x, uint32_t &xs) {
  asm("{\n .reg .pred q0, q1, q2, qs, qx;\n"
      " setp.ge.f32 q0, %2, %3;\n setp.ge.f32 q1, %2, %4;\n setp.ge.f32 q2, %2, %5;\n"
      " setp.ge.f32 qs, %6, 0f00000000;\n xor.pred qx, q0, q1;\n xor.pred qx, qx, q2;\n"
      " @qx or.b32 %0, %0, %7;\n @q1 or.b32 %0, %0, %8;\n @qs or.b32 %1, %1, %7;\n}"
      : "+r"(x), "+r"(xs)
      : "f"(ay), "f"(thr[0]), "f"(thr[1]), "f"(thr[2]), "f"(y), "n"(1u << (4 * R)), "n"(2u << (4 * R)));
}
// turbo2: bit 0 = |y| >= t0, bit 1 = y >= 0
template <int R>
__device__ __forceinline__ void decide2(float ay, float y, const float *thr, uint32_t &x) {
  asm("{\n .reg .pred q0, qs;\n setp.ge.f32 q0, %1, %2;\n setp.ge.f32 qs, %3, 0f00000000;\n"
      " @q0 or.b32 %0, %0, %4;\n @qs or.b32 %0, %0, %5;\n}"
      : "+r"(x)
      : "f"(ay), "f"(thr[0]), "f"(y), "n"(1u << (4 * R)), "n"(2u << (4 * R)));
}
// turbo4: j >= 4, then j & 2 against t5 or t1, then j & 1 against t6, t4, t2 or t0; sign bit 3
template <int R>
__device__ __forceinline__ void decide4(float ay, float y, const float *thr, uint32_t &x) {
  asm("{\n .reg .pred q0, q1, q2, qs;\n .reg .f32 ta, tb, tc;\n"
      " setp.ge.f32 q2, %1, %5;\n selp.f32 ta, %7, %3, q2;\n setp.ge.f32 q1, %1, ta;\n"
      " selp.f32 tb, %8, %6, q1;\n selp.f32 tc, %4, %2, q1;\n selp.f32 tb, tb, tc, q2;\n"
      " setp.ge.f32 q0, %1, tb;\n setp.ge.f32 qs, %9, 0f00000000;\n"
      " @qs or.b32 %0, %0, %10;\n @q2 or.b32 %0, %0, %11;\n @q1 or.b32 %0, %0, %12;\n"
      " @q0 or.b32 %0, %0, %13;\n}"
      : "+r"(x)
      : "f"(ay), "f"(thr[0]), "f"(thr[1]), "f"(thr[2]), "f"(thr[3]), "f"(thr[4]), "f"(thr[5]), "f"(thr[6]),
        "f"(y), "n"(8u << (4 * R)), "n"(4u << (4 * R)), "n"(2u << (4 * R)), "n"(1u << (4 * R)));
}

// One lane's share of a packed block: the norm (binary16 bits), qs words
// (turbo2/3: words 2 l4 and 2 l4 + 1 in w[0], w[1]; turbo4: words 2 i + l4/2 in
// w[i], stored by the even lanes) and, for turbo3, signs word l4.
template <int TYPE>
struct PackedShare {
  uint32_t norm;
  uint32_t w[8];
  uint32_t sg;
};

// Quantise the block whose 32 elements per lane are in v (modified).  All 32
// lanes of the warp must call it (it shuffles within groups of four lanes).
template <int TYPE>
__device__ __forceinline__ void quantise_block4(const DevCodebook &cb, int l4, float v[8][4], PackedShare<TYPE> &out) {
  constexpr int NC = TypeTraits<TYPE>::NC;
  constexpr int HALF = NC / 2;

  // this lane's 32 sign bits: bit 4i + r = sign of element 4 l4 + 16 i + r (bit
  // 16 (i & 1) + 4 l4 + r of sign word i / 2); a set bit flips the float's sign bit
  uint32_t smask = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i)
    smask |= ((cb.sign_bits[i >> 1] >> (16 * (i & 1) + 4 * l4)) & 0xFu) << (4 * i);
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      ss = fmaf(v[i][r], v[i][r], ss);
      v[i][r] = __uint_as_float(__float_as_uint(v[i][r]) ^ ((smask << (31 - (4 * i + r))) & 0x80000000u));
    }
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  ss += __shfl_xor_sync(0xffffffffu, ss, 2);

  // butterflies inside the lane on pairs P[i][r] = (v[i][r], v[i + 4][r]), i < 4: the
  // stages h = 1, 2 (r bits) and h = 16, 32 (i bits 0, 1) combine two pairs elementwise
  // (packed f32x2), h = 64 (i bit 2) the two halves of a pair.  Each element sees the
  // same operations in the same order as one stage at a time on scalars.
  float2 P[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int r = 0; r < 4; ++r) P[i][r] = make_float2(v[i][r], v[i + 4][r]);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 a0 = add2(P[i][0], P[i][1]), a1 = sub2(P[i][0], P[i][1]);
    const float2 a2 = add2(P[i][2], P[i][3]), a3 = sub2(P[i][2], P[i][3]);
    P[i][0] = add2(a0, a2); P[i][2] = sub2(a0, a2); P[i][1] = add2(a1, a3); P[i][3] = sub2(a1, a3);
  }
#pragma unroll
  for (int hb = 1; hb < 4; hb <<= 1)
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (!(i & hb))
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const float2 x = P[i][r], y = P[i | hb][r];
          P[i][r] = add2(x, y);
          P[i | hb][r] = sub2(x, y);
        }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int r = 0; r < 4; ++r) P[i][r] = make_float2(P[i][r].x + P[i][r].y, P[i][r].x - P[i][r].y);
  // across the 4 lanes: h = 4 (lane ^ 1), h = 8 (lane ^ 2); element j takes
  // o = x[j ^ h] and becomes (j & h) ? o - x[j] : x[j] + o
#pragma unroll
  for (int m = 1; m < 4; m <<= 1) {
    const float sg = (l4 & m) ? -1.f : 1.f;
    const float2 sg2 = make_float2(sg, sg);
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float2 o = make_float2(__shfl_xor_sync(0xffffffffu, P[i][r].x, m), __shfl_xor_sync(0xffffffffu, P[i][r].y, m));
        P[i][r] = fma2(sg2, P[i][r], o);
      }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      v[i][r] = P[i][r].x;
      v[i + 4][r] = P[i][r].y;
    }

  // thresholds between positive centroids, scaled to the unnormalised domain
  const float nrm_scale = sqrtf(ss * 128.f);
  float thr[HALF - 1];
#pragma unroll
  for (int k = 0; k < HALF - 1; ++k)
    thr[k] = ss > 0.f ? 0.5f * (cb.c[HALF + k] + cb.c[HALF + k + 1]) * nrm_scale : INFINITY;

  // Decisions |y| >= t_k against the ascending thresholds (and y >= 0 for the sign) as
  // predicates, combined with predicate logic and folded into the packed words with
  // predicated ORs: no mask or select per decision (an unordered compare is false).
  out.norm = __half_as_ushort(__float2half_rn(sqrtf(ss)));
  out.sg = 0;
  if constexpr (TYPE == 4) {
    // word w = 2i + l4/2, element nibble 4*(l4 & 1) + r: code = 8 s + j, j = #{t_k <= |y|}
    // (3 bits by a three-level search over the 7 thresholds); lanes l4, l4^1 share a word.
    // The nibbles are packed with constant shifts and the word moved to its half once.
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t x = 0;
      decide4<0>(fabsf(v[i][0]), v[i][0], thr, x);
      decide4<1>(fabsf(v[i][1]), v[i][1], thr, x);
      decide4<2>(fabsf(v[i][2]), v[i][2], thr, x);
      decide4<3>(fabsf(v[i][3]), v[i][3], thr, x);
      x <<= 16 * (l4 & 1);
      out.w[i] = x | __shfl_xor_sync(0xffffffffu, x, 1);
    }
  } else {
    // qs word i holds elements 16i .. 16i+15; this lane's are 16i + 4*l4 + r.
    // turbo3: 2-bit j in qs, sign in the signs plane; turbo2: 2-bit code 2 s + j in qs.
    uint32_t wq[8];
    uint32_t ws[4] = {0u, 0u, 0u, 0u};
    // element 4 l4 + r of a qs word sits at bit qb + 4 r (qb = qs2_bit(4 l4)); its sign
    // at bit sb[i & 1] + 4 r of its signs word (sb = sg_bit(16 (i & 1) + 4 l4))
    const int qb = 16 * (l4 & 1) + 2 * (l4 >> 1);
    const int sb0 = 2 + 16 * (l4 & 1) + (l4 >> 1), sb1 = 16 * (l4 & 1) + (l4 >> 1);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t x = 0;
      if constexpr (TYPE == 3) {
        uint32_t xs = 0;
        decide3<0>(fabsf(v[i][0]), v[i][0], thr, x, xs);
        decide3<1>(fabsf(v[i][1]), v[i][1], thr, x, xs);
        decide3<2>(fabsf(v[i][2]), v[i][2], thr, x, xs);
        decide3<3>(fabsf(v[i][3]), v[i][3], thr, x, xs);
        ws[i >> 1] |= xs << ((i & 1) ? sb1 : sb0);
      } else {
        decide2<0>(fabsf(v[i][0]), v[i][0], thr, x);
        decide2<1>(fabsf(v[i][1]), v[i][1], thr, x);
        decide2<2>(fabsf(v[i][2]), v[i][2], thr, x);
        decide2<3>(fabsf(v[i][3]), v[i][3], thr, x);
      }
      x <<= qb;
      x |= __shfl_xor_sync(0xffffffffu, x, 1);
      x |= __shfl_xor_sync(0xffffffffu, x, 2);
      wq[i] = x;
    }
    out.w[0] = pick4(wq[0], wq[2], wq[4], wq[6], l4);
    out.w[1] = pick4(wq[1], wq[3], wq[5], wq[7], l4);
    if constexpr (TYPE == 3) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        ws[u] |= __shfl_xor_sync(0xffffffffu, ws[u], 1);
        ws[u] |= __shfl_xor_sync(0xffffffffu, ws[u], 2);
      }
      out.sg = pick4(ws[0], ws[1], ws[2], ws[3], l4);
    }
  }
}

// Store a lane's share of a packed block (global or shared memory; qs 16-byte
// aligned, signs 4-byte aligned).
template <int TYPE>
__device__ __forceinline__ void store_block4(const PackedShare<TYPE> &pb, int l4, uint16_t *norm, uint8_t *qs,
                                             uint8_t *signs) {
  if (l4 == 0) *norm = static_cast<uint16_t>(pb.norm);
  if (TYPE == 4) {
    if ((l4 & 1) == 0) {
#pragma unroll
      for (int i = 0; i < 8; ++i) reinterpret_cast<uint32_t *>(qs)[2 * i + (l4 >> 1)] = pb.w[i];
    }
  } else {
    reinterpret_cast<uint2 *>(qs)[l4] = make_uint2(pb.w[0], pb.w[1]);
    if (TYPE == 3) reinterpret_cast<uint32_t *>(signs)[l4] = pb.sg;
  }
}

}  // namespace tq

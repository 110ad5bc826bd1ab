// Split-KV bookkeeping shared by the decode kernels: tagged per-split partials,
// their log-sum-exp merge and the inverse rotation of the merged output.
#pragma once

#include "tq_common.cuh"
#include "tq_tc.cuh"

namespace tq {

// 2^x for x <= 0 (split weights), approximate to a few ulp.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Order-preserving map of a float to an int (for integer max atomics) and back.
__device__ __forceinline__ int ordered_int(float x) {
  const int b = __float_as_int(x);
  return b >= 0 ? b : b ^ 0x7fffffff;
}
__device__ __forceinline__ float ordered_float(int b) { return __int_as_float(b >= 0 ? b : b ^ 0x7fffffff); }

// Floats of shared memory decode_merge needs.
__host__ __device__ inline int merge_smem_floats(int group, int nbv, int n_splits) {
  return group * QK * nbv + 2 * group * n_splits;
}

// ---- split partials.  Each 32-bit value of a partial (m, l, o') is stored with
// a 32-bit tag in one 64-bit word, which a single access reads or writes whole.
// The tag holds the KV head's launch epoch + 1 (24 bits, never 0, so a
// zero-filled workspace holds no valid word) above the KV head index (8 bits):
// the merging CTA loads every partial of its head in one round trip and knows
// from the tags alone which ones are this launch's, so a CTA that stored its
// partial needs no fence and no second counter, and the arrival counter can be
// bumped before the partial is even computed.  A stale word of this head
// carries an older epoch (the epoch of head hk changes only after all CTAs of
// head hk have read it); a word that another head wrote carries another head
// index, whatever the two heads' epochs -- so calls of different shapes (head
// counts, lengths) may share one workspace.  An older word of this head is
// mistaken for a current one only after 2^24 launches of the head that never
// rewrote its slot.
__device__ __forceinline__ uint32_t split_tag(uint32_t epoch, int hk) {
  uint32_t t = (epoch + 1u) & 0xFFFFFFu;
  if (t == 0u) t = 1u;
  return (t << 8) | static_cast<uint32_t>(hk & 0xFF);
}

__device__ __forceinline__ void st_tagged(uint64_t *p, float v, uint32_t tag) {
  const uint64_t w = (static_cast<uint64_t>(tag) << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}

__device__ __forceinline__ uint64_t ld_tagged(const uint64_t *p) {
  uint64_t w;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
  return w;
}

__device__ __forceinline__ float tagged_value(uint64_t w) { return __uint_as_float(static_cast<uint32_t>(w)); }
__device__ __forceinline__ bool tagged_ok(uint64_t w, uint32_t tag) { return static_cast<uint32_t>(w >> 32) == tag; }

// Epoch of KV head hk for this launch (one thread; the value goes to every
// thread of the CTA through shared memory).
__device__ __forceinline__ uint32_t load_epoch(const DecodeArgs &a, int hk) {
  uint32_t e;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(e) : "l"(a.epochs + hk) : "memory");
  return e;
}

// Arrival of this CTA at its KV head's counter (one thread, before the CTA's
// partial is stored); the returned count says whether it is the last one.
__device__ __forceinline__ int split_arrive(const DecodeArgs &a, int hk) {
  int prev;
  asm volatile("atom.add.relaxed.gpu.s32 %0, [%1], 1;" : "=r"(prev) : "l"(a.counters + hk) : "memory");
  return prev;
}

// Partial of query head h = hk * group + g, split s: (m, l) and o'[d].
// (a.test_drop_split names a split whose partial is skipped: a test's way to make
// the merging CTAs' bounded waits run out; 0 in every product call)
__device__ __forceinline__ void store_partial_ml(const DecodeArgs &a, int h, int s, float m, float l, uint32_t tag) {
  if (s + 1 == a.test_drop_split) return;
  uint64_t *p = a.part_ml + (static_cast<size_t>(h) * a.n_splits + s) * 2;
  st_tagged(p, m, tag);
  st_tagged(p + 1, l, tag);
}
__device__ __forceinline__ void store_partial_o(const DecodeArgs &a, int h, int s, int d, float o, uint32_t tag) {
  if (s + 1 == a.test_drop_split) return;
  st_tagged(a.part + (static_cast<size_t>(h) * a.n_splits + s) * a.part_stride + d, o, tag);
}

// Run, when the grid is larger than the GPU holds at once (no cooperative launch),
// by every thread of the last CTA of KV head hk to arrive (its own partial
// stored and a CTA barrier passed).  Merges the splits
//   M = max_s m_s,  L = sum_s l_s 2^(m_s - M),  o' = sum_s o'_s 2^(m_s - M) / L
// (scores are kept in the log2 domain), rotates back with the V codebook,
//   o = S H o' / sqrt(128)   (R^T for R = H S / sqrt(128)),
// writes out[h][0 .. dv), resets the counter and advances the epoch, so the next
// launch (or graph replay) finds the workspace ready.  Each warp merges 32
// consecutive outputs of one head, 24 splits at a time: lane s < 24 holds split
// s's maximum and sum, every lane loads its output's words of the 24 splits at
// once (one L2 round trip per 24 splits) and the batch is loaded again, a
// bounded number of times, while a word of it still carries another tag.
// `smem` must hold merge_smem_floats(group, nbv, n_splits) floats.
template <int NT>
__device__ void decode_merge(const DecodeArgs &a, int hk, uint32_t epoch, float *smem) {
  const uint32_t tag = split_tag(epoch, hk);
  const int G = a.group, ns = a.n_splits, dvp = QK * a.nbv;
  const int stride = a.part_stride;
  float *orot = smem;                     // [G][dvp]
  const uint64_t *base = a.part + static_cast<size_t>(hk) * G * ns * stride;
  const uint64_t *base_ml = a.part_ml + static_cast<size_t>(hk) * G * ns * 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  bool late = false;
  for (int i0 = warp * 32; i0 < G * dvp; i0 += NT) {     // dvp is a multiple of 32: one head per warp pass
    const int i = i0 + lane, g = i / dvp, d = i % dvp;
    const uint64_t *p = base + static_cast<size_t>(g) * ns * stride;
    const uint64_t *pml = base_ml + static_cast<size_t>(g) * ns * 2;
    float M = -INFINITY, L = 0.f, o = 0.f;
    for (int s0 = 0; s0 < ns; s0 += 24) {
      const int n = min(24, ns - s0);
      const uint64_t *ps = p + static_cast<size_t>(s0) * stride + d;
      uint64_t wm = 0, wl = 0, wo[24];
      for (int tries = 0;; ++tries) {
        if (lane < n) {
          wm = ld_tagged(pml + 2 * (s0 + lane));
          wl = ld_tagged(pml + 2 * (s0 + lane) + 1);
        }
#pragma unroll
        for (int j = 0; j < 24; ++j) wo[j] = (j < n) ? ld_tagged(ps + static_cast<size_t>(j) * stride) : 0;
        bool ok = lane >= n || (tagged_ok(wm, tag) && tagged_ok(wl, tag));
#pragma unroll
        for (int j = 0; j < 24; ++j) ok = ok && (j >= n || tagged_ok(wo[j], tag));
        if (__all_sync(0xffffffffu, ok)) break;
        if (tries >= (1 << 16)) {          // a split never stored its partial: report, merge what is there
          late = true;
          break;
        }
        __nanosleep(100);
      }
      const float ms = (lane < n) ? tagged_value(wm) : -INFINITY, ls = (lane < n) ? tagged_value(wl) : 0.f;
      const float Mn = fmaxf(M, warp_max(ms));
      const float f = (M == -INFINITY) ? 0.f : fast_exp2(M - Mn);
      const float w = (ms == -INFINITY) ? 0.f : fast_exp2(ms - Mn);
      L = L * f + warp_sum(w * ls);
      o *= f;
#pragma unroll
      for (int j = 0; j < 24; ++j) o = fmaf(__shfl_sync(0xffffffffu, w, j), tagged_value(wo[j]), o);
      M = Mn;
    }
    orot[i] = (L > 0.f) ? o / L : 0.f;
  }
  if (late && lane == 0) set_status(a.status, TQ_ERR_TIMEOUT);
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
  if (threadIdx.x == 0) {
    a.counters[hk] = 0;
    a.epochs[hk] = epoch + 1u;
  }
}

// Merge of one output block (query head h = hk * group + g, V block b) over all
// splits by 128 threads of one CTA (warps w0 .. w0 + 3, thread t = output d of
// the block), used when every CTA of the grid is resident (a cooperative launch):
// the block's partial words of all splits are loaded, 24 splits per round trip,
// and loaded again (bounded) until every tag is this launch's, i.e. until every
// split has stored its partial; then the merge, the inverse rotation by warp w0
// and the store of out[h][128 b ..].  `buf` holds 128 floats of shared memory and
// named barrier `bar_id` is free for these 128 threads.  Returns false if a
// split's partial never arrived (the bound ran out).
__device__ __forceinline__ bool merge_block(const DecodeArgs &a, int hk, int g, int b, uint32_t tag, int t, int bar_id, float *buf) {
  const int ns = a.n_splits, G = a.group, lane = t & 31;
  const int h = hk * G + g;
  const uint64_t *pml = a.part_ml + static_cast<size_t>(h) * ns * 2;
  const uint64_t *po = a.part + static_cast<size_t>(h) * ns * a.part_stride + b * QK + t;
  float M = -INFINITY, L = 0.f, o = 0.f;
  bool arrived = true;
  for (int s0 = 0; s0 < ns; s0 += 24) {
    const int n = min(24, ns - s0);
    const uint64_t *ps = po + static_cast<size_t>(s0) * a.part_stride;
    uint64_t wm = 0, wl = 0, wo[24];
    for (int tries = 0;; ++tries) {
      if (lane < n) {
        wm = ld_tagged(pml + 2 * (s0 + lane));
        wl = ld_tagged(pml + 2 * (s0 + lane) + 1);
      }
#pragma unroll
      for (int j = 0; j < 24; ++j) wo[j] = (j < n) ? ld_tagged(ps + static_cast<size_t>(j) * a.part_stride) : 0;
      bool ok = lane >= n || (tagged_ok(wm, tag) && tagged_ok(wl, tag));
#pragma unroll
      for (int j = 0; j < 24; ++j) ok = ok && (j >= n || tagged_ok(wo[j], tag));
      if (__all_sync(0xffffffffu, ok)) break;
      if (tries >= (1 << 16)) {
        arrived = false;
        break;
      }
      __nanosleep(16);
    }
    const float ms = (lane < n) ? tagged_value(wm) : -INFINITY, ls = (lane < n) ? tagged_value(wl) : 0.f;
    const float Mn = fmaxf(M, warp_max(ms));
    const float f = (M == -INFINITY) ? 0.f : fast_exp2(M - Mn);
    const float w = (ms == -INFINITY) ? 0.f : fast_exp2(ms - Mn);
    L = L * f + warp_sum(w * ls);
    o *= f;
#pragma unroll
    for (int j = 0; j < 24; ++j) o = fmaf(__shfl_sync(0xffffffffu, w, j), tagged_value(wo[j]), o);
    M = Mn;
  }
  buf[t] = (L > 0.f) ? o / L : 0.f;
  tc::named_sync(bar_id, 128);
  if (t < 32) {
    float v[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) v[r] = buf[4 * lane + r];
    wht128_warp(v, lane);
#pragma unroll
    for (int r = 0; r < 4; ++r) v[r] *= kInvSqrtQK;
    apply_signs(v, a.cbv, lane);
    float *out = a.out + static_cast<size_t>(h) * a.dv;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int d = b * QK + 4 * lane + r;
      if (d < a.dv) out[d] = v[r];
    }
  }
  tc::named_sync(bar_id, 128);                  // buf free again
  return __all_sync(0xffffffffu, arrived);
}

// The cooperative split merge of KV head hk, run by threads 0..127 of every CTA
// of the head after it stored its partial: CTA `split` merges output blocks
// u = split, split + n_splits, ... of the group * nbv blocks; split 0 advances
// the head's epoch (every CTA of the head has read it by the time its merge
// found all partials).
__device__ __forceinline__ void coop_merge(const DecodeArgs &a, int hk, int split, uint32_t epoch, float *buf) {
  const int t = threadIdx.x;
  bool arrived = true;
  for (int u = split; u < a.group * a.nbv; u += a.n_splits)
    arrived = merge_block(a, hk, u / a.nbv, u % a.nbv, split_tag(epoch, hk), t, 1, buf) && arrived;
  if (!arrived && (t & 31) == 0) set_status(a.status, TQ_ERR_TIMEOUT);
  if (split == 0 && t == 0) a.epochs[hk] = epoch + 1u;
}

// Query block wb = g * nbk + b (head hk * group + g, dims 128 b ..): lane i
// loads dims 4i .. 4i+3 of the block, zero beyond dk.
__device__ __forceinline__ void load_query_block(const DecodeArgs &a, int hk, int wb, int lane, float v[4]) {
  const int g = wb / a.nbk, b = wb % a.nbk;
  const size_t row = static_cast<size_t>(hk * a.group + g) * a.dk;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int d = b * QK + 4 * lane + r;
    if (a.q_type == TQ_F32) {
      v[r] = (d < a.dk) ? a.q[row + d] : 0.f;
    } else {
      const uint16_t bits = (d < a.dk) ? reinterpret_cast<const uint16_t *>(a.q)[row + d] : 0;
      v[r] = a.q_type == TQ_BF16 ? __bfloat162float(__ushort_as_bfloat16(bits)) : __half2float(__ushort_as_half(bits));
    }
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

// Host side of the C ABI: argument checks, workspace layout, codebook
// construction and kernel dispatch.  Nothing here allocates device memory,
// synchronises or reads device memory except tq_workspace_status, so every
// compute call can be captured into a CUDA graph ([HIP#28] "1. Graph-safe
// decode": the page's crash came from cudaMalloc/cudaFree during capture).
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "tq_internal.h"
#include "../../include/tq_testing.h"

namespace tq {

// ---------------------------------------------------------------- device info

int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 152;
  }
  int v = cached[dev].load(std::memory_order_relaxed);
  if (v > 0) return v;
  if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
    cudaGetLastError();
    v = 152;
  }
  cached[dev].store(v, std::memory_order_relaxed);
  return v;
}

static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }


// Raise the kernel's MaxDynamicSharedMemorySize attribute to at least `bytes`,
// calling the driver only when the size is above what was set before on this
// device (a driver call on every launch cost about 0.8 us of host time per eager
// decode call).  The attribute is one value per kernel and is only ever raised,
// so launches of any smaller size stay valid.  It lives as long as the device's
// primary context: a process that resets the device (cudaDeviceReset) must not
// reuse the library.
cudaError_t set_dynamic_smem(const void *kern, int bytes) {
  struct Entry {
    int dev, bytes;
    const void *kern;
  };
  static std::mutex mu;
  static Entry cache[128];
  static int n_cache = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  int slot = -1;
  for (int i = 0; i < n_cache; ++i)
    if (cache[i].dev == dev && cache[i].kern == kern) {
      if (cache[i].bytes >= bytes) return cudaSuccess;
      slot = i;
      break;
    }
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  if (slot >= 0) cache[slot].bytes = bytes;
  else if (n_cache < 128) cache[n_cache++] = Entry{dev, bytes, kern};
  return cudaSuccess;
}

// Whether `kern` can run as clusters of `csize` CTAs (threads, smem each) with
// at least `want` clusters resident at once.  Cached per device and kernel.
bool cluster_merge_ok(const void *kern, int csize, int threads, size_t smem, int want) {
  struct Entry {
    int dev, csize, want;
    const void *kern;
    bool ok;
  };
  static std::mutex mu;
  static Entry cache[64];
  static int n_cache = 0;
  if (csize < 2 || csize > 16) return false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_cache; ++i)
    if (cache[i].dev == dev && cache[i].kern == kern && cache[i].csize == csize && cache[i].want == want)
      return cache[i].ok;
  bool ok = true;
  if (csize > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
    ok = false;
  if (ok) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(csize, want);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = csize;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    ok = cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n >= want;
  }
  cudaGetLastError();
  if (n_cache < 64) cache[n_cache++] = Entry{dev, csize, want, kern, ok};
  return ok;
}

DecodeWorkspaceLayout decode_layout(int n_kv_heads, int n_q_heads, int nbv, int64_t kv_len,
                                    int /*algo*/) {
  DecodeWorkspaceLayout L;
  // about one CTA per SM (with at most 16 splits per KV head the splits run as
  // one thread-block cluster and merge on chip, see the decode kernels)
  // at most one CTA per SM in all, so that the grid can run as one cooperative launch
  const int target_ctas = sm_count();
  int per_head = target_ctas / n_kv_heads;
  if (per_head < 1) per_head = 1;
  if (per_head > 256) per_head = 256;
  int64_t chunk = (kv_len + per_head - 1) / per_head;
  chunk = (chunk + 63) / 64 * 64;
  if (chunk < 128) chunk = 128;
  L.chunk = chunk;
  L.n_splits = kv_len > 0 ? static_cast<int>((kv_len + chunk - 1) / chunk) : 1;
  L.epochs_off = kWsHeader;
  L.counters_off = L.epochs_off + kWsEpochBytes;
  L.ml_off = L.counters_off + round_up(sizeof(int32_t) * n_kv_heads, 256);
  L.part_off = L.ml_off + round_up(sizeof(uint64_t) * 2 * n_q_heads * L.n_splits, 256);
  L.total = L.part_off + round_up(sizeof(uint64_t) * n_q_heads * L.n_splits * 128 * static_cast<size_t>(nbv), 256);
  return L;
}

// Key-range splits of a prefill launch: when the query tiles x KV heads do not
// fill the SMs, each query tile's keys are split over up to 16 work items (at
// least two key tiles each); a second kernel merges the splits.  The split count
// minimises the estimated time of the launch: the rounds of work items over the
// SMs, each item costing its key tiles plus about six tiles' worth of set-up and
// epilogue (measured on the 4K workload: 2.3 us per 64-key tile, ~15 us per item).
// Query tiles that fill the SMs are not split.
PrefillWorkspaceLayout prefill_layout(int nq, int group, int n_kv_heads, int64_t kv_len, int nbk, int nbv) {
  PrefillWorkspaceLayout L;
  const int64_t qt = (static_cast<int64_t>(nq) * group + 127) / 128;
  const int64_t ctas = qt * n_kv_heads;
  const int bn = (nbk == 2) ? 64 : 128;        // the prefill kernel's key tile
  const int64_t tiles = (kv_len + bn - 1) / bn;
  const int64_t sms = sm_count();
  int64_t sp = 1;
  double best = 0.0;
  // (query tiles that fill the SMs are not split: the longest-first queue balances
  // their different lengths, and splits would only add partials)
  for (int64_t c = 1; c <= 16 && ctas > 0 && ctas < sms; ++c) {
    if (c > 1 && c > tiles / 2) break;
    const int64_t rounds = (ctas * c + sms - 1) / sms;
    const double cost = static_cast<double>(rounds) * (static_cast<double>((tiles + c - 1) / c) + 6.0);
    if (c == 1 || cost < best) {
      best = cost;
      sp = c;
    }
  }
  L.n_split = static_cast<int>(sp);
  L.sched_off = kWsHeader + kWsEpochBytes;         // the decode epochs stay untouched
  L.part_off = L.sched_off + 256;
  L.total = L.part_off;
  if (L.n_split > 1)
    L.total += round_up(sizeof(float) * qt * n_kv_heads * L.n_split * 128 * (4 + 128 * static_cast<size_t>(nbv)), 256);
  return L;
}

// ------------------------------------------------------------- binary16 / codebook

// Nearest binary16 value of x (round to nearest, ties to even), as a double.
static double round_to_binary16(double x) {
  if (x == 0.0 || !isfinite(x)) return x;
  const double ax = fabs(x);
  int e = 0;
  frexp(ax, &e);               // ax = m 2^e, m in [0.5, 1)
  const int E = e - 1;         // ax in [2^E, 2^(E+1))
  double q;
  if (E < -14) q = nearbyint(ax * 0x1p24) * 0x1p-24;              // subnormal spacing
  else q = nearbyint(ldexp(ax, 10 - E)) * ldexp(1.0, E - 10);    // 11 significant bits
  if (q > 65504.0) q = INFINITY;
  return copysign(q, x);
}

// P(a < X < b), X ~ N(0,1), from erfc on the side without cancellation.
static double gauss_prob(double a, double b) {
  const double r = 0.70710678118654752440;
  if (a >= 0) return 0.5 * (erfc(a * r) - erfc(b * r));
  if (b <= 0) return 0.5 * (erfc(-b * r) - erfc(-a * r));
  return 1.0 - 0.5 * erfc(-a * r) - 0.5 * erfc(b * r);
}

static double gauss_pdf(double x) {
  return isinf(x) ? 0.0 : exp(-0.5 * x * x) * 0.39894228040143267794;
}

// Lloyd-Max quantiser of N(0,1): thresholds at midpoints, centroids at the
// conditional means E[X | cell], repeated to a fixed point.
static void lloyd_max(int n, double *c) {
  for (int k = 0; k < n; ++k) c[k] = (k - 0.5 * (n - 1)) * (4.0 / n);
  double t[17];
  for (int it = 0; it < 200000; ++it) {
    t[0] = -INFINITY;
    t[n] = INFINITY;
    for (int k = 1; k < n; ++k) t[k] = 0.5 * (c[k - 1] + c[k]);
    double delta = 0.0;
    for (int k = 0; k < n; ++k) {
      const double nk = (gauss_pdf(t[k]) - gauss_pdf(t[k + 1])) / gauss_prob(t[k], t[k + 1]);
      delta = fmax(delta, fabs(nk - c[k]));
      c[k] = nk;
    }
    if (delta < 1e-15) break;
  }
}

static int n_centroids_of(int type) {
  return type == TQ_TURBO2 ? 4 : type == TQ_TURBO3 ? 8 : type == TQ_TURBO4 ? 16 : 0;
}

static bool codebook_ok(const tq_codebook *cb, int type) {
  const int n = n_centroids_of(type);
  if (!cb || n == 0 || cb->n_centroids != n) return false;
  for (int i = 0; i < n; ++i) {
    const float c = cb->centroids[i];
    if (!isfinite(c)) return false;
    if (i + 1 < n && !(c < cb->centroids[i + 1])) return false;
    if (c != -cb->centroids[n - 1 - i]) return false;
    if (round_to_binary16(c) != static_cast<double>(c)) return false;
  }
  return cb->centroids[n / 2] > 0.f;
}

// binary16 bit pattern of a float that is exactly representable in binary16
static uint16_t binary16_bits(float f) {
  if (f == 0.f) return signbit(f) ? 0x8000 : 0;
  uint16_t sign = f < 0 ? 0x8000 : 0;
  double a = fabs(static_cast<double>(f));
  int e = 0;
  const double m = frexp(a, &e);           // a = m 2^e, m in [0.5, 1)
  const int E = e - 1;                     // a in [2^E, 2^(E+1))
  if (E < -14) return sign | static_cast<uint16_t>(nearbyint(a * 0x1p24));            // subnormal
  const uint32_t mant = static_cast<uint32_t>(nearbyint((2.0 * m - 1.0) * 1024.0));
  return sign | static_cast<uint16_t>(((E + 15) << 10) | mant);
}

void code_byte_tables(const tq_codebook *cb, int type, uint32_t t[4]) {
  const int n = cb->n_centroids, half = n / 2;
  uint16_t v[8];
  for (int k = 0; k < 8; ++k) {
    float f = 0.f;
    if (type == TQ_TURBO4) f = cb->centroids[8 + k];                    // magnitudes
    else if (k < n) f = (k & half) ? cb->centroids[half + (k & (half - 1))] : -cb->centroids[half + (k & (half - 1))];
    v[k] = binary16_bits(f);
  }
  t[0] = t[1] = t[2] = t[3] = 0;
  for (int k = 0; k < 4; ++k) {
    t[0] |= static_cast<uint32_t>(v[k] & 0xff) << (8 * k);
    t[1] |= static_cast<uint32_t>(v[4 + k] & 0xff) << (8 * k);
    t[2] |= static_cast<uint32_t>(v[k] >> 8) << (8 * k);
    t[3] |= static_cast<uint32_t>(v[4 + k] >> 8) << (8 * k);
  }
}

static DevCodebook to_dev(const tq_codebook *cb) {
  DevCodebook d;
  memset(&d, 0, sizeof(d));
  for (int i = 0; i < 4; ++i) d.sign_bits[i] = cb->sign_bits[i];
  d.n = cb->n_centroids;
  for (int i = 0; i < cb->n_centroids && i < 16; ++i) d.c[i] = cb->centroids[i];
  return d;
}

// ------------------------------------------------------------------ checks

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static tq_status check_cache(const tq_cache *c) {
  if (!c) return TQ_ERR_INVALID_ARG;
  if (n_centroids_of(c->type) == 0) return TQ_ERR_INVALID_ARG;
  if (c->n_kv_heads <= 0 || c->head_dim <= 0 || c->head_dim % 8 != 0 || c->head_dim > 1 << 16)
    return TQ_ERR_INVALID_ARG;
  if (c->n_blocks != (c->head_dim + 127) / 128) return TQ_ERR_INVALID_ARG;
  if (c->n_cells <= 0 || c->n_cells % 64 != 0) return TQ_ERR_INVALID_ARG;
  if (!c->norms || !c->qs || !aligned16(c->norms) || !aligned16(c->qs)) return TQ_ERR_INVALID_ARG;
  if (c->type == TQ_TURBO3 && (!c->signs || !aligned16(c->signs))) return TQ_ERR_INVALID_ARG;
  return TQ_OK;
}

// A failed launch or call leaves its error in the runtime's last-error slot, where
// the caller's next CUDA call (or another library's launch check) would report it
// as its own: clear it here, the status says what happened.
static tq_status map_cuda(cudaError_t e) {
  if (e == cudaSuccess) return TQ_OK;
  cudaGetLastError();
  return TQ_ERR_CUDA;
}

}  // namespace tq

using namespace tq;

extern "C" {

const char *tq_status_string(int status) {
  switch (status) {
    case TQ_OK: return "ok";
    case TQ_ERR_INVALID_ARG: return "invalid argument";
    case TQ_ERR_UNSUPPORTED: return "unsupported combination";
    case TQ_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case TQ_ERR_CUDA: return "CUDA runtime error";
    case TQ_ERR_TIMEOUT: return "device-side wait timed out";
    case TQ_ERR_DEVICE_CHECK: return "device-side input check failed";
    default: return "unknown status";
  }
}

int tq_version(void) { return 100; }

tq_status tq_codebook_init(int type, const uint32_t sign_bits[4], tq_codebook *out) {
  const int n = n_centroids_of(type);
  if (n == 0 || !sign_bits || !out) return TQ_ERR_INVALID_ARG;
  double c[16];
  lloyd_max(n, c);
  // enforce exact symmetry before rounding: average the mirrored pair
  memset(out, 0, sizeof(*out));
  for (int i = 0; i < 4; ++i) out->sign_bits[i] = sign_bits[i];
  out->n_centroids = n;
  for (int i = 0; i < n / 2; ++i) {
    const double m = 0.5 * (c[n - 1 - i] - c[i]) / sqrt(128.0);
    const float r = static_cast<float>(round_to_binary16(m));
    out->centroids[n - 1 - i] = r;
    out->centroids[i] = -r;
  }
  return TQ_OK;
}

tq_status tq_cache_plane_bytes(int type, int n_kv_heads, int head_dim, int64_t n_cells,
                               size_t *norms_bytes, size_t *qs_bytes, size_t *signs_bytes) {
  if (n_centroids_of(type) == 0 || n_kv_heads <= 0 || head_dim <= 0 || n_cells <= 0 ||
      !norms_bytes || !qs_bytes || !signs_bytes)
    return TQ_ERR_INVALID_ARG;
  const size_t blocks = static_cast<size_t>(n_kv_heads) * n_cells * ((head_dim + 127) / 128);
  *norms_bytes = blocks * 2;
  *qs_bytes = blocks * (type == TQ_TURBO4 ? 64 : 32);
  *signs_bytes = type == TQ_TURBO3 ? blocks * 16 : 0;
  return TQ_OK;
}

tq_status tq_set_rows(const tq_cache *dst, const tq_codebook *cb, const void *src, int src_type,
                      const int64_t *cell_ids, int64_t n_rows, int32_t *dev_status,
                      tq_stream stream) {
  tq_status st = check_cache(dst);
  if (st != TQ_OK) return st;
  if (!codebook_ok(cb, dst->type)) return TQ_ERR_INVALID_ARG;
  if (src_type != TQ_F32 && src_type != TQ_F16 && src_type != TQ_BF16) return TQ_ERR_INVALID_ARG;
  if (n_rows < 0) return TQ_ERR_INVALID_ARG;
  if (n_rows == 0) return TQ_OK;
  if (!src || !aligned16(src) || !cell_ids || (reinterpret_cast<uintptr_t>(cell_ids) & 7u))
    return TQ_ERR_INVALID_ARG;
  if (dev_status && (reinterpret_cast<uintptr_t>(dev_status) & 3u)) return TQ_ERR_INVALID_ARG;
  const int64_t warps = n_rows * dst->n_kv_heads * dst->n_blocks;
  if ((warps + 7) / 8 > 0x7fffffffLL) return TQ_ERR_INVALID_ARG;
  SetRowsArgs a;
  a.src = src;
  a.cell_ids = cell_ids;
  a.dev_status = dev_status;
  a.norms = static_cast<uint16_t *>(dst->norms);
  a.qs = static_cast<uint8_t *>(dst->qs);
  a.signs = static_cast<uint8_t *>(dst->signs);
  a.n_rows = n_rows;
  a.n_cells = dst->n_cells;
  a.n_kv_heads = dst->n_kv_heads;
  a.head_dim = dst->head_dim;
  a.n_blocks = dst->n_blocks;
  a.cb = to_dev(cb);
  return map_cuda(launch_set_rows(dst->type, src_type, a, static_cast<cudaStream_t>(stream)));
}

static tq_status check_kv_pair(const tq_cache *k, const tq_cache *v, int n_q_heads, int64_t kv_len) {
  tq_status st = check_cache(k);
  if (st != TQ_OK) return st;
  st = check_cache(v);
  if (st != TQ_OK) return st;
  if (k->n_kv_heads != v->n_kv_heads || k->n_cells != v->n_cells) return TQ_ERR_INVALID_ARG;
  if (n_q_heads <= 0 || n_q_heads % k->n_kv_heads != 0) return TQ_ERR_INVALID_ARG;
  if (kv_len < 0 || kv_len > k->n_cells) return TQ_ERR_INVALID_ARG;
  return TQ_OK;
}

// Decode also keeps one epoch word per KV head in the workspace header.
static tq_status check_decode_pair(const tq_cache *k, const tq_cache *v, int n_q_heads, int64_t kv_len) {
  const tq_status st = check_kv_pair(k, v, n_q_heads, kv_len);
  if (st != TQ_OK) return st;
  return k->n_kv_heads <= kMaxDecodeKvHeads ? TQ_OK : TQ_ERR_INVALID_ARG;
}

// Launch heads of a decode call: sequences x KV heads x, on the tensor-core
// kernel, group / mma_group(group) launch heads per KV head.
static int64_t decode_launch_heads(int n_kv_heads, int group, int n_seq, int algo) {
  const int rep = (algo == TQ_DECODE_MMA) ? group / mma_group(group) : 1;
  return static_cast<int64_t>(n_seq > 0 ? n_seq : 1) * n_kv_heads * rep;
}

// The tensor-core kernel takes the shape (and its launch heads fit the epoch words).
static bool decode_mma_ok(const tq_cache *k, const tq_cache *v, int n_q_heads, int n_seq) {
  const int group = n_q_heads / k->n_kv_heads;
  return decode_mma_supported(k->type, v->type, group, k->n_blocks, v->n_blocks) &&
         decode_launch_heads(k->n_kv_heads, group, n_seq, TQ_DECODE_MMA) <= kMaxDecodeKvHeads;
}

size_t tq_fattn_decode_workspace(const tq_cache *k, const tq_cache *v, int n_q_heads,
                                 int64_t kv_len) {
  if (check_decode_pair(k, v, n_q_heads, kv_len) != TQ_OK) return 0;
  // large enough for either kernel (their launch heads differ for GQA groups
  // other than 1, 2 and 4)
  size_t total = decode_layout(k->n_kv_heads, n_q_heads, v->n_blocks, kv_len, TQ_DECODE_LUT).total;
  if (decode_mma_ok(k, v, n_q_heads, 0)) {
    const int heads = static_cast<int>(decode_launch_heads(k->n_kv_heads, n_q_heads / k->n_kv_heads, 0, TQ_DECODE_MMA));
    const size_t m = decode_layout(heads, n_q_heads, v->n_blocks, kv_len, TQ_DECODE_MMA).total;
    if (m > total) total = m;
  }
  return total;
}

// Decode, optionally with the new token's rows appended first (k_row != null):
// fused into the tensor-core kernel, else as two SET_ROWS launches before it.
// clear_counters: zero the workspace's split counters on the stream right before
// the decode kernel, after every argument check (the allocation-free entry point,
// whose shared array may hold counters of an interrupted call).
// n_seq > 0: batched decode of n_seq sequences (host arrays seq_cell0 / seq_len,
// kv_len their longest length), tensor-core kernel only.
static tq_status decode_call(const tq_cache *k, const tq_cache *v, const tq_codebook *cbk, const tq_codebook *cbv,
                             const void *k_row, const void *v_row, int src_type, const int64_t *cell_id,
                             const float *q, int n_q_heads, int64_t kv_len, float scale, float v_thresh,
                             int algo, float *out, void *workspace, size_t workspace_bytes, tq_stream stream,
                             bool clear_counters = false, int drop_split = -1, int n_seq = 0,
                             const int64_t *seq_cell0 = nullptr, const int64_t *seq_len = nullptr,
                             int q_type = TQ_F32) {
  tq_status st = check_decode_pair(k, v, n_q_heads, n_seq > 0 ? 0 : kv_len);
  if (st != TQ_OK) return st;
  if (!codebook_ok(cbk, k->type) || !codebook_ok(cbv, v->type)) return TQ_ERR_INVALID_ARG;
  if (!q || !out || !aligned16(q) || !aligned16(out) || !isfinite(scale)) return TQ_ERR_INVALID_ARG;
  if (!(v_thresh >= 0.f) || !isfinite(v_thresh)) return TQ_ERR_INVALID_ARG;
  if (algo != TQ_DECODE_AUTO && algo != TQ_DECODE_LUT && algo != TQ_DECODE_MMA)
    return TQ_ERR_INVALID_ARG;
  const bool append = k_row != nullptr;
  if (append) {
    if (src_type != TQ_F32 && src_type != TQ_F16 && src_type != TQ_BF16) return TQ_ERR_INVALID_ARG;
    if (!v_row || !aligned16(k_row) || !aligned16(v_row) || !cell_id ||
        (reinterpret_cast<uintptr_t>(cell_id) & 7u))
      return TQ_ERR_INVALID_ARG;
  }
  const int group = n_q_heads / k->n_kv_heads;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool ws_ok = workspace && !(reinterpret_cast<uintptr_t>(workspace) & 255u);
  int32_t *status = ws_ok ? static_cast<int32_t *>(workspace) : nullptr;
  const int n_out = (n_seq > 0 ? n_seq : 1) * n_q_heads;       // query heads of all sequences
  if (kv_len == 0) {             // nothing to attend: append only, zero output
    if (append) {
      st = tq_set_rows(k, cbk, k_row, src_type, cell_id, 1, status, stream);
      if (st != TQ_OK) return st;
      st = tq_set_rows(v, cbv, v_row, src_type, cell_id, 1, status, stream);
      if (st != TQ_OK) return st;
    }
    return map_cuda(cudaMemsetAsync(out, 0, sizeof(float) * n_out * v->head_dim, s));
  }
  const bool mma_ok = decode_mma_ok(k, v, n_q_heads, n_seq);
  const bool lut_ok = n_seq == 0 && group <= 8 && k->n_blocks <= 2 && v->n_blocks <= 2;
  int use = algo;
  if (use == TQ_DECODE_AUTO) use = mma_ok ? TQ_DECODE_MMA : TQ_DECODE_LUT;
  if ((use == TQ_DECODE_MMA && !mma_ok) || (use == TQ_DECODE_LUT && !lut_ok)) return TQ_ERR_UNSUPPORTED;
  const int kgroup = (use == TQ_DECODE_MMA) ? mma_group(group) : group;     // query heads per launch head
  const int launch_heads = static_cast<int>(decode_launch_heads(k->n_kv_heads, group, n_seq, use));
  const DecodeWorkspaceLayout L = decode_layout(launch_heads, n_out, v->n_blocks, kv_len, use);
  if (!ws_ok || workspace_bytes < L.total) return TQ_ERR_WORKSPACE;
  if (append && use != TQ_DECODE_MMA) {      // the LUT kernel: SET_ROWS launches first
    st = tq_set_rows(k, cbk, k_row, src_type, cell_id, 1, status, stream);
    if (st != TQ_OK) return st;
    st = tq_set_rows(v, cbv, v_row, src_type, cell_id, 1, status, stream);
    if (st != TQ_OK) return st;
  }

  DecodeArgs a;
  memset(&a, 0, sizeof(a));
  a.kn = static_cast<const uint16_t *>(k->norms);
  a.kqs = static_cast<const uint8_t *>(k->qs);
  a.ksg = static_cast<const uint8_t *>(k->signs);
  a.vn = static_cast<const uint16_t *>(v->norms);
  a.vqs = static_cast<const uint8_t *>(v->qs);
  a.vsg = static_cast<const uint8_t *>(v->signs);
  a.q = q;
  a.out = out;
  a.part = reinterpret_cast<uint64_t *>(static_cast<char *>(workspace) + L.part_off);
  a.part_ml = reinterpret_cast<uint64_t *>(static_cast<char *>(workspace) + L.ml_off);
  a.counters = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + L.counters_off);
  a.epochs = reinterpret_cast<uint32_t *>(static_cast<char *>(workspace) + L.epochs_off);
  a.status = status;
  a.n_cells = k->n_cells;
  a.kv_len = kv_len;
  a.chunk = L.chunk;
  a.n_splits = L.n_splits;
  a.n_kv_heads = launch_heads;
  a.kv_rep = group / kgroup;
  a.hkv = k->n_kv_heads * a.kv_rep;          // launch heads per sequence
  a.n_seq = n_seq;
  a.q_type = q_type;
  for (int i = 0; i < n_seq; ++i) {
    a.seq_cell0[i] = seq_cell0[i];
    a.seq_len[i] = seq_len[i];
  }
  a.group = kgroup;
  a.dk = k->head_dim;
  a.dv = v->head_dim;
  a.nbk = k->n_blocks;
  a.nbv = v->n_blocks;
  a.part_stride = 128 * v->n_blocks;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.v_thresh = v_thresh;
  a.coop = static_cast<int64_t>(L.n_splits) * launch_heads <= sm_count();
  a.test_drop_split = drop_split + 1;
  a.v_log2_thresh = v_thresh > 0.f ? log2f(v_thresh) : -INFINITY;
  a.cbk = to_dev(cbk);
  a.cbv = to_dev(cbv);
  code_byte_tables(cbk, k->type, a.tabk);
  code_byte_tables(cbv, v->type, a.tabv);
  if (append && use == TQ_DECODE_MMA) {
    a.k_src = k_row;
    a.v_src = v_row;
    a.cell_id = cell_id;
    a.src_type = src_type;
    const int es = (src_type == TQ_F32) ? 4 : 2;
    a.row_async = (k->head_dim * es) % 16 == 0 && (v->head_dim * es) % 16 == 0;
  }
  if (clear_counters) {
    const cudaError_t ec = cudaMemsetAsync(static_cast<char *>(workspace) + L.counters_off, 0,
                                           L.ml_off - L.counters_off, s);
    if (ec != cudaSuccess) return map_cuda(ec);
  }
  cudaError_t e = (use == TQ_DECODE_MMA) ? launch_decode_mma(k->type, v->type, a, s)
                                         : launch_decode_lut(k->type, v->type, a, s);
  return map_cuda(e);
}

}  // extern "C"

namespace tq {
tq_status decode_counters_cleared(const tq_cache *k, const tq_cache *v, const tq_codebook *cbk,
                                  const tq_codebook *cbv, const float *q, int n_q_heads, int64_t kv_len,
                                  float scale, int algo, float *out, void *workspace, size_t workspace_bytes,
                                  tq_stream stream) {
  return decode_call(k, v, cbk, cbv, nullptr, nullptr, 0, nullptr, q, n_q_heads, kv_len, scale, 0.f, algo, out,
                     workspace, workspace_bytes, stream, true);
}
}  // namespace tq

extern "C" {

tq_status tq_fattn_decode(const tq_cache *k, const tq_cache *v, const tq_codebook *cbk,
                          const tq_codebook *cbv, const float *q, int n_q_heads, int64_t kv_len,
                          float scale, int algo, float *out, void *workspace,
                          size_t workspace_bytes, tq_stream stream) {
  return decode_call(k, v, cbk, cbv, nullptr, nullptr, 0, nullptr, q, n_q_heads, kv_len, scale, 0.f, algo, out,
                     workspace, workspace_bytes, stream);
}

size_t tq_fattn_decode_batch_workspace(const tq_cache *k, const tq_cache *v, int n_q_heads, int n_seq,
                                       int64_t max_len) {
  if (check_kv_pair(k, v, n_q_heads, 0) != TQ_OK || n_seq < 1 || n_seq > kMaxDecodeSeqs || max_len < 0 ||
      max_len > k->n_cells || !decode_mma_ok(k, v, n_q_heads, n_seq))
    return 0;
  const int heads = static_cast<int>(decode_launch_heads(k->n_kv_heads, n_q_heads / k->n_kv_heads, n_seq,
                                                         TQ_DECODE_MMA));
  return decode_layout(heads, n_seq * n_q_heads, v->n_blocks, max_len, TQ_DECODE_MMA).total;
}

tq_status tq_fattn_decode_batch(const tq_cache *k, const tq_cache *v, const tq_codebook *cbk, const tq_codebook *cbv,
                                const float *q, int n_q_heads, int n_seq, const int64_t *seq_cell0,
                                const int64_t *seq_len, float scale, int algo, float *out, void *workspace,
                                size_t workspace_bytes, tq_stream stream) {
  tq_status st = check_kv_pair(k, v, n_q_heads, 0);
  if (st != TQ_OK) return st;
  if (n_seq < 1 || n_seq > kMaxDecodeSeqs || !seq_cell0 || !seq_len) return TQ_ERR_INVALID_ARG;
  if (algo == TQ_DECODE_LUT || !decode_mma_ok(k, v, n_q_heads, n_seq)) return TQ_ERR_UNSUPPORTED;
  int64_t max_len = 0;
  for (int i = 0; i < n_seq; ++i) {
    // whole 64-cell groups of each sequence lie inside the cache (the kernels
    // copy keys in groups of 32 and 64)
    if (seq_cell0[i] < 0 || seq_cell0[i] % 64 != 0 || seq_len[i] < 0 ||
        seq_cell0[i] + (seq_len[i] + 63) / 64 * 64 > k->n_cells)
      return TQ_ERR_INVALID_ARG;
    if (seq_len[i] > max_len) max_len = seq_len[i];
  }
  return decode_call(k, v, cbk, cbv, nullptr, nullptr, 0, nullptr, q, n_q_heads, max_len, scale, 0.f, algo, out,
                     workspace, workspace_bytes, stream, false, -1, n_seq, seq_cell0, seq_len);
}

tq_status tq_testing_decode_drop_split(const tq_cache *k, const tq_cache *v, const tq_codebook *cbk,
                                       const tq_codebook *cbv, const float *q, int n_q_heads, int64_t kv_len,
                                       float scale, int algo, float *out, void *workspace, size_t workspace_bytes,
                                       int drop_split, tq_stream stream) {
  if (drop_split < 0) return TQ_ERR_INVALID_ARG;
  return decode_call(k, v, cbk, cbv, nullptr, nullptr, 0, nullptr, q, n_q_heads, kv_len, scale, 0.f, algo, out,
                     workspace, workspace_bytes, stream, false, drop_split);
}

tq_status tq_fattn_decode_sparse_v(const tq_cache *k, const tq_cache *v, const tq_codebook *cbk,
                                   const tq_codebook *cbv, const float *q, int n_q_heads, int64_t kv_len,
                                   float scale, float v_threshold, int algo, float *out, void *workspace,
                                   size_t workspace_bytes, tq_stream stream) {
  return decode_call(k, v, cbk, cbv, nullptr, nullptr, 0, nullptr, q, n_q_heads, kv_len, scale, v_threshold, algo,
                     out, workspace, workspace_bytes, stream);
}

tq_status tq_fattn_decode_append(const tq_cache *k, const tq_cache *v, const tq_codebook *cbk,
                                 const tq_codebook *cbv, const void *k_row, const void *v_row, int src_type,
                                 const int64_t *cell_id, const float *q, int n_q_heads, int64_t kv_len,
                                 float scale, int algo, float *out, void *workspace, size_t workspace_bytes,
                                 tq_stream stream) {
  if (!k_row) return TQ_ERR_INVALID_ARG;
  return decode_call(k, v, cbk, cbv, k_row, v_row, src_type, cell_id, q, n_q_heads, kv_len, scale, 0.f, algo, out,
                     workspace, workspace_bytes, stream);
}

// Prefill calls with few query rows (decode steps of speculative verification)
// take the decode kernel ([HIP#28] "1. Graph-safe decode" routes up to two query
// rows to the decode path; here up to eight, where a 128-row prefill tile would
// be mostly empty): query row i becomes one sequence of a batched decode over
// cells 0 .. p_i of the same caches.
constexpr int kPrefillAsDecodeMaxRows = 8;
static bool prefill_as_decode(const tq_cache *k, const tq_cache *v, int nq, int n_q_heads) {
  return nq >= 1 && nq <= kPrefillAsDecodeMaxRows && decode_mma_ok(k, v, n_q_heads, nq);
}

size_t tq_fattn_prefill_workspace(const tq_cache *k, const tq_cache *v, int nq, int n_q_heads,
                                  int64_t kv_len) {
  if (check_kv_pair(k, v, n_q_heads, kv_len) != TQ_OK || nq < 0) return 0;
  size_t total = prefill_layout(nq, n_q_heads / k->n_kv_heads, k->n_kv_heads, kv_len, k->n_blocks, v->n_blocks).total;
  if (prefill_as_decode(k, v, nq, n_q_heads)) {
    const int heads = static_cast<int>(decode_launch_heads(k->n_kv_heads, n_q_heads / k->n_kv_heads, nq,
                                                           TQ_DECODE_MMA));
    const size_t d = decode_layout(heads, nq * n_q_heads, v->n_blocks, kv_len, TQ_DECODE_MMA).total;
    if (d > total) total = d;
  }
  return total;
}

tq_status tq_fattn_prefill(const tq_cache *k, const tq_cache *v, const tq_codebook *cbk,
                           const tq_codebook *cbv, const void *q, int q_type, int nq,
                           int n_q_heads, int64_t kv_len, float scale, int causal, float *out,
                           void *workspace, size_t workspace_bytes, tq_stream stream) {
  tq_status st = check_kv_pair(k, v, n_q_heads, kv_len);
  if (st != TQ_OK) return st;
  if (!codebook_ok(cbk, k->type) || !codebook_ok(cbv, v->type)) return TQ_ERR_INVALID_ARG;
  if (q_type != TQ_F32 && q_type != TQ_F16 && q_type != TQ_BF16) return TQ_ERR_INVALID_ARG;
  if (nq < 0 || (causal && nq > kv_len) || !isfinite(scale)) return TQ_ERR_INVALID_ARG;
  if (nq == 0) return TQ_OK;
  if (!q || !out || !aligned16(q) || !aligned16(out)) return TQ_ERR_INVALID_ARG;
  const int group = n_q_heads / k->n_kv_heads;
  if (prefill_as_decode(k, v, nq, n_q_heads) && kv_len > 0) {
    int64_t cell0[kPrefillAsDecodeMaxRows] = {}, len[kPrefillAsDecodeMaxRows];
    for (int i = 0; i < nq; ++i) len[i] = causal ? kv_len - nq + 1 + i : kv_len;
    return decode_call(k, v, cbk, cbv, nullptr, nullptr, 0, nullptr, static_cast<const float *>(q), n_q_heads,
                       kv_len, scale, 0.f, TQ_DECODE_MMA, out, workspace, workspace_bytes, stream, false, -1, nq,
                       cell0, len, q_type);
  }
  if (!prefill_supported(k->type, v->type, group, k->n_blocks, v->n_blocks)) return TQ_ERR_UNSUPPORTED;
  const PrefillWorkspaceLayout L = prefill_layout(nq, group, k->n_kv_heads, kv_len, k->n_blocks, v->n_blocks);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) || workspace_bytes < L.total)
    return TQ_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (kv_len == 0)
    return map_cuda(cudaMemsetAsync(out, 0, sizeof(float) * nq * n_q_heads * v->head_dim, s));
  if (static_cast<int64_t>(nq) * group > 0x7fffffffLL) return TQ_ERR_INVALID_ARG;
  if ((static_cast<int64_t>(nq) * group + 127) / 128 * k->n_kv_heads * 16 > 0x7fffffffLL) return TQ_ERR_UNSUPPORTED;
  PrefillArgs a;
  memset(&a, 0, sizeof(a));
  a.kn = static_cast<const uint16_t *>(k->norms);
  a.kqs = static_cast<const uint8_t *>(k->qs);
  a.ksg = static_cast<const uint8_t *>(k->signs);
  a.vn = static_cast<const uint16_t *>(v->norms);
  a.vqs = static_cast<const uint8_t *>(v->qs);
  a.vsg = static_cast<const uint8_t *>(v->signs);
  a.q = q;
  a.out = out;
  a.status = static_cast<int32_t *>(workspace);
  a.n_cells = k->n_cells;
  a.kv_len = kv_len;
  a.q_type = q_type;
  a.nq = nq;
  a.n_q_heads = n_q_heads;
  a.n_kv_heads = k->n_kv_heads;
  a.group = group;
  a.dk = k->head_dim;
  a.dv = v->head_dim;
  a.nbk = k->n_blocks;
  a.nbv = v->n_blocks;
  a.causal = causal ? 1 : 0;
  a.n_split = L.n_split;
  a.part = reinterpret_cast<float *>(static_cast<char *>(workspace) + L.part_off);
  a.sched = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + L.sched_off);
  a.n_qt = static_cast<int32_t>((static_cast<int64_t>(nq) * group + 127) / 128);
  a.n_items = a.n_qt * k->n_kv_heads * L.n_split;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.cbk = to_dev(cbk);
  a.cbv = to_dev(cbv);
  code_byte_tables(cbk, k->type, a.tabk);
  code_byte_tables(cbv, v->type, a.tabv);
  cudaError_t e = launch_prefill(k->type, a, s);
  if (e == cudaSuccess) e = launch_prefill_merge(a, s);       // split partials, if any
  return map_cuda(e);
}

tq_status tq_checksum_fnv1a64(const void *host_bytes, size_t n_bytes, uint64_t *out) {
  if (!out || (!host_bytes && n_bytes > 0)) return TQ_ERR_INVALID_ARG;
  const unsigned char *p = static_cast<const unsigned char *>(host_bytes);
  uint64_t h = 0xcbf29ce484222325ull;
  for (size_t i = 0; i < n_bytes; ++i) {
    h ^= p[i];
    h *= 0x100000001b3ull;
  }
  *out = h;
  return TQ_OK;
}

tq_status tq_workspace_status(void *workspace, size_t workspace_bytes, int32_t *status_out,
                              tq_stream stream) {
  if (!workspace || workspace_bytes < kWsHeader || !status_out) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess ||
      cudaMemsetAsync(workspace, 0, sizeof(v), s) != cudaSuccess)
    return map_cuda(cudaErrorUnknown);
  *status_out = v;
  return TQ_OK;
}

}  // extern "C"

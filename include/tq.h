/*
 * tq.h -- C ABI of the GB300 (sm_103a) library for attention over a
 * TurboQuant-compressed KV cache.
 *
 * Sources restated here (no code was taken from them):
 *   [TQ#36]    llama-cpp-turboquant pull request #36, four commit messages:
 *              "shuffle WHT" (SET_ROWS butterflies, stages h = 1..64),
 *              "asymmetric D" (K head dim 192 with V head dim 128, padding),
 *              "Q x centroid LUT" (per-step LUT of q[d] * centroid[c] for the
 *              single-query decode; 4/8/16 centroids; 2 qs bytes + 1 signs byte
 *              per 8 turbo3 elements), "VEC tuning" (results table; turbo2 7.5x).
 *   [HIP#28]   atomic-llama-cpp-turboquant pull request #28, "HIP/turbo3:
 *              graph-safe decode + inline-dequant TILE prefill": section
 *              "1. Graph-safe decode" (no allocation while a stream is being
 *              captured; decode with at most 2 query rows takes the VEC path),
 *              section "2. Inline-dequant TILE prefill" (dequantise K/V while
 *              loading tiles, never materialise f16 K/V), "Correctness".
 *   [QSA#1821] "qsa_prompt_attn: int8 K/V prefetched in registers and sharing
 *              one buffer": sections "What" and "Change" (prompt attention over
 *              scattered int8 K/V rows with per-row scales).
 *
 * Conventions for every call:
 *   - Pointers marked "device" are CUDA device pointers owned by the caller;
 *     the library keeps no state and allocates nothing.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream) and may be captured into a CUDA graph.
 *   - Arguments are checked on the host before anything is launched; a bad
 *     argument returns an error code and launches nothing.  A failed launch
 *     returns TQ_ERR_CUDA.  Device-side checks (e.g. a cell id out of range)
 *     write a tq_status value into a caller-provided device word and skip the
 *     offending access; they never trap.
 *   - All device buffers must be 16-byte aligned.
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or shape       */
  TQ_ERR_UNSUPPORTED = 2,   /* valid but not implemented combination            */
  TQ_ERR_WORKSPACE = 3,     /* workspace missing, misaligned or too small       */
  TQ_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed             */
  TQ_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up               */
  TQ_ERR_DEVICE_CHECK = 6   /* a device-side range check rejected an input      */
} tq_status;

typedef enum { TQ_TURBO2 = 2, TQ_TURBO3 = 3, TQ_TURBO4 = 4 } tq_type;
typedef enum { TQ_F32 = 0, TQ_F16 = 1, TQ_BF16 = 2 } tq_dtype;

/* Decode kernel choice.  LUT: the pages' per-step Q x centroid shared-memory
 * table ([TQ#36] "Q x centroid LUT").  MMA: codes unpacked in registers straight
 * into tensor-core operand fragments.  AUTO picks MMA when it supports the
 * shape, else LUT.  Both compute the same attention.
 * Shapes: MMA takes K and V of one code type, any GQA group (groups other than
 * 1, 2 and 4 run as group/4, group/2 or group launch heads per KV head, each
 * re-reading the head's cache planes; at most 256 launch heads per call), and
 * 1 or 2 blocks per row (K two and V one allowed).  LUT takes mixed types,
 * groups up to 8 and 1 or 2 blocks per row; it is the only kernel for mixed
 * K / V code types. */
typedef enum { TQ_DECODE_AUTO = 0, TQ_DECODE_LUT = 1, TQ_DECODE_MMA = 2 } tq_decode_algo;

typedef void *tq_stream; /* cudaStream_t */

/* Codebook of one cache ([TQ#36] "Q x centroid LUT": 4, 8 or 16 centroids).
 * sign_bits: the 128-entry +-1 diagonal S of the rotation; bit i of the
 *            little-endian 128-bit value set means s_i = -1.
 * centroids: n_centroids values, strictly ascending, exactly symmetric
 *            (c[i] == -c[n-1-i]) and each exactly representable in binary16.
 * tq_codebook_init fills the canonical table. */
typedef struct tq_codebook {
  uint32_t sign_bits[4];
  int32_t n_centroids;
  float centroids[16];
} tq_codebook;

/* One compressed cache (K or V) in three device planes, head-major:
 *   norms  binary16 [n_kv_heads][n_cells][n_blocks]        block L2 norms
 *   qs     uint8    [n_kv_heads][n_cells][n_blocks][32]    turbo2 / turbo3
 *                   [n_kv_heads][n_cells][n_blocks][64]    turbo4
 *   signs  uint8    [n_kv_heads][n_cells][n_blocks][16]    turbo3 only (else NULL)
 * n_blocks = ceil(head_dim / 128); head_dim is the logical width (a partial last
 * block is zero-padded before quantisation, [TQ#36] "asymmetric D").
 * n_cells must be a positive multiple of 64.
 * Codes are sign-magnitude: code k = s*(n/2) + j has value (s ? +1 : -1) *
 * centroids[n/2 + j].  Bit layout of one 128-element block:
 *   qs (turbo2/3): 8 little-endian u32 words; word w holds elements 16w..16w+15;
 *      element 16w+i (i < 8) at bits 4i..4i+1, element 16w+8+i at bits 4i+2..4i+3
 *      (turbo2: the 2-bit code; turbo3: the magnitude index j).
 *   qs (turbo4): 16 words; word w holds elements 8w..8w+7, element 8w+i at
 *      bits 4i..4i+3 (the 4-bit code).
 *   signs (turbo3): 4 words; word u holds elements 32u..32u+31; element 32u+r at
 *      bit 4(r%8) + 2 + r/8 for r < 16 and at bit 4((r-16)%8) + (r-16)/8 for r >= 16.
 * Stored size: 2.125 / 3.125 / 4.125 bits per element (turbo2 / 3 / 4); turbo2
 * is 7.5x smaller than f16 ([TQ#36] "VEC tuning"). */
typedef struct tq_cache {
  int32_t type;        /* tq_type */
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t n_blocks;
  int64_t n_cells;
  void *norms;         /* device */
  void *qs;            /* device */
  void *signs;         /* device, turbo3 only */
} tq_cache;

/* Human-readable name of a status code (static string, never NULL). */
const char *tq_status_string(int status);

/* Library ABI version (major * 100 + minor). */
int tq_version(void);

/* Host only.  Canonical codebook for `type`: the Lloyd-Max quantiser of
 * N(0, 1) (Lloyd iteration in double precision) scaled by 1/sqrt(128), each
 * centroid rounded to the nearest binary16 value; sign_bits copied in.
 * Errors: TQ_ERR_INVALID_ARG for an unknown type or NULL pointers. */
tq_status tq_codebook_init(int type, const uint32_t sign_bits[4], tq_codebook *out);

/* Host only.  Bytes of the norms / qs / signs planes for a cache of this shape
 * (signs = 0 unless turbo3).  Errors: TQ_ERR_INVALID_ARG. */
tq_status tq_cache_plane_bytes(int type, int n_kv_heads, int head_dim, int64_t n_cells,
                               size_t *norms_bytes, size_t *qs_bytes, size_t *signs_bytes);

/* SET_ROWS, quantise-on-write ([TQ#36] "shuffle WHT"): for every row r and KV
 * head h, each 128-element block x of src[r][h][:] (zero-padded to a multiple
 * of 128) is written to cell cell_ids[r] as
 *   norm  = binary16(|x|)                      (round to nearest even)
 *   y     = H S x / (|x| sqrt(128))            H: 128-point Walsh-Hadamard
 *   code  = nearest centroid of each y_i       (ties: the higher centroid)
 * src      device, src_type (TQ_F32 / TQ_F16 / TQ_BF16) [n_rows][n_kv_heads][head_dim]
 * cell_ids device int64 [n_rows]; distinct; each in [0, n_cells)
 * dev_status device int32 or NULL: a row whose cell id is out of range is
 *          skipped and TQ_ERR_DEVICE_CHECK is stored here.
 * n_rows = 0 is a no-op.  Errors: TQ_ERR_INVALID_ARG, TQ_ERR_CUDA. */
tq_status tq_set_rows(const tq_cache *dst, const tq_codebook *cb, const void *src, int src_type,
                      const int64_t *cell_ids, int64_t n_rows, int32_t *dev_status,
                      tq_stream stream);

/* Bytes of workspace tq_fattn_decode needs for this shape (0 if the shape is
 * invalid, including more than 256 KV heads).  The workspace must be 256-byte
 * aligned and zero-filled before its first use; every call leaves it ready for
 * the next one (the split counters reset themselves and a per-KV-head launch
 * epoch advances), so it can be reused across calls, shapes and graph replays
 * but not by two calls that run concurrently.  The split partials are stored
 * with a tag made of the KV head's epoch and the head's index, and the merging
 * CTA takes a value only when its tag is this launch's: decode calls of
 * different shapes (head counts, lengths, types) may share one workspace, and
 * a prefill or prompt-attention call may share it between decode calls (their
 * data never carries a decode tag, short of a 32-bit pattern coincidence) and
 * keeps the epoch words intact. */
size_t tq_fattn_decode_workspace(const tq_cache *k, const tq_cache *v, int n_q_heads,
                                 int64_t kv_len);

/* Single-query decode attention over cells 0..kv_len-1 ([TQ#36] "Q x centroid
 * LUT", "VEC tuning"; [HIP#28] "1. Graph-safe decode"):
 *   out[h][:] = softmax_t(scale * q[h] . k_t) v_t      k_t, v_t dequantised rows
 * with query head h reading KV head h / (n_q_heads / n_kv_heads).  The key range
 * is split across CTAs; each split keeps a running max/sum and the merge is a
 * log-sum-exp combination (in a cluster over distributed shared memory; else,
 * when the grid fits on the GPU at once, a cooperative launch in which each
 * output block is merged by one CTA; else by the last CTA of each KV head).
 * q    device f32 [n_q_heads][k->head_dim]
 * out  device f32 [n_q_heads][v->head_dim]
 * algo tq_decode_algo.  kv_len = 0 writes zeros.
 * Errors: TQ_ERR_INVALID_ARG (shapes, kv_len > n_cells, codebooks),
 *         TQ_ERR_UNSUPPORTED (algo cannot take this shape), TQ_ERR_WORKSPACE,
 *         TQ_ERR_CUDA. */
tq_status tq_fattn_decode(const tq_cache *k, const tq_cache *v, const tq_codebook *cbk,
                          const tq_codebook *cbv, const float *q, int n_q_heads, int64_t kv_len,
                          float scale, int algo, float *out, void *workspace,
                          size_t workspace_bytes, tq_stream stream);

/* SET_ROWS of one new token followed by decode, in one launch:
 *   tq_set_rows(k, cbk, k_row, src_type, cell_id, 1, <workspace status>);
 *   tq_set_rows(v, cbv, v_row, src_type, cell_id, 1, <workspace status>);
 *   tq_fattn_decode(k, v, cbk, cbv, q, n_q_heads, kv_len, scale, algo, out, ...);
 * with the same cache bytes and the same output as those three calls.  The
 * pages run the two SET_ROWS ops and FLASH_ATTN_EXT as separate graph nodes
 * ([TQ#36] "shuffle WHT", [HIP#28] "1. Graph-safe decode"); the tensor-core
 * decode kernel quantises the token's rows itself (in the CTA whose key range
 * holds the cell), writes them to the cache and attends the fresh codes, so
 * a decode step costs one launch instead of three.  With the LUT kernel (or
 * kv_len = 0) the three launches are issued in order instead.
 * k_row    device, src_type [k->n_kv_heads][k->head_dim], 16-byte aligned
 * v_row    device, src_type [v->n_kv_heads][v->head_dim], 16-byte aligned
 * cell_id  device int64 [1], 8-byte aligned: the cell the token is written to;
 *          it is attended when cell < kv_len.  A cell outside [0, n_cells)
 *          writes nothing and stores TQ_ERR_DEVICE_CHECK in the workspace
 *          status word (tq_workspace_status).
 * Other arguments, results and errors as tq_fattn_decode; the workspace is the
 * one tq_fattn_decode_workspace sizes. */
tq_status tq_fattn_decode_append(const tq_cache *k, const tq_cache *v, const tq_codebook *cbk,
                                 const tq_codebook *cbv, const void *k_row, const void *v_row, int src_type,
                                 const int64_t *cell_id, const float *q, int n_q_heads, int64_t kv_len,
                                 float scale, int algo, float *out, void *workspace, size_t workspace_bytes,
                                 tq_stream stream);

/* tq_fattn_decode with sparse V ([TQ#36] "VEC tuning", item 3: thresholds
 * 5e-3 for turbo3 / turbo4 and 1e-2 for turbo2).  A key whose softmax weight
 * relative to the running maximum score, exp(s - m), is below v_threshold for
 * every query head of its GQA group adds nothing to the weighted sum of V rows;
 * its weight still counts in the normaliser.  The tensor-core kernel decides per
 * group of 16 keys, the LUT kernel per key.  The running maximum is at most the
 * final one, so every key left out has exp(s - max) < v_threshold for each of
 * those heads; which of those keys are left out depends on the key order and the
 * launch shape.  v_threshold = 0 gives exactly tq_fattn_decode's result.
 * Errors: as tq_fattn_decode, and TQ_ERR_INVALID_ARG for a negative or
 * non-finite v_threshold. */
tq_status tq_fattn_decode_sparse_v(const tq_cache *k, const tq_cache *v, const tq_codebook *cbk,
                                   const tq_codebook *cbv, const float *q, int n_q_heads, int64_t kv_len,
                                   float scale, float v_threshold, int algo, float *out, void *workspace,
                                   size_t workspace_bytes, tq_stream stream);

/* Bytes of workspace tq_fattn_decode_batch needs for n_seq sequences of at
 * most max_len cells (0 if the shape is invalid: n_seq outside 1..32 or more
 * than 256 sequence x KV head pairs).  Same alignment and zero-fill rule as
 * the decode workspace. */
size_t tq_fattn_decode_batch_workspace(const tq_cache *k, const tq_cache *v, int n_q_heads, int n_seq,
                                       int64_t max_len);

/* Single-query decode of several sequences in one launch ([HIP#28]
 * "1. Graph-safe decode": decode steps of up to two query rows per sequence
 * take the decode path; here a batch of sequences, one new token each):
 * sequence s owns cells seq_cell0[s] .. seq_cell0[s] + seq_len[s] - 1 of the
 * caches and
 *   out[s][h][:] = softmax_t(scale * q[s][h] . k_t) v_t   over its cells,
 * each (sequence, KV head) pair splitting its key range over CTAs like
 * tq_fattn_decode.
 * q          device f32 [n_seq][n_q_heads][k->head_dim]
 * out        device f32 [n_seq][n_q_heads][v->head_dim]
 * seq_cell0, seq_len  HOST int64 [n_seq]: each seq_cell0 a multiple of 64 and
 *            seq_cell0 + seq_len rounded up to 64 within n_cells (copied into the
 *            launch, so a captured graph keeps the values it was captured with)
 * n_seq      1 .. 32, with n_seq * n_kv_heads <= 256.  A sequence of length 0
 *            gets a zero output.
 * algo       TQ_DECODE_AUTO or TQ_DECODE_MMA (the tensor-core kernel; its
 *            supported shapes are those of tq_fattn_decode's MMA kernel).
 * Errors: TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED (LUT kernel, or a shape the
 * tensor-core kernel does not take), TQ_ERR_WORKSPACE, TQ_ERR_CUDA. */
tq_status tq_fattn_decode_batch(const tq_cache *k, const tq_cache *v, const tq_codebook *cbk,
                                const tq_codebook *cbv, const float *q, int n_q_heads, int n_seq,
                                const int64_t *seq_cell0, const int64_t *seq_len, float scale, int algo,
                                float *out, void *workspace, size_t workspace_bytes, tq_stream stream);

/* tq_fattn_decode without a caller workspace, for callers that cannot
 * allocate device memory (code inside an allocator or memory-pool callback, a
 * runtime that has reserved all device memory up front, a plugin host that only
 * passes input and output buffers).  The pages have no counterpart: this is an
 * addition of this library.
 * The split partials, counters and status word live in one fixed 4 MiB device
 * array inside the library; every GPU that loads the library keeps those 4 MiB
 * until the process exits.  Shapes whose decode workspace
 * (tq_fattn_decode_workspace) exceeds 4 MiB return TQ_ERR_WORKSPACE and launch
 * nothing.  The first call on a device looks up the array's address with that
 * device current; make it before any stream capture.  Each call clears the
 * split counters on `stream` just before the kernel, after its argument checks
 * (a rejected call writes nothing).  Device-side errors (a bounded wait that
 * timed out) collect in a status word at the start of the array, which
 * tq_noalloc_status reads.  All calls share the array, so calls that overlap
 * on the GPU (different streams) race and give wrong results.  Other
 * arguments, results and errors as tq_fattn_decode. */
tq_status tq_fattn_decode_noalloc(const tq_cache *k, const tq_cache *v, const tq_codebook *cbk,
                                  const tq_codebook *cbv, const float *q, int n_q_heads,
                                  int64_t kv_len, float scale, int algo, float *out,
                                  tq_stream stream);

/* Reads and clears the status word of the array tq_fattn_decode_noalloc uses
 * on the current device, like tq_workspace_status: waits for `stream`, so it
 * must not be called while the stream is being captured.  *status_out
 * receives TQ_OK or the first device-side error of the calls since the last
 * read (TQ_ERR_TIMEOUT).  Like the entry point it serves, an addition of this
 * library with no counterpart on the pages.  Errors: TQ_ERR_INVALID_ARG,
 * TQ_ERR_CUDA. */
tq_status tq_noalloc_status(int32_t *status_out, tq_stream stream);

/* Bytes of workspace tq_fattn_prefill needs (0 if the shape is invalid);
 * same alignment and zero-fill rule as the decode workspace. */
size_t tq_fattn_prefill_workspace(const tq_cache *k, const tq_cache *v, int nq, int n_q_heads,
                                  int64_t kv_len);

/* Multi-query (prefill / verify) attention with inline dequantisation
 * ([HIP#28] "2. Inline-dequant TILE prefill"): packed K/V tiles are expanded
 * to fp16 operand tiles in shared memory and multiplied on the tcgen05 tensor
 * cores; no f16 copy of the cache is ever written to global memory.
 *   out[i][h][:] = softmax_{t <= p_i}(scale * q[i][h] . k_t) v_t,
 *   p_i = kv_len - nq + i when causal, else every t < kv_len.
 * q    device, q_type (TQ_BF16, TQ_F16 or TQ_F32) [nq][n_q_heads][k->head_dim]
 * out  device f32 [nq][n_q_heads][v->head_dim]
 * Requires nq <= kv_len when causal.  Calls with nq <= 8 (decode steps that
 * verify draft tokens) run on the decode kernel instead when it takes the
 * shape ([HIP#28] "1. Graph-safe decode" sends up to two query rows down the
 * decode path; a 128-row prefill tile would be mostly empty up to eight), each
 * query row as one sequence of a batched decode; the workspace size returned
 * below covers both.  When the query tiles do not fill the GPU, the key range
 * of each is split; the call then issues a second kernel on `stream` that
 * merges the splits (both are captured alike in a CUDA graph).
 * Errors: TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_WORKSPACE, TQ_ERR_CUDA. */
tq_status tq_fattn_prefill(const tq_cache *k, const tq_cache *v, const tq_codebook *cbk,
                           const tq_codebook *cbv, const void *q, int q_type, int nq,
                           int n_q_heads, int64_t kv_len, float scale, int causal, float *out,
                           void *workspace, size_t workspace_bytes, tq_stream stream);

/* Bytes of workspace tq_int8_prompt_attn needs (0 if the shape is invalid). */
size_t tq_int8_prompt_attn_workspace(int nq, int n_q_heads, int n_kv_heads, int head_dim,
                                     int64_t ctx);

/* Prompt attention over an int8 KV cache with per-row scales whose rows are
 * scattered over the cells ([QSA#1821] "What", "Change"):
 *   k_t = k[cell_of_pos[t]][hk][:] * float(k_scale[cell_of_pos[t]][hk])   (v alike)
 *   out[i][h][:] = softmax_{t <= p_i}(scale * q[i][h] . k_t) v_t,  p_i = ctx - nq + i
 * (every t < ctx when causal = 0).
 * k, v        device int8 [n_cells][n_kv_heads][head_dim]
 * k_scale, v_scale device binary16 [n_cells][n_kv_heads]
 * cell_of_pos device int32 [ctx], each in [0, n_cells)
 * q           device binary16 [nq][n_q_heads][head_dim]
 * out         device f32 [nq][n_q_heads][head_dim]
 * head_dim must be 128.  A cell id out of range is read as a zero row and
 * TQ_ERR_DEVICE_CHECK is stored in the workspace status word (tq_workspace_status).
 * Errors: TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED, TQ_ERR_WORKSPACE, TQ_ERR_CUDA. */
tq_status tq_int8_prompt_attn(const int8_t *k, const uint16_t *k_scale, const int8_t *v,
                              const uint16_t *v_scale, int64_t n_cells, const int32_t *cell_of_pos,
                              int64_t ctx, const uint16_t *q, int nq, int n_q_heads,
                              int n_kv_heads, int head_dim, float scale, int causal, float *out,
                              void *workspace, size_t workspace_bytes, tq_stream stream);

/* The same prompt attention over a binary16 KV cache (the other cache mode of
 * [QSA#1821], whose output checksums the page compares alongside int8): rows
 *   k_t = k[cell_of_pos[t]][hk][:],  v_t = v[cell_of_pos[t]][hk][:]   (no scales)
 * k, v   device binary16 [n_cells][n_kv_heads][head_dim], 16-byte aligned
 * Other arguments, the workspace (tq_int8_prompt_attn_workspace), results and
 * errors as tq_int8_prompt_attn. */
tq_status tq_f16_prompt_attn(const uint16_t *k, const uint16_t *v, int64_t n_cells,
                             const int32_t *cell_of_pos, int64_t ctx, const uint16_t *q, int nq,
                             int n_q_heads, int n_kv_heads, int head_dim, float scale, int causal,
                             float *out, void *workspace, size_t workspace_bytes, tq_stream stream);

/* Host only.  64-bit FNV-1a hash of n_bytes host bytes (offset basis
 * 0xcbf29ce484222325, prime 0x100000001b3), so that two builds' outputs can be
 * compared bit for bit from one printed number ([QSA#1821] "Measured": each
 * mode prints a checksum of its output).  Errors: TQ_ERR_INVALID_ARG for a
 * NULL pointer with n_bytes > 0 or a NULL out. */
tq_status tq_checksum_fnv1a64(const void *host_bytes, size_t n_bytes, uint64_t *out);

/* Reads (and clears) the device status word kept in a workspace of the
 * calls above: waits for `stream`, so it must not be called while the stream
 * is being captured.  *status_out receives TQ_OK or the first device-side
 * error (TQ_ERR_DEVICE_CHECK, TQ_ERR_TIMEOUT).  Errors: TQ_ERR_INVALID_ARG,
 * TQ_ERR_CUDA. */
tq_status tq_workspace_status(void *workspace, size_t workspace_bytes, int32_t *status_out,
                              tq_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H */

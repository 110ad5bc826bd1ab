// Internal declarations shared by the host API and the kernel translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/tq.h"

namespace tq {

constexpr int kMaxDecodeSeqs = 32;   // sequences of one batched decode launch

// Codebook as the kernels receive it (by value, in the launch parameters).
struct DevCodebook {
  uint32_t sign_bits[4];
  int32_t n;
  float c[16];
};

struct SetRowsArgs {
  const void *src;
  const int64_t *cell_ids;
  int32_t *dev_status;
  uint16_t *norms;
  uint8_t *qs;
  uint8_t *signs;
  int64_t n_rows;
  int64_t n_cells;
  int32_t n_kv_heads;
  int32_t head_dim;
  int32_t n_blocks;
  DevCodebook cb;
};

// Everything a decode kernel needs; the partial results of split s of query
// head h are m (log2 domain), l at part_ml + 2 (h * n_splits + s) and
// o'[0 .. 128 nbv) (unnormalised, rotated domain) at part + (h * n_splits + s) * part_stride,
// each value in a 64-bit word with its launch tag (tq_decode_common.cuh).
struct DecodeArgs {
  const uint16_t *kn;
  const uint8_t *kqs;
  const uint8_t *ksg;
  const uint16_t *vn;
  const uint8_t *vqs;
  const uint8_t *vsg;
  const float *q;
  float *out;
  uint64_t *part;         // split outputs o'[h][split][part_stride], tagged words
  uint64_t *part_ml;      // split maxima and sums [h][split][2], tagged words
  int32_t *counters;      // [kv head] arrivals, self-resetting
  uint32_t *epochs;       // [kv head] launch epochs (tags of the partials)
  int32_t *status;        // workspace status word (device-side errors)
  int64_t n_cells;
  int64_t kv_len;
  int64_t chunk;
  int32_t n_splits;
  int32_t n_kv_heads;
  int32_t group;          // query heads per launch head (tensor-core kernel: 1, 2 or 4)
  int32_t kv_rep;         // launch heads per cache head (query heads per KV head / group)
  int32_t dk, dv;         // logical head dims
  int32_t nbk, nbv;       // 128-blocks of K / V rows
  int32_t part_stride;    // words per (head, split) partial output (128 nbv)
  float scale_log2;       // softmax scale * log2(e)
  float v_thresh;         // sparse V: weight relative to the running maximum below which V is skipped (0 = off)
  float v_log2_thresh;    // log2(v_thresh)
  DevCodebook cbk, cbv;
  uint32_t tabk[4], tabv[4];   // binary16 byte tables of the code values (see code_byte_tables)
  // append: the new token's K / V rows ([n_kv_heads][dk], [n_kv_heads][dv] of
  // src_type) are quantised into cell *cell_id before it is attended; null = none
  const void *k_src;
  const void *v_src;
  const int64_t *cell_id;
  int32_t src_type;
  int32_t row_async;      // every head's source rows start 16-byte aligned: staged by cp.async
  int32_t coop;           // the grid fits on the GPU at once: cooperative launch, merge by every CTA
  int32_t test_drop_split;  // 1 + a split whose partial is never stored (0: none); set only by
                            // tq_testing_decode_drop_split, to make the merge's bounded waits run out
  // several sequences in one launch (tq_fattn_decode_batch; n_seq = 0 otherwise):
  // launch head y = sequence y / hkv, head y % hkv of the sequence's hkv launch
  // heads (KV head (y % hkv) / kv_rep); sequence s attends its
  // seq_len[s] cells starting at cell seq_cell0[s]; q, out and the split
  // bookkeeping are indexed by launch head (sequence-major)
  int32_t n_seq;
  int32_t hkv;
  int32_t q_type;         // TQ_F32 (0, decode's own calls), TQ_F16 or TQ_BF16: element type of q
  int64_t seq_cell0[kMaxDecodeSeqs];
  int64_t seq_len[kMaxDecodeSeqs];
};

struct PrefillArgs {
  const uint16_t *kn;
  const uint8_t *kqs;
  const uint8_t *ksg;
  const uint16_t *vn;
  const uint8_t *vqs;
  const uint8_t *vsg;
  const void *q;
  float *out;
  int32_t *status;
  float *part;            // split partials [q tile][kv head][split][128 rows][4 + 128 nbv]
  int32_t *sched;         // [0] next work item, [1] CTAs done (both reset by the last CTA)
  int64_t n_cells;
  int64_t kv_len;
  int32_t q_type;
  int32_t nq;
  int32_t n_q_heads;
  int32_t n_kv_heads;
  int32_t group;
  int32_t dk, dv;
  int32_t nbk, nbv;
  int32_t causal;
  int32_t n_split;        // key-range splits per query tile
  int32_t n_qt;           // query tiles of 128 rows
  int32_t n_items;        // work items: query tiles x KV heads x splits, longest first
  float scale_log2;
  DevCodebook cbk, cbv;
  uint32_t tabk[4], tabv[4];
};

struct DecodeWorkspaceLayout {
  size_t epochs_off, counters_off, ml_off, part_off, total;
  int n_splits;
  int64_t chunk;
};

constexpr size_t kWsHeader = 256;   // status word lives at offset 0
// Decode epochs of KV heads 0 .. 255 sit at a fixed place after the header in
// every workspace layout, so no other use of a shared workspace overwrites them
// and a change of decode shape keeps each head's epoch word.
constexpr size_t kWsEpochBytes = 1024;
constexpr int kMaxDecodeKvHeads = 256;

int sm_count();
bool cluster_merge_ok(const void *kern, int csize, int threads, size_t smem, int want);
cudaError_t set_dynamic_smem(const void *kern, int bytes);
// prmt byte tables of a codebook's binary16 code values: t[0], t[1] low bytes of
// codes 0..3 / 4..7, t[2], t[3] high bytes (turbo4: magnitudes 0..7).
void code_byte_tables(const tq_codebook *cb, int type, uint32_t t[4]);
DecodeWorkspaceLayout decode_layout(int n_kv_heads, int n_q_heads, int nbv, int64_t kv_len, int algo);

cudaError_t launch_set_rows(int type, int src_type, const SetRowsArgs &a, cudaStream_t s);
cudaError_t launch_decode_lut(int ktype, int vtype, const DecodeArgs &a, cudaStream_t s);
// The tensor-core decode kernel serves 1, 2 or 4 query heads per launch head.
// A GQA group of another size runs as group / mma_group(group) launch heads per
// KV head, all of them reading that head's cache planes.
constexpr int mma_group(int group) { return group % 4 == 0 ? 4 : (group % 2 == 0 ? 2 : 1); }
bool decode_mma_supported(int ktype, int vtype, int group, int nbk, int nbv);
cudaError_t launch_decode_mma(int ktype, int vtype, const DecodeArgs &a, cudaStream_t s);
cudaError_t launch_decode_mma_t2(const DecodeArgs &a, cudaStream_t s);
cudaError_t launch_decode_mma_t3(const DecodeArgs &a, cudaStream_t s);
cudaError_t launch_decode_mma_t4(const DecodeArgs &a, cudaStream_t s);
bool prefill_supported(int ktype, int vtype, int group, int nbk, int nbv);
struct PrefillWorkspaceLayout {
  int n_split;
  size_t sched_off, part_off, total;
};
PrefillWorkspaceLayout prefill_layout(int nq, int group, int n_kv_heads, int64_t kv_len, int nbk, int nbv);
// merge of a prefill launch's key-range splits (a no-op without splits)
cudaError_t launch_prefill_merge(const PrefillArgs &a, cudaStream_t s);
cudaError_t launch_prefill(int ktype, const PrefillArgs &a, cudaStream_t s);
// tq_fattn_decode that also zeroes the workspace's split counters on the stream
// just before the kernel, once every argument has been checked.
tq_status decode_counters_cleared(const tq_cache *k, const tq_cache *v, const tq_codebook *cbk,
                                  const tq_codebook *cbv, const float *q, int n_q_heads, int64_t kv_len,
                                  float scale, int algo, float *out, void *workspace, size_t workspace_bytes,
                                  tq_stream stream);

}  // namespace tq

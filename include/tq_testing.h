/*
 * tq_testing.h -- a test hook of libtq, not part of the product API.
 *
 * The decode kernels' split merge waits, a bounded number of times, for every
 * split's partial result ([HIP#28] "1. Graph-safe decode": a decode call must
 * never hang a captured graph).  To show that such a wait ends and reports
 * instead of hanging, a test needs a partial that never arrives; this entry
 * point is tq_fattn_decode with one split's partial store left out.
 */
#ifndef TQ_TESTING_H
#define TQ_TESTING_H

#include "tq.h"

#ifdef __cplusplus
extern "C" {
#endif

/* tq_fattn_decode in which split `drop_split` (>= 0) of every KV head computes
 * but never stores its partial result, so the merging CTAs' bounded waits run
 * out (tens of milliseconds): the call returns, the merge uses the words it
 * found, and the workspace status word (tq_workspace_status) reads
 * TQ_ERR_TIMEOUT.  A split index beyond the launch's splits drops nothing.
 * The output is then not the attention result.  Errors: as tq_fattn_decode,
 * and TQ_ERR_INVALID_ARG for a negative drop_split. */
tq_status tq_testing_decode_drop_split(const tq_cache *k, const tq_cache *v, const tq_codebook *cbk,
                                       const tq_codebook *cbv, const float *q, int n_q_heads, int64_t kv_len,
                                       float scale, int algo, float *out, void *workspace, size_t workspace_bytes,
                                       int drop_split, tq_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* TQ_TESTING_H */

"""The decode merge's bounded waits end and report instead of hanging.

A test hook (include/tq_testing.h) leaves one split's partial result unstored,
so every CTA that merges an output block of a KV head waits for a partial that
never arrives.  The wait is bounded (tens of milliseconds): the call returns,
the workspace status word reads TQ_ERR_TIMEOUT, the output stays finite, and
the next regular call on the same workspace is correct again.  No GPU fault,
trap or endless loop is involved: the failure is a partial the host asked the
kernel to leave out."""
import math

import numpy as np
import pytest

import oracle as O
import workloads as W
from tests._helpers import compare_outputs, oracle_cache, upload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("algo", ["mma", "lut"])
def test_merge_wait_times_out_and_reports(algo):
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    from quantized_kv_cache_tq_gb300 import _lib

    sh = W.decode_32k()
    kv_len = 8192                              # 19 splits per KV head: the cooperative merge
    k, v = W.kv_inputs(sh, kv_len)
    sk, sv = W.codebook_signs(sh)
    kc, vc = oracle_cache(3, k, sk), oracle_cache(3, v, sv)
    gk, gv = upload(kc), upload(vc)
    cbk, cbv = tq.codebook(3, sk), tq.codebook(3, sv)
    q = torch.from_numpy(W.to_f32(W.decode_query(sh))).cuda()
    scale = 1.0 / math.sqrt(sh.head_dim_k)
    code = {"mma": tq.TQ_DECODE_MMA, "lut": tq.TQ_DECODE_LUT}[algo]
    ws = tq.workspace(_lib.tq_fattn_decode_workspace(gk.c, gv.c, sh.n_q_heads, kv_len))
    stream = torch.cuda.current_stream().cuda_stream
    out = torch.full((sh.n_q_heads, sh.head_dim_v), float("nan"), device="cuda")

    st = _lib.tq_testing_decode_drop_split(gk.c, gv.c, cbk, cbv, q.data_ptr(), sh.n_q_heads, kv_len, scale, code,
                                           out.data_ptr(), ws.data_ptr(), ws.numel(), 3, stream)
    assert st == _lib.TQ_OK
    torch.cuda.synchronize()
    assert _lib.tq_workspace_status(ws.data_ptr(), ws.numel(), stream) == _lib.TQ_ERR_TIMEOUT
    assert torch.isfinite(out).all()

    # the same workspace serves the next regular call: correct output, clean status
    out2 = tq.fattn_decode(gk, gv, cbk, cbv, q, kv_len, scale, algo=code, ws=ws)
    torch.cuda.synchronize()
    assert _lib.tq_workspace_status(ws.data_ptr(), ws.numel(), stream) == _lib.TQ_OK
    ref = O.decode(kc, vc, sk, sv, O.centroids(3), O.centroids(3), q.cpu().numpy().astype(np.float64), kv_len,
                   scale)
    compare_outputs(out2.cpu().numpy(), ref)


def test_drop_split_rejects_negative_index():
    import quantized_kv_cache_tq_gb300 as tq
    from quantized_kv_cache_tq_gb300 import _lib
    c = tq.TqCache(3, 1, 128, 64)
    cb = tq.codebook(3, [0, 0, 0, 0])
    st = _lib.tq_testing_decode_drop_split(c.c, c.c, cb, cb, 1 << 20, 1, 64, 0.1, 0, 1 << 20, 1 << 20, 1 << 20,
                                           -1, None)
    assert st == _lib.TQ_ERR_INVALID_ARG

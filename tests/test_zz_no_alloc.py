"""The allocation-free decode entry point (for callers that cannot allocate
device memory) against the regular workspace entry point, through the C ABI.

Collected last on purpose: it runs after every other test, and must also pass
on its own in a fresh process."""
import math

import numpy as np
import pytest

import oracle as O
import workloads as W
from tests._helpers import MAX_ABS, MAX_NMSE, oracle_cache, upload

pytestmark = pytest.mark.gpu


def test_noalloc_matches_workspace_decode_twice():
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    from quantized_kv_cache_tq_gb300 import _lib

    sh = W.decode_32k()
    kv_len = 3000
    k, v = W.kv_inputs(sh, kv_len)
    sk, sv = W.codebook_signs(sh)
    gk, gv = upload(oracle_cache(3, k, sk)), upload(oracle_cache(3, v, sv))
    cbk, cbv = tq.codebook(3, sk), tq.codebook(3, sv)
    q = torch.from_numpy(W.to_f32(W.decode_query(sh))).cuda()
    scale = 1.0 / math.sqrt(sh.head_dim_k)
    stream = torch.cuda.current_stream().cuda_stream

    ref = torch.empty(sh.n_q_heads, sh.head_dim_v, device="cuda")
    ws = tq.workspace(_lib.tq_fattn_decode_workspace(gk.c, gv.c, sh.n_q_heads, kv_len))
    st = _lib.tq_fattn_decode(gk.c, gv.c, cbk, cbv, q.data_ptr(), sh.n_q_heads, kv_len, scale,
                              tq.TQ_DECODE_AUTO, ref.data_ptr(), ws.data_ptr(), ws.numel(), stream)
    assert st == _lib.TQ_OK

    for _ in range(2):                       # two calls in a row share the library's array
        out = torch.full((sh.n_q_heads, sh.head_dim_v), float("nan"), device="cuda")
        st = _lib.tq_fattn_decode_noalloc(gk.c, gv.c, cbk, cbv, q.data_ptr(), sh.n_q_heads, kv_len, scale,
                                          tq.TQ_DECODE_AUTO, out.data_ptr(), stream)
        assert st == _lib.TQ_OK, _lib.status_string(st)
        torch.cuda.synchronize()
        a, b = out.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)
        assert np.all(np.isfinite(a))
        assert np.max(np.abs(a - b)) <= MAX_ABS
        assert O.nmse(a, b) <= MAX_NMSE


def test_noalloc_rejects_oversized_shape():
    import quantized_kv_cache_tq_gb300 as tq
    from quantized_kv_cache_tq_gb300 import _lib
    # 512 query heads of width 256 over one KV head: the split partials exceed 4 MiB
    gk, gv = tq.TqCache(3, 1, 256, 1 << 16), tq.TqCache(3, 1, 256, 1 << 16)
    cb = tq.codebook(3, [1, 2, 3, 4])
    need = _lib.tq_fattn_decode_workspace(gk.c, gv.c, 512, 1 << 16)
    assert need > (4 << 20)
    st = _lib.tq_fattn_decode_noalloc(gk.c, gv.c, cb, cb, 1 << 20, 512, 1 << 16, 0.1, 0, 1 << 20, None)
    assert st == _lib.TQ_ERR_WORKSPACE

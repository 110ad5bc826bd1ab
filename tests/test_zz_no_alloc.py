"""The allocation-free decode entry point against the regular workspace entry
point, through the C ABI.

Some callers cannot call cudaMalloc where they run decode: code inside a custom
allocator or memory-pool callback, a runtime that has reserved all device
memory up front, or a plugin host that only hands out input and output
buffers.  tq_fattn_decode_noalloc serves them from a fixed array inside the
library; these tests check that it gives the workspace decode's output, call
after call, and that its status word stays clean.

Collected last on purpose: it runs after every other test, and must also pass
on its own in a fresh process."""
import math

import numpy as np
import pytest

import oracle as O
import workloads as W
from tests._helpers import MAX_ABS, MAX_NMSE, oracle_cache, upload

pytestmark = pytest.mark.gpu


def _algo(name):
    import quantized_kv_cache_tq_gb300 as tq
    return {"mma": tq.TQ_DECODE_MMA, "lut": tq.TQ_DECODE_LUT, "auto": tq.TQ_DECODE_AUTO}[name]


class _Case:
    """One decode shape: caches, codebooks and query on the GPU."""

    def __init__(self, sh, n_rows):
        import torch
        import quantized_kv_cache_tq_gb300 as tq
        k, v = W.kv_inputs(sh, n_rows)
        sk, sv = W.codebook_signs(sh)
        self.sh = sh
        self.gk, self.gv = upload(oracle_cache(3, k, sk)), upload(oracle_cache(3, v, sv))
        self.cbk, self.cbv = tq.codebook(3, sk), tq.codebook(3, sv)
        self.q = torch.from_numpy(W.to_f32(W.decode_query(sh))).cuda()
        self.scale = 1.0 / math.sqrt(sh.head_dim_k)

    def workspace_decode(self, kv_len, algo):
        import torch
        import quantized_kv_cache_tq_gb300 as tq
        from quantized_kv_cache_tq_gb300 import _lib
        sh = self.sh
        ref = torch.empty(sh.n_q_heads, sh.head_dim_v, device="cuda")
        ws = tq.workspace(_lib.tq_fattn_decode_workspace(self.gk.c, self.gv.c, sh.n_q_heads, kv_len))
        st = _lib.tq_fattn_decode(self.gk.c, self.gv.c, self.cbk, self.cbv, self.q.data_ptr(), sh.n_q_heads,
                                  kv_len, self.scale, algo, ref.data_ptr(), ws.data_ptr(), ws.numel(),
                                  torch.cuda.current_stream().cuda_stream)
        assert st == _lib.TQ_OK
        return ref

    def noalloc_decode(self, kv_len, algo):
        import torch
        from quantized_kv_cache_tq_gb300 import _lib
        sh = self.sh
        out = torch.full((sh.n_q_heads, sh.head_dim_v), float("nan"), device="cuda")
        stream = torch.cuda.current_stream().cuda_stream
        st = _lib.tq_fattn_decode_noalloc(self.gk.c, self.gv.c, self.cbk, self.cbv, self.q.data_ptr(),
                                          sh.n_q_heads, kv_len, self.scale, algo, out.data_ptr(), stream)
        assert st == _lib.TQ_OK, _lib.status_string(st)
        assert _lib.tq_noalloc_status(stream) == _lib.TQ_OK      # no bounded wait gave up
        return out


def _same(out, ref):
    import torch
    torch.cuda.synchronize()
    a, b = out.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(a))
    assert np.max(np.abs(a - b)) <= MAX_ABS
    assert O.nmse(a, b) <= MAX_NMSE


@pytest.mark.parametrize("algo", ["mma", "lut"])
def test_noalloc_matches_workspace_decode_twice(algo):
    case = _Case(W.decode_32k(), 3000)
    ref = case.workspace_decode(3000, _algo(algo))
    for _ in range(2):                       # two calls in a row share the library's array
        _same(case.noalloc_decode(3000, _algo(algo)), ref)


@pytest.mark.parametrize("algo", ["mma", "lut"])
def test_noalloc_shape_changes_between_calls(algo):
    # large, small, large again on one stream, then another head count: split
    # partials an earlier call left in the array carry an older epoch and are
    # never taken by a later call
    big = _Case(W.decode_32k(), 8192)
    other = _Case(W.AttnShape("noalloc_2kv", 2, 8, 128, 128, 1500, seed=41), 1500)
    seq = [(big, 8192), (big, 700), (big, 8192), (other, 1500), (big, 129), (other, 1500)]
    refs = {(id(c), n): c.workspace_decode(n, _algo(algo)) for c, n in seq}
    for c, n in seq:
        _same(c.noalloc_decode(n, _algo(algo)), refs[(id(c), n)])


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

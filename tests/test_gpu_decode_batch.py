"""Decode of several sequences in one launch (tq_fattn_decode_batch) on the GPU:
each sequence's output against the f64 oracle's decode over that sequence's own
cells (max-abs <= 2e-3, NMSE <= 1e-6).  Sequences sit at different cell offsets
of one cache and have ragged lengths (including 0 and 1)."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests._helpers import compare_outputs, oracle_cache, scale_of

pytestmark = pytest.mark.gpu


def _batch(tq_type, hkv, hq, dk, dv, lens, offs, n_cells, seed):
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    sh = W.AttnShape("batch", hkv, hq, dk, dv, max(lens), seed=seed)
    sk, sv = W.codebook_signs(sh)
    gk, gv = tq.TqCache(tq_type, hkv, dk, n_cells), tq.TqCache(tq_type, hkv, dv, n_cells)
    refs, qs = [], []
    for s, (n, c0) in enumerate(zip(lens, offs)):
        shs = W.AttnShape("batch", hkv, hq, dk, dv, max(n, 1), seed=seed * 100 + s)
        k, v = W.kv_inputs(shs, max(n, 1))
        kc, vc = oracle_cache(tq_type, k, sk), oracle_cache(tq_type, v, sv)
        rows = (max(n, 1) + 63) // 64 * 64
        for g, o in ((gk, kc), (gv, vc)):              # this sequence's planes at cells c0 ..
            g.norms[:, c0:c0 + rows].copy_(torch.from_numpy(o.norms[:, :rows].view(np.int16)))
            g.qs[:, c0:c0 + rows].copy_(torch.from_numpy(o.qs[:, :rows]))
            if o.signs is not None:
                g.signs[:, c0:c0 + rows].copy_(torch.from_numpy(o.signs[:, :rows]))
        q = W.to_f32(W.decode_query(shs))
        qs.append(q)
        refs.append(O.decode(kc, vc, sk, sv, O.centroids(tq_type), O.centroids(tq_type), q.astype(np.float64), n,
                             scale_of(dk)))
    cbk, cbv = tq.codebook(tq_type, sk), tq.codebook(tq_type, sv)
    q = torch.from_numpy(np.stack(qs)).cuda()
    out = tq.fattn_decode_batch(gk, gv, cbk, cbv, q, offs, lens, scale_of(dk))
    torch.cuda.synchronize()
    return out.cpu().numpy(), np.stack(refs)


@pytest.mark.parametrize("tq_type", [3, 2, 4])
def test_ragged_batch(tq_type):
    lens = [3000, 1, 0, 2049, 130]
    offs = [0, 3008, 3072, 3136, 5248]
    out, ref = _batch(tq_type, 8, 32, 128, 128, lens, offs, 5440, seed=51)
    for s in range(len(lens)):
        compare_outputs(out[s], ref[s])


def test_batch_asymmetric_192_128():
    lens = [1500, 700]
    offs = [64, 1600]
    out, ref = _batch(3, 4, 4, 192, 128, lens, offs, 2304, seed=52)
    for s in range(len(lens)):
        compare_outputs(out[s], ref[s])


def test_batch_of_eight_at_8k():
    # eight sequences of 8192 cells, 8 KV x 32 query heads: two splits per (sequence, head)
    lens = [8192] * 8
    offs = [8192 * s for s in range(8)]
    out, ref = _batch(3, 8, 32, 128, 128, lens, offs, 8192 * 8, seed=53)
    for s in range(len(lens)):
        err, nm = compare_outputs(out[s], ref[s])
    print(f"batch 8 x 8K: last max-abs {err:.2e} nmse {nm:.2e}")


def test_batch_gqa8():
    # group 8: two launch heads per (sequence, KV head)
    lens = [2000, 65, 1024]
    offs = [0, 2048, 2176]
    out, ref = _batch(3, 4, 32, 128, 128, lens, offs, 3200, seed=54)
    for s in range(len(lens)):
        compare_outputs(out[s], ref[s])


def test_batch_rejects_bad_arguments():
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    from quantized_kv_cache_tq_gb300 import _lib
    gk = tq.TqCache(3, 8, 128, 1024)
    cb = tq.codebook(3, [1, 2, 3, 4])
    q = torch.zeros((2, 32, 128), device="cuda")
    out = torch.zeros((2, 32, 128), device="cuda")
    ws = tq.workspace(_lib.tq_fattn_decode_batch_workspace(gk.c, gk.c, 32, 2, 1024))
    args = lambda c0, ln, algo=0: _lib.tq_fattn_decode_batch(gk.c, gk.c, cb, cb, q.data_ptr(), 32, c0, ln, 0.1,
                                                             algo, out.data_ptr(), ws.data_ptr(), ws.numel(), None)
    assert args([0, 100], [64, 64]) == _lib.TQ_ERR_INVALID_ARG        # offset not a multiple of 64
    assert args([0, 960], [64, 100]) == _lib.TQ_ERR_INVALID_ARG       # past the cells
    assert args([0, 64], [64, 64], algo=tq.TQ_DECODE_LUT) == _lib.TQ_ERR_UNSUPPORTED
    assert args([0, 64], [64, 64]) == _lib.TQ_OK
    assert _lib.tq_fattn_decode_batch_workspace(gk.c, gk.c, 32, 33, 64) == 0

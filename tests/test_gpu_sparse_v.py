"""Sparse-V decode ([TQ#36] "VEC tuning", item 3) on the GPU vs the oracle.

The kernels leave out of the V sum keys whose weights relative to a running
maximum are below the threshold; the oracle names the largest such set (weights
relative to the final maximum) and bounds how far leaving out any subset of it
can move the result.  So:
  * threshold 0 gives tq_fattn_decode's result bit for bit;
  * on scores with a wide gap (a few hot keys, the rest e^-40 below) every key
    left out is negligible, and the result must match the exact one to the usual
    tolerance while most key groups are skipped;
  * on the decode_32k inputs the result lies within the bound of both the exact
    result and the oracle's sparse result."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests._helpers import MAX_ABS, compare_outputs, oracle_cache, scale_of, upload

pytestmark = pytest.mark.gpu


def _algo(tq, name):
    return {"lut": tq.TQ_DECODE_LUT, "mma": tq.TQ_DECODE_MMA}[name]


def _gapped_inputs(seed, n_kv, n_q, d, L, hot_every=64):
    """K rows +-3 along one direction per KV head (+3 for the hot keys, about one
    in hot_every) plus N(0, 0.1) noise; queries 75 times that direction plus
    N(0, 0.1) noise: hot scores near +20, the others near -20."""
    e = W.normal(seed, W.S_EXTRA, n_kv * d).reshape(n_kv, d)
    e /= np.linalg.norm(e, axis=1, keepdims=True)
    u = W.uniform(W.stream_key(seed, W.S_EXTRA + 1), np.arange(L * n_kv, dtype=np.uint64)).reshape(L, n_kv)
    hot = u < 1.0 / hot_every
    k = 0.1 * W.normal(seed, W.S_K, L * n_kv * d).reshape(L, n_kv, d)
    k += np.where(hot, 3.0, -3.0)[..., None] * e[None]
    v = W.normal(seed, W.S_V, L * n_kv * d).reshape(L, n_kv, d)
    g = n_q // n_kv
    q = 75.0 * np.repeat(e, g, axis=0) + 0.1 * W.normal(seed, W.S_Q, n_q * d).reshape(n_q, d)
    return k, v, q, hot


def _run(kc, vc, sk, sv, q, L, thr, algo):
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    gk, gv = upload(kc), upload(vc)
    cbk, cbv = tq.codebook(kc.tq_type, sk), tq.codebook(vc.tq_type, sv)
    qt = torch.from_numpy(W.to_f32(q)).cuda()
    out = tq.fattn_decode(gk, gv, cbk, cbv, qt, L, scale_of(kc.head_dim), algo=_algo(tq, algo), sparse_v=thr)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("algo", ["mma", "lut"])
def test_threshold_zero_is_plain_decode(algo):
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    sh = W.decode_32k(4096)
    k, v = W.kv_inputs(sh)
    sk, sv = W.codebook_signs(sh)
    gk, gv = upload(oracle_cache(3, k, sk)), upload(oracle_cache(3, v, sv))
    cbk, cbv = tq.codebook(3, sk), tq.codebook(3, sv)
    q = torch.from_numpy(W.to_f32(W.decode_query(sh))).cuda()
    a = tq.fattn_decode(gk, gv, cbk, cbv, q, 4096, algo=_algo(tq, algo))
    from quantized_kv_cache_tq_gb300 import _lib
    b = torch.empty_like(a)
    ws = tq.workspace(_lib.tq_fattn_decode_workspace(gk.c, gv.c, q.shape[0], 4096))
    st = _lib.tq_fattn_decode_sparse_v(gk.c, gv.c, cbk, cbv, q.data_ptr(), q.shape[0], 4096, scale_of(128), 0.0,
                                       _algo(tq, algo), b.data_ptr(), ws.data_ptr(), ws.numel(),
                                       torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert torch.equal(a, b)


@pytest.mark.parametrize("algo", ["mma", "lut"])
def test_gapped_scores_match_exact(algo):
    L = 32768
    k, v, q, hot = _gapped_inputs(31, 8, 32, 128, L)
    q = W.to_f32(q).astype(np.float64)
    sk, sv = W.codebook_signs(W.decode_32k())
    kc, vc = oracle_cache(3, k, sk), oracle_cache(3, v, sv)
    c = O.centroids(3)
    o_skip, o_exact, bound = O.decode_sparse_v(kc, vc, sk, sv, c, c, q, L, scale_of(128), 5e-3, slack=1.01)
    assert float(bound.max()) < 1e-9                     # what may be left out is negligible
    out = _run(kc, vc, sk, sv, q, L, 5e-3, algo)
    err, nm = compare_outputs(out, o_exact)
    print(f"sparse-V gapped ({algo}): hot keys {hot.mean():.4f} of all, max-abs {err:.2e} nmse {nm:.2e}")


@pytest.mark.parametrize("tq_type,thr", [(3, 5e-3), (2, 1e-2), (4, 5e-3)])
def test_decode_32k_within_bound(tq_type, thr):
    sh = W.decode_32k()
    k, v = W.kv_inputs(sh)
    sk, sv = W.codebook_signs(sh)
    kc, vc = oracle_cache(tq_type, k, sk), oracle_cache(tq_type, v, sv)
    c = O.centroids(tq_type)
    q = W.to_f32(W.decode_query(sh)).astype(np.float64)
    o_skip, o_exact, bound = O.decode_sparse_v(kc, vc, sk, sv, c, c, q, sh.kv_len, scale_of(128), thr, slack=1.01)
    out = _run(kc, vc, sk, sv, q, sh.kv_len, thr, "mma")
    assert np.all(np.isfinite(out))
    d_exact = np.abs(out - o_exact)
    d_skip = np.abs(out - o_skip)
    assert np.all(d_exact <= bound + MAX_ABS), float(np.max(d_exact - bound))
    assert np.all(d_skip <= bound + MAX_ABS), float(np.max(d_skip - bound))
    print(f"sparse-V turbo{tq_type} thr {thr}: bound max {bound.max():.2e}, |gpu-exact| max {d_exact.max():.2e}, "
          f"|gpu-skip| max {d_skip.max():.2e}")

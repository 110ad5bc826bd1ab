"""Split-KV single-query decode on the GPU vs the f64 oracle, on the same
oracle-quantised cache (max-abs <= 2e-3, NMSE <= 1e-6)."""
import functools

import numpy as np
import pytest

import oracle as O
import workloads as W
from tests._helpers import compare_outputs, oracle_cache, scale_of, upload

pytestmark = pytest.mark.gpu

ALGOS = ["lut", "mma"]


def _algo(name):
    import quantized_kv_cache_tq_gb300 as tq
    return {"lut": tq.TQ_DECODE_LUT, "mma": tq.TQ_DECODE_MMA, "auto": tq.TQ_DECODE_AUTO}[name]


def _setup(sh, ktype, vtype, n_rows=None):
    k, v = W.kv_inputs(sh, n_rows)
    sk, sv = W.codebook_signs(sh)
    kc = oracle_cache(ktype, k, sk)
    vc = oracle_cache(vtype, v, sv)
    return kc, vc, sk, sv


def _decode_pair(kc, vc, sk, sv, q, kv_len, algo):
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    gk, gv = upload(kc), upload(vc)
    cbk, cbv = tq.codebook(kc.tq_type, sk), tq.codebook(vc.tq_type, sv)
    out = tq.fattn_decode(gk, gv, cbk, cbv, torch.from_numpy(W.to_f32(q)).cuda(), kv_len,
                          scale_of(kc.head_dim), algo=_algo(algo))
    torch.cuda.synchronize()
    ref = O.decode(kc, vc, sk, sv, O.centroids(kc.tq_type), O.centroids(vc.tq_type),
                   W.to_f32(q).astype(np.float64), kv_len, scale_of(kc.head_dim))
    return out.cpu().numpy(), ref


@pytest.mark.parametrize("algo", ALGOS)
def test_tiny_decode(algo):
    sh = W.tiny_decode()
    kc, vc, sk, sv = _setup(sh, 3, 3)
    q = W.decode_query(sh)
    out, ref = _decode_pair(kc, vc, sk, sv, q, sh.kv_len, algo)
    compare_outputs(out, ref)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("kv_len", [1, 63, 127, 129, 1000, 2049])
def test_ragged_lengths(algo, kv_len):
    sh = W.decode_32k()
    kc, vc, sk, sv = _setup(sh, 3, 3, n_rows=2112)
    q = W.decode_query(sh)
    out, ref = _decode_pair(kc, vc, sk, sv, q, kv_len, algo)
    compare_outputs(out, ref)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("types", [(2, 2), (4, 4), (3, 2), (2, 4)])
def test_types(algo, types):
    if algo == "mma" and types[0] != types[1]:
        pytest.skip("the tensor-core decode takes K and V of one type (AUTO falls back to the LUT kernel)")
    sh = W.decode_32k()
    kc, vc, sk, sv = _setup(sh, types[0], types[1], n_rows=3000)
    q = W.decode_query(sh)
    out, ref = _decode_pair(kc, vc, sk, sv, q, 3000, algo)
    compare_outputs(out, ref)


@pytest.mark.parametrize("algo", ALGOS)
def test_asymmetric_192_128(algo):
    sh = W.asym_8k()
    kc, vc, sk, sv = _setup(sh, 3, 3, n_rows=1500)
    q = W.decode_query(sh)
    out, ref = _decode_pair(kc, vc, sk, sv, q, 1500, algo)
    compare_outputs(out, ref)


def test_kv_len_zero_gives_zeros():
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    sk = W.sign_bits(0, W.S_SIGNS_K)
    gk, gv = tq.TqCache(3, 2, 128, 64), tq.TqCache(3, 2, 128, 64)
    cb = tq.codebook(3, sk)
    out = torch.full((4, 128), 7.0, device="cuda")
    tq.fattn_decode(gk, gv, cb, cb, torch.ones(4, 128, device="cuda"), 0, out=out)
    torch.cuda.synchronize()
    assert torch.all(out == 0)


@pytest.mark.parametrize("algo", ALGOS)
def test_full_decode_32k(algo):
    # the full 32K-context workload: 8 KV heads x 32 query heads, turbo3 K and V
    sh = W.decode_32k()
    kc, vc, sk, sv = _setup(sh, 3, 3)
    q = W.decode_query(sh)
    out, ref = _decode_pair(kc, vc, sk, sv, q, sh.kv_len, algo)
    err, nm = compare_outputs(out, ref)
    print(f"decode 32K {algo}: max-abs {err:.2e} nmse {nm:.2e}")


def test_graph_replay_and_workspace_reuse():
    # captured into a CUDA graph; replays reuse the self-resetting workspace
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    sh = W.decode_32k()
    kc, vc, sk, sv = _setup(sh, 3, 3, n_rows=4096)
    gk, gv = upload(kc), upload(vc)
    cbk, cbv = tq.codebook(3, sk), tq.codebook(3, sv)
    q = torch.from_numpy(W.to_f32(W.decode_query(sh))).cuda()
    ws = tq.workspace(tq._lib.tq_fattn_decode_workspace(gk.c, gv.c, 32, 4096))
    out = torch.empty(32, 128, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        tq.fattn_decode(gk, gv, cbk, cbv, q, 4096, out=out, ws=ws)     # warm-up
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    first = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        tq.fattn_decode(gk, gv, cbk, cbv, q, 4096, out=out, ws=ws)
    for _ in range(3):
        out.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, first)
    ref = O.decode(kc, vc, sk, sv, O.centroids(3), O.centroids(3), q.cpu().numpy().astype(np.float64),
                   4096, scale_of(128))
    compare_outputs(out.cpu().numpy(), ref)


@pytest.mark.parametrize("algo", ALGOS)
def test_more_kv_heads_than_sms_uses_last_cta_merge(algo):
    # 160 KV heads of one query head each: one split per head and 160 CTAs, more
    # than the GPU holds at once, so no cooperative launch; the last CTA of each
    # head (here its only one) merges
    sh = W.AttnShape("many_heads", 160, 160, 128, 128, 600, seed=17)
    kc, vc, sk, sv = _setup(sh, 3, 3)
    q = W.decode_query(sh)
    out, ref = _decode_pair(kc, vc, sk, sv, q, sh.kv_len, algo)
    compare_outputs(out, ref)


def test_more_than_256_kv_heads_rejected():
    import quantized_kv_cache_tq_gb300 as tq
    from quantized_kv_cache_tq_gb300 import _lib
    c = tq.TqCache(3, 257, 128, 64)
    assert _lib.tq_fattn_decode_workspace(c.c, c.c, 257, 64) == 0


@functools.lru_cache(maxsize=2)
def _full_32k(tq_type):
    # the 32K decode workload's inputs quantised by the oracle and its result,
    # shared by the two kernels' tests of one code type
    sh = W.decode_32k()
    kc, vc, sk, sv = _setup(sh, tq_type, tq_type)
    q = W.decode_query(sh)
    ref = O.decode(kc, vc, sk, sv, O.centroids(tq_type), O.centroids(tq_type), W.to_f32(q).astype(np.float64),
                   sh.kv_len, scale_of(sh.head_dim_k))
    return kc, vc, sk, sv, q, ref


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("tq_type", [2, 4])
def test_full_decode_32k_turbo2_turbo4(tq_type, algo):
    # the same 32K workload (8 KV x 32 query heads, D = 128) at turbo2 and turbo4
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    kc, vc, sk, sv, q, ref = _full_32k(tq_type)
    gk, gv = upload(kc), upload(vc)
    out = tq.fattn_decode(gk, gv, tq.codebook(tq_type, sk), tq.codebook(tq_type, sv),
                          torch.from_numpy(W.to_f32(q)).cuda(), kc.n_cells, scale_of(128), algo=_algo(algo))
    torch.cuda.synchronize()
    err, nm = compare_outputs(out.cpu().numpy(), ref)
    print(f"decode 32K turbo{tq_type} {algo}: max-abs {err:.2e} nmse {nm:.2e}")


@pytest.mark.parametrize("algo", ALGOS)
def test_full_asym_8k_decode(algo):
    # K head dim 192 (two blocks, the second zero-padded), V 128, 16 = 16 heads, 8192 cells
    sh = W.asym_8k()
    kc, vc, sk, sv = _setup(sh, 3, 3)
    q = W.decode_query(sh)
    out, ref = _decode_pair(kc, vc, sk, sv, q, sh.kv_len, algo)
    err, nm = compare_outputs(out, ref)
    print(f"decode asym 8K {algo}: max-abs {err:.2e} nmse {nm:.2e}")


@pytest.mark.parametrize("algo", ALGOS)
def test_one_workspace_across_shapes(algo):
    # one workspace shared by calls of different shapes (8 and 2 KV heads, long and
    # short contexts): a split partial left by an earlier call is never taken for
    # a later call's, whatever the heads' launch counts
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    cases = {}
    for name, sh, n in (("big", W.decode_32k(), 8192), ("two", W.AttnShape("two_kv", 2, 8, 128, 128, 1500, seed=41),
                                                          1500)):
        kc, vc, sk, sv = _setup(sh, 3, 3, n_rows=n)
        cases[name] = (upload(kc), upload(vc), tq.codebook(3, sk), tq.codebook(3, sv),
                       torch.from_numpy(W.to_f32(W.decode_query(sh))).cuda(), kc, vc, sk, sv)
    ws = tq.workspace(max(tq._lib.tq_fattn_decode_workspace(c[0].c, c[1].c, c[4].shape[0], 8192)
                          for c in cases.values()))
    for name, n in (("big", 8192), ("big", 700), ("big", 8192), ("two", 1500), ("big", 129), ("two", 1500),
                    ("big", 4096)):
        gk, gv, cbk, cbv, q, kc, vc, sk, sv = cases[name]
        out = tq.fattn_decode(gk, gv, cbk, cbv, q, n, scale_of(128), algo=_algo(algo), ws=ws)
        torch.cuda.synchronize()
        ref = O.decode(kc, vc, sk, sv, O.centroids(3), O.centroids(3), q.cpu().numpy().astype(np.float64), n,
                       scale_of(128))
        compare_outputs(out.cpu().numpy(), ref)


@pytest.mark.parametrize("algo", ALGOS)
@pytest.mark.parametrize("group", [3, 6, 8, 16])
def test_gqa_groups_beyond_four(group, algo):
    # GQA groups the tensor-core kernel serves as several launch heads of 1, 2 or
    # 4 query heads per KV head (3 -> 3 x 1, 6 -> 3 x 2, 8 -> 2 x 4, 16 -> 4 x 4);
    # the LUT kernel takes groups up to 8
    import quantized_kv_cache_tq_gb300 as tq
    from quantized_kv_cache_tq_gb300 import _lib
    sh = W.AttnShape(f"gqa{group}", 4, 4 * group, 128, 128, 3000, seed=60 + group)
    kc, vc, sk, sv = _setup(sh, 3, 3)
    q = W.decode_query(sh)
    if algo == "lut" and group > 8:
        import torch
        gk, gv = upload(kc), upload(vc)
        cb = tq.codebook(3, sk)
        ws = tq.workspace(_lib.tq_fattn_decode_workspace(gk.c, gv.c, sh.n_q_heads, 3000))
        out = torch.empty(sh.n_q_heads, 128, device="cuda")
        qg = torch.from_numpy(W.to_f32(q)).cuda()
        assert _lib.tq_fattn_decode(gk.c, gv.c, cb, cb, qg.data_ptr(), sh.n_q_heads, 3000, 0.1, _algo(algo),
                                    out.data_ptr(), ws.data_ptr(), ws.numel(), None) == _lib.TQ_ERR_UNSUPPORTED
        return
    out, ref = _decode_pair(kc, vc, sk, sv, q, 3000, algo)
    err, nm = compare_outputs(out, ref)
    print(f"decode GQA {group} {algo}: max-abs {err:.2e} nmse {nm:.2e}")


def test_gqa8_32k_full():
    # 8 KV x 64 query heads over 32768 cells: 16 launch heads of 4 query heads
    sh = W.AttnShape("gqa8_32k", 8, 64, 128, 128, 32768, seed=69)
    kc, vc, sk, sv = _setup(sh, 3, 3)
    q = W.decode_query(sh)
    out, ref = _decode_pair(kc, vc, sk, sv, q, sh.kv_len, "mma")
    err, nm = compare_outputs(out, ref)
    print(f"decode GQA 8 32K: max-abs {err:.2e} nmse {nm:.2e}")


def test_lut_launch_sizes_alternate():
    # the LUT kernel's dynamic shared memory depends on the split count: calls whose
    # sizes go large, small, large again all launch (the size attribute only grows)
    sh = W.decode_32k()
    kc, vc, sk, sv = _setup(sh, 3, 3, n_rows=3000)
    q = W.decode_query(sh)
    for n in (3000, 64, 3000, 700, 64):
        out, ref = _decode_pair(kc, vc, sk, sv, q, n, "lut")
        compare_outputs(out, ref)

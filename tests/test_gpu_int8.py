"""int8 prompt attention (scattered rows, per-row scales) on the GPU vs the
f64 oracle (max-abs <= 2e-3, NMSE <= 1e-6)."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests._helpers import compare_outputs, scale_of

pytestmark = pytest.mark.gpu


def _inputs(seed, n_cells, ctx, hkv, hq, nq, d=128):
    raw_k = W.gaussian_with_outliers(seed, W.S_K, W.S_K_OUT, n_cells, hkv, d)
    raw_v = W.gaussian_with_outliers(seed, W.S_V, W.S_V_OUT, n_cells, hkv, d)
    ki, ks = W.int8_rows(raw_k)
    vi, vs = W.int8_rows(raw_v)
    perm = W.permutation(seed, W.S_PERM, n_cells)[:ctx].astype(np.int32)
    qb = W.to_f16_bits(W.normal(seed, W.S_Q, nq * hq * d).reshape(nq, hq, d))
    return ki, ks, vi, vs, perm, qb


def _run(ki, ks, vi, vs, perm, qb, ctx, causal=True, rows=None):
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    g = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    out = tq.int8_prompt_attn(g(ki), g(ks.view(np.int16)), g(vi), g(vs.view(np.int16)), g(perm), ctx,
                              g(qb.view(np.int16)).view(torch.float16), scale_of(ki.shape[2]), causal=causal)
    torch.cuda.synchronize()
    q = W.f16_bits_to_f64(qb)
    ref = O.int8_prompt_attn(ki, ks, vi, vs, perm, ctx, q, scale_of(ki.shape[2]), causal, rows=rows)
    out = out.cpu().numpy()
    if rows is not None:
        out, ref = out[rows], ref[rows]
    return out, ref


@pytest.mark.parametrize("causal", [True, False])
def test_small_scattered(causal):
    ki, ks, vi, vs, perm, qb = _inputs(3, 320, 250, 2, 8, 40)
    out, ref = _run(ki, ks, vi, vs, perm, qb, 250, causal)
    err, nm = compare_outputs(out, ref)
    print(f"int8 small causal={causal}: max-abs {err:.2e} nmse {nm:.2e}")


def test_ragged_and_gqa1():
    ki, ks, vi, vs, perm, qb = _inputs(4, 200, 131, 3, 3, 77)
    out, ref = _run(ki, ks, vi, vs, perm, qb, 131)
    compare_outputs(out, ref)


def test_out_of_range_cell_reads_zero_row():
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    from quantized_kv_cache_tq_gb300 import _lib
    ki, ks, vi, vs, perm, qb = _inputs(5, 100, 90, 2, 4, 10)
    bad = perm.copy()
    bad[17] = 1000                                            # beyond n_cells = 100
    g = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    ws = tq.workspace(_lib.tq_int8_prompt_attn_workspace(10, 4, 2, 128, 90))
    out = tq.int8_prompt_attn(g(ki), g(ks.view(np.int16)), g(vi), g(vs.view(np.int16)), g(bad), 90,
                              g(qb.view(np.int16)).view(torch.float16), scale_of(128), ws=ws)
    st = _lib.tq_workspace_status(ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == _lib.TQ_ERR_DEVICE_CHECK
    # oracle: the same positions with position 17 pointing at an all-zero row
    ki2 = np.concatenate([ki, np.zeros((1,) + ki.shape[1:], np.int8)])
    vi2 = np.concatenate([vi, np.zeros((1,) + vi.shape[1:], np.int8)])
    ks2 = np.concatenate([ks, np.zeros((1,) + ks.shape[1:], np.uint16)])
    vs2 = np.concatenate([vs, np.zeros((1,) + vs.shape[1:], np.uint16)])
    p2 = perm.copy()
    p2[17] = 100
    ref = O.int8_prompt_attn(ki2, ks2, vi2, vs2, p2, 90, W.f16_bits_to_f64(qb), scale_of(128), True)
    compare_outputs(out.cpu().numpy(), ref)


def test_int8_prompt_ctx4096_full():
    # 8 KV x 32 query heads, 2048 queries over 4096 scattered cells, every output compared
    sh = W.int8_prompt(4096)
    ki, ks, vi, vs, perm, qb = _inputs(sh.seed, 4096, 4096, 8, 32, 2048)
    out, ref = _run(ki, ks, vi, vs, perm, qb, 4096)
    err, nm = compare_outputs(out, ref)
    print(f"int8 ctx 4096: max-abs {err:.2e} nmse {nm:.2e}")


def test_int8_prompt_ctx40000_sampled_rows():
    sh = W.int8_prompt(40000)
    ki, ks, vi, vs, perm, qb = _inputs(sh.seed, 40000, 40000, 8, 32, 2048)
    # the first and last row of every 128-row query tile (32 positions x 4 heads) and a stride between
    rows = np.unique(np.concatenate([np.arange(0, 2048, 32), np.arange(31, 2048, 32), np.arange(5, 2048, 61)]))
    out, ref = _run(ki, ks, vi, vs, perm, qb, 40000, rows=rows)
    err, nm = compare_outputs(out, ref)
    print(f"int8 ctx 40000 (sampled rows): max-abs {err:.2e} nmse {nm:.2e}")


def test_int8_prompt_ctx140000_sampled_rows():
    sh = W.int8_prompt(140000)
    ki, ks, vi, vs, perm, qb = _inputs(sh.seed, 140000, 140000, 8, 32, 2048)
    # the first and last row of every fourth query tile (32 positions each), and the last rows
    rows = np.unique(np.concatenate([np.arange(0, 2048, 128), np.arange(31, 2048, 128), [1, 517, 2046, 2047]]))
    out, ref = _run(ki, ks, vi, vs, perm, qb, 140000, rows=rows)
    err, nm = compare_outputs(out, ref)
    print(f"int8 ctx 140000 (sampled rows): max-abs {err:.2e} nmse {nm:.2e}")

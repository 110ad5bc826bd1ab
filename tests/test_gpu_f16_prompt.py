"""Prompt attention over a binary16 KV cache (rows scattered over the cells, no
scales) on the GPU vs the f64 oracle (max-abs <= 2e-3, NMSE <= 1e-6)."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests._helpers import compare_outputs, scale_of

pytestmark = pytest.mark.gpu


def _inputs(seed, n_cells, ctx, hkv, hq, nq, d=128):
    kb = W.to_f16_bits(W.gaussian_with_outliers(seed, W.S_K, W.S_K_OUT, n_cells, hkv, d))
    vb = W.to_f16_bits(W.gaussian_with_outliers(seed, W.S_V, W.S_V_OUT, n_cells, hkv, d))
    perm = W.permutation(seed, W.S_PERM, n_cells)[:ctx].astype(np.int32)
    qb = W.to_f16_bits(W.normal(seed, W.S_Q, nq * hq * d).reshape(nq, hq, d))
    return kb, vb, perm, qb


def _run(kb, vb, perm, qb, ctx, causal=True, rows=None, cells=None):
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    g = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    f16 = lambda x: g(x.view(np.int16)).view(torch.float16)
    out = tq.f16_prompt_attn(f16(kb), f16(vb), g(perm if cells is None else cells), ctx, f16(qb),
                             scale_of(kb.shape[2]), causal=causal)
    torch.cuda.synchronize()
    q = W.f16_bits_to_f64(qb)
    ref = O.f16_prompt_attn(kb, vb, perm, ctx, q, scale_of(kb.shape[2]), causal, rows=rows)
    out = out.cpu().numpy()
    if rows is not None:
        out, ref = out[rows], ref[rows]
    return out, ref


@pytest.mark.parametrize("causal", [True, False])
def test_small_scattered(causal):
    kb, vb, perm, qb = _inputs(13, 320, 250, 2, 8, 40)
    out, ref = _run(kb, vb, perm, qb, 250, causal)
    err, nm = compare_outputs(out, ref)
    print(f"f16 small causal={causal}: max-abs {err:.2e} nmse {nm:.2e}")


def test_ragged_and_gqa1():
    kb, vb, perm, qb = _inputs(14, 200, 131, 3, 3, 77)
    out, ref = _run(kb, vb, perm, qb, 131)
    compare_outputs(out, ref)


def test_out_of_range_cell_reads_zero_row():
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    from quantized_kv_cache_tq_gb300 import _lib
    kb, vb, perm, qb = _inputs(15, 100, 90, 2, 4, 10)
    bad = perm.copy()
    bad[17] = 1000                                            # beyond n_cells = 100
    g = lambda x: torch.from_numpy(np.ascontiguousarray(x)).cuda()
    f16 = lambda x: g(x.view(np.int16)).view(torch.float16)
    ws = tq.workspace(_lib.tq_int8_prompt_attn_workspace(10, 4, 2, 128, 90))
    out = tq.f16_prompt_attn(f16(kb), f16(vb), g(bad), 90, f16(qb), scale_of(128), ws=ws)
    st = _lib.tq_workspace_status(ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == _lib.TQ_ERR_DEVICE_CHECK
    # oracle: the same positions with position 17 pointing at an all-zero row
    kb2 = np.concatenate([kb, np.zeros((1,) + kb.shape[1:], np.uint16)])
    vb2 = np.concatenate([vb, np.zeros((1,) + vb.shape[1:], np.uint16)])
    p2 = perm.copy()
    p2[17] = 100
    ref = O.f16_prompt_attn(kb2, vb2, p2, 90, W.f16_bits_to_f64(qb), scale_of(128), True)
    compare_outputs(out.cpu().numpy(), ref)


def test_f16_prompt_ctx4096_full():
    sh = W.int8_prompt(4096)
    kb, vb, perm, qb = _inputs(sh.seed, 4096, 4096, 8, 32, 2048)
    out, ref = _run(kb, vb, perm, qb, 4096)
    err, nm = compare_outputs(out, ref)
    print(f"f16 ctx 4096: max-abs {err:.2e} nmse {nm:.2e}")


def test_f16_prompt_ctx40000_sampled_rows():
    sh = W.int8_prompt(40000)
    kb, vb, perm, qb = _inputs(sh.seed, 40000, 40000, 8, 32, 2048)
    rows = np.concatenate([np.arange(0, 2048, 97), [2047]])
    out, ref = _run(kb, vb, perm, qb, 40000, rows=rows)
    err, nm = compare_outputs(out, ref)
    print(f"f16 ctx 40000 (sampled rows): max-abs {err:.2e} nmse {nm:.2e}")

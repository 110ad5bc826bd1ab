"""tq_fattn_decode_append (SET_ROWS of the new token fused into decode) on the GPU.

The fused launch must leave the same cache bytes and produce the same output,
bit for bit, as the three separate calls it replaces (SET_ROWS K, SET_ROWS V,
decode); the output is also checked against the f64 oracle with the oracle's own
quantisation of the new token."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests._helpers import compare_outputs, oracle_cache, scale_of, upload

pytestmark = pytest.mark.gpu


def _clone(tq, g):
    c = tq.TqCache(g.tq_type, g.n_kv_heads, g.head_dim, g.n_cells)
    c.norms.copy_(g.norms)
    c.qs.copy_(g.qs)
    if g.signs is not None:
        c.signs.copy_(g.signs)
    return c


def _planes_equal(a, b):
    same = bool((a.norms == b.norms).all()) and bool((a.qs == b.qs).all())
    if a.signs is not None:
        same = same and bool((a.signs == b.signs).all())
    return same


def _case(sh, ktype, vtype, n_rows, kv_len, cell, src_dtype="f32", algo="auto", n_cells=None):
    """Returns (fused out, separate out, oracle out or None, status, planes equal)."""
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    from quantized_kv_cache_tq_gb300 import _lib
    k, v = W.kv_inputs(sh, n_rows)
    sk, sv = W.codebook_signs(sh)
    kc = oracle_cache(ktype, k[:n_rows - 1], sk, n_cells)
    vc = oracle_cache(vtype, v[:n_rows - 1], sv, n_cells)
    cbk, cbv = tq.codebook(ktype, sk), tq.codebook(vtype, sv)
    a_k, a_v = upload(kc), upload(vc)
    b_k, b_v = _clone(tq, a_k), _clone(tq, a_v)
    tdt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[src_dtype]
    k_row = torch.from_numpy(W.to_f32(k[n_rows - 1])).cuda().to(tdt).contiguous()
    v_row = torch.from_numpy(W.to_f32(v[n_rows - 1])).cuda().to(tdt).contiguous()
    cell_t = torch.tensor([cell], dtype=torch.int64, device="cuda")
    q = torch.from_numpy(W.to_f32(W.decode_query(sh))).cuda()
    scale = scale_of(sh.head_dim_k)
    algo_id = {"auto": tq.TQ_DECODE_AUTO, "lut": tq.TQ_DECODE_LUT, "mma": tq.TQ_DECODE_MMA}[algo]

    # separate calls
    ws_a = tq.workspace(_lib.tq_fattn_decode_workspace(a_k.c, a_v.c, sh.n_q_heads, kv_len))
    st_a = torch.zeros(1, dtype=torch.int32, device="cuda")
    tq.set_rows(a_k, cbk, k_row.unsqueeze(0), cell_t, dev_status=st_a)
    tq.set_rows(a_v, cbv, v_row.unsqueeze(0), cell_t, dev_status=st_a)
    out_a = tq.fattn_decode(a_k, a_v, cbk, cbv, q, kv_len, scale, algo=algo_id, ws=ws_a)
    # fused
    ws_b = tq.workspace(_lib.tq_fattn_decode_workspace(b_k.c, b_v.c, sh.n_q_heads, kv_len))
    out_b = tq.fattn_decode_append(b_k, b_v, cbk, cbv, k_row, v_row, cell_t, q, kv_len, scale, algo=algo_id,
                                   ws=ws_b)
    torch.cuda.synchronize()
    status = _lib.tq_workspace_status(ws_b.data_ptr(), ws_b.numel(), torch.cuda.current_stream().cuda_stream)
    same = _planes_equal(a_k, b_k) and _planes_equal(a_v, b_v)

    ref = None
    if 0 <= cell < kc.n_cells and src_dtype == "f32":
        O.set_rows(kc, W.to_f32(k[n_rows - 1:n_rows]), np.array([cell]), sk, O.centroids(ktype))
        O.set_rows(vc, W.to_f32(v[n_rows - 1:n_rows]), np.array([cell]), sv, O.centroids(vtype))
        ref = O.decode(kc, vc, sk, sv, O.centroids(ktype), O.centroids(vtype),
                       W.to_f32(W.decode_query(sh)).astype(np.float64), kv_len, scale)
    return out_b.cpu().numpy(), out_a.cpu().numpy(), ref, status, same


@pytest.mark.parametrize("tq_type", [3, 2, 4])
def test_append_last_cell_matches_separate_calls(tq_type):
    sh = W.decode_32k()
    out_b, out_a, ref, st, same = _case(sh, tq_type, tq_type, 3000, 3000, 2999)
    assert st == 0 and same
    assert np.array_equal(out_b, out_a)
    compare_outputs(out_b, ref)


def test_append_32k_full_context():
    sh = W.decode_32k()
    out_b, out_a, ref, st, same = _case(sh, 3, 3, 32768, 32768, 32767)
    assert st == 0 and same
    assert np.array_equal(out_b, out_a)
    err, nm = compare_outputs(out_b, ref)
    print(f"append 32K: max-abs {err:.2e} nmse {nm:.2e}")


@pytest.mark.parametrize("cell", [0, 1234, 2047])
def test_append_cell_inside_context(cell):
    # the token lands in an earlier cell (a rewrite); every split may own it
    sh = W.decode_32k()
    out_b, out_a, ref, st, same = _case(sh, 3, 3, 2112, 2100, cell)
    assert st == 0 and same
    assert np.array_equal(out_b, out_a)
    compare_outputs(out_b, ref)


def test_append_beyond_kv_len_is_written_not_attended():
    sh = W.decode_32k()
    out_b, out_a, ref, st, same = _case(sh, 3, 3, 2112, 1500, 2000)
    assert st == 0 and same
    assert np.array_equal(out_b, out_a)
    compare_outputs(out_b, ref)


def test_append_out_of_range_cell_sets_status_and_writes_nothing():
    import quantized_kv_cache_tq_gb300 as tq
    from quantized_kv_cache_tq_gb300 import _lib
    sh = W.decode_32k()
    out_b, out_a, _, st, same = _case(sh, 3, 3, 2112, 2000, 5000)
    assert st == _lib.TQ_ERR_DEVICE_CHECK
    assert same                                   # neither path wrote a row
    assert np.array_equal(out_b, out_a)


@pytest.mark.parametrize("src", ["f16", "bf16"])
def test_append_half_sources(src):
    sh = W.decode_32k()
    out_b, out_a, _, st, same = _case(sh, 3, 3, 3000, 3000, 2999, src_dtype=src)
    assert st == 0 and same
    assert np.array_equal(out_b, out_a)


def test_append_asymmetric_head_dims():
    sh = W.asym_8k()
    out_b, out_a, ref, st, same = _case(sh, 3, 3, 1000, 1000, 999)
    assert st == 0 and same
    assert np.array_equal(out_b, out_a)
    compare_outputs(out_b, ref)


def test_append_tiny_single_split():
    sh = W.tiny_decode()
    out_b, out_a, ref, st, same = _case(sh, 3, 3, 512, 512, 511)
    assert st == 0 and same
    assert np.array_equal(out_b, out_a)
    compare_outputs(out_b, ref)


def test_append_lut_path_issues_separate_launches():
    sh = W.decode_32k()
    out_b, out_a, ref, st, same = _case(sh, 3, 3, 3000, 3000, 2999, algo="lut")
    assert st == 0 and same
    assert np.array_equal(out_b, out_a)
    compare_outputs(out_b, ref)


@pytest.mark.parametrize("group", [8, 3])
def test_append_gqa_group_with_several_launch_heads(group):
    # two (group 8) or three (group 3) launch heads per KV head each own the cell;
    # the cache row is written once and both outputs agree bit for bit
    sh = W.AttnShape(f"gqa{group}", 4, 4 * group, 128, 128, 3000, seed=70 + group)
    out_b, out_a, ref, st, same = _case(sh, 3, 3, 3000, 3000, 2999)
    assert st == 0 and same
    assert np.array_equal(out_b, out_a)
    compare_outputs(out_b, ref)

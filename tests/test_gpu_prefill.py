"""tcgen05 inline-dequant prefill on the GPU vs the f64 oracle on the same
oracle-quantised cache (max-abs <= 2e-3, NMSE <= 1e-6)."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests._helpers import compare_outputs, oracle_cache, scale_of, upload

pytestmark = pytest.mark.gpu


def _queries(shape, nq, dtype):
    import torch
    q = W.normal(shape.seed, W.S_Q, nq * shape.n_q_heads * shape.head_dim_k).reshape(nq, shape.n_q_heads,
                                                                                     shape.head_dim_k)
    if dtype == "bf16":
        bits = W.to_bf16_bits(q)
        return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16), W.bf16_bits_to_f64(bits)
    if dtype == "f16":
        bits = W.to_f16_bits(q)
        return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.float16), W.f16_bits_to_f64(bits)
    f = W.to_f32(q)
    return torch.from_numpy(f).cuda(), f.astype(np.float64)


def _run(shape, nq, kv_len, tq_type=3, causal=True, dtype="bf16", rows=None, n_rows=None):
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    k, v = W.kv_inputs(shape, n_rows or kv_len)
    sk, sv = W.codebook_signs(shape)
    kc = oracle_cache(tq_type, k, sk)
    vc = oracle_cache(tq_type, v, sv)
    gk, gv = upload(kc), upload(vc)
    cbk, cbv = tq.codebook(tq_type, sk), tq.codebook(tq_type, sv)
    qg, qh = _queries(shape, nq, dtype)
    out = tq.fattn_prefill(gk, gv, cbk, cbv, qg, kv_len, scale_of(shape.head_dim_k), causal=causal)
    torch.cuda.synchronize()
    c = O.centroids(tq_type)
    ref = O.prefill(kc, vc, sk, sv, c, c, qh, kv_len, scale_of(shape.head_dim_k), causal, rows=rows)
    out = out.cpu().numpy()
    if rows is not None:
        out, ref = out[rows], ref[rows]
    return out, ref


@pytest.mark.parametrize("nq", [3, 64, 200])
def test_small_causal_d256(nq):
    sh = W.AttnShape("p", 2, 4, 256, 256, 320, seed=7)
    out, ref = _run(sh, nq, 320)
    err, nm = compare_outputs(out, ref)
    print(f"prefill d256 nq={nq}: max-abs {err:.2e} nmse {nm:.2e}")


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
def test_d128_gqa4_dtypes(dtype):
    sh = W.AttnShape("p", 2, 8, 128, 128, 200, seed=8)
    out, ref = _run(sh, 77, 200, dtype=dtype)
    compare_outputs(out, ref)


def test_full_causal_square():
    # nq == kv_len: query i sees keys 0..i (the first rows see 1, 2, ... keys)
    sh = W.AttnShape("p", 1, 2, 256, 256, 192, seed=9)
    out, ref = _run(sh, 192, 192)
    err, nm = compare_outputs(out, ref)
    print(f"prefill square: max-abs {err:.2e} nmse {nm:.2e}")


def test_non_causal():
    sh = W.AttnShape("p", 2, 4, 128, 128, 130, seed=10)
    out, ref = _run(sh, 50, 130, causal=False)
    compare_outputs(out, ref)


@pytest.mark.parametrize("tq_type", [2, 4])
def test_other_types(tq_type):
    sh = W.AttnShape("p", 2, 4, 256, 256, 260, seed=11)
    out, ref = _run(sh, 100, 260, tq_type=tq_type)
    compare_outputs(out, ref)


def test_asymmetric_192_128():
    sh = W.asym_8k(512)
    out, ref = _run(sh, 96, 700)
    compare_outputs(out, ref)


def test_prefill_4k_nq512_full():
    # the 4K-context prefill workload at nq = 512 (8 KV x 16 query heads, D = 256)
    sh = W.prefill_4k(512)
    out, ref = _run(sh, 512, 4096)
    err, nm = compare_outputs(out, ref)
    print(f"prefill 4K nq=512: max-abs {err:.2e} nmse {nm:.2e}")


@pytest.mark.parametrize("nq", [3, 64, 2048, 4096])
def test_prefill_4k_full(nq):
    # the 4K-context prefill workload (8 KV x 16 query heads, D = 256, causal) at
    # every query count of the sweep but 512 (above), all rows compared
    sh = W.prefill_4k(nq)
    out, ref = _run(sh, nq, 4096)
    err, nm = compare_outputs(out, ref)
    print(f"prefill 4K nq={nq}: max-abs {err:.2e} nmse {nm:.2e}")


def test_asym_8k_prefill_512():
    # K 192 / V 128 over 8192 cells, 512 queries, all rows
    sh = W.asym_8k(512)
    out, ref = _run(sh, 512, 8192)
    err, nm = compare_outputs(out, ref)
    print(f"prefill asym 8K nq=512: max-abs {err:.2e} nmse {nm:.2e}")


@pytest.mark.parametrize("nq", [2, 4, 6])
def test_verify_batches_at_32k_context(nq):
    # speculative-decoding verify batches: a few new tokens attend causally over
    # the 32K decode cache (8 KV x 32 query heads, D = 128, f32 queries)
    sh = W.decode_32k()
    out, ref = _run(sh, nq, 32768, dtype="f32")
    err, nm = compare_outputs(out, ref)
    print(f"verify nq={nq} at 32K: max-abs {err:.2e} nmse {nm:.2e}")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("nq,causal", [(1, True), (2, True), (2, False), (8, True), (9, True)])
def test_few_rows_take_the_decode_path(nq, causal, dtype):
    # nq <= 8 runs on the decode kernel (one batched-decode sequence per query
    # row, the causal row seeing kv_len - nq + 1 + i cells), nq = 9 on the
    # prefill kernel; the same tolerance either way
    sh = W.decode_32k(4096)
    out, ref = _run(sh, nq, 3000, causal=causal, dtype=dtype, n_rows=3000)
    compare_outputs(out, ref)


@pytest.mark.parametrize("nq", [4, 12])
def test_gqa8_queries(nq):
    # group 8, D = 128: 4 query rows take the decode path (two launch heads per
    # KV head and row), 12 the prefill kernel
    sh = W.AttnShape("gqa8_p", 2, 16, 128, 128, 700, seed=75)
    out, ref = _run(sh, nq, 700, dtype="f32")
    compare_outputs(out, ref)

"""SET_ROWS on the GPU vs the oracle: codes bit-exact away from decision
boundaries, norms within one binary16 ulp."""
import numpy as np
import pytest

import oracle as O
import workloads as W
from tests._helpers import compare_caches, download

pytestmark = pytest.mark.gpu


def _run(tq_type, raw, cells, n_cells, sb, src_dtype="f32"):
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    n, H, D = raw.shape
    g = tq.TqCache(tq_type, H, D, n_cells)
    cb = tq.codebook(tq_type, sb)
    if src_dtype == "f32":
        src_np = W.to_f32(raw)
        src = torch.from_numpy(src_np).cuda()
    elif src_dtype == "f16":
        bits = W.to_f16_bits(raw)
        src_np = W.f16_bits_to_f64(bits)
        src = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.float16)
    else:
        bits = W.to_bf16_bits(raw)
        src_np = W.bf16_bits_to_f64(bits)
        src = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tq.set_rows(g, cb, src, torch.from_numpy(cells.astype(np.int64)).cuda(), dev_status=status)
    torch.cuda.synchronize()
    ref = O.empty_cache(tq_type, H, D, n_cells)
    y = O.set_rows(ref, src_np, cells, sb, O.centroids(tq_type))
    return download(g), ref, y, int(status.item())


@pytest.mark.parametrize("tq_type", [2, 3, 4])
def test_tiny_decode_rows(tq_type):
    sh = W.tiny_decode()
    k, _ = W.kv_inputs(sh)
    sb = W.sign_bits(sh.seed, W.S_SIGNS_K)
    cells = np.arange(sh.kv_len)
    g, ref, y, st = _run(tq_type, k, cells, 512, sb)
    assert st == 0
    compare_caches(g, ref, y, cells)


@pytest.mark.parametrize("src_dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("tq_type", [2, 3, 4])
def test_scattered_cells_and_dtypes(tq_type, src_dtype):
    sh = W.decode_32k()
    raw = W.gaussian_with_outliers(sh.seed, W.S_K, W.S_K_OUT, 700, 8, 128)
    cells = W.permutation(sh.seed, W.S_CELLS, 1024)[:700]
    sb = W.sign_bits(sh.seed, W.S_SIGNS_V)
    g, ref, y, st = _run(tq_type, raw, cells, 1024, sb, src_dtype)
    assert st == 0
    compare_caches(g, ref, y, cells)
    untouched = np.setdiff1d(np.arange(1024), cells)
    assert not g.qs[:, untouched].any() and not g.norms[:, untouched].any()


def test_asymmetric_192_padded_blocks():
    sh = W.asym_8k()
    k, _ = W.kv_inputs(sh, n_rows=300)
    sb = W.sign_bits(sh.seed, W.S_SIGNS_K)
    cells = np.arange(300)
    g, ref, y, st = _run(3, k, cells, 320, sb)
    compare_caches(g, ref, y, cells)


def test_zero_rows_and_bad_cell_id():
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    sb = W.sign_bits(1, W.S_SIGNS_K)
    raw = np.zeros((3, 2, 128))
    raw[1] = W.normal(1, 1, 256).reshape(2, 128)
    g = tq.TqCache(3, 2, 128, 64)
    cb = tq.codebook(3, sb)
    cells = torch.tensor([5, 64, 7], dtype=torch.int64, device="cuda")     # 64 is out of range
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    tq.set_rows(g, cb, torch.from_numpy(W.to_f32(raw)).cuda(), cells, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 6                       # TQ_ERR_DEVICE_CHECK
    d = download(g)
    # zero row -> norm 0 and every code = +smallest centroid (code 4)
    assert not d.norms[:, 5].any()
    assert np.all(O.unpack_codes(d.qs[:, 5], d.signs[:, 5], 3) == 4)
    ref = O.empty_cache(3, 2, 128, 64)
    y = O.set_rows(ref, W.to_f32(raw[2:3]), np.array([7]), sb, O.centroids(3))
    compare_caches(d, ref, y, np.array([7]))


@pytest.mark.parametrize("tq_type", [3])
def test_full_decode_32k_cache(tq_type):
    # the whole 32768 x 8 x 128 K cache of the 32K decode workload
    sh = W.decode_32k()
    k, _ = W.kv_inputs(sh)
    sb = W.sign_bits(sh.seed, W.S_SIGNS_K)
    cells = np.arange(sh.kv_len)
    g, ref, y, st = _run(tq_type, k, cells, sh.kv_len, sb)
    assert st == 0
    flips, norm_ulps = compare_caches(g, ref, y, cells)
    print(f"boundary flips {flips}, norms off by one ulp {norm_ulps}")

"""The seeded input generators shared by the CUDA path's tests and the oracle,
pinned to facts outside themselves (no GPU needed)."""
import math

import numpy as np
import pytest
import torch

import workloads as W


def test_counter_stream_is_splitmix64():
    # bits(0, i) is output i + 1 of SplitMix64 (Vigna) started from state 0; its first
    # three outputs are the generator's published test values
    b = W.bits(0, np.arange(3, dtype=np.uint64))
    assert [int(x) for x in b] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    # the scalar finaliser used for stream keys is the same function
    assert W._mix64_scalar(0x9E3779B97F4A7C15) == 0xE220A8397B1DCDAF


def test_uniform_is_open_unit_interval_of_the_top_53_bits():
    key = W.stream_key(5, 1)
    i = np.arange(1000, dtype=np.uint64)
    u = W.uniform(key, i)
    top = (W.bits(key, i) >> np.uint64(11)).astype(np.float64)
    assert np.array_equal(u, (top + 0.5) / 2.0 ** 53)
    assert np.all((u > 0) & (u < 1))


def test_normal_is_box_muller_of_consecutive_uniforms():
    key = W.stream_key(3, 2)
    x = W.normal(3, 2, 11)                       # odd length: the last pair is cut
    assert x.shape == (11,)
    for p in range(5):
        u1, u2 = W.uniform(key, np.array([2 * p, 2 * p + 1], dtype=np.uint64))
        r, t = math.sqrt(-2 * math.log(u1)), 2 * math.pi * u2
        assert x[2 * p] == pytest.approx(r * math.cos(t), abs=1e-15)
        assert x[2 * p + 1] == pytest.approx(r * math.sin(t), abs=1e-15)
    # chunked and unchunked draws agree, and the moments are those of N(0, 1)
    y = W.normal(4, 1, 1_000_000)
    assert np.array_equal(y[:4097], W.normal(4, 1, 4097, chunk=1000)[:4097])
    assert abs(y.mean()) < 5e-3 and abs(y.var() - 1) < 5e-3
    assert abs(np.mean(y ** 4) - 3) < 3e-2


def test_streams_and_seeds_are_independent_draws():
    a, b, c = W.normal(1, 1, 1000), W.normal(1, 2, 1000), W.normal(2, 1, 1000)
    assert not np.array_equal(a, b) and not np.array_equal(a, c)
    assert abs(np.corrcoef(a, b)[0, 1]) < 0.1 and abs(np.corrcoef(a, c)[0, 1]) < 0.1
    assert np.array_equal(a, W.normal(1, 1, 1000))            # deterministic


def test_permutation_outliers_and_signs():
    p = W.permutation(9, W.S_PERM, 5000)
    assert p.dtype == np.int32 and np.array_equal(np.sort(p), np.arange(5000))
    assert W.permutation(9, W.S_PERM, 0).shape == (0,)
    ch = W.outlier_channels(2, W.S_K_OUT, 8, 192)
    assert ch.shape == (8, 6)                                 # 4 per 128 channels
    for row in ch:
        assert len(set(row.tolist())) == 6 and row.min() >= 0 and row.max() < 192
    sb = W.sign_bits(1, W.S_SIGNS_K)
    assert sb.dtype == np.uint32 and sb.shape == (4,)
    ones = sum(bin(int(w)).count("1") for w in sb)
    assert 40 < ones < 88                                     # 128 fair bits
    x = W.gaussian_with_outliers(2, W.S_K, W.S_K_OUT, 300, 8, 192)
    plain = W.normal(2, W.S_K, 300 * 8 * 192).reshape(300, 8, 192)
    for h in range(8):
        assert np.array_equal(x[:, h, ch[h]], 8 * plain[:, h, ch[h]])
        rest = np.setdiff1d(np.arange(192), ch[h])
        assert np.array_equal(x[:, h, rest], plain[:, h, rest])


def test_half_and_bfloat16_rounding_match_torch():
    x = np.concatenate([W.normal(6, 1, 20000) * 10.0 ** W.normal(6, 2, 20000),
                        [1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 65504.0, 1e-8, 0.0, -0.0]])
    f32 = torch.tensor(x.astype(np.float32))
    assert np.array_equal(W.to_bf16_bits(x), f32.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))
    # binary16 from f64 directly (numpy) equals torch's f64 -> f16 for every value here
    assert np.array_equal(W.to_f16_bits(x), torch.tensor(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16))
    b = W.to_bf16_bits(np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8]))
    assert np.array_equal(W.bf16_bits_to_f64(b), [1.0, 1 + 2.0 ** -6])   # ties to even
    assert np.array_equal(W.f16_bits_to_f64(W.to_f16_bits(np.array([0.5, -2.0]))), [0.5, -2.0])


def test_int8_rows_format():
    x = W.gaussian_with_outliers(8, W.S_K, W.S_K_OUT, 50, 2, 128)
    x[3, 1] = 0.0                                             # a zero row
    q, sbits = W.int8_rows(x)
    s = W.f16_bits_to_f64(sbits)
    assert q.dtype == np.int8 and sbits.dtype == np.uint16
    assert np.all(np.abs(q.astype(np.int64)) <= 127)
    assert np.array_equal(sbits, W.to_f16_bits(np.abs(x).max(axis=-1) / 127))
    assert s[3, 1] == 0 and not q[3, 1].any()
    err = np.abs(q * s[..., None] - x)
    # half a step, plus the clamp of the largest element when the binary16 scale rounds down
    assert np.all(err <= 0.5 * s[..., None] + 2.0 ** -11 * np.abs(x).max(axis=-1, keepdims=True) + 1e-12)

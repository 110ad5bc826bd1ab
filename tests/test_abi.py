"""C-ABI library checks that need no GPU: it loads, exports every declared
symbol, and its host-side logic (codebook, sizes, argument checks) is right."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle as O
import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _lib():
    try:
        from quantized_kv_cache_tq_gb300 import _lib
    except ImportError as e:
        pytest.fail(f"libtq.so not built: {e}")
    return _lib


def _declared():
    src = "".join(open(os.path.join(ROOT, "include", h)).read() for h in ("tq.h", "tq_testing.h"))
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tq_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol():
    L = _lib()
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L.lib, n), f"{n} not exported"
    assert set(names) == set(L.EXPORTED)


def test_nm_lists_symbols_as_extern_c():
    import subprocess
    L = _lib()
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH], capture_output=True, text=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for n in _declared():
        assert n in syms


@pytest.mark.parametrize("t", [2, 3, 4])
def test_codebook_matches_oracle(t):
    L = _lib()
    sb = W.sign_bits(3, W.S_SIGNS_K)
    cb = L.tq_codebook_init(t, sb)
    n = O.N_CENTROIDS[t]
    assert cb.n_centroids == n
    assert list(cb.sign_bits) == [int(x) for x in sb]
    lib_c = np.array(cb.centroids[:n], dtype=np.float64)
    assert np.array_equal(lib_c, O.centroids(t))


def test_plane_bytes():
    L = _lib()
    assert L.tq_cache_plane_bytes(3, 8, 128, 32768) == (8 * 32768 * 2, 8 * 32768 * 32, 8 * 32768 * 16)
    assert L.tq_cache_plane_bytes(4, 16, 192, 64) == (16 * 64 * 2 * 2, 16 * 64 * 2 * 64, 0)
    assert L.tq_cache_plane_bytes(2, 1, 128, 64)[2] == 0


def test_status_strings():
    L = _lib()
    for s in range(7):
        assert L.status_string(s)
    assert L.status_string(0) == "ok"


def _fake_cache(L, t=3, h=2, d=128, n=64, ptr=1 << 20):
    return L.tq_cache(t, h, d, (d + 127) // 128, n, ptr, ptr + (1 << 16), ptr + (1 << 18))


def test_host_argument_checks_reject_before_launch():
    # every call below must be rejected on the host: no device is touched
    L = _lib()
    cb = L.tq_codebook_init(3, [1, 2, 3, 4])
    good = _fake_cache(L)
    bad_cells = _fake_cache(L, n=100)                 # not a multiple of 64
    bad_blocks = L.tq_cache(3, 2, 128, 2, 64, 1 << 20, 1 << 21, 1 << 22)
    misaligned = _fake_cache(L, ptr=(1 << 20) + 8)
    no_signs = L.tq_cache(3, 2, 128, 1, 64, 1 << 20, 1 << 21, 0)
    for c in (bad_cells, bad_blocks, misaligned, no_signs):
        assert L.tq_set_rows(c, cb, 1 << 23, L.TQ_F32, 1 << 24, 4, None, None) == L.TQ_ERR_INVALID_ARG
    # wrong codebook for the type, non-symmetric or non-binary16 centroids
    cb2 = L.tq_codebook_init(2, [0, 0, 0, 0])
    assert L.tq_set_rows(good, cb2, 1 << 23, L.TQ_F32, 1 << 24, 4, None, None) == L.TQ_ERR_INVALID_ARG
    cb3 = L.tq_codebook_init(3, [0, 0, 0, 0])
    cb3.centroids[0] = cb3.centroids[0] * 1.0001
    assert L.tq_set_rows(good, cb3, 1 << 23, L.TQ_F32, 1 << 24, 4, None, None) == L.TQ_ERR_INVALID_ARG
    # null source, bad dtype, negative rows; zero rows is a no-op
    assert L.tq_set_rows(good, cb, None, L.TQ_F32, 1 << 24, 4, None, None) == L.TQ_ERR_INVALID_ARG
    assert L.tq_set_rows(good, cb, 1 << 23, 7, 1 << 24, 4, None, None) == L.TQ_ERR_INVALID_ARG
    assert L.tq_set_rows(good, cb, 1 << 23, L.TQ_F32, 1 << 24, -1, None, None) == L.TQ_ERR_INVALID_ARG
    assert L.tq_set_rows(good, cb, 1 << 23, L.TQ_F32, 1 << 24, 0, None, None) == L.TQ_OK
    # decode: kv_len beyond the cache, head-count mismatch, workspace too small
    k, v = _fake_cache(L), _fake_cache(L)
    assert L.tq_fattn_decode_workspace(k, v, 4, 65) == 0
    assert L.tq_fattn_decode(k, v, cb, cb, 1 << 23, 4, 65, 0.1, 0, 1 << 24, 1 << 25, 1 << 20,
                             None) == L.TQ_ERR_INVALID_ARG
    assert L.tq_fattn_decode(k, v, cb, cb, 1 << 23, 3, 64, 0.1, 0, 1 << 24, 1 << 25, 1 << 20,
                             None) == L.TQ_ERR_INVALID_ARG
    need = L.tq_fattn_decode_workspace(k, v, 4, 64)
    assert need > 0
    assert L.tq_fattn_decode(k, v, cb, cb, 1 << 23, 4, 64, 0.1, 0, 1 << 24, 1 << 25, need - 1,
                             None) == L.TQ_ERR_WORKSPACE
    assert L.tq_fattn_decode(k, v, cb, cb, 1 << 23, 4, 64, 0.1, 0, 1 << 24, (1 << 25) + 16, need,
                             None) == L.TQ_ERR_WORKSPACE
    assert L.tq_fattn_decode(k, v, cb, cb, 1 << 23, 4, 64, 0.1, 9, 1 << 24, 1 << 25, need,
                             None) == L.TQ_ERR_INVALID_ARG


def test_decode_workspace_grows_with_splits():
    L = _lib()
    k = _fake_cache(L, h=8, n=32768)
    small = L.tq_fattn_decode_workspace(k, k, 32, 512)
    big = L.tq_fattn_decode_workspace(k, k, 32, 32768)
    assert 0 < small < big
    assert big % 256 == 0


def test_sparse_v_and_head_limit_checks_reject_before_launch():
    L = _lib()
    cb = L.tq_codebook_init(3, [1, 2, 3, 4])
    k, v = _fake_cache(L), _fake_cache(L)
    need = L.tq_fattn_decode_workspace(k, v, 4, 64)
    assert need >= 256 + 1024                      # status header + the per-head epoch words
    for thr in (-1e-3, float("nan"), float("inf")):
        assert L.tq_fattn_decode_sparse_v(k, v, cb, cb, 1 << 23, 4, 64, 0.1, thr, 0, 1 << 24, 1 << 25, need,
                                          None) == L.TQ_ERR_INVALID_ARG
    # more than 256 KV heads: no decode workspace, decode rejected
    big = _fake_cache(L, h=257)
    assert L.tq_fattn_decode_workspace(big, big, 257, 64) == 0
    assert L.tq_fattn_decode(big, big, cb, cb, 1 << 23, 257, 64, 0.1, 0, 1 << 24, 1 << 25, 1 << 30,
                             None) == L.TQ_ERR_INVALID_ARG
    assert L.tq_fattn_decode_workspace(_fake_cache(L, h=256), _fake_cache(L, h=256), 256, 64) > 0


def test_fnv1a64_known_values():
    # published FNV-1a 64 test vectors: "" and "a"
    L = _lib()
    assert L.tq_checksum_fnv1a64(None, 0) == 0xcbf29ce484222325
    buf = C.create_string_buffer(b"a", 1)
    assert L.tq_checksum_fnv1a64(C.addressof(buf), 1) == 0xaf63dc4c8601ec8c
    buf = C.create_string_buffer(b"foobar", 6)
    assert L.tq_checksum_fnv1a64(C.addressof(buf), 6) == 0x85944171f73967e8


def test_batch_decode_workspace_limits():
    L = _lib()
    c = L.tq_cache(3, 8, 128, 1, 1024, 1 << 20, 1 << 20, 1 << 20)
    assert L.tq_fattn_decode_batch_workspace(c, c, 32, 32, 1024) > 0
    assert L.tq_fattn_decode_batch_workspace(c, c, 32, 33, 1024) == 0      # more than 32 sequences
    big = L.tq_cache(3, 16, 128, 1, 1024, 1 << 20, 1 << 20, 1 << 20)
    assert L.tq_fattn_decode_batch_workspace(big, big, 16, 17, 64) == 0    # 272 sequence x head pairs
    assert L.tq_fattn_decode_batch_workspace(c, c, 32, 2, 2048) == 0       # longer than the cache
    # a GQA group of 8 runs as two launch heads of 4 query heads per KV head:
    # 16 sequences x 8 KV heads x 2 = 256 launch heads fit, 17 sequences do not
    assert L.tq_fattn_decode_batch_workspace(c, c, 64, 16, 1024) > 0
    assert L.tq_fattn_decode_batch_workspace(c, c, 64, 17, 1024) == 0


def test_decode_workspace_covers_both_kernels_for_large_groups():
    # group 8 (8 KV x 64 query heads): the tensor-core kernel's 16 launch heads and
    # the LUT kernel's 8 give different layouts; the query returns the larger
    L = _lib()
    c = L.tq_cache(3, 8, 128, 1, 32768, 1 << 20, 1 << 20, 1 << 20)
    need8 = L.tq_fattn_decode_workspace(c, c, 64, 32768)
    assert need8 > 0 and need8 % 256 == 0
    # group 16 needs no more epochs than 256 launch heads: 16 KV heads x 4 = 64
    c16 = L.tq_cache(3, 16, 128, 1, 4096, 1 << 20, 1 << 20, 1 << 20)
    assert L.tq_fattn_decode_workspace(c16, c16, 256, 4096) > 0


def _sm_count_is_152():
    # the split choices below assume 152 SMs: the library's own fallback without a
    # GPU, and the GB300's count
    try:
        import torch
        if torch.cuda.is_available():
            return torch.cuda.get_device_properties(0).multi_processor_count == 152
    except Exception:
        pass
    return True


def test_prefill_split_choice_in_workspace_size():
    # The prefill workspace holds (m, l, O') of 128 rows per query tile and split
    # (rows of 4 + 128 nbv floats) after a 1536-byte header.  On the 4K workload
    # (8 KV x 16 query heads, D = 256, 4096 cells; 152 SMs) the split count minimises
    # rounds x (key tiles per item + 6): nq = 64 -> 1 query tile x 16 splits, 200 -> 4 x 4,
    # 512 -> 8 x 2 (one round of 128 items, not 8 x 3 in two), and the query tiles of
    # nq >= 2048 fill the SMs and are not split.
    if not _sm_count_is_152():
        pytest.skip("split choices computed for 152 SMs")
    L = _lib()
    c = _fake_cache(L, h=8, d=256, n=4096)
    tiles_x_splits = {64: 16, 200: 16, 512: 16}
    for nq, ts in tiles_x_splits.items():
        part = 4 * ts * 8 * 128 * (4 + 256)
        assert L.tq_fattn_prefill_workspace(c, c, nq, 16, 4096) == 1536 + (part + 255) // 256 * 256, nq
    for nq in (2048, 4096):
        assert L.tq_fattn_prefill_workspace(c, c, nq, 16, 4096) == 1536


def test_int8_split_choice_in_workspace_size():
    # int8 prompt attention (8 KV x 32 query heads, 2048 queries): ctx 4096 has too
    # few key tiles to split (status word only); ctx 40000 and 140000 take 5 splits,
    # the first count within 1% of the best wave efficiency on 152 SMs.  Layout:
    # status word, merge counters of the 64 x 8 query tiles, partials.
    if not _sm_count_is_152():
        pytest.skip("split choices computed for 152 SMs")
    L = _lib()
    assert L.tq_int8_prompt_attn_workspace(2048, 32, 8, 128, 4096) == 256
    part = 4 * 512 * 5 * 128 * (4 + 128)
    for ctx in (40000, 140000):
        assert L.tq_int8_prompt_attn_workspace(2048, 32, 8, 128, ctx) == 256 + 4 * 512 + part


def test_set_rows_prefill_and_prompt_attention_checks_reject_before_launch():
    # more host checks: each call below returns before any device work
    L = _lib()
    cb = L.tq_codebook_init(3, [1, 2, 3, 4])
    good = _fake_cache(L)
    # SET_ROWS: source rows 16-byte aligned, cell ids 8-byte aligned, status word 4-byte aligned
    assert L.tq_set_rows(good, cb, (1 << 23) + 8, L.TQ_F32, 1 << 24, 4, None, None) == L.TQ_ERR_INVALID_ARG
    assert L.tq_set_rows(good, cb, 1 << 23, L.TQ_F32, (1 << 24) + 4, 4, None, None) == L.TQ_ERR_INVALID_ARG
    assert L.tq_set_rows(good, cb, 1 << 23, L.TQ_F32, 1 << 24, 4, (1 << 25) + 2, None) == L.TQ_ERR_INVALID_ARG
    # prefill (nq = 64 > 8, so not the batched-decode route): query type, counts, scale, alignment, workspace
    k, v = _fake_cache(L), _fake_cache(L)
    need = L.tq_fattn_prefill_workspace(k, v, 64, 4, 64)
    assert need > 0

    def pf(q=1 << 23, q_type=L.TQ_F32, nq=64, kv_len=64, scale=0.1, causal=1, out=1 << 24, ws=1 << 25, wsb=need):
        return L.tq_fattn_prefill(k, v, cb, cb, q, q_type, nq, 4, kv_len, scale, causal, out, ws, wsb, None)

    assert pf(q_type=7) == L.TQ_ERR_INVALID_ARG
    assert pf(nq=-1) == L.TQ_ERR_INVALID_ARG
    assert pf(nq=64, kv_len=63) == L.TQ_ERR_INVALID_ARG          # causal rows need nq <= kv_len
    assert pf(scale=float("nan")) == L.TQ_ERR_INVALID_ARG
    assert pf(scale=float("inf")) == L.TQ_ERR_INVALID_ARG
    assert pf(nq=0) == L.TQ_OK
    assert pf(q=(1 << 23) + 4) == L.TQ_ERR_INVALID_ARG
    assert pf(out=0) == L.TQ_ERR_INVALID_ARG
    assert pf(wsb=need - 1) == L.TQ_ERR_WORKSPACE
    assert pf(ws=(1 << 25) + 64) == L.TQ_ERR_WORKSPACE
    # int8 / binary16 prompt attention
    ctx, nq = 40000, 2048
    wneed = L.tq_int8_prompt_attn_workspace(nq, 32, 8, 128, ctx)
    assert wneed > 256
    assert L.tq_int8_prompt_attn_workspace(nq, 30, 8, 128, ctx) == 0       # heads not a multiple
    assert L.tq_int8_prompt_attn_workspace(nq, 32, 8, 64, ctx) == 0        # head_dim other than 128
    assert L.tq_int8_prompt_attn_workspace(-1, 32, 8, 128, ctx) == 0

    def i8(k=1 << 23, ks=1 << 24, v=1 << 25, vs=1 << 26, n_cells=ctx, cells=1 << 27, ctx_=ctx, q=1 << 28, nq_=nq,
           hq=32, hkv=8, d=128, scale=0.1, causal=1, out=1 << 29, ws=1 << 30, wsb=wneed):
        return L.tq_int8_prompt_attn(k, ks, v, vs, n_cells, cells, ctx_, q, nq_, hq, hkv, d, scale, causal, out,
                                     ws, wsb, None)

    assert i8(hq=30) == L.TQ_ERR_INVALID_ARG
    assert i8(hq=24) == L.TQ_ERR_UNSUPPORTED                           # GQA group 3
    assert i8(d=64) == L.TQ_ERR_UNSUPPORTED
    assert i8(nq_=-1) == L.TQ_ERR_INVALID_ARG
    assert i8(ctx_=-1) == L.TQ_ERR_INVALID_ARG
    assert i8(n_cells=0) == L.TQ_ERR_INVALID_ARG
    assert i8(nq_=nq, ctx_=nq - 1) == L.TQ_ERR_INVALID_ARG              # causal rows need nq <= ctx
    assert i8(scale=float("nan")) == L.TQ_ERR_INVALID_ARG
    assert i8(nq_=0) == L.TQ_OK
    assert i8(out=(1 << 29) + 4) == L.TQ_ERR_INVALID_ARG
    assert i8(q=0) == L.TQ_ERR_INVALID_ARG
    assert i8(wsb=wneed - 1) == L.TQ_ERR_WORKSPACE
    assert i8(ws=(1 << 30) + 128) == L.TQ_ERR_WORKSPACE
    assert i8(k=(1 << 23) + 8) == L.TQ_ERR_INVALID_ARG
    assert i8(cells=0) == L.TQ_ERR_INVALID_ARG
    assert i8(cells=(1 << 27) + 2) == L.TQ_ERR_INVALID_ARG
    assert i8(ks=0) == L.TQ_ERR_INVALID_ARG                            # int8 rows need their scales
    assert i8(vs=(1 << 26) + 1) == L.TQ_ERR_INVALID_ARG
    # binary16 rows have no scales; the other checks are shared
    f16 = lambda **kw: L.tq_f16_prompt_attn(kw.get("k", 1 << 23), 1 << 25, ctx, 1 << 27, ctx, 1 << 28, nq, 32, 8,
                                            128, 0.1, 1, 1 << 29, 1 << 30, kw.get("wsb", wneed), None)
    assert f16(k=(1 << 23) + 8) == L.TQ_ERR_INVALID_ARG
    assert f16(wsb=wneed - 1) == L.TQ_ERR_WORKSPACE

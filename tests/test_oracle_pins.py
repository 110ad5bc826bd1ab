"""Pins of the CPU oracle to facts outside itself: closed forms, published
tables, invariants, brute force and special cases (no GPU needed)."""
import math
import os

import numpy as np
import pytest
from scipy.integrate import quad

import oracle as O
import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_table(name):
    rows = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                parts = line.split()
                rows[parts[0]] = parts[1:]
    return rows


# --------------------------------------------------------------------- rotation

def test_hadamard_orthogonal_and_symmetric():
    H = O.hadamard()
    assert np.array_equal(H @ H.T, 128 * np.eye(128))
    assert np.array_equal(H, H.T)
    assert set(np.unique(H)) == {-1.0, 1.0}


def test_hadamard_matches_butterfly_recursion():
    # column j of H is the butterfly transform of the unit vector e_j
    H = O.hadamard()
    eye = np.eye(128)
    assert np.array_equal(O.butterfly_wht(eye), H)           # rows: transforms of e_j
    # 7 stages h = 1..64 as printed on the page
    facts = _read_table("page_format_facts.txt")
    assert int(facts["wht_stages"][0]) == int(math.log2(128))


def test_hadamard_small_known():
    # Sylvester H_4 written out by hand
    H4 = np.array([[1, 1, 1, 1], [1, -1, 1, -1], [1, 1, -1, -1], [1, -1, -1, 1]], float)
    assert np.array_equal(O.hadamard(4), H4)


def test_rotation_orthonormal_norm_preserving():
    sb = W.sign_bits(1, W.S_SIGNS_K)
    R = O.rotation(sb)
    assert np.allclose(R @ R.T, np.eye(128), atol=1e-14)
    S = np.diag(O.sign_vector(sb))
    assert np.array_equal(S @ S, np.eye(128))
    u = W.normal(3, 1, 128 * 50).reshape(50, 128)
    assert np.allclose(np.linalg.norm(u @ R.T, axis=1), np.linalg.norm(u, axis=1), rtol=1e-14)


def test_sign_bits_order():
    sb = np.array([0b101, 0, 0, 1 << 31], dtype=np.uint32)
    s = O.sign_vector(sb)
    neg = np.nonzero(s < 0)[0].tolist()
    assert neg == [0, 2, 127]


# -------------------------------------------------------------------- codebooks

@pytest.mark.parametrize("n", [4, 8, 16])
def test_lloyd_max_matches_max_1960(n):
    table = _read_table("lloyd_max_gaussian.txt")[str(n)]
    dist, levels = float(table[0]), np.array([float(v) for v in table[1:]])
    c = O.lloyd_max_normal(n)
    assert np.allclose(c[n // 2:], levels, atol=6e-4)
    assert abs(O.lloyd_max_distortion(c) - dist) / dist < 5e-4


@pytest.mark.parametrize("n", [4, 8, 16])
def test_lloyd_max_fixed_point_by_quadrature(n):
    c = O.lloyd_max_normal(n)
    assert np.allclose(c, -c[::-1], atol=1e-14)
    t = np.concatenate(([-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]))
    pdf = lambda x: math.exp(-x * x / 2) / math.sqrt(2 * math.pi)
    d = 0.0
    for k in range(n):
        m0 = quad(pdf, t[k], t[k + 1], epsabs=1e-14)[0]
        m1 = quad(lambda x: x * pdf(x), t[k], t[k + 1], epsabs=1e-14)[0]
        assert abs(m1 / m0 - c[k]) < 1e-10             # centroid condition
        d += quad(lambda x: (x - c[k]) ** 2 * pdf(x), t[k], t[k + 1], epsabs=1e-14)[0]
    assert abs(d - O.lloyd_max_distortion(c)) < 1e-12


@pytest.mark.parametrize("t", [2, 3, 4])
def test_canonical_codebook(t):
    c = O.centroids(t)
    facts = _read_table("page_format_facts.txt")
    assert len(c) == int(facts[f"turbo{t}_centroids"][0])
    assert np.all(np.diff(c) > 0)
    assert np.array_equal(c, -c[::-1])
    assert np.array_equal(c.astype(np.float16).astype(np.float64), c)
    exact = O.lloyd_max_normal(len(c)) / math.sqrt(128)
    assert np.max(np.abs(c - exact) / np.abs(exact)) <= 2.0 ** -11


# --------------------------------------------------------------- codes, layout

@pytest.mark.parametrize("t", [2, 3, 4])
def test_code_mapping_roundtrip(t):
    c = O.centroids(t)
    n = len(c)
    i = np.arange(n)
    codes = O.index_to_code(i, n)
    assert sorted(codes.tolist()) == list(range(n))
    assert np.array_equal(O.code_to_value(codes, c), c)
    # sign-magnitude: top bit = sign, low bits = magnitude rank
    assert np.all((O.code_to_value(np.arange(n), c) > 0) == (np.arange(n) >= n // 2))


@pytest.mark.parametrize("t", [2, 3, 4])
def test_pack_unpack_roundtrip(t):
    n = O.N_CENTROIDS[t]
    codes = (W.bits(7, np.arange(64 * 128, dtype=np.uint64)) % np.uint64(n)).astype(np.int64)
    codes = codes.reshape(64, 128)
    qs, signs = O.pack_codes(codes, t)
    assert qs.shape == (64, O.QS_BYTES[t])
    assert np.array_equal(O.unpack_codes(qs, signs, t), codes)


def test_bit_positions_by_hand():
    def one(t, e, k):
        codes = np.zeros((1, 128), np.int64)
        codes[0, e] = k
        qs, signs = O.pack_codes(codes, t)
        return qs[0], (None if signs is None else signs[0])

    qs, sg = one(3, 0, 7)            # j = 3, s = 1
    assert qs[0] == 0x03 and sg[0] == 0x04
    qs, sg = one(3, 8, 7)            # second half of word 0: bits 2..3, sign bit 3
    assert qs[0] == 0x0C and sg[0] == 0x08
    qs, sg = one(3, 5, 2)            # element 5: bits 20..21 -> byte 2 bits 4..5
    assert qs[2] == 0x20 and not sg.any()
    qs, sg = one(3, 13, 2)           # element 13 = 8 + 5: bits 22..23 -> byte 2 bits 6..7
    assert qs[2] == 0x80 and not sg.any()
    qs, sg = one(3, 16, 4)           # word 1, sign at bit 0 of signs word 0
    assert qs[4] == 0x00 and sg[0] == 0x01
    qs, sg = one(3, 24, 5)           # element 24: r = 24 -> bit 1 of signs word 0
    assert qs[4] == 0x04 and sg[0] == 0x02
    qs, sg = one(3, 127, 4)          # last element: signs word 3, r = 31 -> bit 4*7+1
    assert sg[15] == 0x20
    qs, _ = one(4, 9, 0xB)           # turbo4: word 1 nibble 1
    assert qs[4] == 0xB0
    qs, _ = one(2, 127, 3)           # turbo2: element 127 -> word 7, i = 7, bits 30..31
    assert qs[31] == 0xC0


def test_format_sizes_match_pages():
    facts = _read_table("page_format_facts.txt")
    assert O.bits_per_element(2) == 2.125
    assert O.bits_per_element(3) == 3.125
    assert O.bits_per_element(4) == 4.125
    assert round(16 / O.bits_per_element(2), 1) == float(facts["turbo2_compression_vs_f16"][0])
    per8 = (O.QS_BYTES[3] / 16, O.SIGN_BYTES / 16)
    assert per8 == (float(facts["turbo3_qs_bytes_per_8"][0]), float(facts["turbo3_sign_bytes_per_8"][0]))


# --------------------------------------------------------------------- encoder

@pytest.mark.parametrize("t", [2, 3, 4])
def test_brute_force_equals_threshold_search(t):
    c = O.centroids(t)
    y = W.normal(11, 2, 1_000_000) / math.sqrt(128)
    mids = 0.5 * (c[:-1] + c[1:])
    away = np.min(np.abs(y[:, None] - mids[None, :]), axis=1) > 1e-12
    by_threshold = np.searchsorted(mids, y, side="right")        # y >= t  => upper cell
    brute = O.nearest_centroid(y, c)
    assert np.array_equal(brute[away], by_threshold[away])
    assert np.array_equal(O.nearest_centroid(mids, c), np.arange(1, len(c)))   # exact ties -> upper
    # the oracle's encoder on exact midpoints picks the upper centroid
    sb = np.zeros(4, np.uint32)
    x = np.zeros(128)
    x[0] = 1.0                                  # y = (1/sqrt(128)) * H[:,0] = all +1/sqrt(128)
    _, codes, y0 = O.quantize_blocks(x, sb, c)
    assert np.allclose(y0, 1 / math.sqrt(128))


def test_zero_block():
    c = O.centroids(3)
    nb, codes, y = O.quantize_blocks(np.zeros(128), np.zeros(4, np.uint32), c)
    assert nb == 0 and np.all(y == 0)
    # exact tie between -c4 and +c4 at 0 goes to the upper centroid: code s=1, j=0
    assert np.all(codes == 4)
    assert np.all(O.dequantize_blocks(nb, codes, np.zeros(4, np.uint32), c) == 0)


@pytest.mark.parametrize("t", [2, 3, 4])
def test_quantiser_distortion_matches_lloyd_max(t):
    c = O.centroids(t)
    sb = W.sign_bits(5, W.S_SIGNS_K)
    x = W.normal(5, 1, 4000 * 128).reshape(4000, 128)
    nb, codes, y = O.quantize_blocks(x, sb, c)
    mse = np.mean((y - O.code_to_value(codes, c)) ** 2) * 128
    d = O.lloyd_max_distortion(O.lloyd_max_normal(len(c)))
    assert abs(mse - d) / d < 0.03
    # full round trip: relative error of x_hat is the same distortion
    xh = O.dequantize_blocks(nb, codes, sb, c)
    rel = np.sum((xh - x) ** 2) / np.sum(x * x)
    assert abs(rel - d) / d < 0.05


def test_dequantize_structure():
    c = O.centroids(3)
    sb = W.sign_bits(9, W.S_SIGNS_V)
    codes = (W.bits(3, np.arange(128, dtype=np.uint64)) % np.uint64(8)).astype(np.int64)
    nb = np.array(np.float16(2.5)).view(np.uint16)
    xh = O.dequantize_blocks(nb, codes, sb, c)
    vals = O.code_to_value(codes, c)
    assert abs(np.linalg.norm(xh) - 2.5 * np.linalg.norm(vals)) < 1e-12
    assert np.allclose(O.rotation(sb) @ xh / 2.5, vals, atol=1e-14)


def test_norm_is_fp16_rne():
    x = np.zeros(128)
    x[3] = 1.0 + 2.0 ** -11          # exactly half an fp16 ulp above 1 -> ties to even (1.0)
    nb, _, _ = O.quantize_blocks(x, np.zeros(4, np.uint32), O.centroids(3))
    assert nb == np.array(np.float16(1.0)).view(np.uint16)
    x[3] = 1.0 + 3 * 2.0 ** -11      # 1.5 ulp -> rounds up to 1 + 2 ulp
    nb, _, _ = O.quantize_blocks(x, np.zeros(4, np.uint32), O.centroids(3))
    assert nb == np.array(np.float16(1.0 + 2.0 ** -9)).view(np.uint16)


def test_set_rows_padding_and_cells():
    c = O.centroids(3)
    sb = W.sign_bits(2, W.S_SIGNS_K)
    cache = O.empty_cache(3, 2, 192, 64)
    src = W.normal(2, 3, 5 * 2 * 192).reshape(5, 2, 192)
    cells = np.array([7, 0, 63, 12, 30])
    O.set_rows(cache, src, cells, sb, c)
    # block 1 of a 192-wide row = channels 128..191 followed by 64 zeros
    blk = np.concatenate([src[2, 1, 128:], np.zeros(64)])
    nb, codes, _ = O.quantize_blocks(blk, sb, c)
    assert cache.norms[1, 63, 1] == nb
    assert np.array_equal(O.unpack_codes(cache.qs[1, 63, 1], cache.signs[1, 63, 1], 3), codes)
    assert not cache.qs[0, 1].any()                      # untouched cell


# -------------------------------------------------------------------- attention

def _loop_attention(q, k, v, scale):
    # plain scalar loops with math.exp
    out = []
    for qi in q:
        s = [scale * sum(a * b for a, b in zip(qi, kt)) for kt in k]
        m = max(s)
        e = [math.exp(x - m) for x in s]
        z = sum(e)
        out.append([sum(e[t] * v[t][d] for t in range(len(k))) / z for d in range(len(v[0]))])
    return np.array(out)


def test_attention_special_cases():
    rng_q = W.normal(1, 1, 3 * 8).reshape(3, 8)
    k = W.normal(1, 2, 5 * 8).reshape(5, 8)
    v = W.normal(1, 3, 5 * 4).reshape(5, 4)
    # one key -> output = that value row
    assert np.allclose(O.softmax_attention(rng_q, k[:1], v[:1], 0.3), np.repeat(v[:1], 3, 0), atol=1e-15)
    # equal scores (q = 0) -> mean of V
    assert np.allclose(O.softmax_attention(np.zeros((1, 8)), k, v, 1.0), v.mean(0, keepdims=True), atol=1e-15)
    # brute-force loops
    assert np.allclose(O.softmax_attention(rng_q, k, v, 0.37), _loop_attention(rng_q, k, v, 0.37), atol=1e-13)
    # empty key set -> zeros
    assert np.all(O.softmax_attention(rng_q, k[:0], v[:0], 1.0) == 0)


def test_causal_equals_prefix_attention():
    q = W.normal(4, 1, 6 * 16).reshape(6, 16)
    k = W.normal(4, 2, 10 * 16).reshape(10, 16)
    v = W.normal(4, 3, 10 * 16).reshape(10, 16)
    pos = np.arange(4, 10)
    o = O.softmax_attention(q, k, v, 0.25, pos)
    for i, p in enumerate(pos):
        assert np.allclose(o[i], O.softmax_attention(q[i:i + 1], k[:p + 1], v[:p + 1], 0.25)[0], atol=1e-14)


def test_split_lse_merge_equals_unsplit():
    q = W.normal(6, 1, 2 * 32).reshape(2, 32) * 3
    k = W.normal(6, 2, 100 * 32).reshape(100, 32)
    v = W.normal(6, 3, 100 * 32).reshape(100, 32)
    full = O.softmax_attention(q, k, v, 0.2)
    parts = [O.lse_partial(q, k[a:b], v[a:b], 0.2) for a, b in [(0, 7), (7, 64), (64, 100)]]
    assert np.allclose(O.lse_merge(parts), full, atol=1e-14)


def test_sparse_v_special_cases_and_bound():
    # [TQ#36 "VEC tuning"] item 3: keys with exp(s - max) < threshold leave the V sum
    q = W.normal(11, 1, 2 * 16).reshape(2, 16)
    k = W.normal(11, 2, 40 * 16).reshape(40, 16) * 2
    v = W.normal(11, 3, 40 * 8).reshape(40, 8)
    exact = O.softmax_attention(q, k, v, 0.7)
    # threshold 0 leaves nothing out
    o_skip, o_exact, bound = O.sparse_v_attention(q, k, v, 0.7, 0.0)
    assert np.allclose(o_exact, exact, atol=1e-14) and np.array_equal(o_skip, o_exact) and np.all(bound == 0)
    # a threshold above 1 leaves every key out (the maximum has weight 1): zero output,
    # and the bound is the whole |V|-weighted mass
    o_skip, _, bound = O.sparse_v_attention(q, k, v, 0.7, 1.5)
    assert np.all(o_skip == 0)
    assert np.allclose(bound, O.softmax_attention(q, k, np.abs(v), 0.7), atol=1e-14)
    # any threshold: the left-out keys move the result by at most the bound
    for thr in (1e-3, 5e-3, 1e-2, 0.2):
        o_skip, o_exact, bound = O.sparse_v_attention(q, k, v, 0.7, thr)
        assert np.all(np.abs(o_skip - o_exact) <= bound + 1e-15)
        assert np.all(bound >= 0)


def test_sparse_v_by_hand():
    # scores 0, -10, -1 (natural log units): weights 1, e^-10, e^-1; threshold 1e-3
    # leaves key 1 out of the V sum only
    q = np.array([[1.0, 0.0]])
    k = np.array([[0.0, 0.0], [-10.0, 0.0], [-1.0, 0.0]])
    v = np.array([[1.0, 2.0], [3.0, -4.0], [5.0, 6.0]])
    w = np.array([1.0, math.exp(-10.0), math.exp(-1.0)])
    o_skip, o_exact, bound = O.sparse_v_attention(q, k, v, 1.0, 1e-3)
    assert np.allclose(o_skip[0], (v[0] + w[2] * v[2]) / w.sum(), atol=1e-15)
    assert np.allclose(o_exact[0], (w[:, None] * v).sum(0) / w.sum(), atol=1e-15)
    assert np.allclose(bound[0], w[1] * np.abs(v[1]) / w.sum(), atol=1e-18)
    # a slack of 50 moves the cut to 0.05, still between e^-10 and e^-1
    o2, _, _ = O.sparse_v_attention(q, k, v, 1.0, 1e-3, slack=50.0)
    assert np.array_equal(o2, o_skip)
    # a slack of 400 moves it to 0.4, above e^-1: key 2 leaves the V sum as well, and
    # the bound takes both left-out keys (the normaliser still counts every key)
    o3, _, b3 = O.sparse_v_attention(q, k, v, 1.0, 1e-3, slack=400.0)
    assert np.allclose(o3[0], v[0] / w.sum(), atol=1e-15)
    assert np.allclose(b3[0], (w[1] * np.abs(v[1]) + w[2] * np.abs(v[2])) / w.sum(), atol=1e-15)


def test_decode_sparse_v_matches_per_head_attention():
    shape = W.AttnShape("t", 2, 4, 128, 128, 70, seed=5)
    c = O.centroids(3)
    sk, sv = W.codebook_signs(shape)
    kr, vr = W.kv_inputs(shape)
    kc = O.empty_cache(3, 2, 128, 128)
    vc = O.empty_cache(3, 2, 128, 128)
    O.set_rows(kc, kr, np.arange(70), sk, c)
    O.set_rows(vc, vr, np.arange(70), sv, c)
    q = W.decode_query(shape) * 4
    o_skip, o_exact, bound = O.decode_sparse_v(kc, vc, sk, sv, c, c, q, 70, 1 / math.sqrt(128), 5e-3)
    assert np.allclose(o_exact, O.decode(kc, vc, sk, sv, c, c, q, 70, 1 / math.sqrt(128)), atol=1e-13)
    kh = O.dequantize_cache(kc, sk, c, 70)
    vh = O.dequantize_cache(vc, sv, c, 70)
    for h in range(4):
        s = (q[h] @ kh[h // 2].T) / math.sqrt(128)
        p = np.exp(s - s.max())
        keep = p >= 5e-3
        ref = (p[keep] @ vh[h // 2][keep]) / p.sum()
        assert np.allclose(o_skip[h], ref, atol=1e-13)
    assert np.all(np.abs(o_skip - o_exact) <= bound + 1e-15)


def test_decode_gqa_and_dequant_path():
    shape = W.AttnShape("t", 2, 4, 128, 128, 70, seed=3)
    c = O.centroids(3)
    sk, sv = W.codebook_signs(shape)
    kr, vr = W.kv_inputs(shape)
    kc = O.empty_cache(3, 2, 128, 128)
    vc = O.empty_cache(3, 2, 128, 128)
    O.set_rows(kc, kr, np.arange(70), sk, c)
    O.set_rows(vc, vr, np.arange(70), sv, c)
    q = W.decode_query(shape)
    out = O.decode(kc, vc, sk, sv, c, c, q, 70, 1 / math.sqrt(128))
    kh = O.dequantize_cache(kc, sk, c, 70)
    vh = O.dequantize_cache(vc, sv, c, 70)
    for h in range(4):
        ref = _loop_attention(q[h:h + 1], kh[h // 2], vh[h // 2], 1 / math.sqrt(128))
        assert np.allclose(out[h], ref[0], atol=1e-12)
    # quantised attention is close to unquantised attention (sanity, loose)
    exact = np.stack([O.softmax_attention(q[h:h + 1], kr[:, h // 2], vr[:, h // 2], 1 / math.sqrt(128))[0]
                      for h in range(4)])
    assert O.nmse(out, exact) < 0.2


def test_int8_dequantised_attention_and_permutation():
    n_cells, hkv, d = 40, 2, 128
    raw = W.gaussian_with_outliers(8, W.S_K, W.S_K_OUT, n_cells, hkv, d)
    rawv = W.gaussian_with_outliers(8, W.S_V, W.S_V_OUT, n_cells, hkv, d)
    ki, ks = W.int8_rows(raw)
    vi, vs = W.int8_rows(rawv)
    q = W.normal(8, W.S_Q, 5 * 4 * d).reshape(5, 4, d)
    ident = np.arange(n_cells, dtype=np.int32)
    o1 = O.int8_prompt_attn(ki, ks, vi, vs, ident, n_cells, q, 0.1)
    # scatter the rows through a permutation: same logical content -> same output
    perm = W.permutation(8, W.S_PERM, n_cells)            # cell_of_pos
    ki2 = np.zeros_like(ki); ks2 = np.zeros_like(ks); vi2 = np.zeros_like(vi); vs2 = np.zeros_like(vs)
    ki2[perm] = ki; ks2[perm] = ks; vi2[perm] = vi; vs2[perm] = vs
    o2 = O.int8_prompt_attn(ki2, ks2, vi2, vs2, perm, n_cells, q, 0.1)
    assert np.allclose(o1, o2, atol=1e-13)
    # equals attention over q_int * scale computed with plain loops (one head, last query)
    kk = [[float(ki[t, 0, j]) * float(np.float16(ks[t, 0].view(np.float16))) for j in range(d)] for t in range(n_cells)]
    vv = [[float(vi[t, 0, j]) * float(np.float16(vs[t, 0].view(np.float16))) for j in range(d)] for t in range(n_cells)]
    ref = _loop_attention(q[4:5, 1], kk, vv, 0.1)
    assert np.allclose(o1[4, 1], ref[0], atol=1e-12)
    # int8 rows reconstruct the raw values within half a quantisation step
    recon = O.int8_dequantize(ki, ks)
    step = ks.view(np.float16).astype(np.float64)
    assert np.all(np.abs(recon - raw) <= 0.5 * step[..., None] * (1 + 1e-3) + 1e-3 * np.abs(raw))


def test_f16_prompt_attention_loops_and_causality():
    # binary16 rows through a permutation: plain-loop attention over the gathered
    # rows, the causal horizon of each query, and the non-causal case
    n_cells, hkv, d, nq, hq = 24, 2, 128, 4, 4
    kb = W.to_f16_bits(W.gaussian_with_outliers(9, W.S_K, W.S_K_OUT, n_cells, hkv, d))
    vb = W.to_f16_bits(W.gaussian_with_outliers(9, W.S_V, W.S_V_OUT, n_cells, hkv, d))
    perm = W.permutation(9, W.S_PERM, n_cells)
    ctx = 20
    q = W.normal(9, W.S_Q, nq * hq * d).reshape(nq, hq, d)
    out = O.f16_prompt_attn(kb, vb, perm, ctx, q, 0.05, causal=True)
    kf = kb.view(np.float16).astype(np.float64)
    vf = vb.view(np.float16).astype(np.float64)
    for i in range(nq):
        p_i = ctx - nq + i                                  # keys 0..p_i are visible
        for h in range(hq):
            hk = h // (hq // hkv)
            kk = [[kf[perm[t], hk, j] for j in range(d)] for t in range(p_i + 1)]
            vv = [[vf[perm[t], hk, j] for j in range(d)] for t in range(p_i + 1)]
            ref = _loop_attention(q[i:i + 1, h], kk, vv, 0.05)
            assert np.allclose(out[i, h], ref[0], atol=1e-12)
    full = O.f16_prompt_attn(kb, vb, perm, ctx, q, 0.05, causal=False)
    kk = [[kf[perm[t], 0, j] for j in range(d)] for t in range(ctx)]
    vv = [[vf[perm[t], 0, j] for j in range(d)] for t in range(ctx)]
    assert np.allclose(full[0, 1], _loop_attention(q[0:1, 1], kk, vv, 0.05)[0], atol=1e-12)


def test_f16_rows_of_integers_match_int8_rows_with_unit_scales():
    # the two cache modes agree when the binary16 rows hold the int8 values and
    # every scale is 1
    n_cells, hkv, d = 16, 1, 128
    raw = W.gaussian_with_outliers(10, W.S_K, W.S_K_OUT, n_cells, hkv, d)
    ki, _ = W.int8_rows(raw)
    vi, _ = W.int8_rows(W.gaussian_with_outliers(10, W.S_V, W.S_V_OUT, n_cells, hkv, d))
    ones = W.to_f16_bits(np.ones((n_cells, hkv)))
    q = W.normal(10, W.S_Q, 3 * 2 * d).reshape(3, 2, d) * 0.01
    perm = W.permutation(10, W.S_PERM, n_cells)
    a = O.int8_prompt_attn(ki, ones, vi, ones, perm, n_cells, q, 0.1)
    b = O.f16_prompt_attn(W.to_f16_bits(ki.astype(np.float64)), W.to_f16_bits(vi.astype(np.float64)), perm,
                          n_cells, q, 0.1)
    assert np.allclose(a, b, atol=1e-12)


def test_nmse_definition():
    b = np.array([1.0, 2.0, 2.0])
    a = b + np.array([0.0, 0.3, 0.0])
    assert abs(O.nmse(a, b) - 0.09 / 9.0) < 1e-15


# ---------------------------------------------- rotation order and prefill pins

def test_rotation_applies_signs_before_the_hadamard():
    # y = H S x / sqrt(128): for x = e_j with sign bit j set, S e_j = -e_j, so
    # y = -H[:, j] / sqrt(128); with bit j clear and another bit set, y = +H[:, j] / sqrt(128)
    # (the other order, S H x, would flip one element of H[:, j] instead)
    H = O.hadamard()
    for j, bits in ((5, {5}), (5, {9}), (77, {77, 3}), (0, {0, 127})):
        sb = np.zeros(4, np.uint32)
        for b in bits:
            sb[b // 32] |= np.uint32(1 << (b % 32))
        x = np.zeros(128)
        x[j] = 1.0
        want = (-1.0 if j in bits else 1.0) * H[:, j] / math.sqrt(128)
        assert np.array_equal(O.rotation(sb) @ x, want)
        _, _, y = O.quantize_blocks(x, sb, O.centroids(3))
        assert np.allclose(y, want, atol=1e-15)
    # random x against the page's butterfly applied to the sign-flipped input
    sb = W.sign_bits(12, W.S_SIGNS_K)
    x = W.normal(12, 1, 6 * 128).reshape(6, 128)
    s = np.where([(int(sb[i // 32]) >> (i % 32)) & 1 for i in range(128)], -1.0, 1.0)
    assert np.allclose(x @ O.rotation(sb).T, O.butterfly_wht(x * s) / math.sqrt(128), atol=1e-14)


def _dequant_rows_by_loops(cache, sign_bits, cents, n, head):
    """Rows of cells 0..n-1 of one head, rebuilt element by element: value of each
    code (sign-magnitude), the page's butterfly on the block, the sign flips, the
    norm, and the padding columns dropped."""
    s = [-1.0 if (int(sign_bits[i // 32]) >> (i % 32)) & 1 else 1.0 for i in range(128)]
    half = len(cents) // 2
    rows = []
    for t in range(n):
        row = []
        for b in range(cache.n_blocks):
            codes = O.unpack_codes(cache.qs[head, t, b], None if cache.signs is None else cache.signs[head, t, b],
                                   cache.tq_type)
            vals = [(1.0 if k >= half else -1.0) * cents[half + (k % half)] for k in codes]
            hv = O.butterfly_wht(np.array(vals))          # H is symmetric: H^T c = H c
            nrm = float(np.array(cache.norms[head, t, b], np.uint16).view(np.float16))
            row += [nrm * s[i] * hv[i] / math.sqrt(128) for i in range(128)]
        rows.append(row[:cache.head_dim])
    return np.array(rows)


def _tiny_asym_caches(seed):
    # 2 KV heads, Dk = 192 (two blocks, the second zero-padded), Dv = 128; 12 cells
    # written, of which the calls below attend the first kv_len
    c = O.centroids(3)
    sk, sv = W.sign_bits(seed, W.S_SIGNS_K), W.sign_bits(seed, W.S_SIGNS_V)
    kc = O.empty_cache(3, 2, 192, 64)
    vc = O.empty_cache(3, 2, 128, 64)
    O.set_rows(kc, W.gaussian_with_outliers(seed, W.S_K, W.S_K_OUT, 12, 2, 192), np.arange(12), sk, c)
    O.set_rows(vc, W.gaussian_with_outliers(seed, W.S_V, W.S_V_OUT, 12, 2, 128), np.arange(12), sv, c)
    return kc, vc, sk, sv, c


def test_prefill_causal_gqa_asymmetric_by_loops():
    # C2's causal rule: query i of nq sits at position kv_len - nq + i and sees keys
    # 0 .. kv_len - nq + i; query head h reads KV head h // (Hq / Hkv); Dk = 192, Dv = 128
    kc, vc, sk, sv, c = _tiny_asym_caches(31)
    kv_len, nq, hq = 9, 3, 4
    q = W.normal(31, W.S_Q, nq * hq * 192).reshape(nq, hq, 192) * 2.0
    scale = 1 / math.sqrt(192)
    out = O.prefill(kc, vc, sk, sv, c, c, q, kv_len, scale, causal=True)
    assert out.shape == (nq, hq, 128)
    for hk in range(2):
        k = _dequant_rows_by_loops(kc, sk, c, kv_len, hk)
        v = _dequant_rows_by_loops(vc, sv, c, kv_len, hk)
        for h in (2 * hk, 2 * hk + 1):
            for i in range(nq):
                last = kv_len - nq + i                   # 6, 7, 8
                ref = _loop_attention(q[i:i + 1, h], k[:last + 1], v[:last + 1], scale)[0]
                assert np.allclose(out[i, h], ref, atol=1e-12)
    # the rows= subset gives the same rows and zeros elsewhere
    sub = O.prefill(kc, vc, sk, sv, c, c, q, kv_len, scale, causal=True, rows=np.array([2]))
    assert np.allclose(sub[2], out[2], atol=1e-14) and not sub[:2].any()


def test_prefill_non_causal_by_loops():
    kc, vc, sk, sv, c = _tiny_asym_caches(32)
    kv_len, nq, hq = 10, 4, 2                            # GQA 1: head h reads KV head h
    q = W.normal(32, W.S_Q, nq * hq * 192).reshape(nq, hq, 192)
    scale = 0.11
    out = O.prefill(kc, vc, sk, sv, c, c, q, kv_len, scale, causal=False)
    for h in range(hq):
        k = _dequant_rows_by_loops(kc, sk, c, kv_len, h)
        v = _dequant_rows_by_loops(vc, sv, c, kv_len, h)
        assert np.allclose(out[:, h], _loop_attention(q[:, h], k, v, scale), atol=1e-12)


def test_dequantize_cache_matches_loops():
    kc, vc, sk, sv, c = _tiny_asym_caches(33)
    for hk in range(2):
        assert np.allclose(O.dequantize_cache(kc, sk, c, 12, hk), _dequant_rows_by_loops(kc, sk, c, 12, hk),
                           atol=1e-13)
        assert np.allclose(O.dequantize_cache(vc, sv, c, 12, hk), _dequant_rows_by_loops(vc, sv, c, 12, hk),
                           atol=1e-13)


def test_empty_key_range_gives_zero_output():
    # kv_len = 0: nothing to attend, the output is zero (decode and prefill)
    kc, vc, sk, sv, c = _tiny_asym_caches(34)
    q = W.normal(34, W.S_Q, 4 * 192).reshape(4, 192)
    assert O.dequantize_cache(kc, sk, c, 0).shape == (2, 0, 192)
    out = O.decode(kc, vc, sk, sv, c, c, q, 0, 0.1)
    assert out.shape == (4, 128) and not out.any()
    assert not O.prefill(kc, vc, sk, sv, c, c, q.reshape(1, 4, 192), 0, 0.1, causal=False).any()


def test_sparse_v_slack_reaches_decode_and_empty_keys():
    # decode_sparse_v hands its slack to every head: a slack that lifts the cut above
    # most weights changes the result exactly as the per-head call with that slack
    shape = W.AttnShape("t", 2, 4, 128, 128, 40, seed=6)
    c = O.centroids(3)
    sk, sv = W.codebook_signs(shape)
    kr, vr = W.kv_inputs(shape)
    kc = O.empty_cache(3, 2, 128, 64)
    vc = O.empty_cache(3, 2, 128, 64)
    O.set_rows(kc, kr, np.arange(40), sk, c)
    O.set_rows(vc, vr, np.arange(40), sv, c)
    q = W.decode_query(shape) * 4
    scale = 1 / math.sqrt(128)
    o1, _, _ = O.decode_sparse_v(kc, vc, sk, sv, c, c, q, 40, scale, 1e-2)
    o2, _, b2 = O.decode_sparse_v(kc, vc, sk, sv, c, c, q, 40, scale, 1e-2, slack=50.0)
    kh = O.dequantize_cache(kc, sk, c, 40)
    vh = O.dequantize_cache(vc, sv, c, 40)
    for h in range(4):
        ref, _, rb = O.sparse_v_attention(q[h:h + 1], kh[h // 2], vh[h // 2], scale, 1e-2, slack=50.0)
        assert np.allclose(o2[h], ref[0], atol=1e-14) and np.allclose(b2[h], rb[0], atol=1e-14)
    assert not np.allclose(o1, o2)                        # the cut at 0.5 leaves more keys out
    # no keys: zero output and zero bound
    z = O.sparse_v_attention(q[:1], np.zeros((0, 128)), np.zeros((0, 128)), scale, 1e-3)
    assert all(x.shape == (1, 128) and not x.any() for x in z)


def test_lse_partial_pieces():
    # (m, l, o) of a key range: m the maximum score, l = sum exp(s - m), o the
    # softmax-weighted values of that range alone
    q = W.normal(12, 1, 3 * 16).reshape(3, 16)
    k = W.normal(12, 2, 30 * 16).reshape(30, 16)
    v = W.normal(12, 3, 30 * 8).reshape(30, 8)
    m, l, o = O.lse_partial(q, k, v, 0.3)
    s = 0.3 * (q @ k.T)
    assert np.array_equal(m, s.max(axis=1))
    assert np.allclose(l, np.exp(s - s.max(axis=1, keepdims=True)).sum(axis=1), rtol=1e-15)
    assert np.allclose(o, O.softmax_attention(q, k, v, 0.3), atol=1e-14)


def test_set_rows_keeps_f64_inputs_exact():
    # the rotated values set_rows reports are R x / |x| of the f64 rows as given (no
    # rounding of the source to a narrower type on the way)
    c = O.centroids(3)
    sb = W.sign_bits(3, W.S_SIGNS_K)
    src = W.normal(3, 4, 3 * 2 * 128).reshape(3, 2, 128) * (1 + 2.0 ** -40)
    cache = O.empty_cache(3, 2, 128, 8)
    y = O.set_rows(cache, src, np.array([5, 1, 6]), sb, c)
    ref = src @ O.rotation(sb).T / np.linalg.norm(src, axis=-1, keepdims=True)
    assert np.allclose(y[:, :, 0], ref, rtol=0, atol=1e-15)


@pytest.mark.parametrize("mode", ["int8", "f16", "prefill"])
def test_rows_subset_is_the_full_rows_and_zero_elsewhere(mode):
    # the rows= argument of the multi-query functions: the chosen rows equal the
    # full computation, every other row is zero
    nq, hq, d = 5, 4, 128
    rows = np.array([1, 4])
    q = W.normal(13, W.S_Q, nq * hq * d).reshape(nq, hq, d)
    if mode == "prefill":
        shape = W.AttnShape("t", 2, hq, d, d, 24, seed=13)
        c = O.centroids(3)
        sk, sv = W.codebook_signs(shape)
        kr, vr = W.kv_inputs(shape)
        kc = O.empty_cache(3, 2, d, 32)
        vc = O.empty_cache(3, 2, d, 32)
        O.set_rows(kc, kr, np.arange(24), sk, c)
        O.set_rows(vc, vr, np.arange(24), sv, c)
        run = lambda r: O.prefill(kc, vc, sk, sv, c, c, q, 24, 0.1, causal=True, rows=r)
    else:
        n_cells = 24
        raw = W.gaussian_with_outliers(13, W.S_K, W.S_K_OUT, n_cells, 2, d)
        rawv = W.gaussian_with_outliers(13, W.S_V, W.S_V_OUT, n_cells, 2, d)
        perm = W.permutation(13, W.S_PERM, n_cells)
        if mode == "int8":
            ki, ks = W.int8_rows(raw)
            vi, vs = W.int8_rows(rawv)
            run = lambda r: O.int8_prompt_attn(ki, ks, vi, vs, perm, 20, q, 0.1, causal=True, rows=r)
        else:
            kb, vb = W.to_f16_bits(raw), W.to_f16_bits(rawv)
            run = lambda r: O.f16_prompt_attn(kb, vb, perm, 20, q, 0.1, causal=True, rows=r)
    full, sub = run(None), run(rows)
    assert np.array_equal(sub[rows], full[rows])
    others = np.setdiff1d(np.arange(nq), rows)
    assert not sub[others].any() and full[others].any()

"""CPU oracle for attention over a TurboQuant-compressed KV cache (plain numpy, f64).

TEST INFRASTRUCTURE.  Only the tests, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  It shares no code with the CUDA library: the rotation is a dense
Hadamard matrix built from its closed form, the encoder is a brute-force
nearest-centroid search, and attention is dequantise-then-exact-softmax.

Sources (the pages this restates; no code was taken from them):

  [TQ#36]   llama-cpp-turboquant pull request #36 -- four commit messages:
            "shuffle WHT" (butterfly stages h=1..64 and the update
            o = x[j^h]; x[j] = (j&h) ? o - x[j] : x[j] + o),
            "asymmetric D" (K head dim 192, V head dim 128, padding),
            "Q x centroid LUT" (4/8/16 centroids; 2 qs bytes + 1 signs byte
            per 8 elements), "VEC tuning" (results table; turbo2 = 7.5x;
            item 3: sparse V thresholds 5e-3 for turbo3/4, 1e-2 for turbo2).
  [HIP#28]  atomic-llama-cpp-turboquant pull request #28, "HIP/turbo3:
            graph-safe decode + inline-dequant TILE prefill" -- sections
            "Two coupled changes" and "Correctness" (NMSE vs a CPU reference).
  [QSA#1821] "qsa_prompt_attn: int8 K/V prefetched in registers and sharing
            one buffer" -- sections "What", "Change" (scattered int8 rows with
            per-row scales, 32-cell chunks) and "Measured".

Readings where the pages are silent (each is a rule both sides follow):

  * block = 128 elements; one fp16 (round-to-nearest-even) L2 norm per block;
    the block is divided by its exact norm, multiplied by a seeded +-1 sign
    vector S, rotated by the unnormalised Hadamard H and scaled by 1/sqrt(128):
    y = H S x / (|x| sqrt(128)).  A zero block keeps y = 0.
  * centroids: the Lloyd-Max quantiser of N(0,1) (Lloyd iteration in f64),
    divided by sqrt(128), each rounded to the nearest binary16 value; the
    rounded values are the codebook.
  * nearest centroid: argmin |y - c_i|; on an exact tie the higher centroid.
  * codes are sign-magnitude: code k = s * n/2 + j, value (+1 if s else -1) *
    c[n/2 + j] with the positive centroids ascending in j.  turbo3 stores j in
    the qs plane (2 bits) and s in the signs plane; turbo2 stores the 2-bit
    code and turbo4 the 4-bit code in the qs plane.
  * bit layout: see ``pack_codes``.
  * attention is exact softmax(scale * q.k) v over the dequantised rows with
    scale given by the caller; causal query i of nq sits at position
    kv_len - nq + i; query head h reads KV head h // (Hq / Hkv).
  * kv_len = 0 gives a zero output.
  * sparse V ([TQ#36 "VEC tuning"] item 3 names only the thresholds): a key whose
    softmax weight relative to the maximum score, exp(s - max), is below the
    threshold adds nothing to the weighted sum of V rows; the normaliser still
    sums every key.  A kernel sees only a running maximum, which is at most the
    final one, so the keys it leaves out are a subset of those this rule names
    with the final maximum: ``sparse_v_attention`` returns the result without
    them, the exact result and the bound on the distance of any such subset's
    result from both.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
from scipy.special import ndtr

QK = 128                      # elements per quantisation block
QS_BYTES = {2: 32, 3: 32, 4: 64}
SIGN_BYTES = 16
N_CENTROIDS = {2: 4, 3: 8, 4: 16}


# ---------------------------------------------------------------------------
# rotation  [TQ#36 "shuffle WHT"]
# ---------------------------------------------------------------------------

def hadamard(n: int = QK) -> np.ndarray:
    """Sylvester Hadamard matrix, H[i][j] = (-1)^popcount(i & j)."""
    i = np.arange(n)
    a = i[:, None] & i[None, :]
    parity = np.zeros_like(a)
    while a.any():
        parity ^= a & 1
        a >>= 1
    return np.where(parity == 0, 1.0, -1.0)


def sign_vector(sign_bits) -> np.ndarray:
    """+-1 diagonal of S: bit i of the 128-bit little-endian word set => -1."""
    s = np.ones(QK)
    for i in range(QK):
        if (int(sign_bits[i // 32]) >> (i % 32)) & 1:
            s[i] = -1.0
    return s


def rotation(sign_bits) -> np.ndarray:
    """R = H S / sqrt(128) (orthonormal)."""
    return hadamard() * sign_vector(sign_bits)[None, :] / math.sqrt(QK)


def butterfly_wht(x: np.ndarray) -> np.ndarray:
    """The pages' butterfly recursion, stage by stage (h = 1, 2, ..., 64):
    element j takes o = x[j ^ h] and becomes (j & h) ? o - x[j] : x[j] + o.
    Used only as an independent pin of the dense ``hadamard``."""
    x = np.array(x, dtype=np.float64)
    n = x.shape[-1]
    j = np.arange(n)
    h = 1
    while h < n:
        o = x[..., j ^ h]
        x = np.where((j & h) != 0, o - x, x + o)
        h *= 2
    return x


# ---------------------------------------------------------------------------
# codebooks  [TQ#36 "Q x centroid LUT": 4 / 8 / 16 centroids]
# ---------------------------------------------------------------------------

def _interval_prob(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    # P(a < X < b) for X ~ N(0,1), evaluated on the side that avoids cancellation
    return np.where(a >= 0, ndtr(-a) - ndtr(-b), ndtr(b) - ndtr(a))


def _phi(x: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore", invalid="ignore"):
        return np.where(np.isinf(x), 0.0, np.exp(-0.5 * x * x) / math.sqrt(2 * math.pi))


def lloyd_max_normal(n_levels: int, tol: float = 1e-15, max_iter: int = 200000) -> np.ndarray:
    """Lloyd-Max quantiser of N(0,1): alternate midpoint thresholds and
    conditional-mean centroids until a fixed point.  Returns ascending f64."""
    c = np.array([-(n_levels - 1) / 2 + k for k in range(n_levels)], dtype=np.float64)
    c *= 3.0 / n_levels
    for _ in range(max_iter):
        t = np.concatenate(([-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]))
        a, b = t[:-1], t[1:]
        new = (_phi(a) - _phi(b)) / _interval_prob(a, b)
        if np.max(np.abs(new - c)) < tol:
            c = new
            break
        c = new
    return c


def lloyd_max_distortion(c: np.ndarray) -> float:
    """E[(X - Q(X))^2] for X ~ N(0,1) and nearest-centroid Q with centroids c."""
    t = np.concatenate(([-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]))
    a, b = t[:-1], t[1:]
    p = _interval_prob(a, b)
    # E[X^2; a<X<b] = P + a phi(a) - b phi(b)   (with x phi(x) -> 0 at +-inf)
    with np.errstate(invalid="ignore"):
        aphi = np.where(np.isinf(a), 0.0, a * _phi(a))
        bphi = np.where(np.isinf(b), 0.0, b * _phi(b))
    ex2 = p + aphi - bphi
    ex = _phi(a) - _phi(b)
    return float(np.sum(ex2 - 2 * c * ex + c * c * p))


def centroids(tq_type: int) -> np.ndarray:
    """Canonical centroid table (ascending f64 values, each binary16-exact)."""
    c = lloyd_max_normal(N_CENTROIDS[tq_type]) / math.sqrt(QK)
    return c.astype(np.float16).astype(np.float64)


# ---------------------------------------------------------------------------
# codes and bit layout  [TQ#36 "Q x centroid LUT": 2 qs bytes + 1 signs byte
# per 8 elements for turbo3]
# ---------------------------------------------------------------------------

def index_to_code(i: np.ndarray, n: int) -> np.ndarray:
    half = n // 2
    return np.where(i >= half, i, half - 1 - i)


def code_to_value(k: np.ndarray, cents: np.ndarray) -> np.ndarray:
    n = len(cents)
    half = n // 2
    s = k // half
    j = k % half
    mag = cents[half + j]
    return np.where(s == 1, mag, -mag)


def _qs_field(tq_type: int, e: int):
    """(byte offset, bit shift, width) of element e's field in the qs plane."""
    if tq_type == 4:
        w, i = divmod(e, 8)
        bit = 4 * i
        return 4 * w + bit // 8, bit % 8, 4
    w, r = divmod(e, 16)
    bit = 4 * r if r < 8 else 4 * (r - 8) + 2
    return 4 * w + bit // 8, bit % 8, 2


def _sign_bit(e: int):
    """(byte offset, bit shift) of element e's sign bit in the turbo3 signs plane."""
    u, r = divmod(e, 32)
    if r < 16:
        bit = 4 * (r % 8) + 2 + r // 8
    else:
        rr = r - 16
        bit = 4 * (rr % 8) + rr // 8
    return 4 * u + bit // 8, bit % 8


def pack_codes(codes: np.ndarray, tq_type: int):
    """codes [..., 128] (sign-magnitude) -> (qs [..., QS_BYTES], signs [..., 16] or None).

    qs plane, turbo2/turbo3: 8 little-endian 32-bit words; word w holds elements
    16w..16w+15; element 16w+i (i<8) at bits 4i..4i+1, element 16w+8+i at bits
    4i+2..4i+3.  turbo2 stores the whole 2-bit code there, turbo3 the magnitude
    index j.  turbo4: 16 words; word w holds elements 8w..8w+7, element 8w+i at
    bits 4i..4i+3 (the 4-bit code).  signs plane (turbo3): 4 words; word u holds
    elements 32u..32u+31; element 32u+r for r<16 at bit 4(r%8)+2+(r//8), for
    r>=16 at bit 4((r-16)%8)+((r-16)//8).
    """
    codes = np.asarray(codes, dtype=np.int64)
    lead = codes.shape[:-1]
    qs = np.zeros(lead + (QS_BYTES[tq_type],), dtype=np.uint8)
    signs = np.zeros(lead + (SIGN_BYTES,), dtype=np.uint8) if tq_type == 3 else None
    for e in range(QK):
        byte, shift, width = _qs_field(tq_type, e)
        k = codes[..., e]
        field_val = (k & 3) if tq_type == 3 else k
        qs[..., byte] |= ((field_val << shift) & 0xFF).astype(np.uint8)
        if tq_type == 3:
            sb, ss = _sign_bit(e)
            signs[..., sb] |= (((k >> 2) & 1) << ss).astype(np.uint8)
    return qs, signs


def unpack_codes(qs: np.ndarray, signs, tq_type: int) -> np.ndarray:
    qs = np.asarray(qs, dtype=np.int64)
    codes = np.zeros(qs.shape[:-1] + (QK,), dtype=np.int64)
    for e in range(QK):
        byte, shift, width = _qs_field(tq_type, e)
        v = (qs[..., byte] >> shift) & ((1 << width) - 1)
        if tq_type == 3:
            sb, ss = _sign_bit(e)
            v = v | (((np.asarray(signs[..., sb], dtype=np.int64) >> ss) & 1) << 2)
        codes[..., e] = v
    return codes


# ---------------------------------------------------------------------------
# quantise / dequantise one 128-element block
# ---------------------------------------------------------------------------

def quantize_blocks(x: np.ndarray, sign_bits, cents: np.ndarray):
    """x [..., 128] -> (norm fp16 bits, codes [..., 128], rotated y [..., 128] f64).

    norm = fp16_rne(|x|); y = R x / |x| with the exact norm; code = nearest
    centroid (ties to the higher one), sign-magnitude encoded."""
    x = np.asarray(x, dtype=np.float64)
    nrm = np.sqrt(np.sum(x * x, axis=-1))
    norm_bits = nrm.astype(np.float16).view(np.uint16)
    safe = np.where(nrm > 0, nrm, 1.0)
    u = np.where(nrm[..., None] > 0, x / safe[..., None], 0.0)
    y = u @ rotation(sign_bits).T
    return norm_bits, index_to_code(nearest_centroid(y, cents), len(cents)), y


def nearest_centroid(y: np.ndarray, cents: np.ndarray) -> np.ndarray:
    """Brute force: index of the closest centroid to each y (ties -> higher index)."""
    dist = np.abs(np.asarray(y)[..., None] - cents)          # [..., n]
    return len(cents) - 1 - np.argmin(dist[..., ::-1], axis=-1)


def dequantize_blocks(norm_bits: np.ndarray, codes: np.ndarray, sign_bits, cents: np.ndarray):
    """x_hat = n * R^T c[code] for every block; returns [..., 128] f64."""
    n = np.asarray(norm_bits, dtype=np.uint16).view(np.float16).astype(np.float64)
    vals = code_to_value(codes, cents)
    return n[..., None] * (vals @ rotation(sign_bits))


# ---------------------------------------------------------------------------
# cache planes and SET_ROWS
# ---------------------------------------------------------------------------

@dataclass
class Cache:
    tq_type: int
    n_kv_heads: int
    head_dim: int
    n_cells: int
    norms: np.ndarray            # uint16 [H][n_cells][nb]
    qs: np.ndarray               # uint8  [H][n_cells][nb][QS_BYTES]
    signs: np.ndarray | None     # uint8  [H][n_cells][nb][16]  (turbo3)

    @property
    def n_blocks(self) -> int:
        return (self.head_dim + QK - 1) // QK


def empty_cache(tq_type: int, n_kv_heads: int, head_dim: int, n_cells: int) -> Cache:
    nb = (head_dim + QK - 1) // QK
    return Cache(tq_type, n_kv_heads, head_dim, n_cells,
                 np.zeros((n_kv_heads, n_cells, nb), np.uint16),
                 np.zeros((n_kv_heads, n_cells, nb, QS_BYTES[tq_type]), np.uint8),
                 np.zeros((n_kv_heads, n_cells, nb, SIGN_BYTES), np.uint8) if tq_type == 3 else None)


def _pad_blocks(x: np.ndarray, head_dim: int) -> np.ndarray:
    nb = (head_dim + QK - 1) // QK
    pad = nb * QK - head_dim
    if pad:
        x = np.concatenate([x, np.zeros(x.shape[:-1] + (pad,))], axis=-1)
    return x.reshape(x.shape[:-1] + (nb, QK))


def set_rows(cache: Cache, src: np.ndarray, cell_ids: np.ndarray, sign_bits, cents: np.ndarray):
    """Quantise rows src [n_rows][H][D] into cells cell_ids (in place); returns
    the rotated values y [n_rows][H][nb][128] for boundary-distance checks.
    Cell ids must be distinct."""
    src = np.asarray(src)
    cell_ids = np.asarray(cell_ids, dtype=np.int64)
    ys = []
    for lo in range(0, src.shape[0], 2048):              # row batches bound the memory use
        blocks = _pad_blocks(np.asarray(src[lo:lo + 2048], dtype=np.float64), cache.head_dim)
        norm_bits, codes, y = quantize_blocks(blocks, sign_bits, cents)   # [n][H][nb][...]
        qs, signs = pack_codes(codes, cache.tq_type)
        cells = cell_ids[lo:lo + 2048]
        cache.norms[:, cells] = norm_bits.transpose(1, 0, 2)
        cache.qs[:, cells] = qs.transpose(1, 0, 2, 3)
        if signs is not None:
            cache.signs[:, cells] = signs.transpose(1, 0, 2, 3)
        ys.append(y)
    return np.concatenate(ys) if ys else np.zeros((0, cache.n_kv_heads, cache.n_blocks, QK))


def dequantize_cache(cache: Cache, sign_bits, cents: np.ndarray, n: int, head: int | None = None):
    """Dequantised rows of cells 0..n-1: [H][n][D] (or [n][D] for one head)."""
    heads = range(cache.n_kv_heads) if head is None else [head]
    out = []
    for h in heads:
        codes = unpack_codes(cache.qs[h, :n], None if cache.signs is None else cache.signs[h, :n],
                             cache.tq_type)
        x = dequantize_blocks(cache.norms[h, :n], codes, sign_bits, cents)
        out.append(x.reshape(n, cache.n_blocks * QK)[:, :cache.head_dim])
    return out[0] if head is not None else np.stack(out)


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def softmax_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                      q_pos: np.ndarray | None = None) -> np.ndarray:
    """Exact softmax(scale * q k^T) v in f64.  q [nq][Dk], k [L][Dk], v [L][Dv];
    with q_pos, query i sees keys 0..q_pos[i] only."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    if k.shape[0] == 0:
        return np.zeros((q.shape[0], v.shape[1]))
    s = scale * (q @ k.T)
    if q_pos is not None:
        mask = np.arange(k.shape[0])[None, :] > np.asarray(q_pos)[:, None]
        s = np.where(mask, -np.inf, s)
    m = np.max(s, axis=1, keepdims=True)
    e = np.exp(s - m)
    return (e @ v) / np.sum(e, axis=1, keepdims=True)


def sparse_v_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                       threshold: float, slack: float = 1.0):
    """Sparse-V decode attention of queries q [nq][Dk] over k [L][Dk], v [L][Dv]
    (f64).  With p_t = exp(s_t - max_t s_t), s = scale q.k, the keys with
    p_t < threshold * slack are left out of the V sum (the normaliser keeps them):
        o_skip  = sum_{kept t} p_t v_t / sum_t p_t
        o_exact = sum_t p_t v_t / sum_t p_t
        bound_d = sum_{left-out t} p_t |v_t,d| / sum_t p_t.
    Any result that leaves out a subset of those keys is within bound of both.
    Returns (o_skip, o_exact, bound), each [nq][Dv]."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    if k.shape[0] == 0:
        z = np.zeros((q.shape[0], v.shape[1]))
        return z, z.copy(), z.copy()
    s = scale * (q @ k.T)
    p = np.exp(s - np.max(s, axis=1, keepdims=True))
    total = np.sum(p, axis=1, keepdims=True)
    out = p < threshold * slack
    p_kept = np.where(out, 0.0, p)
    p_out = np.where(out, p, 0.0)
    return (p_kept @ v) / total, (p @ v) / total, (p_out @ np.abs(v)) / total


def lse_partial(q, k, v, scale):
    """(m, l, o) of one key range: m = max score, l = sum exp(s - m),
    o = sum exp(s - m) v / l  (the pieces a split-KV pass keeps)."""
    s = scale * (np.asarray(q, np.float64) @ np.asarray(k, np.float64).T)
    m = np.max(s, axis=-1)
    e = np.exp(s - m[..., None])
    l = np.sum(e, axis=-1)
    return m, l, (e @ np.asarray(v, np.float64)) / l[..., None]


def lse_merge(parts):
    """Combine (m_s, l_s, o_s) partials into the full softmax-weighted output."""
    ms = np.stack([p[0] for p in parts])
    M = np.max(ms, axis=0)
    w = np.stack([p[1] * np.exp(p[0] - M) for p in parts])
    o = sum(w[i][..., None] * parts[i][2] for i in range(len(parts)))
    return o / np.sum(w, axis=0)[..., None]


def decode(kc: Cache, vc: Cache, k_signs, v_signs, k_cents, v_cents,
           q: np.ndarray, kv_len: int, scale: float) -> np.ndarray:
    """Single-query decode: q [Hq][Dk] -> out [Hq][Dv] over cells 0..kv_len-1."""
    n_q = q.shape[0]
    g = n_q // kc.n_kv_heads
    out = np.zeros((n_q, vc.head_dim))
    for hk in range(kc.n_kv_heads):
        k = dequantize_cache(kc, k_signs, k_cents, kv_len, hk)
        v = dequantize_cache(vc, v_signs, v_cents, kv_len, hk)
        for h in range(hk * g, (hk + 1) * g):
            out[h] = softmax_attention(q[h][None, :], k, v, scale)[0]
    return out


def decode_sparse_v(kc: Cache, vc: Cache, k_signs, v_signs, k_cents, v_cents,
                    q: np.ndarray, kv_len: int, scale: float, threshold: float, slack: float = 1.0):
    """Single-query decode with sparse V (see ``sparse_v_attention``):
    q [Hq][Dk] -> (o_skip, o_exact, bound), each [Hq][Dv]."""
    n_q = q.shape[0]
    g = n_q // kc.n_kv_heads
    res = [np.zeros((n_q, vc.head_dim)) for _ in range(3)]
    for hk in range(kc.n_kv_heads):
        k = dequantize_cache(kc, k_signs, k_cents, kv_len, hk)
        v = dequantize_cache(vc, v_signs, v_cents, kv_len, hk)
        for h in range(hk * g, (hk + 1) * g):
            for r, x in zip(res, sparse_v_attention(q[h][None, :], k, v, scale, threshold, slack)):
                r[h] = x[0]
    return tuple(res)


def prefill(kc: Cache, vc: Cache, k_signs, v_signs, k_cents, v_cents,
            q: np.ndarray, kv_len: int, scale: float, causal: bool = True,
            rows: np.ndarray | None = None) -> np.ndarray:
    """Multi-query attention: q [nq][Hq][Dk] -> out [nq][Hq][Dv].  Causal query i
    sits at position kv_len - nq + i.  ``rows`` restricts the work to some query
    rows (the output keeps all rows; the others are zero)."""
    nq, n_q, _ = q.shape
    g = n_q // kc.n_kv_heads
    rows = np.arange(nq) if rows is None else np.asarray(rows)
    pos = (kv_len - nq + rows) if causal else None
    out = np.zeros((nq, n_q, vc.head_dim))
    for hk in range(kc.n_kv_heads):
        k = dequantize_cache(kc, k_signs, k_cents, kv_len, hk)
        v = dequantize_cache(vc, v_signs, v_cents, kv_len, hk)
        for h in range(hk * g, (hk + 1) * g):
            out[rows, h] = softmax_attention(q[rows, h], k, v, scale, pos)
    return out


def int8_dequantize(rows_i8: np.ndarray, scale_bits: np.ndarray) -> np.ndarray:
    """value * float(scale) for int8 rows [..., D] with fp16 scales [...]."""
    s = np.asarray(scale_bits, np.uint16).view(np.float16).astype(np.float64)
    return np.asarray(rows_i8, np.float64) * s[..., None]


def int8_prompt_attn(k_i8, k_scale, v_i8, v_scale, cell_of_pos, ctx: int,
                     q: np.ndarray, scale: float, causal: bool = True,
                     rows: np.ndarray | None = None) -> np.ndarray:
    """[QSA#1821 "What"/"Change"]: attention of q [nq][Hq][D] over the logical
    positions 0..ctx-1, position p reading cell cell_of_pos[p] of the int8 cache
    k_i8/v_i8 [n_cells][Hkv][D] with fp16 scales [n_cells][Hkv]."""
    nq, n_q, _ = q.shape
    hkv = k_i8.shape[1]
    g = n_q // hkv
    rows = np.arange(nq) if rows is None else np.asarray(rows)
    pos = (ctx - nq + rows) if causal else None
    cells = np.asarray(cell_of_pos[:ctx], dtype=np.int64)
    out = np.zeros((nq, n_q, v_i8.shape[2]))
    for hk in range(hkv):
        k = int8_dequantize(k_i8[cells, hk], k_scale[cells, hk])
        v = int8_dequantize(v_i8[cells, hk], v_scale[cells, hk])
        for h in range(hk * g, (hk + 1) * g):
            out[rows, h] = softmax_attention(q[rows, h], k, v, scale, pos)
    return out


def f16_prompt_attn(k_bits, v_bits, cell_of_pos, ctx: int, q: np.ndarray, scale: float, causal: bool = True,
                    rows: np.ndarray | None = None) -> np.ndarray:
    """The other cache mode of [QSA#1821] ("Measured": output checksums for int8
    and fp16): the same attention with rows k, v read as binary16 values
    [n_cells][Hkv][D] (uint16 bit patterns), no scales."""
    nq, n_q, _ = q.shape
    kv = np.asarray(k_bits, dtype=np.uint16).view(np.float16).astype(np.float64)
    vv = np.asarray(v_bits, dtype=np.uint16).view(np.float16).astype(np.float64)
    hkv = kv.shape[1]
    g = n_q // hkv
    rows = np.arange(nq) if rows is None else np.asarray(rows)
    pos = (ctx - nq + rows) if causal else None
    cells = np.asarray(cell_of_pos[:ctx], dtype=np.int64)
    out = np.zeros((nq, n_q, vv.shape[2]))
    for hk in range(hkv):
        k = kv[cells, hk]
        v = vv[cells, hk]
        for h in range(hk * g, (hk + 1) * g):
            out[rows, h] = softmax_attention(q[rows, h], k, v, scale, pos)
    return out


def nmse(a: np.ndarray, b: np.ndarray) -> float:
    """sum (a - b)^2 / sum b^2, b the reference ([HIP#28 "Correctness"])."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    den = float(np.sum(b * b))
    return float(np.sum((a - b) ** 2)) / den if den > 0 else float(np.sum((a - b) ** 2))


def bits_per_element(tq_type: int) -> float:
    """Stored bits per element: qs + signs + one fp16 norm per 128 elements."""
    b = QS_BYTES[tq_type] + (SIGN_BYTES if tq_type == 3 else 0) + 2
    return 8.0 * b / QK

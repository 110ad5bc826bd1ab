"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module only draws random numbers and lays them out in the shapes of the
workloads; it holds none of the quantiser's or the attention's arithmetic.

Random numbers come from one counter-based generator, defined here once:

    mix64(z)        the splitmix64 finaliser
                    z ^= z >> 30; z *= 0xBF58476D1CE4E5B9;
                    z ^= z >> 27; z *= 0x94D049BB133111EB; z ^= z >> 31
    key(seed, s)    mix64(mix64(seed) ^ (s * 0xD1B54A32D192ED03))
    bits(k, i)      mix64(k + (i + 1) * 0x9E3779B97F4A7C15)        (mod 2**64)
    uniform(k, i)   ((bits(k, i) >> 11) + 0.5) * 2**-53            in (0, 1)
    normal(k, 2i)   sqrt(-2 ln uniform(k, 2i)) * cos(2 pi uniform(k, 2i+1))
    normal(k, 2i+1) sqrt(-2 ln uniform(k, 2i)) * sin(2 pi uniform(k, 2i+1))

Workload shapes (named after what they are):

    tiny_decode      1 KV head, 1 query head, D=128, 512 cells, turbo3
    decode_32k       8 KV heads, 32 query heads (GQA 4), D=128, 32768 cells,
                     turbo3 (also turbo2 / turbo4 on the same inputs)
    prefill_4k       8 KV heads, 16 query heads, D=256, 4096 cells,
                     nq in {3, 64, 512, 2048, 4096}, causal, bf16 Q
    asym_8k          16 KV = 16 query heads, Dk=192, Dv=128, 8192 cells,
                     decode (fp32 Q) and prefill nq=512 (bf16 Q)
    int8_prompt      8 KV heads, 32 query heads, D=128, 2048 queries,
                     contexts 4096 / 40000 / 140000, fp16 Q, int8 rows
                     gathered through a seeded permutation of the cells

K/V (and the decode queries) are N(0,1) with 4 outlier channels per 128
channels scaled by 8 for every token; the outlier channels are drawn per
(tensor, head) by a seeded partial Fisher-Yates shuffle.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

_M64 = (1 << 64) - 1
_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_C1 = np.uint64(0xBF58476D1CE4E5B9)
_C2 = np.uint64(0x94D049BB133111EB)
_STREAM_MUL = 0xD1B54A32D192ED03

# stream ids: one per independent draw
S_Q, S_K, S_V = 1, 2, 3
S_Q_OUT, S_K_OUT, S_V_OUT = 4, 5, 6
S_SIGNS_K, S_SIGNS_V = 7, 8
S_PERM = 9
S_CELLS = 10
S_EXTRA = 11

OUTLIER_SCALE = 8.0
OUTLIERS_PER_128 = 4


def _mix64_scalar(z: int) -> int:
    z &= _M64
    z ^= z >> 30
    z = (z * 0xBF58476D1CE4E5B9) & _M64
    z ^= z >> 27
    z = (z * 0x94D049BB133111EB) & _M64
    z ^= z >> 31
    return z


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z ^ (z >> np.uint64(30))
    z = z * _C1
    z = z ^ (z >> np.uint64(27))
    z = z * _C2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> int:
    return _mix64_scalar(_mix64_scalar(seed) ^ ((stream * _STREAM_MUL) & _M64))


def bits(key: int, idx: np.ndarray) -> np.ndarray:
    """64 random bits for each counter value in ``idx`` (uint64 array)."""
    idx = np.asarray(idx, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return _mix64(np.uint64(key) + (idx + np.uint64(1)) * _GAMMA)


def uniform(key: int, idx: np.ndarray) -> np.ndarray:
    b = bits(key, idx)
    return ((b >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def normal(seed: int, stream: int, n: int, chunk: int = 1 << 22) -> np.ndarray:
    """n standard normal f64 values: pair i (values 2i, 2i+1) is the Box-Muller
    pair r cos(t), r sin(t) with r = sqrt(-2 ln uniform(k, 2i)), t = 2 pi uniform(k, 2i+1)."""
    key = stream_key(seed, stream)
    n_pairs = (n + 1) // 2
    out = np.empty(2 * n_pairs, dtype=np.float64)
    for lo in range(0, n_pairs, chunk):
        hi = min(n_pairs, lo + chunk)
        i = np.arange(lo, hi, dtype=np.uint64)
        r = np.sqrt(-2.0 * np.log(uniform(key, 2 * i)))
        t = 2.0 * math.pi * uniform(key, 2 * i + np.uint64(1))
        out[2 * lo:2 * hi:2] = r * np.cos(t)
        out[2 * lo + 1:2 * hi:2] = r * np.sin(t)
    return out[:n]


def outlier_channels(seed: int, stream: int, n_heads: int, dim: int) -> np.ndarray:
    """[n_heads][n_out] distinct channel indices per head (partial Fisher-Yates)."""
    n_out = max(1, round(OUTLIERS_PER_128 * dim / 128))
    key = stream_key(seed, stream)
    out = np.empty((n_heads, n_out), dtype=np.int64)
    for h in range(n_heads):
        perm = list(range(dim))
        r = bits(key, np.arange(h * dim, h * dim + n_out, dtype=np.uint64))
        for i in range(n_out):
            j = i + int(r[i] % np.uint64(dim - i))
            perm[i], perm[j] = perm[j], perm[i]
        out[h] = perm[:n_out]
    return out


def gaussian_with_outliers(seed: int, stream: int, out_stream: int, n_rows: int,
                           n_heads: int, dim: int, outliers: bool = True) -> np.ndarray:
    """f64 [n_rows][n_heads][dim]: N(0,1), outlier channels scaled by 8."""
    x = normal(seed, stream, n_rows * n_heads * dim).reshape(n_rows, n_heads, dim)
    if outliers:
        ch = outlier_channels(seed, out_stream, n_heads, dim)
        for h in range(n_heads):
            x[:, h, ch[h]] *= OUTLIER_SCALE
    return x


def sign_bits(seed: int, stream: int) -> np.ndarray:
    """128 random sign bits as 4 little-endian uint32 words (bit i set => -1)."""
    b = bits(stream_key(seed, stream), np.arange(2, dtype=np.uint64))
    words = []
    for v in b:
        v = int(v)
        words += [v & 0xFFFFFFFF, v >> 32]
    return np.array(words, dtype=np.uint32)


def permutation(seed: int, stream: int, n: int) -> np.ndarray:
    """A seeded permutation of range(n) (argsort of random 64-bit keys), int32."""
    if n == 0:
        return np.zeros(0, dtype=np.int32)
    b = bits(stream_key(seed, stream), np.arange(n, dtype=np.uint64))
    return np.argsort(b, kind="stable").astype(np.int32)


def to_f32(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32)


def to_f16_bits(x: np.ndarray) -> np.ndarray:
    """Round to IEEE binary16 (round-to-nearest-even) and return the bit patterns."""
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float16)).view(np.uint16)


def f16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return np.asarray(b, dtype=np.uint16).view(np.float16).astype(np.float64)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round f64 -> f32 -> bfloat16 (round-to-nearest-even); returns uint16 patterns."""
    f = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = ((f >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((f + rounding) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def int8_rows(x: np.ndarray):
    """Input format of the int8 prompt-attention cache.

    Per row of the last axis: scale = fp16(absmax / 127) (round-to-nearest-even),
    value = clamp(rint(x / scale), -127, 127) with ties to even; a zero row has
    scale 0 and values 0.  Returns (int8 values, uint16 fp16 scale bits).
    """
    x = np.asarray(x, dtype=np.float64)
    amax = np.abs(x).max(axis=-1)
    scale_bits = to_f16_bits(amax / 127.0)
    scale = f16_bits_to_f64(scale_bits)
    safe = np.where(scale > 0, scale, 1.0)
    q = np.clip(np.rint(x / safe[..., None]), -127, 127)
    q = np.where(scale[..., None] > 0, q, 0.0)
    return q.astype(np.int8), scale_bits


# --------------------------------------------------------------------------
# workload descriptions
# --------------------------------------------------------------------------

@dataclass
class AttnShape:
    name: str
    n_kv_heads: int
    n_q_heads: int
    head_dim_k: int
    head_dim_v: int
    kv_len: int
    nq: int = 1
    types: tuple = (3,)
    causal: bool = False
    seed: int = 0
    extra: dict = field(default_factory=dict)


def tiny_decode() -> AttnShape:
    return AttnShape("tiny_decode", 1, 1, 128, 128, 512, 1, (3,), False, 20260)


def decode_32k(kv_len: int = 32768) -> AttnShape:
    return AttnShape("decode_32k", 8, 32, 128, 128, kv_len, 1, (3, 2, 4), False, 20261)


def prefill_4k(nq: int = 4096) -> AttnShape:
    return AttnShape("prefill_4k", 8, 16, 256, 256, 4096, nq, (3,), True, 20262)


def asym_8k(nq: int = 1) -> AttnShape:
    return AttnShape("asym_8k", 16, 16, 192, 128, 8192, nq, (3,), nq > 1, 20263)


def int8_prompt(ctx: int = 40000) -> AttnShape:
    return AttnShape("int8_prompt", 8, 32, 128, 128, ctx, 2048, (), True, 20264)


def kv_inputs(shape: AttnShape, n_rows: int | None = None):
    """Raw K and V rows (f64 [n_rows][n_kv_heads][D]) with outlier channels."""
    n = shape.kv_len if n_rows is None else n_rows
    k = gaussian_with_outliers(shape.seed, S_K, S_K_OUT, n, shape.n_kv_heads, shape.head_dim_k)
    v = gaussian_with_outliers(shape.seed, S_V, S_V_OUT, n, shape.n_kv_heads, shape.head_dim_v)
    return k, v


def decode_query(shape: AttnShape) -> np.ndarray:
    """f64 [n_q_heads][Dk] query with outlier channels (its own channels)."""
    return gaussian_with_outliers(shape.seed, S_Q, S_Q_OUT, 1, shape.n_q_heads, shape.head_dim_k)[0]


def prompt_queries(shape: AttnShape) -> np.ndarray:
    """f64 [nq][n_q_heads][Dk] ~ N(0,1), no outliers."""
    return normal(shape.seed, S_Q, shape.nq * shape.n_q_heads * shape.head_dim_k).reshape(
        shape.nq, shape.n_q_heads, shape.head_dim_k)


def codebook_signs(shape: AttnShape):
    return sign_bits(shape.seed, S_SIGNS_K), sign_bits(shape.seed, S_SIGNS_V)

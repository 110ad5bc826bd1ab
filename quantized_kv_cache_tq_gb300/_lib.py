"""ctypes binding of libtq.so: the C ABI of include/tq.h under the same names.

Argument marshalling only; every step of the path runs in the library's CUDA
kernels.  There is no fallback: if libtq.so is missing or fails to load, the
import raises.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libtq.so")

TQ_OK = 0
TQ_ERR_INVALID_ARG = 1
TQ_ERR_UNSUPPORTED = 2
TQ_ERR_WORKSPACE = 3
TQ_ERR_CUDA = 4
TQ_ERR_TIMEOUT = 5
TQ_ERR_DEVICE_CHECK = 6

TQ_TURBO2, TQ_TURBO3, TQ_TURBO4 = 2, 3, 4
TQ_F32, TQ_F16, TQ_BF16 = 0, 1, 2
TQ_DECODE_AUTO, TQ_DECODE_LUT, TQ_DECODE_MMA = 0, 1, 2


class tq_codebook(C.Structure):
    _fields_ = [("sign_bits", C.c_uint32 * 4), ("n_centroids", C.c_int32),
                ("centroids", C.c_float * 16)]


class tq_cache(C.Structure):
    _fields_ = [("type", C.c_int32), ("n_kv_heads", C.c_int32), ("head_dim", C.c_int32),
                ("n_blocks", C.c_int32), ("n_cells", C.c_int64), ("norms", C.c_void_p),
                ("qs", C.c_void_p), ("signs", C.c_void_p)]


class TQError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


def _load() -> C.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                          "(the CUDA library has no fallback)")
    return C.CDLL(LIB_PATH)


lib = _load()

_P = C.c_void_p
_SIGS = {
    "tq_status_string": (C.c_char_p, [C.c_int]),
    "tq_version": (C.c_int, []),
    "tq_codebook_init": (C.c_int, [C.c_int, C.POINTER(C.c_uint32), C.POINTER(tq_codebook)]),
    "tq_cache_plane_bytes": (C.c_int, [C.c_int, C.c_int, C.c_int, C.c_int64, C.POINTER(C.c_size_t),
                                       C.POINTER(C.c_size_t), C.POINTER(C.c_size_t)]),
    "tq_set_rows": (C.c_int, [C.POINTER(tq_cache), C.POINTER(tq_codebook), _P, C.c_int, _P,
                              C.c_int64, _P, _P]),
    "tq_fattn_decode_workspace": (C.c_size_t, [C.POINTER(tq_cache), C.POINTER(tq_cache), C.c_int,
                                               C.c_int64]),
    "tq_fattn_decode": (C.c_int, [C.POINTER(tq_cache), C.POINTER(tq_cache), C.POINTER(tq_codebook),
                                  C.POINTER(tq_codebook), _P, C.c_int, C.c_int64, C.c_float, C.c_int,
                                  _P, _P, C.c_size_t, _P]),
    "tq_fattn_decode_sparse_v": (C.c_int, [C.POINTER(tq_cache), C.POINTER(tq_cache), C.POINTER(tq_codebook),
                                           C.POINTER(tq_codebook), _P, C.c_int, C.c_int64, C.c_float, C.c_float,
                                           C.c_int, _P, _P, C.c_size_t, _P]),
    "tq_fattn_decode_append": (C.c_int, [C.POINTER(tq_cache), C.POINTER(tq_cache), C.POINTER(tq_codebook),
                                         C.POINTER(tq_codebook), _P, _P, C.c_int, _P, _P, C.c_int, C.c_int64,
                                         C.c_float, C.c_int, _P, _P, C.c_size_t, _P]),
    "tq_fattn_decode_noalloc": (C.c_int, [C.POINTER(tq_cache), C.POINTER(tq_cache), C.POINTER(tq_codebook),
                                          C.POINTER(tq_codebook), _P, C.c_int, C.c_int64, C.c_float, C.c_int,
                                          _P, _P]),
    "tq_fattn_prefill_workspace": (C.c_size_t, [C.POINTER(tq_cache), C.POINTER(tq_cache), C.c_int,
                                                C.c_int, C.c_int64]),
    "tq_fattn_prefill": (C.c_int, [C.POINTER(tq_cache), C.POINTER(tq_cache), C.POINTER(tq_codebook),
                                   C.POINTER(tq_codebook), _P, C.c_int, C.c_int, C.c_int, C.c_int64,
                                   C.c_float, C.c_int, _P, _P, C.c_size_t, _P]),
    "tq_int8_prompt_attn_workspace": (C.c_size_t, [C.c_int, C.c_int, C.c_int, C.c_int, C.c_int64]),
    "tq_int8_prompt_attn": (C.c_int, [_P, _P, _P, _P, C.c_int64, _P, C.c_int64, _P, C.c_int, C.c_int,
                                      C.c_int, C.c_int, C.c_float, C.c_int, _P, _P, C.c_size_t, _P]),
    "tq_f16_prompt_attn": (C.c_int, [_P, _P, C.c_int64, _P, C.c_int64, _P, C.c_int, C.c_int, C.c_int, C.c_int,
                                     C.c_float, C.c_int, _P, _P, C.c_size_t, _P]),
    "tq_workspace_status": (C.c_int, [_P, C.c_size_t, C.POINTER(C.c_int32), _P]),
    "tq_noalloc_status": (C.c_int, [C.POINTER(C.c_int32), _P]),
    "tq_checksum_fnv1a64": (C.c_int, [_P, C.c_size_t, C.POINTER(C.c_uint64)]),
    "tq_fattn_decode_batch_workspace": (C.c_size_t, [C.POINTER(tq_cache), C.POINTER(tq_cache), C.c_int, C.c_int,
                                                     C.c_int64]),
    "tq_fattn_decode_batch": (C.c_int, [C.POINTER(tq_cache), C.POINTER(tq_cache), C.POINTER(tq_codebook),
                                        C.POINTER(tq_codebook), _P, C.c_int, C.c_int, C.POINTER(C.c_int64),
                                        C.POINTER(C.c_int64), C.c_float, C.c_int, _P, _P, C.c_size_t, _P]),
    # test hook (include/tq_testing.h)
    "tq_testing_decode_drop_split": (C.c_int, [C.POINTER(tq_cache), C.POINTER(tq_cache), C.POINTER(tq_codebook),
                                               C.POINTER(tq_codebook), _P, C.c_int, C.c_int64, C.c_float, C.c_int,
                                               _P, _P, C.c_size_t, C.c_int, _P]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_SIGS)


def status_string(status: int) -> str:
    return lib.tq_status_string(status).decode()


def check(fn: str, status: int) -> None:
    if status != TQ_OK:
        raise TQError(fn, status)


def tq_status_string(status: int) -> str:
    return status_string(status)


def tq_version() -> int:
    return lib.tq_version()


def tq_codebook_init(tq_type: int, sign_bits) -> tq_codebook:
    cb = tq_codebook()
    sb = (C.c_uint32 * 4)(*[int(x) for x in sign_bits])
    check("tq_codebook_init", lib.tq_codebook_init(tq_type, sb, C.byref(cb)))
    return cb


def tq_cache_plane_bytes(tq_type: int, n_kv_heads: int, head_dim: int, n_cells: int):
    a, b, c = C.c_size_t(), C.c_size_t(), C.c_size_t()
    check("tq_cache_plane_bytes", lib.tq_cache_plane_bytes(tq_type, n_kv_heads, head_dim, n_cells,
                                                           C.byref(a), C.byref(b), C.byref(c)))
    return a.value, b.value, c.value


def tq_set_rows(dst: tq_cache, cb: tq_codebook, src: int, src_type: int, cell_ids: int,
                n_rows: int, dev_status: int | None, stream: int | None) -> int:
    return lib.tq_set_rows(C.byref(dst), C.byref(cb), src, src_type, cell_ids, n_rows, dev_status,
                           stream)


def tq_fattn_decode_workspace(k: tq_cache, v: tq_cache, n_q_heads: int, kv_len: int) -> int:
    return lib.tq_fattn_decode_workspace(C.byref(k), C.byref(v), n_q_heads, kv_len)


def tq_fattn_decode(k: tq_cache, v: tq_cache, cbk: tq_codebook, cbv: tq_codebook, q: int,
                    n_q_heads: int, kv_len: int, scale: float, algo: int, out: int, ws: int,
                    ws_bytes: int, stream: int | None) -> int:
    return lib.tq_fattn_decode(C.byref(k), C.byref(v), C.byref(cbk), C.byref(cbv), q, n_q_heads,
                               kv_len, scale, algo, out, ws, ws_bytes, stream)


def tq_fattn_decode_sparse_v(k: tq_cache, v: tq_cache, cbk: tq_codebook, cbv: tq_codebook, q: int,
                             n_q_heads: int, kv_len: int, scale: float, v_threshold: float, algo: int,
                             out: int, ws: int, ws_bytes: int, stream: int | None) -> int:
    return lib.tq_fattn_decode_sparse_v(C.byref(k), C.byref(v), C.byref(cbk), C.byref(cbv), q, n_q_heads,
                                        kv_len, scale, v_threshold, algo, out, ws, ws_bytes, stream)


def tq_fattn_decode_append(k: tq_cache, v: tq_cache, cbk: tq_codebook, cbv: tq_codebook, k_row: int,
                           v_row: int, src_type: int, cell_id: int, q: int, n_q_heads: int, kv_len: int,
                           scale: float, algo: int, out: int, ws: int, ws_bytes: int,
                           stream: int | None) -> int:
    return lib.tq_fattn_decode_append(C.byref(k), C.byref(v), C.byref(cbk), C.byref(cbv), k_row, v_row,
                                      src_type, cell_id, q, n_q_heads, kv_len, scale, algo, out, ws, ws_bytes,
                                      stream)


def tq_fattn_decode_noalloc(k: tq_cache, v: tq_cache, cbk: tq_codebook, cbv: tq_codebook, q: int,
                            n_q_heads: int, kv_len: int, scale: float, algo: int, out: int,
                            stream: int | None) -> int:
    return lib.tq_fattn_decode_noalloc(C.byref(k), C.byref(v), C.byref(cbk), C.byref(cbv), q, n_q_heads,
                                       kv_len, scale, algo, out, stream)


def tq_fattn_prefill_workspace(k: tq_cache, v: tq_cache, nq: int, n_q_heads: int, kv_len: int) -> int:
    return lib.tq_fattn_prefill_workspace(C.byref(k), C.byref(v), nq, n_q_heads, kv_len)


def tq_fattn_prefill(k: tq_cache, v: tq_cache, cbk: tq_codebook, cbv: tq_codebook, q: int,
                     q_type: int, nq: int, n_q_heads: int, kv_len: int, scale: float, causal: int,
                     out: int, ws: int, ws_bytes: int, stream: int | None) -> int:
    return lib.tq_fattn_prefill(C.byref(k), C.byref(v), C.byref(cbk), C.byref(cbv), q, q_type, nq,
                                n_q_heads, kv_len, scale, causal, out, ws, ws_bytes, stream)


def tq_int8_prompt_attn_workspace(nq: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                                  ctx: int) -> int:
    return lib.tq_int8_prompt_attn_workspace(nq, n_q_heads, n_kv_heads, head_dim, ctx)


def tq_int8_prompt_attn(k: int, k_scale: int, v: int, v_scale: int, n_cells: int, cell_of_pos: int,
                        ctx: int, q: int, nq: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                        scale: float, causal: int, out: int, ws: int, ws_bytes: int,
                        stream: int | None) -> int:
    return lib.tq_int8_prompt_attn(k, k_scale, v, v_scale, n_cells, cell_of_pos, ctx, q, nq,
                                   n_q_heads, n_kv_heads, head_dim, scale, causal, out, ws, ws_bytes,
                                   stream)


def tq_f16_prompt_attn(k: int, v: int, n_cells: int, cell_of_pos: int, ctx: int, q: int, nq: int,
                       n_q_heads: int, n_kv_heads: int, head_dim: int, scale: float, causal: int, out: int,
                       ws: int, ws_bytes: int, stream: int | None) -> int:
    return lib.tq_f16_prompt_attn(k, v, n_cells, cell_of_pos, ctx, q, nq, n_q_heads, n_kv_heads, head_dim,
                                  scale, causal, out, ws, ws_bytes, stream)


def tq_workspace_status(ws: int, ws_bytes: int, stream: int | None) -> int:
    st = C.c_int32()
    check("tq_workspace_status", lib.tq_workspace_status(ws, ws_bytes, C.byref(st), stream))
    return st.value


def tq_noalloc_status(stream: int | None) -> int:
    st = C.c_int32()
    check("tq_noalloc_status", lib.tq_noalloc_status(C.byref(st), stream))
    return st.value


def tq_testing_decode_drop_split(k: tq_cache, v: tq_cache, cbk: tq_codebook, cbv: tq_codebook, q: int,
                                 n_q_heads: int, kv_len: int, scale: float, algo: int, out: int, ws: int,
                                 ws_bytes: int, drop_split: int, stream: int | None) -> int:
    return lib.tq_testing_decode_drop_split(C.byref(k), C.byref(v), C.byref(cbk), C.byref(cbv), q, n_q_heads,
                                            kv_len, scale, algo, out, ws, ws_bytes, drop_split, stream)


def tq_checksum_fnv1a64(host_ptr: int, n_bytes: int) -> int:
    h = C.c_uint64()
    check("tq_checksum_fnv1a64", lib.tq_checksum_fnv1a64(host_ptr, n_bytes, C.byref(h)))
    return h.value


def tq_fattn_decode_batch_workspace(k: tq_cache, v: tq_cache, n_q_heads: int, n_seq: int, max_len: int) -> int:
    return lib.tq_fattn_decode_batch_workspace(C.byref(k), C.byref(v), n_q_heads, n_seq, max_len)


def tq_fattn_decode_batch(k: tq_cache, v: tq_cache, cbk: tq_codebook, cbv: tq_codebook, q: int, n_q_heads: int,
                          seq_cell0, seq_len, scale: float, algo: int, out: int, ws: int, ws_bytes: int,
                          stream: int | None) -> int:
    n = len(seq_cell0)
    c0 = (C.c_int64 * n)(*[int(x) for x in seq_cell0])
    ln = (C.c_int64 * n)(*[int(x) for x in seq_len])
    return lib.tq_fattn_decode_batch(C.byref(k), C.byref(v), C.byref(cbk), C.byref(cbv), q, n_q_heads, n, c0, ln,
                                     scale, algo, out, ws, ws_bytes, stream)

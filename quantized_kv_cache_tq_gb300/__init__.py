"""Attention over a TurboQuant-compressed KV cache on GB300 (sm_103a).

The compute lives in libtq.so (C ABI, include/tq.h); ``_lib`` binds it with
ctypes under the same names.  The helpers below only hold PyTorch tensors for
device memory and pass their pointers and the current CUDA stream through.
"""
from __future__ import annotations

import math

from . import _lib
from ._lib import (TQ_BF16, TQ_DECODE_AUTO, TQ_DECODE_LUT, TQ_DECODE_MMA, TQ_F16, TQ_F32,
                   TQ_TURBO2, TQ_TURBO3, TQ_TURBO4, TQError, tq_cache, tq_codebook)

QS_BYTES = {2: 32, 3: 32, 4: 64}


def _torch():
    import torch
    return torch


def _stream(stream=None):
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


class TqCache:
    """Device planes of one compressed cache (K or V), allocated with PyTorch."""

    def __init__(self, tq_type: int, n_kv_heads: int, head_dim: int, n_cells: int, device="cuda"):
        torch = _torch()
        nb = (head_dim + 127) // 128
        self.tq_type, self.n_kv_heads, self.head_dim, self.n_cells, self.n_blocks = (
            tq_type, n_kv_heads, head_dim, n_cells, nb)
        self.norms = torch.zeros((n_kv_heads, n_cells, nb), dtype=torch.int16, device=device)
        self.qs = torch.zeros((n_kv_heads, n_cells, nb, QS_BYTES[tq_type]), dtype=torch.uint8, device=device)
        self.signs = (torch.zeros((n_kv_heads, n_cells, nb, 16), dtype=torch.uint8, device=device)
                      if tq_type == 3 else None)
        self.c = tq_cache(tq_type, n_kv_heads, head_dim, nb, n_cells, self.norms.data_ptr(),
                          self.qs.data_ptr(), 0 if self.signs is None else self.signs.data_ptr())

    def planes(self):
        return self.norms, self.qs, self.signs


def codebook(tq_type: int, sign_bits) -> tq_codebook:
    return _lib.tq_codebook_init(tq_type, sign_bits)


def workspace(nbytes: int, device="cuda"):
    """Zero-filled, 256-byte aligned workspace (PyTorch allocations are)."""
    torch = _torch()
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def set_rows(cache: TqCache, cb: tq_codebook, src, cell_ids, dev_status=None, stream=None):
    torch = _torch()
    src_type = {torch.float32: TQ_F32, torch.float16: TQ_F16, torch.bfloat16: TQ_BF16}[src.dtype]
    assert src.is_contiguous() and cell_ids.dtype == torch.int64 and cell_ids.is_contiguous()
    st = _lib.tq_set_rows(cache.c, cb, src.data_ptr(), src_type, cell_ids.data_ptr(),
                          cell_ids.numel(), None if dev_status is None else dev_status.data_ptr(),
                          _stream(stream))
    _lib.check("tq_set_rows", st)


def fattn_decode(kc: TqCache, vc: TqCache, cbk, cbv, q, kv_len: int, scale: float | None = None,
                 algo: int = TQ_DECODE_AUTO, out=None, ws=None, stream=None, sparse_v: float = 0.0):
    """Decode over cells 0..kv_len-1; ``sparse_v`` > 0 leaves out of the V sum the
    keys whose weights relative to the running maximum are below it."""
    torch = _torch()
    n_q = q.shape[0]
    scale = 1.0 / math.sqrt(kc.head_dim) if scale is None else scale
    if out is None:
        out = torch.empty((n_q, vc.head_dim), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(_lib.tq_fattn_decode_workspace(kc.c, vc.c, n_q, kv_len), q.device)
    if sparse_v:
        st = _lib.tq_fattn_decode_sparse_v(kc.c, vc.c, cbk, cbv, q.data_ptr(), n_q, kv_len, scale, sparse_v,
                                           algo, out.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream))
        _lib.check("tq_fattn_decode_sparse_v", st)
    else:
        st = _lib.tq_fattn_decode(kc.c, vc.c, cbk, cbv, q.data_ptr(), n_q, kv_len, scale, algo,
                                  out.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream))
        _lib.check("tq_fattn_decode", st)
    return out


def fattn_decode_append(kc: TqCache, vc: TqCache, cbk, cbv, k_row, v_row, cell_id, q, kv_len: int,
                        scale: float | None = None, algo: int = TQ_DECODE_AUTO, out=None, ws=None, stream=None):
    """SET_ROWS of one token's K/V rows ([n_kv_heads][head_dim]) into cell ``cell_id``
    (a device int64 tensor of one element), then decode over cells 0..kv_len-1."""
    torch = _torch()
    n_q = q.shape[0]
    src_type = {torch.float32: TQ_F32, torch.float16: TQ_F16, torch.bfloat16: TQ_BF16}[k_row.dtype]
    assert v_row.dtype == k_row.dtype and k_row.is_contiguous() and v_row.is_contiguous()
    assert cell_id.dtype == torch.int64 and cell_id.numel() == 1
    scale = 1.0 / math.sqrt(kc.head_dim) if scale is None else scale
    if out is None:
        out = torch.empty((n_q, vc.head_dim), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(_lib.tq_fattn_decode_workspace(kc.c, vc.c, n_q, kv_len), q.device)
    st = _lib.tq_fattn_decode_append(kc.c, vc.c, cbk, cbv, k_row.data_ptr(), v_row.data_ptr(), src_type,
                                     cell_id.data_ptr(), q.data_ptr(), n_q, kv_len, scale, algo,
                                     out.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream))
    _lib.check("tq_fattn_decode_append", st)
    return out


def fattn_decode_batch(kc: TqCache, vc: TqCache, cbk, cbv, q, seq_cell0, seq_len, scale: float | None = None,
                       algo: int = TQ_DECODE_AUTO, out=None, ws=None, stream=None):
    """Decode of several sequences in one launch: q [n_seq][n_q_heads][Dk];
    sequence s attends cells seq_cell0[s] .. + seq_len[s] - 1 (host integers)."""
    torch = _torch()
    n_seq, n_q, _ = q.shape
    scale = 1.0 / math.sqrt(kc.head_dim) if scale is None else scale
    if out is None:
        out = torch.empty((n_seq, n_q, vc.head_dim), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(_lib.tq_fattn_decode_batch_workspace(kc.c, vc.c, n_q, n_seq, max(seq_len)), q.device)
    st = _lib.tq_fattn_decode_batch(kc.c, vc.c, cbk, cbv, q.data_ptr(), n_q, list(seq_cell0), list(seq_len), scale,
                                    algo, out.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream))
    _lib.check("tq_fattn_decode_batch", st)
    return out


def fattn_prefill(kc: TqCache, vc: TqCache, cbk, cbv, q, kv_len: int, scale: float | None = None,
                  causal: bool = True, out=None, ws=None, stream=None):
    torch = _torch()
    nq, n_q, _ = q.shape
    q_type = {torch.float32: TQ_F32, torch.float16: TQ_F16, torch.bfloat16: TQ_BF16}[q.dtype]
    scale = 1.0 / math.sqrt(kc.head_dim) if scale is None else scale
    if out is None:
        out = torch.empty((nq, n_q, vc.head_dim), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(_lib.tq_fattn_prefill_workspace(kc.c, vc.c, nq, n_q, kv_len), q.device)
    st = _lib.tq_fattn_prefill(kc.c, vc.c, cbk, cbv, q.data_ptr(), q_type, nq, n_q, kv_len, scale,
                               int(causal), out.data_ptr(), ws.data_ptr(), ws.numel(), _stream(stream))
    _lib.check("tq_fattn_prefill", st)
    return out


def int8_prompt_attn(k, k_scale, v, v_scale, cell_of_pos, ctx: int, q, scale: float | None = None,
                     causal: bool = True, out=None, ws=None, stream=None):
    torch = _torch()
    n_cells, n_kv, d = k.shape
    nq, n_q, _ = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if out is None:
        out = torch.empty((nq, n_q, d), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(_lib.tq_int8_prompt_attn_workspace(nq, n_q, n_kv, d, ctx), q.device)
    st = _lib.tq_int8_prompt_attn(k.data_ptr(), k_scale.data_ptr(), v.data_ptr(), v_scale.data_ptr(),
                                  n_cells, cell_of_pos.data_ptr(), ctx, q.data_ptr(), nq, n_q, n_kv, d,
                                  scale, int(causal), out.data_ptr(), ws.data_ptr(), ws.numel(),
                                  _stream(stream))
    _lib.check("tq_int8_prompt_attn", st)
    return out


def f16_prompt_attn(k, v, cell_of_pos, ctx: int, q, scale: float | None = None, causal: bool = True, out=None,
                    ws=None, stream=None):
    """Prompt attention over binary16 K/V rows [n_cells][n_kv_heads][128] gathered
    through cell_of_pos (the int8 path's other cache mode, no scales)."""
    torch = _torch()
    assert k.dtype == torch.float16 and v.dtype == torch.float16
    n_cells, n_kv, d = k.shape
    nq, n_q, _ = q.shape
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    if out is None:
        out = torch.empty((nq, n_q, d), dtype=torch.float32, device=q.device)
    if ws is None:
        ws = workspace(_lib.tq_int8_prompt_attn_workspace(nq, n_q, n_kv, d, ctx), q.device)
    st = _lib.tq_f16_prompt_attn(k.data_ptr(), v.data_ptr(), n_cells, cell_of_pos.data_ptr(), ctx, q.data_ptr(),
                                 nq, n_q, n_kv, d, scale, int(causal), out.data_ptr(), ws.data_ptr(), ws.numel(),
                                 _stream(stream))
    _lib.check("tq_f16_prompt_attn", st)
    return out


def checksum(t) -> str:
    """FNV-1a 64 of a tensor's bytes (copied to the host), as 16 hex digits."""
    import numpy as np
    a = np.ascontiguousarray(t.detach().cpu().numpy())
    return f"{_lib.tq_checksum_fnv1a64(a.ctypes.data, a.nbytes):016x}"

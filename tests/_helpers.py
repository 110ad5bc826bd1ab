"""Shared test plumbing: oracle caches uploaded to the GPU, comparisons."""
from __future__ import annotations

import math

import numpy as np

import oracle as O
import workloads as W

MAX_ABS = 2e-3          # attention output tolerance (absolute)
MAX_NMSE = 1e-6         # attention output tolerance (normalised MSE, vs the oracle)
BAND = 1e-6             # codes may differ only this close to a decision boundary
MAX_FLIP_FRAC = 1e-5    # ... and on at most this fraction of elements


def oracle_cache(tq_type, raw, sign_bits, n_cells=None):
    """Oracle-quantised cache of raw rows [L][H][D] into cells 0..L-1."""
    L, H, D = raw.shape
    n_cells = n_cells or max(64, (L + 63) // 64 * 64)
    c = O.empty_cache(tq_type, H, D, n_cells)
    O.set_rows(c, W.to_f32(raw), np.arange(L), sign_bits, O.centroids(tq_type))
    return c


def upload(oc: O.Cache):
    """Copy an oracle cache's planes into a GPU TqCache."""
    import torch
    import quantized_kv_cache_tq_gb300 as tq
    g = tq.TqCache(oc.tq_type, oc.n_kv_heads, oc.head_dim, oc.n_cells)
    g.norms.copy_(torch.from_numpy(oc.norms.view(np.int16)))
    g.qs.copy_(torch.from_numpy(oc.qs))
    if oc.signs is not None:
        g.signs.copy_(torch.from_numpy(oc.signs))
    return g


def download(g) -> O.Cache:
    return O.Cache(g.tq_type, g.n_kv_heads, g.head_dim, g.n_cells,
                   g.norms.cpu().numpy().view(np.uint16), g.qs.cpu().numpy(),
                   None if g.signs is None else g.signs.cpu().numpy())


def compare_outputs(gpu, ref, max_abs=MAX_ABS, max_nmse=MAX_NMSE):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape
    assert np.all(np.isfinite(gpu)), "non-finite output"
    err = float(np.max(np.abs(gpu - ref))) if gpu.size else 0.0
    nm = O.nmse(gpu, ref)
    assert err <= max_abs, f"max-abs {err:.3e} > {max_abs}"
    assert nm <= max_nmse, f"nmse {nm:.3e} > {max_nmse}"
    return err, nm


def compare_caches(gpu: O.Cache, ref: O.Cache, y: np.ndarray, cells: np.ndarray):
    """Codes bit-exact except within BAND of a decision boundary (counted);
    norms within one binary16 ulp.  y = oracle's rotated values [n][H][nb][128]."""
    cents = O.centroids(ref.tq_type)
    mids = 0.5 * (cents[:-1] + cents[1:])
    g_codes = O.unpack_codes(gpu.qs[:, cells], None if gpu.signs is None else gpu.signs[:, cells], gpu.tq_type)
    r_codes = O.unpack_codes(ref.qs[:, cells], None if ref.signs is None else ref.signs[:, cells], ref.tq_type)
    yy = y.transpose(1, 0, 2, 3)                                    # [H][n][nb][128]
    near = np.min(np.abs(yy[..., None] - mids), axis=-1) < BAND
    diff = g_codes != r_codes
    assert not np.any(diff & ~near), f"{int(np.sum(diff & ~near))} codes differ away from a boundary"
    flips = int(np.sum(diff))
    assert flips <= MAX_FLIP_FRAC * diff.size, f"{flips} boundary flips of {diff.size}"
    gn = gpu.norms[:, cells].astype(np.int64)
    rn = ref.norms[:, cells].astype(np.int64)
    assert np.max(np.abs(gn - rn)) <= 1, "norm differs by more than one binary16 ulp"
    return flips, int(np.sum(gn != rn))


def scale_of(d):
    return 1.0 / math.sqrt(d)

"""Mutation check of the oracle's pins (run by hand: ``python tests/oracle_mutants.py``).

Each entry below is a plausible mistake in ``oracle/__init__.py`` (a dropped term, a
wrong sign, bit position, index or offset, a transposed operand, an ignored argument).
For each one a copy of the oracle with that single change is checked against
``tests/test_oracle_pins.py``; the script lists every mistake the pins fail to
catch and exits non-zero if there is one.  It takes a few minutes (one pytest run
per mistake), so it is not part of the test suite.
"""
import os
import shutil
import subprocess
import sys
import tempfile

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = open(os.path.join(ROOT, "oracle", "__init__.py")).read()
M = [
 ("hadamard sign", "return np.where(parity == 0, 1.0, -1.0)", "return np.where(parity == 0, -1.0, 1.0)"),
 ("sign bit order", "if (int(sign_bits[i // 32]) >> (i % 32)) & 1:", "if (int(sign_bits[i // 32]) >> (31 - i % 32)) & 1:"),
 ("sign word index", "if (int(sign_bits[i // 32]) >> (i % 32)) & 1:", "if (int(sign_bits[i % 4]) >> (i // 4)) & 1:"),
 ("S before H", "return hadamard() * sign_vector(sign_bits)[None, :] / math.sqrt(QK)", "return hadamard() * sign_vector(sign_bits)[:, None] / math.sqrt(QK)"),
 ("rotation scale", "return hadamard() * sign_vector(sign_bits)[None, :] / math.sqrt(QK)", "return hadamard() * sign_vector(sign_bits)[None, :] / QK"),
 ("butterfly sign", "x = np.where((j & h) != 0, o - x, x + o)", "x = np.where((j & h) != 0, x - o, x + o)"),
 ("lloyd midpoint", "        t = np.concatenate(([-np.inf], 0.5 * (c[:-1] + c[1:]), [np.inf]))\n        a, b = t[:-1], t[1:]\n        new", "        t = np.concatenate(([-np.inf], 0.4 * (c[:-1] + c[1:]), [np.inf]))\n        a, b = t[:-1], t[1:]\n        new"),
 ("distortion cross term", "return float(np.sum(ex2 - 2 * c * ex + c * c * p))", "return float(np.sum(ex2 - c * ex + c * c * p))"),
 ("centroid scale", "c = lloyd_max_normal(N_CENTROIDS[tq_type]) / math.sqrt(QK)", "c = lloyd_max_normal(N_CENTROIDS[tq_type]) / QK"),
 ("centroid fp16 rounding", "return c.astype(np.float16).astype(np.float64)", "return c"),
 ("index_to_code", "return np.where(i >= half, i, half - 1 - i)", "return np.where(i >= half, i, half - i)"),
 ("code_to_value sign", "return np.where(s == 1, mag, -mag)", "return np.where(s == 1, -mag, mag)"),
 ("qs field hi half", "bit = 4 * r if r < 8 else 4 * (r - 8) + 2", "bit = 4 * r if r < 8 else 4 * (r - 8) + 1"),
 ("qs field turbo4 order", "        bit = 4 * i\n", "        bit = 4 * (7 - i)\n"),
 ("sign bit low half", "bit = 4 * (r % 8) + 2 + r // 8", "bit = 4 * (r % 8) + 3 - r // 8"),
 ("sign bit high half", "bit = 4 * (rr % 8) + rr // 8", "bit = 4 * (rr % 8) + 1 - rr // 8"),
 ("turbo3 qs field mask", "field_val = (k & 3) if tq_type == 3 else k", "field_val = (k & 1) if tq_type == 3 else k"),
 ("norm precision", "norm_bits = nrm.astype(np.float16).view(np.uint16)", "norm_bits = (nrm * 1.001).astype(np.float16).view(np.uint16)"),
 ("quantise R^T", "y = u @ rotation(sign_bits).T", "y = u @ rotation(sign_bits)"),
 ("tie to lower", "return len(cents) - 1 - np.argmin(dist[..., ::-1], axis=-1)", "return np.argmin(dist, axis=-1)"),
 ("dequantise R", "return n[..., None] * (vals @ rotation(sign_bits))", "return n[..., None] * (vals @ rotation(sign_bits).T)"),
 ("causal >=", "mask = np.arange(k.shape[0])[None, :] > np.asarray(q_pos)[:, None]", "mask = np.arange(k.shape[0])[None, :] >= np.asarray(q_pos)[:, None]"),
 ("no scale", "    s = scale * (q @ k.T)\n    if q_pos", "    s = (q @ k.T)\n    if q_pos"),
 ("sparse normaliser", "return (p_kept @ v) / total, (p @ v) / total, (p_out @ np.abs(v)) / total", "return (p_kept @ v) / np.sum(p_kept, axis=1, keepdims=True), (p @ v) / total, (p_out @ np.abs(v)) / total"),
 ("sparse bound abs", "(p_out @ np.abs(v)) / total", "(p_out @ v) / total"),
 ("sparse threshold slack", "out = p < threshold * slack", "out = p < threshold"),
 ("lse merge sign", "w = np.stack([p[1] * np.exp(p[0] - M) for p in parts])", "w = np.stack([p[1] * np.exp(M - p[0]) for p in parts])"),
 ("lse partial l", "    l = np.sum(e, axis=-1)\n    return m, l,", "    l = np.sum(e, axis=-1) + 1e-3\n    return m, l,"),
 ("decode gqa", "        for h in range(hk * g, (hk + 1) * g):\n            out[h] = softmax_attention", "        for h in range(hk, n_q, kc.n_kv_heads):\n            out[h] = softmax_attention"),
 ("prefill causal offset", "pos = (kv_len - nq + rows) if causal else None", "pos = (kv_len - nq + rows - 1) if causal else None"),
 ("prefill gqa", "            out[rows, h] = softmax_attention(q[rows, h], k, v, scale, pos)\n    return out\n\n\ndef int8_dequantize", "            out[rows, h] = softmax_attention(q[rows, (h % g) * kc.n_kv_heads + h // g], k, v, scale, pos)\n    return out\n\n\ndef int8_dequantize"),
 ("int8 dequant", "return np.asarray(rows_i8, np.float64) * s[..., None]", "return np.asarray(rows_i8, np.float64) / s[..., None]"),
 ("int8 causal", "    pos = (ctx - nq + rows) if causal else None\n    cells = np.asarray(cell_of_pos[:ctx], dtype=np.int64)\n    out = np.zeros((nq, n_q, v_i8", "    pos = (ctx - nq + rows + 1) if causal else None\n    cells = np.asarray(cell_of_pos[:ctx], dtype=np.int64)\n    out = np.zeros((nq, n_q, v_i8"),
 ("int8 ignores permutation", "    cells = np.asarray(cell_of_pos[:ctx], dtype=np.int64)\n    out = np.zeros((nq, n_q, v_i8", "    cells = np.arange(ctx)\n    out = np.zeros((nq, n_q, v_i8"),
 ("int8 v scale from k", "        v = int8_dequantize(v_i8[cells, hk], v_scale[cells, hk])", "        v = int8_dequantize(v_i8[cells, hk], k_scale[cells, hk])"),
 ("f16 ignores permutation", "    cells = np.asarray(cell_of_pos[:ctx], dtype=np.int64)\n    out = np.zeros((nq, n_q, vv", "    cells = np.arange(ctx)\n    out = np.zeros((nq, n_q, vv"),
 ("f16 causal", "    pos = (ctx - nq + rows) if causal else None\n    cells = np.asarray(cell_of_pos[:ctx], dtype=np.int64)\n    out = np.zeros((nq, n_q, vv", "    pos = (ctx - nq + rows - 1) if causal else None\n    cells = np.asarray(cell_of_pos[:ctx], dtype=np.int64)\n    out = np.zeros((nq, n_q, vv"),
 ("nmse denominator", "den = float(np.sum(b * b))", "den = float(np.sum(a * a))"),
 ("bits per element", "b = QS_BYTES[tq_type] + (SIGN_BYTES if tq_type == 3 else 0) + 2", "b = QS_BYTES[tq_type] + (SIGN_BYTES if tq_type == 3 else 0)"),
 ("pad with ones", "x = np.concatenate([x, np.zeros(x.shape[:-1] + (pad,))], axis=-1)", "x = np.concatenate([x, np.ones(x.shape[:-1] + (pad,))], axis=-1)"),
 ("set_rows cell ids ignored", "        cells = cell_ids[lo:lo + 2048]\n", "        cells = np.arange(lo, lo + len(cell_ids[lo:lo + 2048]))\n"),
 ("dequantize_cache truncation", "out.append(x.reshape(n, cache.n_blocks * QK)[:, :cache.head_dim])", "out.append(x.reshape(n, cache.n_blocks * QK)[:, -cache.head_dim:])"),
 ("decode kv_len", "        k = dequantize_cache(kc, k_signs, k_cents, kv_len, hk)\n        v = dequantize_cache(vc, v_signs, v_cents, kv_len, hk)\n        for h in range(hk * g, (hk + 1) * g):\n            out[h]", "        k = dequantize_cache(kc, k_signs, k_cents, kv_len - 1, hk)\n        v = dequantize_cache(vc, v_signs, v_cents, kv_len - 1, hk)\n        for h in range(hk * g, (hk + 1) * g):\n            out[h]"),
 ("prefill noncausal", "pos = (kv_len - nq + rows) if causal else None", "pos = (kv_len - nq + rows)"),
 ("f16 v from k", "vv = np.asarray(v_bits, dtype=np.uint16).view(np.float16).astype(np.float64)", "vv = np.asarray(k_bits, dtype=np.uint16).view(np.float16).astype(np.float64)"),
 ("int8 gqa", "        v = int8_dequantize(v_i8[cells, hk], v_scale[cells, hk])\n        for h in range(hk * g, (hk + 1) * g):", "        v = int8_dequantize(v_i8[cells, hk], v_scale[cells, hk])\n        for h in range(hk, n_q, hkv):"),
 ("f16 gqa", "        v = vv[cells, hk]\n        for h in range(hk * g, (hk + 1) * g):", "        v = vv[cells, hk]\n        for h in range(hk, n_q, hkv):"),
 ("sparse decode gqa", "        for h in range(hk * g, (hk + 1) * g):\n            for r, x in zip", "        for h in range(hk, n_q, kc.n_kv_heads):\n            for r, x in zip"),
 ("sparse decode slack dropped", "sparse_v_attention(q[h][None, :], k, v, scale, threshold, slack)", "sparse_v_attention(q[h][None, :], k, v, scale, threshold)"),
 ("pack turbo3 sign bit", "signs[..., sb] |= (((k >> 2) & 1) << ss).astype(np.uint8)", "signs[..., sb] |= (((k >> 1) & 1) << ss).astype(np.uint8)"),
 ("unpack turbo3 sign shift", "v = v | (((np.asarray(signs[..., sb], dtype=np.int64) >> ss) & 1) << 2)", "v = v | (((np.asarray(signs[..., sb], dtype=np.int64) >> ss) & 1) << 1)"),
 ("code_to_value magnitude", "    j = k % half\n", "    j = (k + 1) % half\n"),
 ("index_to_code boundary", "return np.where(i >= half, i, half - 1 - i)", "return np.where(i > half, i, half - 1 - i)"),
 ("norm of zero block", "u = np.where(nrm[..., None] > 0, x / safe[..., None], 0.0)", "u = np.where(nrm[..., None] > 0, x / safe[..., None], 1.0)"),
 ("dequant norm decode", "n = np.asarray(norm_bits, dtype=np.uint16).view(np.float16).astype(np.float64)", "n = np.asarray(norm_bits, dtype=np.uint16).view(np.float16).astype(np.float32).astype(np.float64) * (1 + 2**-12)"),
 ("lse partial max", "    m = np.max(s, axis=-1)\n    e = np.exp(s - m[..., None])", "    m = np.max(s, axis=-1) * 0.5\n    e = np.exp(s - m[..., None])"),
 ("softmax empty keys", "        return np.zeros((q.shape[0], v.shape[1]))\n    s = scale", "        return np.ones((q.shape[0], v.shape[1]))\n    s = scale"),
 ("sparse empty keys", "        z = np.zeros((q.shape[0], v.shape[1]))\n        return z, z.copy(), z.copy()", "        z = np.ones((q.shape[0], v.shape[1]))\n        return z, z.copy(), z.copy()"),
 ("set_rows batch src", "blocks = _pad_blocks(np.asarray(src[lo:lo + 2048], dtype=np.float64), cache.head_dim)", "blocks = _pad_blocks(np.asarray(src[lo:lo + 2048], dtype=np.float32).astype(np.float64), cache.head_dim)"),
 ("int8 rows restriction", "    pos = (ctx - nq + rows) if causal else None\n    cells = np.asarray(cell_of_pos[:ctx], dtype=np.int64)\n    out = np.zeros((nq, n_q, v_i8", "    pos = (ctx - nq + rows) if causal else None\n    rows = np.arange(nq)\n    pos = (ctx - nq + rows) if causal else None\n    cells = np.asarray(cell_of_pos[:ctx], dtype=np.int64)\n    out = np.zeros((nq, n_q, v_i8"),
 ("hadamard index", "a = i[:, None] & i[None, :]", "a = i[:, None] | i[None, :]"),
 ("distortion p term", "return float(np.sum(ex2 - 2 * c * ex + c * c * p))", "return float(np.sum(ex2 - 2 * c * ex + c * p))"),
]


def main(only):
    tmp = tempfile.mkdtemp()
    try:
        for d in ("tests", "oracle", "workloads"):
            shutil.copytree(os.path.join(ROOT, d), os.path.join(tmp, d), ignore=shutil.ignore_patterns("__pycache__"))
        missed = []
        for name, before, after in M:
            if only and name not in only:
                continue
            if SRC.count(before) != 1:                  # the list no longer matches the oracle
                print("STALE   ", name, flush=True)
                missed.append(name)
                continue
            with open(os.path.join(tmp, "oracle", "__init__.py"), "w") as f:
                f.write(SRC.replace(before, after))
            r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_oracle_pins.py", "-x", "-q",
                                "-p", "no:cacheprovider"], cwd=tmp, capture_output=True, text=True, timeout=600)
            caught = r.returncode != 0
            last = (r.stdout.strip().splitlines() or [""])[-1]
            print("caught  " if caught else "MISSED  ", name, "|", last[:90], flush=True)
            if not caught:
                missed.append(name)
        print(f"{len(missed)} of {len(M) if not only else len(only)} mistakes not caught:", missed)
        return 1 if missed else 0
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


if __name__ == "__main__":
    sys.exit(main(sys.argv[1:]))

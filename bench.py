#!/usr/bin/env python
"""Benchmark of the compressed-KV-cache attention hot path on GB300.

Workload (decode at 32K context): 8 KV heads x 32 query heads (GQA 4), head_dim
128, 32768 cells, turbo3 K and V.  One step = T new tokens (default 64) through
B independent layers (B caches sized so the working set exceeds 4x L2); each
token-layer quantises the token's K and V rows into its cache (SET_ROWS) and
runs the single-query decode attention over the 32768 cells, both in one
tq_fattn_decode_append launch.  The metric is
decode-attention tokens per second for one layer (token-layer calls / s).

Prints one JSON line.  --impl reference times the CPU oracle instead.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode attn tokens/s at 32K ctx (one layer, batch 1, turbo3 K/V, incl. SET_ROWS of the new token)"
UNIT = "tokens/s"
KV_LEN = 32768
N_KV, N_Q, D = 8, 32, 128


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="tq", choices=["tq", "reference"])
    p.add_argument("--algo", default="auto", choices=["auto", "lut", "mma"])
    p.add_argument("--tokens-per-step", type=int, default=64)
    p.add_argument("--no-extras", action="store_true")
    p.add_argument("--extras", default="set_rows,decode,sparse_v,prefill,int8,f16",
                   help="comma-separated extras to run after the main measurement")
    p.add_argument("--prefill-nq", default="3,64,512,2048,4096", help="query counts of the prefill extra")
    p.add_argument("--int8-ctx", default="4096,40000,140000", help="contexts of the int8 extra")
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


# ------------------------------------------------------------------ helpers

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.lines = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: int, world: int, seconds_max: float) -> float:
    """Units all ranks processed, divided by the slowest rank's time (weak scaling)."""
    return units_per_rank * world / seconds_max


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


DECODE_SOURCES = ("tq_decode_mma.cuh", "tq_decode_mma_t3.cu", "tq_decode_mma.cu", "tq_decode_common.cuh",
                  "tq_common.cuh", "tq_tc.cuh", "tq_quant.cuh", "tq_internal.h", "tq_host.cu")
DECODE_PROFILE = os.path.join(ROOT, "profiles", "decode_mma_32k_turbo3_ncu.md")


def decode_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, or None when the
    decode sources changed since that capture (hash of the sources recorded there)."""
    import hashlib
    import re
    try:
        text = open(DECODE_PROFILE).read()
        h = hashlib.sha256()
        for f in DECODE_SOURCES:
            with open(os.path.join(ROOT, "quantized_kv_cache_tq_gb300", "csrc", f), "rb") as fh:
                h.update(fh.read())
    except OSError:
        return None
    m_bytes = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    m_hash = re.search(r"decode_sources_sha256_16:\s*([0-9a-f]{16})", text)
    if not (m_bytes and m_hash) or m_hash.group(1) != h.hexdigest()[:16]:
        return None
    return int(m_bytes.group(1))


def per_cache_bytes(tq_type=3):
    per_block = {2: 34, 3: 50, 4: 66}[tq_type]
    return 2 * N_KV * KV_LEN * per_block


# ------------------------------------------------------------------ CPU oracle

def _oracle_worker(head, conn):
    """One KV head of the oracle in its own process: its K/V rows quantised into
    32768 cells, its 4 query heads and the new token's rows; each "step" message
    runs one token-layer (SET_ROWS of the new token's K and V rows into the last
    cell, then decode of the 4 query heads over 32768 cells)."""
    import numpy as np
    import oracle as O
    import workloads as W
    sh = W.decode_32k()
    k = W.gaussian_with_outliers(sh.seed, W.S_K, W.S_K_OUT, KV_LEN, N_KV, D)[:, head:head + 1]
    v = W.gaussian_with_outliers(sh.seed, W.S_V, W.S_V_OUT, KV_LEN, N_KV, D)[:, head:head + 1]
    sk, sv = W.codebook_signs(sh)
    c = O.centroids(3)
    kc, vc = O.empty_cache(3, 1, D, KV_LEN), O.empty_cache(3, 1, D, KV_LEN)
    O.set_rows(kc, W.to_f32(k), np.arange(KV_LEN), sk, c)
    O.set_rows(vc, W.to_f32(v), np.arange(KV_LEN), sv, c)
    q = W.to_f32(W.decode_query(sh))[4 * head:4 * head + 4].astype(np.float64)
    newk, newv = W.to_f32(k[-1:]), W.to_f32(v[-1:])
    cell = np.array([KV_LEN - 1])
    conn.send("ready")
    while conn.recv() == "step":
        O.set_rows(kc, newk, cell, sk, c)
        O.set_rows(vc, newv, cell, sv, c)
        O.decode(kc, vc, sk, sv, c, c, q, KV_LEN, 1 / math.sqrt(D))
        conn.send("done")


class OracleSample:
    """The CPU oracle on the decode_32k workload, one single-threaded process per
    KV head (8 processes, started with spawn): one step = SET_ROWS of the new
    token's K/V rows, then decode over all 32768 cells, for all 8 KV heads and 32
    query heads."""

    def __init__(self):
        import multiprocessing as mp
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
            os.environ[var] = "1"        # one core per worker process
        ctx = mp.get_context("spawn")
        self.conns, self.procs = [], []
        for h in range(N_KV):
            a, b = ctx.Pipe()
            p = ctx.Process(target=_oracle_worker, args=(h, b), daemon=True)
            p.start()
            self.conns.append(a)
            self.procs.append(p)
        for a in self.conns:
            assert a.recv() == "ready"

    def step(self):
        for a in self.conns:
            a.send("step")
        for a in self.conns:
            assert a.recv() == "done"

    def timed(self, steps, budget_s):
        done, t0 = 0, time.perf_counter()
        while True:
            self.step()
            done += 1
            el = time.perf_counter() - t0
            if done >= steps or el >= budget_s:
                break
        return done / el, el, done

    def cores(self):
        return N_KV

    def describe(self, done):
        return (f"{done} oracle steps of the whole workload (SET_ROWS of the new token's K/V rows + decode over "
                f"32768 cells, 8 KV x 32 query heads), one single-threaded process per KV head")

    def close(self):
        for a in self.conns:
            a.send("stop")
        for p in self.procs:
            p.join(timeout=30)


def run_reference(args):
    rank, world, _ = dist_setup()
    if rank != 0:
        return
    sample = OracleSample()
    warm = max(0, args.warmup)
    for _ in range(warm):
        sample.step()
    tok_s, el, done = sample.timed(max(1, args.steps), budget_s=90.0)
    sample.close()
    line = {
        "impl": "reference", "metric": METRIC, "value": tok_s, "unit": UNIT, "n_gpus": args.gpus,
        "steps": done, "warmup": warm, "ms_per_step": 1000 * el / done, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "decode_32k", "kv_heads": N_KV, "q_heads": N_Q, "head_dim": D,
                   "kv_len": KV_LEN, "type": "turbo3"},
        "cpu_baseline": {"value": tok_s, "unit": UNIT, "cores": sample.cores(), "kind": "oracle",
                         "sample": sample.describe(done)},
        "e2e": {"value": tok_s, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ GPU path

def run_tq(args):
    import numpy as np
    import torch

    import quantized_kv_cache_tq_gb300 as tq
    import workloads as W

    rank, world, local = dist_setup()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    algo = {"auto": tq.TQ_DECODE_AUTO, "lut": tq.TQ_DECODE_LUT, "mma": tq.TQ_DECODE_MMA}[args.algo]
    sh = W.decode_32k()
    sk, sv = W.codebook_signs(sh)
    cbk, cbv = tq.codebook(3, sk), tq.codebook(3, sv)

    # bulk quantisation of the whole cache (also timed as an extra: SET_ROWS at scale)
    k_raw, v_raw = W.kv_inputs(sh)
    k_src = torch.from_numpy(W.to_f32(k_raw)).to(dev)
    v_src = torch.from_numpy(W.to_f32(v_raw)).to(dev)
    del k_raw, v_raw
    cells_all = torch.arange(KV_LEN, dtype=torch.int64, device=dev)
    base_k = tq.TqCache(3, N_KV, D, KV_LEN, dev)
    base_v = tq.TqCache(3, N_KV, D, KV_LEN, dev)
    tq.set_rows(base_k, cbk, k_src, cells_all)
    tq.set_rows(base_v, cbv, v_src, cells_all)
    torch.cuda.synchronize()

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    cache_bytes = per_cache_bytes(3)
    B = max(2, math.ceil(4 * l2 / cache_bytes))
    ks, vs = [], []
    for _ in range(B):
        a, b = tq.TqCache(3, N_KV, D, KV_LEN, dev), tq.TqCache(3, N_KV, D, KV_LEN, dev)
        for dst, src in ((a, base_k), (b, base_v)):
            dst.norms.copy_(src.norms)
            dst.qs.copy_(src.qs)
            dst.signs.copy_(src.signs)
        ks.append(a)
        vs.append(b)

    # per-layer inputs: query and the new token's K/V rows
    q_all = torch.from_numpy(W.to_f32(W.normal(sh.seed, W.S_EXTRA, B * N_Q * D)).reshape(B, N_Q, D)).to(dev)
    newk = torch.from_numpy(W.to_f32(W.normal(sh.seed, W.S_EXTRA + 1, B * N_KV * D)).reshape(B, 1, N_KV, D)).to(dev)
    newv = torch.from_numpy(W.to_f32(W.normal(sh.seed, W.S_EXTRA + 2, B * N_KV * D)).reshape(B, 1, N_KV, D)).to(dev)
    cell = torch.tensor([KV_LEN - 1], dtype=torch.int64, device=dev)
    out = torch.empty((B, N_Q, D), dtype=torch.float32, device=dev)
    ws_bytes = tq._lib.tq_fattn_decode_workspace(ks[0].c, vs[0].c, N_Q, KV_LEN)
    ws = tq.workspace(ws_bytes, dev)
    scale = 1.0 / math.sqrt(D)

    def token(decode_only=False, qs=q_all, kr=newk, vr=newv):
        for b in range(B):
            if decode_only:
                tq.fattn_decode(ks[b], vs[b], cbk, cbv, qs[b], KV_LEN, scale, algo=algo, out=out[b], ws=ws)
            else:   # SET_ROWS of the token's K and V rows + decode, one call
                tq.fattn_decode_append(ks[b], vs[b], cbk, cbv, kr[b][0], vr[b][0], cell, qs[b], KV_LEN,
                                       scale, algo=algo, out=out[b], ws=ws)

    def capture(fn):
        s = torch.cuda.Stream(dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g

    T = args.tokens_per_step
    # one graph per step: T tokens x B layers of launches
    g_step = capture(lambda: [token() for _ in range(T)])
    g_decode = capture(lambda: token(decode_only=True))

    def step():
        g_step.replay()

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        ms = e0.elapsed_time(e1)
        # dominant kernel alone: B decode launches per replay, distinct caches
        R = 200
        d0, d1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for _ in range(5):
            g_decode.replay()
        d0.record(stream)
        for _ in range(R):
            g_decode.replay()
        d1.record(stream)
        torch.cuda.synchronize()
    ms = max_over_ranks(ms, world, dev)
    dec_us = d0.elapsed_time(d1) * 1000.0 / (R * B)

    calls = args.steps * T * B
    value = whole_job_rate(calls, world, ms / 1000.0)
    dec_bytes = cache_bytes + 4 * (N_Q * D * 2)
    achieved = dec_bytes / (dec_us * 1e-6) / 1e9
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        pass
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    peak_src = "measured" if "hbm_gbs" in peaks else "fallback"

    # e2e through the public API with host buffers: per step the T tokens' inputs go
    # host->device from pinned memory into the step's device buffers, which the step
    # graph reads (token t of layer b from d_q[t][b], d_k[t][b], d_v[t][b]), and the
    # last token's outputs come back
    h_q = torch.empty((T, B, N_Q, D), dtype=torch.float32).pin_memory()
    h_k = torch.empty((T, B, 1, N_KV, D), dtype=torch.float32).pin_memory()
    h_v = torch.empty((T, B, 1, N_KV, D), dtype=torch.float32).pin_memory()
    h_out = torch.empty((B, N_Q, D), dtype=torch.float32).pin_memory()
    h_q.copy_(q_all.cpu().unsqueeze(0).expand(T, -1, -1, -1))
    h_k.copy_(newk.cpu().unsqueeze(0).expand(T, -1, -1, -1, -1))
    h_v.copy_(newv.cpu().unsqueeze(0).expand(T, -1, -1, -1, -1))
    d_q = torch.empty((T, B, N_Q, D), dtype=torch.float32, device=dev)
    d_k = torch.empty((T, B, 1, N_KV, D), dtype=torch.float32, device=dev)
    d_v = torch.empty((T, B, 1, N_KV, D), dtype=torch.float32, device=dev)
    d_q.copy_(h_q)
    d_k.copy_(h_k)
    d_v.copy_(h_v)
    g_step_e2e = capture(lambda: [token(qs=d_q[t], kr=d_k[t], vr=d_v[t]) for t in range(T)])

    def e2e_step():
        d_q.copy_(h_q, non_blocking=True)
        d_k.copy_(h_k, non_blocking=True)
        d_v.copy_(h_v, non_blocking=True)
        g_step_e2e.replay()
        h_out.copy_(out, non_blocking=True)

    e2e_step()
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    h2d = h_q.numel() * 4 + h_k.numel() * 4 + h_v.numel() * 4
    d2h = h_out.numel() * 4

    # the same, without a graph: every token-layer is its own tq_fattn_decode_append
    # call through the C ABI (host argument checks and launch on each call)
    from quantized_kv_cache_tq_gb300 import _lib
    cstream = stream.cuda_stream
    ws_ptr, ws_n = ws.data_ptr(), ws.numel()
    call_args = [[(ks[b].c, vs[b].c, d_k[t][b][0].data_ptr(), d_v[t][b][0].data_ptr(), d_q[t][b].data_ptr(),
                   out[b].data_ptr()) for b in range(B)] for t in range(T)]
    algo_code = algo

    def e2e_eager_step():
        d_q.copy_(h_q, non_blocking=True)
        d_k.copy_(h_k, non_blocking=True)
        d_v.copy_(h_v, non_blocking=True)
        for t in range(T):
            for kc_, vc_, kr_, vr_, q_, o_ in call_args[t]:
                st = _lib.tq_fattn_decode_append(kc_, vc_, cbk, cbv, kr_, vr_, tq.TQ_F32, cell.data_ptr(), q_, N_Q,
                                                 KV_LEN, scale, algo_code, o_, ws_ptr, ws_n, cstream)
                if st:
                    raise RuntimeError(_lib.status_string(st))
        h_out.copy_(out, non_blocking=True)

    e2e_eager_step()
    torch.cuda.synchronize()
    eager_steps = max(1, args.steps // 4)
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(eager_steps):
        e2e_eager_step()
    torch.cuda.synchronize()
    eager_s = max_over_ranks(time.perf_counter() - t0, world, dev)
    out_checksum = tq.checksum(out)

    extras = {}
    if not args.no_extras and rank == 0:
        extras = run_extras(tq, torch, dev, base_k, base_v, k_src, v_src, cells_all, cbk, cbv, hbm_peak,
                            float(peaks.get("bf16_tflops", 1900.0)), args)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sample = OracleSample()
        sample.step()
        tok_s, el, done = sample.timed(100, budget_s=20.0)
        sample.close()
        cpu = {"value": tok_s, "unit": UNIT, "cores": sample.cores(), "kind": "oracle",
               "sample": sample.describe(done)}

    if rank == 0:
        clocks = clk.summary()
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "u8 codes; f16 tensor-core operands, f32 accumulate" if args.algo != "lut" else "u8 codes; f32",
            "data": "synthetic",
            "config": {"workload": "decode_32k", "kv_heads": N_KV, "q_heads": N_Q, "head_dim": D,
                       "kv_len": KV_LEN, "type": "turbo3", "layers_cycled": B, "tokens_per_step": T,
                       "algo": args.algo, "l2": f"working set {B} caches x {cache_bytes / 1e6:.1f} MB > 4x L2 "
                                                 f"({l2 / 1e6:.0f} MB); no flush"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": decode_traffic(), "kernel": "decode",
                         "kernel_us": dec_us, "bytes_per_launch": dec_bytes, "peak_source": peak_src},
            "e2e": {"value": calls * world / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "how": "step graph of the C-ABI calls replayed, pinned copies of "
                                                    "the step's inputs and outputs inside the timed region"},
            "e2e_eager": {"value": eager_steps * T * B * world / eager_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
                          "d2h_bytes_per_step": d2h, "steps": eager_steps,
                          "how": "one tq_fattn_decode_append C-ABI call per token-layer from Python (ctypes), no "
                                 "graph; pinned copies of the step's inputs and outputs inside the timed region"},
            "checksum": {"out_last_step": out_checksum, "hash": "FNV-1a 64 of the output bytes"},
            "gpu_launches": calls * (1 if args.algo != "lut" else 3),
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        line.update(extras)
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def time_graph(torch, fn, reps=20, warm=3):
    s = torch.cuda.current_stream()
    for _ in range(warm):
        fn()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(s)
    for _ in range(reps):
        fn()
    b.record(s)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps / 1000.0


class L2Flush:
    """Writes a buffer of twice the L2 size: called before every timed launch of
    an extra, so that no launch finds its inputs in L2."""

    def __init__(self, torch, dev):
        l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.buf = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
        self.note = f"L2 flushed before every timed launch (write of {2 * l2 / 1e6:.0f} MB)"

    def __call__(self):
        self.buf.fill_(1.0)


def time_flushed(torch, fn, flush, reps=10, warm=3):
    """Median device time (s) of fn() over `reps` launches, each after an L2 flush,
    with CUDA events on the current stream right around fn()."""
    s = torch.cuda.current_stream()
    for _ in range(warm):
        fn()
    evs = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(s)
        fn()
        b.record(s)
        evs.append((a, b))
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in evs) / 1000.0


def _device_gaussian(torch, gen, shape, dev, outliers=True):
    """N(0,1) on the device with 4 outlier channels per 128 scaled by 8 (per head)."""
    x = torch.randn(shape, generator=gen, device=dev)
    if outliers:
        n_heads, dim = shape[-2], shape[-1]
        n_out = max(1, round(4 * dim / 128))
        for h in range(n_heads):
            ch = torch.randperm(dim, generator=gen, device=dev)[:n_out]
            x[..., h, ch] *= 8.0
    return x


def _copy_cache(tq, src, dev):
    c = tq.TqCache(src.tq_type, src.n_kv_heads, src.head_dim, src.n_cells, dev)
    for d, s_ in zip(c.planes(), src.planes()):
        if d is not None:
            d.copy_(s_)
    return c


def decode_config(tq, torch, dev, kc, vc, cbk, cbv, q, algo, hbm_peak, name, l2):
    """Decode kernel time on one workload: a graph of B launches over B copies of
    the cache pair (B so that the copies exceed 4x L2), replayed 20 times."""
    from quantized_kv_cache_tq_gb300 import _lib
    kv_len = kc.n_cells
    per_block = {2: 34, 3: 50, 4: 66}
    nbytes = kc.n_kv_heads * kv_len * (kc.n_blocks * per_block[kc.tq_type] + vc.n_blocks * per_block[vc.tq_type])
    B = max(2, math.ceil(4 * l2 / nbytes))
    pairs = [(kc, vc)] + [(_copy_cache(tq, kc, dev), _copy_cache(tq, vc, dev)) for _ in range(B - 1)]
    n_q = q.shape[0]
    out = torch.empty((B, n_q, vc.head_dim), dtype=torch.float32, device=dev)
    ws = tq.workspace(_lib.tq_fattn_decode_workspace(kc.c, vc.c, n_q, kv_len), dev)
    scale = 1.0 / math.sqrt(kc.head_dim)

    def once():
        for b, (k_, v_) in enumerate(pairs):
            tq.fattn_decode(k_, v_, cbk, cbv, q, kv_len, scale, algo=algo, out=out[b], ws=ws)
    once()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        once()
    t = time_graph(torch, g.replay, reps=20) / B
    nbytes += 4 * n_q * (kc.head_dim + vc.head_dim)
    res = {"workload": name, "us": t * 1e6, "GB/s": nbytes / t / 1e9, "frac_hbm": nbytes / t / 1e9 / hbm_peak,
           "tokens/s": 1.0 / t, "bytes_per_launch": nbytes,
           "l2": f"{B} cache copies x {nbytes / 1e6:.1f} MB cycled (> 4x L2)", "checksum": tq.checksum(out[0])}
    del pairs
    return res


def run_decode_configs(tq, torch, dev, k_src, v_src, cells_all, hbm_peak, flush):
    """Decode on every workload of the sweep: tiny_decode; decode_32k at turbo3,
    turbo2 and turbo4 on the same inputs with the tensor-core kernel and with the
    shared-memory Q x centroid LUT kernel; asym_8k (K 192 / V 128)."""
    import workloads as W
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    res = {}
    sh = W.decode_32k()
    sk, sv = W.codebook_signs(sh)
    q = torch.from_numpy(W.to_f32(W.normal(sh.seed, W.S_EXTRA, N_Q * D)).reshape(N_Q, D)).to(dev)
    for t in (3, 2, 4):
        cbk, cbv = tq.codebook(t, sk), tq.codebook(t, sv)
        kc, vc = tq.TqCache(t, N_KV, D, KV_LEN, dev), tq.TqCache(t, N_KV, D, KV_LEN, dev)
        tq.set_rows(kc, cbk, k_src, cells_all)
        tq.set_rows(vc, cbv, v_src, cells_all)
        for algo, code in (("mma", tq.TQ_DECODE_MMA), ("lut", tq.TQ_DECODE_LUT)):
            res[f"decode_32k_turbo{t}_{algo}"] = decode_config(
                tq, torch, dev, kc, vc, cbk, cbv, q, code, hbm_peak,
                f"decode_32k turbo{t}, 8 KV x 32 Q heads, D=128, 32768 cells, {algo} kernel", l2)
        del kc, vc
    # batched decode: 8 sequences of 32768 cells each in one launch (one new token
    # per sequence), K/V of the decode_32k inputs in every sequence's cells
    cbk3, cbv3 = tq.codebook(3, sk), tq.codebook(3, sv)
    n_seq = 8
    per_pair = n_seq * 2 * N_KV * KV_LEN * 50
    n_sets = max(2, math.ceil(4 * l2 / per_pair))
    sets = []
    for _ in range(n_sets):
        kc, vc = tq.TqCache(3, N_KV, D, n_seq * KV_LEN, dev), tq.TqCache(3, N_KV, D, n_seq * KV_LEN, dev)
        for sq in range(n_seq):
            cells = torch.arange(sq * KV_LEN, (sq + 1) * KV_LEN, dtype=torch.int64, device=dev)
            tq.set_rows(kc, cbk3, k_src, cells)
            tq.set_rows(vc, cbv3, v_src, cells)
        sets.append((kc, vc))
    qb = q.unsqueeze(0).repeat(n_seq, 1, 1).contiguous()
    outb = torch.empty((n_seq, N_Q, D), device=dev)
    offs, lens = [sq * KV_LEN for sq in range(n_seq)], [KV_LEN] * n_seq
    wsb = tq.workspace(tq._lib.tq_fattn_decode_batch_workspace(sets[0][0].c, sets[0][1].c, N_Q, n_seq, KV_LEN), dev)

    def once_b():
        for kc, vc in sets:
            tq.fattn_decode_batch(kc, vc, cbk3, cbv3, qb, offs, lens, 1.0 / math.sqrt(D), out=outb, ws=wsb)
    once_b()
    torch.cuda.synchronize()
    gb = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gb):
        once_b()
    t = time_graph(torch, gb.replay, reps=20) / n_sets
    nbytes = per_pair + 4 * n_seq * N_Q * D * 2
    res["decode_batch8_32k"] = {"workload": "8 sequences x 32768 cells, 8 KV x 32 Q heads, D=128, turbo3, one launch",
                                "us": t * 1e6, "tokens/s": n_seq / t, "GB/s": nbytes / t / 1e9,
                                "frac_hbm": nbytes / t / 1e9 / hbm_peak,
                                "l2": f"{n_sets} cache pairs x {per_pair / 1e6:.0f} MB cycled (> 4x L2)",
                                "checksum": tq.checksum(outb)}
    del sets
    # asym_8k: K head dim 192 (two blocks), V 128, 16 = 16 heads, 8192 cells
    gen = torch.Generator(device=dev)
    gen.manual_seed(20263)
    sha = W.asym_8k()
    ska, sva = W.codebook_signs(sha)
    cbk, cbv = tq.codebook(3, ska), tq.codebook(3, sva)
    L = sha.kv_len
    kc, vc = tq.TqCache(3, 16, 192, L, dev), tq.TqCache(3, 16, 128, L, dev)
    cells = torch.arange(L, dtype=torch.int64, device=dev)
    tq.set_rows(kc, cbk, _device_gaussian(torch, gen, (L, 16, 192), dev), cells)
    tq.set_rows(vc, cbv, _device_gaussian(torch, gen, (L, 16, 128), dev), cells)
    qa = _device_gaussian(torch, gen, (1, 16, 192), dev)[0].contiguous()
    res["decode_asym_8k"] = decode_config(tq, torch, dev, kc, vc, cbk, cbv, qa, tq.TQ_DECODE_AUTO, hbm_peak,
                                          "asym_8k decode: Dk=192 / Dv=128, 16 = 16 heads, 8192 cells, turbo3", l2)
    # tiny_decode: 1 KV head, 512 cells (25.6 KB of cache: launch-bound), L2 flushed
    sht = W.tiny_decode()
    skt, svt = W.codebook_signs(sht)
    cbk, cbv = tq.codebook(3, skt), tq.codebook(3, svt)
    kr, vr = W.kv_inputs(sht)
    kc, vc = tq.TqCache(3, 1, 128, 512, dev), tq.TqCache(3, 1, 128, 512, dev)
    cells = torch.arange(512, dtype=torch.int64, device=dev)
    tq.set_rows(kc, cbk, torch.from_numpy(W.to_f32(kr)).to(dev), cells)
    tq.set_rows(vc, cbv, torch.from_numpy(W.to_f32(vr)).to(dev), cells)
    qt = torch.from_numpy(W.to_f32(W.decode_query(sht))).to(dev)
    out = torch.empty((1, 128), device=dev)
    ws = tq.workspace(tq._lib.tq_fattn_decode_workspace(kc.c, vc.c, 1, 512), dev)
    t = time_flushed(torch, lambda: tq.fattn_decode(kc, vc, cbk, cbv, qt, 512, out=out, ws=ws), flush, reps=50)
    res["decode_tiny"] = {"workload": "tiny_decode: 1 KV / 1 Q head, D=128, 512 cells, turbo3", "us": t * 1e6,
                          "tokens/s": 1.0 / t, "l2": flush.note, "checksum": tq.checksum(out),
                          "note": "launch-bound (25.6 KB of cache)"}
    return res


def run_sparse_v_extra(tq, torch, dev, n_sets=6, thr=5e-3):
    """Decode at 32K over caches whose scores have a wide gap: about one key in 64
    scores near +20, the rest near -20 (K rows +-3 along one direction per KV head
    plus N(0, 0.1) noise, queries 75 times that direction).  Decode without and
    with sparse V (threshold 5e-3): the groups of cold keys leave the V work.
    n_sets cache pairs (26 MB each) are cycled so that the working set exceeds L2."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(20263)
    L, HK, HQ, DD = KV_LEN, N_KV, N_Q, D
    import workloads as W
    sk, sv = W.codebook_signs(W.decode_32k())
    cbk, cbv = tq.codebook(3, sk), tq.codebook(3, sv)
    cells = torch.arange(L, dtype=torch.int64, device=dev)
    sets = []
    for _ in range(n_sets):
        e = torch.randn((HK, DD), generator=gen, device=dev)
        e /= e.norm(dim=1, keepdim=True)
        hot = torch.rand((L, HK), generator=gen, device=dev) < 1.0 / 64
        krow = 0.1 * torch.randn((L, HK, DD), generator=gen, device=dev) + torch.where(hot, 3.0, -3.0)[..., None] * e
        kc, vc = tq.TqCache(3, HK, DD, L, dev), tq.TqCache(3, HK, DD, L, dev)
        tq.set_rows(kc, cbk, krow.contiguous(), cells)
        tq.set_rows(vc, cbv, torch.randn((L, HK, DD), generator=gen, device=dev), cells)
        q = 75.0 * e.repeat_interleave(HQ // HK, dim=0) + 0.1 * torch.randn((HQ, DD), generator=gen, device=dev)
        sets.append((kc, vc, q.contiguous(), torch.empty((HQ, DD), dtype=torch.float32, device=dev)))
    ws = tq.workspace(tq._lib.tq_fattn_decode_workspace(sets[0][0].c, sets[0][1].c, HQ, L), dev)
    res = {"workload": f"decode_32k turbo3 over gapped scores (1/64 hot keys), {n_sets} cache sets cycled",
           "threshold": thr}
    for name, t_ in (("exact_us", 0.0), ("sparse_v_us", thr)):
        def once(t_=t_):
            for kc, vc, q, out in sets:
                tq.fattn_decode(kc, vc, cbk, cbv, q, L, 1.0 / math.sqrt(DD), out=out, ws=ws, sparse_v=t_)
        g = torch.cuda.CUDAGraph()
        once()
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            once()
        res[name] = time_graph(torch, g.replay, reps=50) / n_sets * 1e6
    return res


def _prefill_flop(nq, kv_len, n_q, dk, dv, causal=True):
    pairs = sum(min(kv_len, kv_len - nq + i + 1) for i in range(nq)) if causal else nq * kv_len
    return 2.0 * (dk + dv) * pairs * n_q


def run_prefill_extra(tq, torch, dev, tflops_peak, flush, nqs=(3, 64, 512, 2048, 4096)):
    """Prefill over the 4K-context turbo3 cache (8 KV x 16 query heads, D = 256,
    causal) at every query count of the sweep, and the asym_8k prefill (K 192 /
    V 128, 16 = 16 heads, 8192 cells, 512 queries)."""
    import workloads as W
    gen = torch.Generator(device=dev)
    gen.manual_seed(20262)
    L, HK, HQ, DD = 4096, 8, 16, 256
    sh = W.prefill_4k()
    sk, sv = W.codebook_signs(sh)
    cbk, cbv = tq.codebook(3, sk), tq.codebook(3, sv)
    kc, vc = tq.TqCache(3, HK, DD, L, dev), tq.TqCache(3, HK, DD, L, dev)
    cells = torch.arange(L, dtype=torch.int64, device=dev)
    tq.set_rows(kc, cbk, _device_gaussian(torch, gen, (L, HK, DD), dev), cells)
    tq.set_rows(vc, cbv, _device_gaussian(torch, gen, (L, HK, DD), dev), cells)
    res = {"workload": "prefill_4k: 8 KV x 16 Q heads, D=256, 4096 cells, turbo3, causal, bf16 Q",
           "flops": "2 (Dk + Dv) per visible (query, key) pair per query head; hi/lo fp16 operand splits not counted",
           "l2": flush.note}
    for nq in nqs:
        q = torch.randn((nq, HQ, DD), generator=gen, device=dev).to(torch.bfloat16)
        out = torch.empty((nq, HQ, DD), device=dev)
        ws = tq.workspace(tq._lib.tq_fattn_prefill_workspace(kc.c, vc.c, nq, HQ, L), dev)
        t = time_flushed(torch, lambda: tq.fattn_prefill(kc, vc, cbk, cbv, q, L, out=out, ws=ws), flush, reps=7)
        flop = _prefill_flop(nq, L, HQ, DD, DD)
        res[f"nq{nq}"] = {"ms": t * 1e3, "TFLOP/s": flop / t / 1e12, "frac_bf16_peak": flop / t / 1e12 / tflops_peak,
                          "algorithmic_GFLOP": flop / 1e9, "tokens/s": nq / t, "checksum": tq.checksum(out)}
    # speculative-decoding verify batches: nq new tokens over the 32K decode cache
    # (8 KV x 32 query heads, D = 128, f32 queries), through the prefill kernel
    sh32 = W.decode_32k()
    sk32, sv32 = W.codebook_signs(sh32)
    cbk32, cbv32 = tq.codebook(3, sk32), tq.codebook(3, sv32)
    kc32, vc32 = tq.TqCache(3, 8, 128, 32768, dev), tq.TqCache(3, 8, 128, 32768, dev)
    cells32 = torch.arange(32768, dtype=torch.int64, device=dev)
    tq.set_rows(kc32, cbk32, _device_gaussian(torch, gen, (32768, 8, 128), dev), cells32)
    tq.set_rows(vc32, cbv32, _device_gaussian(torch, gen, (32768, 8, 128), dev), cells32)
    for nq in (2, 4, 6):
        q = torch.randn((nq, 32, 128), generator=gen, device=dev)
        out = torch.empty((nq, 32, 128), device=dev)
        ws = tq.workspace(tq._lib.tq_fattn_prefill_workspace(kc32.c, vc32.c, nq, 32, 32768), dev)
        t = time_flushed(torch, lambda: tq.fattn_prefill(kc32, vc32, cbk32, cbv32, q, 32768, out=out, ws=ws), flush,
                         reps=10)
        nbytes = 2 * 8 * 32768 * 50
        res[f"verify_nq{nq}_32k"] = {"us": t * 1e6, "tokens/s": nq / t, "GB/s": nbytes / t / 1e9,
                                     "workload": f"verify batch: {nq} tokens over the 32K turbo3 cache, causal",
                                     "checksum": tq.checksum(out)}
    del kc32, vc32
    # asym_8k prefill, nq = 512
    sha = W.asym_8k(512)
    ska, sva = W.codebook_signs(sha)
    cbk, cbv = tq.codebook(3, ska), tq.codebook(3, sva)
    La = sha.kv_len
    kc, vc = tq.TqCache(3, 16, 192, La, dev), tq.TqCache(3, 16, 128, La, dev)
    cells = torch.arange(La, dtype=torch.int64, device=dev)
    tq.set_rows(kc, cbk, _device_gaussian(torch, gen, (La, 16, 192), dev), cells)
    tq.set_rows(vc, cbv, _device_gaussian(torch, gen, (La, 16, 128), dev), cells)
    q = torch.randn((512, 16, 192), generator=gen, device=dev).to(torch.bfloat16)
    out = torch.empty((512, 16, 128), device=dev)
    ws = tq.workspace(tq._lib.tq_fattn_prefill_workspace(kc.c, vc.c, 512, 16, La), dev)
    t = time_flushed(torch, lambda: tq.fattn_prefill(kc, vc, cbk, cbv, q, La, out=out, ws=ws), flush, reps=7)
    flop = _prefill_flop(512, La, 16, 192, 128)
    res["asym_8k_nq512"] = {"workload": "asym_8k prefill: Dk=192 / Dv=128, 16 = 16 heads, 8192 cells, 512 queries",
                            "ms": t * 1e3, "TFLOP/s": flop / t / 1e12, "frac_bf16_peak": flop / t / 1e12 / tflops_peak,
                            "algorithmic_GFLOP": flop / 1e9, "checksum": tq.checksum(out)}
    return res


def _int8_cache(torch, gen, ctx, dev, HK=8, DD=128):
    raw = _device_gaussian(torch, gen, (ctx, HK, DD), dev)
    sk = (raw.abs().amax(-1) / 127).to(torch.float16)
    k = torch.clamp(torch.round(raw / sk.float().unsqueeze(-1)), -127, 127).to(torch.int8)
    raw = _device_gaussian(torch, gen, (ctx, HK, DD), dev)
    sv = (raw.abs().amax(-1) / 127).to(torch.float16)
    v = torch.clamp(torch.round(raw / sv.float().unsqueeze(-1)), -127, 127).to(torch.int8)
    return k, sk, v, sv


def run_int8_extra(tq, torch, dev, tflops_peak, flush, ctxs=(4096, 40000, 140000), nq=2048):
    """int8 prompt attention: 8 KV x 32 Q heads, D = 128, 2048 queries over each
    context of the sweep, rows gathered through a random permutation of the cells."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(20264)
    HK, HQ, DD = 8, 32, 128
    res = {"workload": "int8_prompt: 8 KV x 32 Q heads, D=128, 2048 queries, scattered int8 rows + fp16 scales, "
                       "fp16 Q, causal", "l2": flush.note}
    for ctx in ctxs:
        k, sk, v, sv = _int8_cache(torch, gen, ctx, dev)
        perm = torch.randperm(ctx, generator=gen, device=dev).to(torch.int32)
        q = torch.randn((nq, HQ, DD), generator=gen, device=dev).to(torch.float16)
        out = torch.empty((nq, HQ, DD), device=dev)
        ws = tq.workspace(tq._lib.tq_int8_prompt_attn_workspace(nq, HQ, HK, DD, ctx), dev)
        t = time_flushed(torch, lambda: tq.int8_prompt_attn(k, sk, v, sv, perm, ctx, q, out=out, ws=ws), flush,
                         reps=5)
        flop = _prefill_flop(nq, ctx, HQ, DD, DD)
        res[f"ctx{ctx}"] = {"ms": t * 1e3, "TFLOP/s": flop / t / 1e12, "frac_bf16_peak": flop / t / 1e12 / tflops_peak,
                            "algorithmic_GFLOP": flop / 1e9, "checksum": tq.checksum(out)}
        del k, v, sk, sv
    return res


def run_f16_prompt_extra(tq, torch, dev, tflops_peak, flush, ctxs=(4096, 40000), nq=2048):
    """Prompt attention over binary16 rows (the int8 path's other cache mode)."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(20265)
    HK, HQ, DD = 8, 32, 128
    res = {"workload": "f16_prompt: 8 KV x 32 Q heads, D=128, 2048 queries, scattered binary16 rows, causal",
           "l2": flush.note}
    for ctx in ctxs:
        k = _device_gaussian(torch, gen, (ctx, HK, DD), dev).to(torch.float16)
        v = _device_gaussian(torch, gen, (ctx, HK, DD), dev).to(torch.float16)
        perm = torch.randperm(ctx, generator=gen, device=dev).to(torch.int32)
        q = torch.randn((nq, HQ, DD), generator=gen, device=dev).to(torch.float16)
        out = torch.empty((nq, HQ, DD), device=dev)
        ws = tq.workspace(tq._lib.tq_int8_prompt_attn_workspace(nq, HQ, HK, DD, ctx), dev)
        t = time_flushed(torch, lambda: tq.f16_prompt_attn(k, v, perm, ctx, q, out=out, ws=ws), flush, reps=5)
        flop = _prefill_flop(nq, ctx, HQ, DD, DD)
        res[f"ctx{ctx}"] = {"ms": t * 1e3, "TFLOP/s": flop / t / 1e12, "frac_bf16_peak": flop / t / 1e12 / tflops_peak,
                            "algorithmic_GFLOP": flop / 1e9, "checksum": tq.checksum(out)}
    return res


def run_extras(tq, torch, dev, base_k, base_v, k_src, v_src, cells_all, cbk, cbv, hbm_peak, tflops_peak, args):
    """Other rows of the hot path and the other workloads of the sweep, each on its own inputs."""
    flush = L2Flush(torch, dev)
    want = set(args.extras.split(","))
    nqs = tuple(int(x) for x in args.prefill_nq.split(",") if x)
    ctxs = tuple(int(x) for x in args.int8_ctx.split(",") if x)
    ex = {}
    # SET_ROWS over the whole 32K cache (K and V): read fp32 rows, write packed planes
    def bulk():
        tq.set_rows(base_k, cbk, k_src, cells_all)
        tq.set_rows(base_v, cbv, v_src, cells_all)
    if "set_rows" in want:
        t = time_flushed(torch, bulk, flush, reps=10)
        nbytes = 2 * (k_src.numel() * 4 + N_KV * KV_LEN * 50) + 2 * KV_LEN * 8
        ex["set_rows_bulk"] = {"workload": "32768 rows x 8 KV heads x 128, K and V, f32 -> turbo3",
                               "ms": t * 1e3, "GB/s": nbytes / t / 1e9, "frac_hbm": nbytes / t / 1e9 / hbm_peak,
                               "l2": flush.note, "checksum": tq.checksum(base_k.qs)}
    if "decode" in want:
        ex["decode_configs"] = run_decode_configs(tq, torch, dev, k_src, v_src, cells_all, hbm_peak, flush)
    if "sparse_v" in want:
        ex["sparse_v"] = run_sparse_v_extra(tq, torch, dev)
    if "prefill" in want:
        ex["prefill"] = run_prefill_extra(tq, torch, dev, tflops_peak, flush, nqs=nqs)
    if "int8" in want:
        ex["int8_prompt"] = run_int8_extra(tq, torch, dev, tflops_peak, flush, ctxs=ctxs)
    if "f16" in want:
        ex["f16_prompt"] = run_f16_prompt_extra(tq, torch, dev, tflops_peak, flush)
    return ex


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_tq(args)


if __name__ == "__main__":
    main()

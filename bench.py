#!/usr/bin/env python
"""Benchmark of the A16W4 MXFP4 MoE layer on GB300 (one JSON line on stdout).

Headline: one MoE layer call at the Kimi-K3 expert-parallel decode shape
(1 token, 112 local experts, H=3584, I=3072, top-15), MXFP4 weights resident in
HBM, in microseconds per call.  A step is one call of the whole forward path
(grouping, gate_up GEMM + SiLU gating, down GEMM, top-k combine).  Four
rotating copies of the 1.97 GB expert weights keep every step's weight reads
out of L2.  The K timed steps are replayed from one CUDA graph.

Also reported (``rows``): the decode sweep (T = 4, 7, 16, 32), the
int4_per_group_32 requantiser over all 112 experts, the int4 MoE at T = 1, 7,
32, and the tensor-core prefill path at T = 4096 when built.  ``e2e`` is the
headline measured through the Python binding of the C ABI with inputs copied
from pinned host memory and the output copied back every step.  ``roofline``
is the dominant decode kernel (both GEMMs of a T=1 call) against measured HBM
bandwidth, its duration taken with CUDA events in a separate 8-step graph (the
timed graph carries no events).  ``cpu_baseline`` is the CPU oracle on a
bounded sample, extrapolated.

--impl reference times the CPU oracle alone on the same workload.
Multi-GPU (torchrun): independent replicas, one per GPU (the layer has no
cross-GPU step at this shape); ``value`` is the aggregate time per call.
"""

from __future__ import annotations

import os

import argparse  # noqa: E402
import ctypes  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE layer us/call (Kimi-K3 EP decode, T=1, MXFP4 A16W4)"
UNIT = "us/call"
SHAPE = synth.k3(1)
W13_BYTES = 2 * SHAPE.I * SHAPE.H // 2 + 2 * SHAPE.I * SHAPE.H // 32  # per expert
W2_BYTES = SHAPE.H * SHAPE.I // 2 + SHAPE.H * SHAPE.I // 32
N_COPIES = 4
ROTATE = 8


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-rows", action="store_true", help="skip the secondary measurements")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--copies", type=int, default=4, help="rotating weight copies (L2 defeat)")
    ap.add_argument("--no-soak", action="store_true", help="skip the 1 s clock soak before the timed region")
    ap.add_argument("--rows", default="sweep,requant,int4,prefill,actquant",
                    help="comma list of secondary measurements to run (sweep, requant, int4, prefill, actquant)")
    ap.add_argument("--prefill-tokens", type=int, default=4096, help="tokens of the prefill row")
    return ap.parse_args()


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("decode.cu", "common.cuh"):
        with open(os.path.join(ROOT, "mxfp4_weight_only_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def fused_decode(H, I):
    """True when the library runs both decode GEMMs in one launch: its fused
    kernel holds activation fragments for at most 8 blocks of 32 per consumer
    warp (14 warps), i.e. H and I at most 3584."""
    nbw = lambda K: 2 * ((K // 32 + 27) // 28)
    return nbw(H) <= 8 and nbw(I) <= 8


def committed_traffic():
    """Per-launch DRAM bytes of the fused decode kernel from the committed ncu
    summary, if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "decode_fused_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_hash") != kernel_source_hash():
        return None
    return d.get("bytes_per_launch")


# ----------------------------------------------------------------------------- CPU oracle


def blas_threads():
    """Threads of numpy's BLAS pool (None when threadpoolctl is not installed)."""
    try:
        from threadpoolctl import threadpool_info
    except ImportError:
        return None
    n = [i.get("num_threads") for i in threadpool_info() if i.get("user_api") == "blas"]
    return max(n) if n else None


def oracle_sample(x, ids, w, weights, n_pairs: int):
    """Time the oracle's ``moe_forward`` on one T=1 call restricted to its first
    ``n_pairs`` (token, expert) pairs (the other ids set to -1, which the layer
    skips).  Returns (seconds measured, microseconds extrapolated to all of the
    call's pairs by pair count: every pair dequantises and multiplies one whole
    expert)."""
    from oracle import moe

    w13, s13, w2, s2 = weights
    sub = np.array(ids, copy=True)
    sub[:, n_pairs:] = -1
    t0 = time.perf_counter()
    moe.moe_forward(x, sub, w, w13, s13, w2, s2)
    dt = time.perf_counter() - t0
    n_valid = int(((ids >= 0) & (ids < w13.shape[0])).sum())
    return dt, dt * 1e6 * n_valid / n_pairs


def cpu_baseline_entry(us_per_call, n_pairs):
    cores = os.cpu_count()
    bt = blas_threads()
    return {"value": round(us_per_call, 1), "unit": UNIT, "cores": bt if bt else cores, "kind": "oracle",
            "host_cpu_count": cores, "blas_threads": bt,
            "sample": (f"{n_pairs} of the {SHAPE.topk} (token, expert) pairs of one T=1 call (the other ids set to "
                       f"-1) through the float64 numpy oracle's moe_forward (whole experts: dequantise, GEMV, SiLU "
                       f"gate, GEMV, weighted sum), extrapolated by pair count to the whole call; BLAS on the host's "
                       f"default thread pool, dequantisation single-threaded numpy")}


def host_weights(seed: int = 100):
    g = synth.rng(seed)
    w13, s13 = synth.random_mxfp4_bytes(g, SHAPE.E, 2 * SHAPE.I, SHAPE.H)
    w2, s2 = synth.random_mxfp4_bytes(g, SHAPE.E, SHAPE.H, SHAPE.I)
    return w13, s13, w2, s2


def host_batch(seed: int, T: int, bias_std=None):
    g = synth.rng(seed)
    x = synth.activations_bf16(g, T, SHAPE.H)
    ids, w = synth.router_topk(g, T, SHAPE.E, SHAPE.topk, bias_std)
    return x, ids, w


REF_PAIRS = 1  # pairs of the 15 per reference-arm step (about half a second of oracle work each)


def run_reference(args, rank: int):
    if rank != 0:
        return
    weights = host_weights()
    batches = [host_batch(1000 + i, 1) for i in range(ROTATE)]
    for i in range(args.warmup):
        x, ids, w = batches[i % ROTATE]
        oracle_sample(x, ids, w, weights, REF_PAIRS)
    secs, vals = [], []
    t0 = time.perf_counter()
    for i in range(args.steps):
        x, ids, w = batches[i % ROTATE]
        s, v = oracle_sample(x, ids, w, weights, REF_PAIRS)
        secs.append(s)
        vals.append(v)
    wall = time.perf_counter() - t0
    v = statistics.mean(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        # the time each step actually took (a sample of one call), not the extrapolated call
        "ms_per_step": round(1000.0 * statistics.mean(secs), 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(),
        "cpu_baseline": cpu_baseline_entry(v, REF_PAIRS),
        "e2e": {"value": round(v, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": round(wall, 2),
    }
    print(json.dumps(line), flush=True)


def workload_config(n_copies=N_COPIES):
    return {"workload": "kimi-k3 ep decode: T=1, E=112 local experts, H=3584, I=3072, topk=15, "
                        "mxfp4 w13[112,6144,1792]+e8m0 / w2[112,3584,1536]+e8m0, x bf16 N(0,1), "
                        "router logits N(0,1) top-15 renormalised",
            "weights": "uniform random E2M1 codes, E8M0 scales uniform in [116,121]",
            "l2": f"{n_copies} rotating weight copies ({n_copies * 1.97:.1f} GB) > L2",
            "launch": "one CUDA graph of the K timed steps"}


# ----------------------------------------------------------------------------- GPU arm


def run_ours(args, rank: int, world: int):
    import torch

    import mxfp4_weight_only_gb300 as m
    from mxfp4_weight_only_gb300 import _native, build

    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    build.build()
    lib = _native.load()
    dev = torch.device("cuda", local)
    peaks = read_peaks()

    # ---- weights: one host copy, three more derived on the device by byte XOR masks
    w13_h, s13_h, w2_h, s2_h = host_weights()
    base = [torch.from_numpy(a).to(dev) for a in (w13_h, s13_h, w2_h, s2_h)]
    copies = [tuple(base)]
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    n_copies = args.copies
    for c in range(1, n_copies):
        mask = torch.randint(0, 256, (1,), generator=gen, device=dev, dtype=torch.int32).to(torch.uint8)
        copies.append((base[0] ^ mask, base[1].clone(), base[2] ^ mask, base[3].clone()))
    torch.cuda.synchronize()

    def dev_batch(T, seed, bias=None):
        x, ids, w = host_batch(seed, T, bias)
        return (torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16), torch.from_numpy(ids).to(dev),
                torch.from_numpy(w).to(dev), ids)

    def distinct(ids):
        v = ids[(ids >= 0) & (ids < SHAPE.E)]
        return len(np.unique(v))

    stream = torch.cuda.Stream(device=dev)

    def capture(T, n_steps, kind="mxfp4", timing_steps=0, weights=None, seed0=1000, path=0, opts=None):
        """Capture n_steps MoE calls (rotating weight copies and batches) into one graph;
        ``opts``: optional layer inputs (keyword arguments of the binding)."""
        opts = opts or {}
        weights = weights or copies
        batches = [dev_batch(T, seed0 + i) for i in range(ROTATE)]
        d = m.dims(SHAPE.E, SHAPE.H, SHAPE.I, SHAPE.topk, T, path)
        # zeroed once: the status word read after the timed region starts clean
        ws = torch.zeros(m.moe_workspace_bytes(d), dtype=torch.uint8, device=dev)
        out = torch.empty((T, SHAPE.H), dtype=torch.bfloat16, device=dev)
        fn = m.moe_a16w4_mxfp4 if kind == "mxfp4" else m.moe_a16w4_int4g32
        ev = []
        with torch.cuda.stream(stream):
            for i in range(2):  # eager warm-up outside capture (kernel attributes, module load)
                x, ids, w, _ = batches[i % ROTATE]
                fn(x, ids, w, *weights[i % len(weights)], out=out, workspace=ws, path=path, **opts)
        stream.synchronize()
        # timing events exist before capture; the library records them as graph nodes
        pre = []
        with torch.cuda.stream(stream):
            for _ in range(timing_steps):
                evs = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
                for e in evs:
                    e.record()
                pre.append(evs)
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        bytes_total = 0
        with torch.cuda.graph(graph, stream=stream, capture_error_mode="thread_local"):
            for i in range(n_steps):
                x, ids, w, ids_h = batches[i % ROTATE]
                # per-kernel events on the first timing_steps steps (only in the
                # graphs built for them: an event between two kernels stops
                # their programmatic overlap)
                if i < timing_steps:
                    evs = pre[i]
                    arr = (ctypes.c_void_p * 8)(*[e.cuda_event for e in evs])
                    _native.check("moe_set_timing_events", lib.moe_set_timing_events(arr, 4))
                    ev.append((evs, distinct(ids_h)))
                fn(x, ids, w, *weights[i % len(weights)], out=out, workspace=ws, path=path, **opts)
                bytes_total += distinct(ids_h) * (W13_BYTES + W2_BYTES)
        return graph, ev, bytes_total, (d, ws)

    def time_graph(graph, reps=1):
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            s_ev.record()
            for _ in range(reps):
                graph.replay()
            e_ev.record()
        e_ev.synchronize()
        return s_ev.elapsed_time(e_ev)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    # ---- headline: K steps in one graph that carries no timing events (an
    # event between two kernels stops their programmatic overlap); the
    # per-kernel durations come from a separate 8-step graph with events on
    # every step, replayed after the timed region
    K, W = args.steps, args.warmup
    g_main, _, bytes_main, (d1, ws1) = capture(1, K)
    g_ev, kev, _, _ = capture(1, 8, timing_steps=8, seed0=3000)
    g_warm, _, _, _ = capture(1, max(W, 1))
    for _ in range(max(W, 3)):
        time_graph(g_warm)
    # clock soak: keep the GPU busy ~1 s while the sampler runs, then the timed region
    with ClockSampler(local) as clk:
        t_end = time.time() + (0.0 if args.no_soak else 1.0)
        while time.time() < t_end:
            time_graph(g_warm, reps=20)
        barrier()
        t0 = time.perf_counter()
        ms = time_graph(g_main)
        wall = time.perf_counter() - t0
        barrier()
    clocks = clk.summary()
    status = m.moe_read_status(d1, ws1)
    ms = max_over_ranks(ms, world, dev)
    us_per_call = ms * 1000.0 / (K * world)
    # per-kernel durations: the event graph, replayed twice, read after the second
    time_graph(g_ev)
    time_graph(g_ev)
    fused = fused_decode(SHAPE.H, SHAPE.I)
    names = ["route", "gemm_fused_gate_up_down" if fused else "gemm1_gate_up", None if fused else "gemm2_down",
             "combine"]
    kt = {n: [] for n in names if n}
    g1_bytes = 0
    for evs, dd in kev:
        for j, n in enumerate(names):
            if n:
                kt[n].append(evs[2 * j].elapsed_time(evs[2 * j + 1]) * 1000.0)
        g1_bytes += dd * (W13_BYTES + W2_BYTES if fused else W13_BYTES)
    kavg = {n: statistics.mean(v) for n, v in kt.items()}
    g1_gbs = g1_bytes / (sum(kt[names[1]]) * 1e-6) / 1e9
    layer_gbs = bytes_main / (ms * 1e-3) / 1e9
    # launches of one T=1 step: grouping inside the GEMM kernels (15 pairs), the
    # GEMM launch(es), the combine
    launches_per_step = (1 if SHAPE.topk > 128 else 0) + (1 if fused else 2) + 1

    # ---- e2e through the Python binding, host buffers, copies in the timed region
    T = 1
    hb = [host_batch(1000 + i, T) for i in range(ROTATE)]
    # one pinned host buffer per step holds x | topk ids | topk weights, so a
    # step's inputs travel in one host-to-device copy
    nbx, nbi = T * SHAPE.H * 2, T * SHAPE.topk * 4
    hin = [torch.from_numpy(np.concatenate([b[0].view(np.uint8).ravel(), b[1].view(np.uint8).ravel(),
                                            b[2].view(np.uint8).ravel()])).pin_memory() for b in hb]
    hout = [torch.empty((T, SHAPE.H), dtype=torch.int16).pin_memory() for _ in range(ROTATE)]
    din = torch.empty(nbx + 2 * nbi, dtype=torch.uint8, device=dev)
    dx = din[:nbx].view(torch.bfloat16).view(T, SHAPE.H)
    dids = din[nbx:nbx + nbi].view(torch.int32).view(T, SHAPE.topk)
    dw = din[nbx + nbi:].view(torch.float32).view(T, SHAPE.topk)
    dout = torch.empty((T, SHAPE.H), dtype=torch.bfloat16, device=dev)

    def e2e_steps(n):
        for i in range(n):
            r = i % ROTATE
            din.copy_(hin[r], non_blocking=True)
            m.moe_a16w4_mxfp4(dx, dids, dw, *copies[i % len(copies)], out=dout, workspace=ws1)
            hout[r].copy_(dout.view(torch.int16), non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_steps(max(W, 3))
        stream.synchronize()
        barrier()
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_ev.record()
        e2e_steps(K)
        e_ev.record()
        stream.synchronize()
    e2e_ms = max_over_ranks(s_ev.elapsed_time(e_ev), world, dev)
    e2e_us = e2e_ms * 1000.0 / (K * world)
    h2d = T * SHAPE.H * 2 + T * SHAPE.topk * 8
    d2h = T * SHAPE.H * 2

    rows = {}
    if not args.no_rows and rank == 0:
        rows = secondary_rows(torch, m, lib, dev, copies, capture, time_graph, peaks, distinct, dev_batch,
                              set(args.rows.split(",")), args.prefill_tokens)

    cpu = None
    if rank == 0 and not args.no_cpu:
        n = 2
        vals = [oracle_sample(*host_batch(1000 + i, 1), (w13_h, s13_h, w2_h, s2_h), n)[1] for i in range(2)]
        cpu = cpu_baseline_entry(statistics.mean(vals), n)

    if rank != 0:
        return
    traffic = committed_traffic()
    line = {
        "metric": METRIC, "value": round(us_per_call, 2), "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(us_per_call / 1000.0, 5), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 mma operands, f32 accumulate, bf16 out", "data": "synthetic",
        "config": workload_config(args.copies),
        "weight_stream_TBps": round(layer_gbs / 1000.0, 3),
        "hbm_frac_layer": round(layer_gbs / peaks["hbm_gbs"], 3),
        "roofline": {"bound": "hbm",
                     "kernel": "decode_fused gate_up+down (mxfp4)" if fused else "decode_gemm gate_up (mxfp4)",
                     "achieved": round(g1_gbs, 1),
                     "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(g1_gbs / peaks["hbm_gbs"], 3),
                     "traffic": traffic if fused else None, "peak_source": peaks["source"],
                     "algorithmic_bytes": ("distinct active experts x 17,547,264 B (w13 + w2 + E8M0 scales) "
                                           "per launch" if fused else
                                           "distinct active experts x 11,698,176 B (w13 + E8M0 scales) per launch")},
        "kernels_us": {k: round(v, 2) for k, v in kavg.items()},
        "gpu_launches": launches_per_step * K,
        "e2e": {"value": round(e2e_us, 2), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "clocks": clocks, "status": status, "wall_s": round(wall, 4),
        "cpu_baseline": cpu, "rows": rows,
    }
    print(json.dumps(line), flush=True)


def prefill_row(torch, m, dev, copies, peaks, dev_batch, prefill_tokens, kind="mxfp4", opts=None, label=None):
    """Tensor-core (prefill) path: skewed routing, median of 4 timed calls."""
    opts = opts or {}
    rows = {}
    T = prefill_tokens
    pb = [dev_batch(T, 2000 + i, bias=2.0) for i in range(2)]
    d = m.dims(SHAPE.E, SHAPE.H, SHAPE.I, SHAPE.topk, T, m.MOE_PATH_PREFILL)
    ws = torch.empty(m.moe_workspace_bytes(d), dtype=torch.uint8, device=dev)
    out = torch.empty((T, SHAPE.H), dtype=torch.bfloat16, device=dev)
    flops = 2.0 * T * SHAPE.topk * 3 * SHAPE.H * SHAPE.I
    ms_list = []
    s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    kev = [torch.cuda.Event(enable_timing=True) for _ in range(12)]
    for ev in kev:
        ev.record()
    lib = m._native.load()
    for i in range(6):
        x, ids, w, _ = pb[i % 2]
        if i == 5:  # per-kernel times of the last call
            arr = (ctypes.c_void_p * 12)(*[ev.cuda_event for ev in kev])
            m._native.check("moe_set_timing_events", lib.moe_set_timing_events(arr, 6))
        s_ev.record()
        fn = m.moe_a16w4_mxfp4 if kind == "mxfp4" else m.moe_a16w4_int4g32
        fn(x, ids, w, *copies[i % len(copies)], out=out, workspace=ws, path=m.MOE_PATH_PREFILL, **opts)
        e_ev.record()
        e_ev.synchronize()
        if i >= 2:
            ms_list.append(s_ev.elapsed_time(e_ev))
    ms = statistics.median(ms_list)
    tf = flops / (ms * 1e-3) / 1e12
    names = ["route", "gather", "gemm1_gate_up_tc", "convert_f16", "gemm2_down_tc", "cast"]
    kms = {n: round(kev[2 * q].elapsed_time(kev[2 * q + 1]), 3) for q, n in enumerate(names)}
    rows[label or f"{'mxfp4' if kind == 'mxfp4' else 'int4g32'}_prefill_T{T}_skewed"] = {
        "ms_per_call": round(ms, 3), "TFLOPs_useful": round(tf, 1), "kernels_ms": kms,
        "bf16_frac_burst": round(tf / peaks["bf16_tflops"], 3),
        "bf16_frac_sustained": round(tf / (peaks["bf16_tflops_sustained"] or peaks["bf16_tflops"]), 3),
        "useful_flops": flops}
    del ws, out
    torch.cuda.empty_cache()
    return rows


def secondary_rows(torch, m, lib, dev, copies, capture, time_graph, peaks, distinct, dev_batch, which,
                   prefill_tokens):
    rows = {}
    reps = 10
    if "prefill" in which:
        rows.update(prefill_row(torch, m, dev, copies, peaks, dev_batch, prefill_tokens))
    # decode sweep
    sweep = {}
    for T in ((4, 7, 16, 32) if "sweep" in which else ()):
        g, _, nbytes, _ = capture(T, 8)
        time_graph(g, 2)
        ms = time_graph(g, reps) / reps
        us = ms * 1000 / 8
        gbs = nbytes / (ms * 1e-3) / 1e9
        sweep[f"T{T}"] = {"us_per_call": round(us, 2), "GBps": round(gbs, 1), "hbm_frac": round(gbs / peaks["hbm_gbs"], 3)}
    if sweep:
        rows["mxfp4_decode_sweep"] = sweep
    if "actquant" in which:
        # quantised activations (W4A8: static FP8 scales sized for x ~ N(0, 1);
        # W4A4: MXFP4), same weights and batches as the A16W4 lines
        schemes = {"w4a8_fp8": {"act_quant": "fp8", "w13_input_scale": 0.02, "w2_input_scale": 0.004},
                   "w4a4_mxfp4": {"act_quant": "mxfp4"}}
        aq = {}
        for name, opts in schemes.items():
            for T in (1, 32):
                g, _, nbytes, _ = capture(T, 8, opts=opts)
                time_graph(g, 2)
                ms = time_graph(g, reps) / reps
                gbs = nbytes / (ms * 1e-3) / 1e9
                aq[f"{name}_T{T}"] = {"us_per_call": round(ms * 1000 / 8, 2), "GBps": round(gbs, 1),
                                      "hbm_frac": round(gbs / peaks["hbm_gbs"], 3)}
            if "prefill" in which:
                rows.update(prefill_row(torch, m, dev, copies, peaks, dev_batch, prefill_tokens, opts=opts,
                                        label=f"mxfp4_{name}_prefill_T{prefill_tokens}_skewed"))
        rows["mxfp4_act_quant_decode"] = aq
        # the quantiser as a call, on the prefill intermediate's shape (T=4096
        # x top-15 rows of I floats, > L2): HBM-bound, bytes = input + codes
        nrows = prefill_tokens * SHAPE.topk
        xa = torch.randn((nrows, SHAPE.I), dtype=torch.float32, device=dev)
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        qa = {}
        for name, (mode, per_val) in {"mxfp4": ("mxfp4", 0.5 + 1 / 32), "fp8": ("fp8", 1.0)}.items():
            tl = []
            m.moe_quantize_act(xa, mode, 0.02)  # warm-up
            for i in range(4):
                # ten calls back to back: the binding's host work (output
                # allocation, the call) overlaps the previous kernels
                s_ev.record()
                for _ in range(10):
                    m.moe_quantize_act(xa, mode, 0.02)
                e_ev.record()
                e_ev.synchronize()
                tl.append(s_ev.elapsed_time(e_ev) / 10)
            ms = statistics.median(tl)
            nb = nrows * SHAPE.I * (4 + per_val)
            qa[name] = {"ms": round(ms, 4), "GBps": round(nb / (ms * 1e-3) / 1e9, 1),
                        "hbm_frac": round(nb / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 3), "bytes": int(nb),
                        "rows": nrows, "K": SHAPE.I, "src": "float32"}
        rows["moe_quantize_act"] = qa
        del xa
        torch.cuda.empty_cache()
    if not ({"requant", "int4"} & which):
        return rows
    # requantiser over all experts (w13 and w2), then the int4 MoE
    q_copies = []
    s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    req_ms = []
    for c in range(len(copies)):
        w13, s13, w2, s2 = copies[c]
        # outputs allocated before the timed region (an allocation inside it
        # would time the allocator, not the kernel)
        q13, q2 = torch.empty_like(w13), torch.empty_like(w2)
        f13 = torch.empty(s13.shape, dtype=torch.float32, device=dev)
        f2 = torch.empty(s2.shape, dtype=torch.float32, device=dev)
        torch.cuda.synchronize()
        s_ev.record()
        m.requant_mxfp4_to_int4g32(w13, s13, q13, f13, experts_per_chunk=8)
        m.requant_mxfp4_to_int4g32(w2, s2, q2, f2, experts_per_chunk=8)
        e_ev.record()
        e_ev.synchronize()
        req_ms.append(s_ev.elapsed_time(e_ev))
        q_copies.append((q13, f13, q2, f2))
    rms = statistics.median(req_ms[1:] or req_ms)
    rbytes = SHAPE.E * (W13_BYTES + W2_BYTES) + SHAPE.E * (2 * SHAPE.I * SHAPE.H // 2 + 2 * SHAPE.I * SHAPE.H // 8
                                                          + SHAPE.H * SHAPE.I // 2 + SHAPE.H * SHAPE.I // 8)
    rows["requant_112_experts"] = {"ms": round(rms, 3), "GBps": round(rbytes / (rms * 1e-3) / 1e9, 1),
                                   "hbm_frac": round(rbytes / (rms * 1e-3) / 1e9 / peaks["hbm_gbs"], 3),
                                   "bytes": rbytes, "experts_per_chunk": 8}
    i4 = {}
    i4_bytes = 2 * SHAPE.I * SHAPE.H // 2 + 2 * SHAPE.I * SHAPE.H // 8 + SHAPE.H * SHAPE.I // 2 + SHAPE.H * SHAPE.I // 8
    for T in (1, 7, 32):
        g, _, nbytes, _ = capture(T, 8, kind="int4", weights=q_copies)
        nbytes = nbytes // (W13_BYTES + W2_BYTES) * i4_bytes
        time_graph(g, 2)
        ms = time_graph(g, reps) / reps
        gbs = nbytes / (ms * 1e-3) / 1e9
        i4[f"T{T}"] = {"us_per_call": round(ms * 1000 / 8, 2), "GBps": round(gbs, 1),
                       "hbm_frac": round(gbs / peaks["hbm_gbs"], 3)}
    rows["int4g32_decode"] = i4
    if "prefill" in which:
        rows.update(prefill_row(torch, m, dev, q_copies, peaks, dev_batch, prefill_tokens, kind="int4"))
    del q_copies
    torch.cuda.empty_cache()
    # the same with bfloat16 group scales (half the scale bytes)
    b_copies, breq_ms = [], []
    for c in range(len(copies)):
        w13, s13, w2, s2 = copies[c]
        q13, q2 = torch.empty_like(w13), torch.empty_like(w2)
        b13 = torch.empty(s13.shape, dtype=torch.bfloat16, device=dev)
        b2 = torch.empty(s2.shape, dtype=torch.bfloat16, device=dev)
        torch.cuda.synchronize()
        s_ev.record()
        m.requant_mxfp4_to_int4g32(w13, s13, q13, b13, experts_per_chunk=8, scale_dtype=torch.bfloat16)
        m.requant_mxfp4_to_int4g32(w2, s2, q2, b2, experts_per_chunk=8, scale_dtype=torch.bfloat16)
        e_ev.record()
        e_ev.synchronize()
        breq_ms.append(s_ev.elapsed_time(e_ev))
        b_copies.append((q13, b13, q2, b2))
    bms = statistics.median(breq_ms[1:] or breq_ms)
    bbytes = rbytes - SHAPE.E * (2 * SHAPE.I * SHAPE.H // 16 + SHAPE.H * SHAPE.I // 16)
    rows["requant_112_experts_bf16_scales"] = {"ms": round(bms, 3), "GBps": round(bbytes / (bms * 1e-3) / 1e9, 1),
                                               "hbm_frac": round(bbytes / (bms * 1e-3) / 1e9 / peaks["hbm_gbs"], 3),
                                               "bytes": bbytes, "experts_per_chunk": 8}
    ib = {}
    ib_bytes = 2 * SHAPE.I * SHAPE.H // 2 + 2 * SHAPE.I * SHAPE.H // 16 + SHAPE.H * SHAPE.I // 2 + SHAPE.H * SHAPE.I // 16
    for T in (1, 7, 32):
        g, _, nbytes, _ = capture(T, 8, kind="int4", weights=b_copies)
        nbytes = nbytes // (W13_BYTES + W2_BYTES) * ib_bytes
        time_graph(g, 2)
        ms = time_graph(g, reps) / reps
        gbs = nbytes / (ms * 1e-3) / 1e9
        ib[f"T{T}"] = {"us_per_call": round(ms * 1000 / 8, 2), "GBps": round(gbs, 1),
                       "hbm_frac": round(gbs / peaks["hbm_gbs"], 3)}
    rows["int4g32_bf16_scales_decode"] = ib
    if "prefill" in which:
        rows.update(prefill_row(torch, m, dev, b_copies, peaks, dev_batch, prefill_tokens, kind="int4",
                                label=f"int4g32_bf16_scales_prefill_T{prefill_tokens}_skewed"))
    del b_copies
    torch.cuda.empty_cache()
    return rows


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest ``value`` over all ranks (the slowest replica sets the job time)."""
    if world <= 1:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1:
        import torch

        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        torch.distributed.init_process_group(backend=backend)
    try:
        if args.impl == "reference":
            run_reference(args, rank)
        else:
            run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch

            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

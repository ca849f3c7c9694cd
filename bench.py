"""Benchmark: W4A16 weight-stream GB/s at M=1 and TFLOP/s at M=4096 on B300.

Workload (Qwen2.5-32B-shaped, INT4 asymmetric, group 128, bf16 activations):
the four linears of one decoder layer -- qkv 5120->7168, o 5120->5120,
gate_up 5120->55296, down 27648->5120 -- stacked 64 times.

* decode step (the headline ``value``): one token (M=1) through all 64 x 4
  linears, i.e. 256 launches of the split-K decode kernel that together stream
  the stack's 16.21 GB of packed weights, scales and zeros.  Timed as CUDA-graph
  replays with CUDA events; value = weight bytes / time (GB/s).
* prefill step (``prefill``): M=4096 tokens through one layer's 4 linears on the
  tcgen05 kernel (a different layer each step); TFLOP/s = 2*M*N*K / time.

Every input is synthetic and seeded: weights W ~ N(0, 0.02) drawn by the
shared generators, quantized on the GPU by the library's round-to-nearest
kernel; the 64 layers are 64 distinct device copies of those four quantized
linears (16.2 GB, far larger than the 126 MB L2, so no L2 flush is needed).

* config sweep (``sweep``): every workload's shapes and token counts (single
  linear, decode sweep, act-order, Qwen shapes, NF4), each timed alone as a
  CUDA graph rotating through weight copies that exceed 4x L2; us per call,
  GB/s of algorithmic weight bytes, TFLOP/s and both roofline fractions.

``--impl reference`` times the CPU oracle instead (dequantize + fp64 product)
on a bounded sample of the same workload on the host cores.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

LINEARS = (("qkv", 5120, 7168), ("o", 5120, 5120), ("gate_up", 5120, 55296), ("down", 27648, 5120))
LAYERS = 64
GROUP = 128
M_PREFILL = 4096
METRIC = "W4A16 M=1 weight-stream GB/s (Qwen2.5-32B-shaped 64-layer INT4 g128 stack)"


def int4_bytes(K, N):
    G = K // GROUP
    return K * N // 2 + G * N * 2 + G * N // 2


STACK_BYTES = LAYERS * sum(int4_bytes(K, N) for _, K, N in LINEARS)
# the decode step's activations and outputs: X [1, K] read and Y [1, N]
# written once per launch, 16-bit
STACK_XY_BYTES = LAYERS * sum(2 * (K + N) for _, K, N in LINEARS)
LAYER_FLOPS = sum(2 * M_PREFILL * K * N for _, K, N in LINEARS)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    return 6400.0, 1800.0, 1400.0, "fallback"


# ------------------------------------------------------------------ clocks
_REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons during a timed region."""

    def __init__(self, index=0, path=None):
        self.index = index
        self.proc = None
        # the raw samples: a kept file when a path is given, else a temporary one
        self.path = path or os.path.join(tempfile.gettempdir(), f"w4a16_clocks_{os.getpid()}.csv")

    def __enter__(self):
        os.makedirs(os.path.dirname(os.path.abspath(self.path)), exist_ok=True)
        q = "clocks.sm,clocks.max.sm,power.draw," + ",".join("clocks_event_reasons." + r for r in _REASONS)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            self.proc.wait()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], [], set()
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 3 + len(_REASONS):
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for name, v in zip(_REASONS, f[3:]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------- CPU oracle
# The oracle (dequantize + fp64 product), as it stands, on every host core:
# the output columns are cut into one slab per core and each slab runs in its
# own process (started with `spawn`, before this process touches the GPU), one
# BLAS thread each.
ORACLE_K, ORACLE_N = 5120, 5120  # the o projection of the Qwen2.5-32B-shaped stack


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _oracle_slab(job):
    """Worker: quantize one column slab with the oracle, then repeat its
    dequantization and product for ``seconds``; returns (passes, seconds, bytes
    per pass, flops per pass)."""
    c0, c1, M, seconds = job
    from oracle import int4, product
    from synth import activations, gaussian_weights

    K = ORACLE_K
    W = gaussian_weights(K, ORACLE_N, 0.02, 0)[:, c0:c1]
    q, s, z = int4.rtn_quantize(W)
    X = activations(M, K, "bf16", 1).double().numpy()
    n = c1 - c0
    done, t0 = 0, time.perf_counter()
    while True:
        w_hat = int4.dequant(q, s, z, "bf16")
        wf = (w_hat.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        product.reference(X, wf)
        done += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return done, time.perf_counter() - t0, int4_bytes(K, n), 2 * M * n * K


def oracle_all_cores(seconds: float = 12.0, M: int = 1):
    """The oracle on the o projection (5120 x 5120) at M tokens, one column slab
    per host core, for about ``seconds``.  Returns (GB/s of packed weight bytes,
    TFLOP/s, cores, sample description)."""
    import multiprocessing as mp

    cores = host_cores()
    edges = [ORACLE_N * i // cores // 8 * 8 for i in range(cores)] + [ORACLE_N]
    jobs = [(edges[i], edges[i + 1], M, seconds) for i in range(cores) if edges[i + 1] > edges[i]]
    saved = {k: os.environ.get(k) for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
    for k in saved:
        os.environ[k] = "1"
    try:
        with mp.get_context("spawn").Pool(len(jobs)) as pool:
            res = pool.map(_oracle_slab, jobs)
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    # every slab ran for about the same wall time; the job's rate is the sum
    gbs = sum(d * b / t for d, t, b, _ in res) / 1e9
    tflops = sum(d * f / t for d, t, _, f in res) / 1e12
    passes = sum(d for d, _, _, _ in res)
    sample = (f"o_proj {ORACLE_K}x{ORACLE_N} INT4 g128 at M={M}: dequantize + fp64 product, {len(jobs)} column "
              f"slabs in parallel processes, {passes} slab passes in {seconds:.0f} s")
    return gbs, tflops, len(jobs), sample


def cpu_baselines(seconds: float):
    """Decode (M = 1) and prefill (M = 4096, timed on 64 rows and scaled by
    4096/64: the product's rows are independent) oracle rates on all cores."""
    v, _, cores, sample = oracle_all_cores(seconds, 1)
    _, tf64, _, sample64 = oracle_all_cores(max(2.0, seconds / 3), 64)
    return {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample,
            "prefill_tflops": round(tf64, 5),
            "prefill_sample": sample64 + "; M=4096 extrapolated from these 64 rows (time x 4096/64)"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    steps, warm = args.steps, args.warmup
    per = max(2.0, 60.0 / max(1, steps + warm))
    for _ in range(warm):
        oracle_all_cores(per / 2)
    vals = []
    t0 = time.perf_counter()
    for _ in range(steps):
        v, _, cores, sample = oracle_all_cores(per)
        vals.append(v)
    wall = time.perf_counter() - t0
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": warm, "ms_per_step": round(wall * 1e3 / steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "CPU oracle (RTN INT4 dequantize + fp64 product), bounded sample of the "
                               "Qwen2.5-32B-shaped decode stack", "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------- multi-rank (replicas)
def max_over_ranks(ms: float, dist, device) -> float:
    """The slowest rank's time: every rank runs its own replica of the
    workload, so the job takes as long as its slowest rank (no data-path
    exchange between ranks; this is the only collective)."""
    if dist is None:
        return ms
    import torch

    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(world: int, bytes_per_step: int, steps: int, max_ms: float) -> float:
    """Whole-job GB/s: the bytes every rank streamed over the slowest rank's time."""
    return world * bytes_per_step * steps / (max_ms * 1e-3) / 1e9


# ------------------------------------------------------------ config sweep
# The five workloads' shapes and token counts, each timed on its own (CUDA
# graph of calls that rotate through enough weight copies to exceed 4x L2).
SWEEP = (
    # (config, K, N, Ms, dtype, kind)
    ("C1 single linear", 4096, 4096, (16,), "f16", "int4"),
    ("C2 decode sweep qkv", 4096, 12288, (1, 4, 16), "bf16", "int4_salient"),
    ("C2 decode sweep o", 4096, 4096, (1, 4, 16), "bf16", "int4_salient"),
    ("C2 decode sweep gate_up", 4096, 22016, (1, 4, 16), "bf16", "int4_salient"),
    ("C2 decode sweep down", 11008, 4096, (1, 4, 16), "bf16", "int4_salient"),
    ("C3 act-order up", 8192, 28672, (1, 16, 64), "f16", "int4_act"),
    ("C3 act-order down", 28672, 8192, (1, 16, 64), "f16", "int4_act"),
    ("C4 Qwen qkv", 5120, 7168, (1, 256, 1024, 4096), "bf16", "int4"),
    ("C4 Qwen o", 5120, 5120, (1, 256, 1024, 4096), "bf16", "int4"),
    ("C4 Qwen gate_up", 5120, 55296, (1, 256, 1024, 4096), "bf16", "int4"),
    ("C4 Qwen down", 27648, 5120, (1, 256, 1024, 4096), "bf16", "int4"),
    ("C5 NF4", 8192, 8192, (1, 64, 1024), "bf16", "nf4"),
)
L2_BYTES = 126 * 2**20  # used when the device does not report its L2 size


def sweep_weights(torch, w4, K, N, kind, seed, dev):
    """Quantized weights of one linear, generated and quantized on the GPU:
    N(0, 0.02) (C2: 1% of the K rows x10; C3: 0.01 * Student-t(5), drawn as
    Z / sqrt(chi2_5 / 5) one column slab at a time; C3's g_idx is a seeded
    permutation of the rows into groups of 128)."""
    g = torch.Generator(device=dev).manual_seed(seed)
    if kind == "int4_act":
        W = torch.empty((K, N), dtype=torch.float32, device=dev)
        for c0 in range(0, N, 4096):
            c1 = min(N, c0 + 4096)
            z = torch.randn((K, c1 - c0), generator=g, device=dev)
            chi2 = sum(torch.randn((K, c1 - c0), generator=g, device=dev) ** 2 for _ in range(5))
            W[:, c0:c1] = 0.01 * z / torch.sqrt(chi2 / 5)
    else:
        W = torch.randn((K, N), generator=g, device=dev) * 0.02
        if kind == "int4_salient":
            rows = torch.randperm(K, generator=g, device=dev)[: round(0.01 * K)]
            W[rows] *= 10
    if kind == "nf4":
        qw, am = w4.nf4_quantize(W, w4.nf4_codebook(dev))
        return (qw, am), K * N // 2 + (K // 64) * N * 4
    qw, sc, qz = w4.quantize(W)
    nbytes = int4_bytes(K, N)
    if kind == "int4_act":
        perm = torch.randperm(K, generator=g, device=dev)
        gi = torch.empty(K, dtype=torch.int32, device=dev)
        gi[perm] = (torch.arange(K, device=dev) // GROUP).to(torch.int32)
        return (qw, sc, qz, gi), nbytes + 4 * K
    return (qw, sc, qz), nbytes


def sweep_entry(name, K, N, M, dt, us, nbytes, hbm_peak, tc_peak):
    """One timed configuration: weight bytes (codes and their group metadata)
    per second, the same with X read and Y written once (16-bit) included, and
    the product's FLOP rate, each against its roofline."""
    gbs = nbytes / us / 1e3
    tf = 2 * M * N * K / us / 1e6
    xy = 2 * M * (K + N)
    return {"config": name, "K": K, "N": N, "M": M, "dtype": dt, "us": round(us, 2), "GBs": round(gbs, 1),
            "GBs_incl_xy": round((nbytes + xy) / us / 1e3, 1), "TFLOPs": round(tf, 1),
            "hbm_frac": round(gbs / hbm_peak, 4), "tc_frac": round(tf / tc_peak, 4),
            "bound": "hbm" if M <= 16 else ("both" if M < 256 else "tensor")}


def sweep_summary(entries):
    """A short digest of the sweep for the bench line (the full entries are
    the sweep_entry JSON lines printed before it): how many entries, each
    configuration's M=1 fraction of the HBM peak, and its largest-M fraction
    of the tensor peak."""
    if not entries:
        return None
    m1, top = {}, {}
    for e in entries:
        name = f"{e['config']} {e['K']}x{e['N']} {e['dtype']}"
        if e["M"] == 1:
            m1[name] = round(e["hbm_frac"], 3)
        if name not in top or e["M"] > top[name][0]:
            top[name] = (e["M"], round(e["tc_frac"], 3))
    return {"entries": len(entries), "lines": "one sweep_entry JSON line per entry, before this line",
            "hbm_frac_at_M1": m1, "tc_frac_at_largest_M": {f"{k} M={v[0]}": v[1] for k, v in top.items() if v[0] > 16}}


def config_sweep(torch, w4, dev, hbm_peak, tc_peak):
    out = []
    # weight copies rotated through: more than 4x the device's L2 (queried)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or L2_BYTES
    for ci, (name, K, N, Ms, dt, kind) in enumerate(SWEEP):
        w, nbytes = sweep_weights(torch, w4, K, N, kind, 1000 + ci, dev)
        copies = max(2, -(-4 * l2 // nbytes))
        sets = [w] + [tuple(t.clone() for t in w) for _ in range(copies - 1)]
        cb = w4.nf4_codebook(dev) if kind == "nf4" else None
        tdt = torch.bfloat16 if dt == "bf16" else torch.float16
        # act-order runs twice: on the g_idx map as stored, and prepacked
        # (rows reordered by group once, before timing; X gathered per call)
        runs = [(name, kind, sets)]
        if kind == "int4_act":
            packed = []
            for t in sets:
                q_sorted, perm = w4.act_order_prepack(t[0], t[3])
                packed.append((q_sorted, t[1], t[2], perm))
            runs.append((name + " (prepacked)", "int4_prepacked", packed))
        for name, kind, sets, M in [(n, k, st, M) for (n, k, st) in runs for M in Ms]:
            X = torch.randn((M, K), device=dev).to(tdt)
            Y = torch.empty((M, N), dtype=tdt, device=dev)
            ws = w4.workspace(M, N, K, dev)
            pws = w4.workspace(M, N, K, dev, nbytes=w4.prepacked_workspace_bytes(M, N, K))
            # everything above was made on the default stream; the calls below
            # run on a side stream
            torch.cuda.synchronize()

            def call(i):
                t = sets[i % copies]
                if kind == "nf4":
                    w4.nf4_gemm(X, t[0], t[1], cb, out=Y, ws=ws)
                elif kind == "int4_prepacked":
                    w4.gemm_prepacked(X, t[0], t[1], t[2], t[3], out=Y, ws=pws)
                else:
                    w4.gemm(X, t[0], t[1], t[2], g_idx=t[3] if kind == "int4_act" else None, out=Y, ws=ws)

            reps = max(copies, 8 if M >= 1024 else 20)
            s = torch.cuda.Stream(dev)
            with torch.cuda.stream(s):
                for i in range(3):
                    call(i)
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr, stream=s):
                    for i in range(reps):
                        call(i)
            torch.cuda.synchronize()
            gr.replay()
            torch.cuda.synchronize()
            cur = torch.cuda.current_stream(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            n_rep = 3 if M >= 1024 else 5
            e0.record(cur)
            for _ in range(n_rep):
                gr.replay()
            e1.record(cur)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / (n_rep * reps)
            out.append(sweep_entry(name, K, N, M, dt, us, nbytes, hbm_peak, tc_peak))
            del gr, X, Y
        del sets, w, runs
        torch.cuda.empty_cache()
    return out


# ------------------------------------------------------------------- GPU
# the decode kernel's complete source: the ncu traffic figure in profiles/ is
# used only while these files are unchanged since the capture
DECODE_SOURCES = ("gemv_ws.cu", "gemv_common.cuh", "dq_common.cuh", "sm100.cuh")


def decode_source_sha256() -> str:
    import hashlib

    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        h.update(open(os.path.join(ROOT, "bit_weight_only_wise_b300", "csrc", f), "rb").read())
    return h.hexdigest()


def traffic_from_profiles(kernel: str):
    """dram read+write bytes per launch from the committed ncu summary, if it
    was taken on the current source of the kernel; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    ent = json.load(open(p)).get(kernel)
    if not ent or ent.get("source_sha256") != decode_source_sha256():
        return None
    return ent


def run_gpu(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    # the CPU baseline runs first: its worker processes start before this
    # process makes any CUDA call
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baselines(args.cpu_seconds)

    import torch

    import bit_weight_only_wise_b300 as w4
    from synth import activations, gaussian_weights

    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    hbm_peak, tc_peak, tc_sustained, peak_src = load_peaks()

    # ---- weights: four linears quantized on the GPU, 64 distinct copies
    base = []
    for i, (name, K, N) in enumerate(LINEARS):
        W = torch.from_numpy(gaussian_weights(K, N, 0.02, 100 + i)).to(dev)
        base.append(w4.quantize(W))
        del W
    torch.cuda.synchronize()
    stack = [[tuple(t.clone() for t in base[i]) for i in range(4)] for _ in range(LAYERS)]
    del base
    torch.cuda.synchronize()

    # ---- decode (M = 1): 256 launches per step, captured once in a graph
    xs = [activations(1, K, "bf16", 7 + i).to(dev) for i, (_, K, _) in enumerate(LINEARS)]
    ys = [torch.empty((1, N), dtype=torch.bfloat16, device=dev) for (_, _, N) in LINEARS]
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))  # the inputs were made on the default stream
    with torch.cuda.stream(s):
        wss = [w4.workspace(1, N, K, dev) for (_, K, N) in LINEARS]
        ws = max(wss, key=lambda t: -1 if t is None else t.numel())

        def decode_step():
            for layer in stack:
                for i in range(4):
                    w4.gemv(xs[i], *layer[i], out=ys[i], ws=ws)

        decode_step()  # attribute setup, first-call work
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            decode_step()
    torch.cuda.synchronize()

    def timed(fn, steps, warm, stream):
        for _ in range(warm):
            fn()
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        return max_over_ranks(e0.elapsed_time(e1), dist, dev)

    cur = torch.cuda.current_stream(dev)
    with ClockSampler(local, args.clock_log) as clk:
        dec_ms = timed(g.replay, args.steps, args.warmup, cur)
    clocks = clk.summary()
    dec_step_ms = dec_ms / args.steps
    value = aggregate_gbs(world, STACK_BYTES, args.steps, dec_ms)
    per_gpu = STACK_BYTES / (dec_step_ms * 1e-3) / 1e9
    launches = args.steps * LAYERS * 4

    # ---- e2e: through the API call by call, X from pinned host memory each
    # step and every output read back
    xh = [x.cpu().pin_memory() for x in xs]
    yh = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in ys]
    h2d = sum(x.numel() * x.element_size() for x in xh)
    d2h = sum(y.numel() * y.element_size() for y in yh)

    # the stack's 256 products as one list, launched by one library call
    # (w4a16_gemv_batch) per step
    with torch.cuda.stream(s):
        batch = w4.GemvBatch([(xs[i], *layer[i], ys[i]) for layer in stack for i in range(4)], ws=ws)

    def e2e_step():
        for i in range(4):
            xs[i].copy_(xh[i], non_blocking=True)
        batch()
        for i in range(4):
            yh[i].copy_(ys[i], non_blocking=True)

    e2e_steps = max(3, min(args.steps, 20))
    with torch.cuda.stream(s):
        e2e_ms = timed(e2e_step, e2e_steps, max(args.warmup, 3), s)
    e2e_val = world * STACK_BYTES * e2e_steps / (e2e_ms * 1e-3) / 1e9

    # ---- prefill (M = 4096): one layer's four linears per step
    xp = [activations(M_PREFILL, K, "bf16", 11 + i).to(dev) for i, (_, K, _) in enumerate(LINEARS)]
    yp = [torch.empty((M_PREFILL, N), dtype=torch.bfloat16, device=dev) for (_, _, N) in LINEARS]
    pre_state = {"layer": 0}
    lin_ms = [0.0] * 4

    def prefill_step(record=False):
        layer = stack[pre_state["layer"] % LAYERS]
        pre_state["layer"] += 1
        for i in range(4):
            w4.gemm(xp[i], *layer[i], out=yp[i])

    # gate_up timed alone first (the GPU idle before it): the burst peak applies
    torch.cuda.synchronize()
    time.sleep(0.5)
    gate_layer = stack[0][2]
    for _ in range(2):
        w4.gemm(xp[2], *gate_layer, out=yp[2])
    torch.cuda.synchronize()
    b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    b0.record(cur)
    for _ in range(3):
        w4.gemm(xp[2], *gate_layer, out=yp[2])
    b1.record(cur)
    torch.cuda.synchronize()
    gate_burst = 2 * M_PREFILL * 5120 * 55296 / (b0.elapsed_time(b1) / 3 * 1e-3) / 1e12

    pre_steps = max(3, min(args.steps, 20))
    pre_ms = timed(prefill_step, pre_steps, max(args.warmup, 3), cur)
    tflops = world * LAYER_FLOPS * pre_steps / (pre_ms * 1e-3) / 1e12
    # per-linear times (events around each linear, for the roofline of the kernel)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(4)]
    torch.cuda.synchronize()
    for rep in range(3):
        layer = stack[(rep * 7) % LAYERS]
        for i in range(4):
            evs[i][0].record(cur)
            w4.gemm(xp[i], *layer[i], out=yp[i])
            evs[i][1].record(cur)
        torch.cuda.synchronize()
        for i in range(4):
            lin_ms[i] += evs[i][0].elapsed_time(evs[i][1]) / 3
    gate = 2 * M_PREFILL * 5120 * 55296 / (lin_ms[2] * 1e-3) / 1e12

    if rank != 0:
        if dist:
            dist.destroy_process_group()
        return 0

    sweep = None if args.no_sweep else config_sweep(torch, w4, dev, hbm_peak, tc_peak)
    if sweep:
        # one line per timed configuration ahead of the bench line (for the log)
        for e in sweep:
            print(json.dumps({"sweep_entry": e}), flush=True)

    traffic = traffic_from_profiles("gemv_ws_kernel")
    achieved = per_gpu  # algorithmic bytes per launch / mean launch time == stack bytes / step time
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(dec_step_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,0.02) weights, RTN INT4 g128 on the GPU; N(0,1) bf16 activations)",
        "config": {
            "workload": "Qwen2.5-32B-shaped decode: M=1 through 64 layers x {qkv 5120x7168, o 5120x5120, "
                        "gate_up 5120x55296, down 27648x5120}, INT4 asymmetric g128, bf16 X/Y",
            "stack_bytes": STACK_BYTES,
            "launches_per_step": LAYERS * 4,
            "timing": "CUDA graph replay of the 256 launches, CUDA events; inputs (16.2 GB) larger than L2",
            "parallelism": f"replicas x{world}",
        },
        "roofline": {
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "achieved_incl_xy": round(achieved * (STACK_BYTES + STACK_XY_BYTES) / STACK_BYTES, 1),
            "peak": hbm_peak,
            "unit": "GB/s",
            "frac": round(achieved / hbm_peak, 4),
            "peak_source": peak_src,
            "traffic": None if traffic is None else traffic.get("bytes_per_launch"),
            "kernel": "gemv_ws_kernel (warp-specialized split-K decode)",
            "algorithmic_bytes_per_launch": STACK_BYTES // (LAYERS * 4),
        },
        "prefill": {
            "metric": "W4A16 M=4096 TFLOP/s (one Qwen2.5-32B-shaped layer, 4 linears)",
            "value": round(tflops, 1),
            "unit": "TFLOP/s",
            "ms_per_step": round(pre_ms / pre_steps, 3),
            "per_linear_ms": {n: round(t, 4) for (n, _, _), t in zip(LINEARS, lin_ms)},
            # gate_up timed right after the long prefill loop: a kernel inside a
            # long step, so the sustained (power-capped) peak is the denominator
            "roofline": {"bound": "tensor", "achieved": round(gate, 1),
                         "peak": tc_sustained if tc_sustained else tc_peak, "unit": "TFLOP/s",
                         "peak_kind": "sustained" if tc_sustained else "burst",
                         "frac": round(gate / (tc_sustained if tc_sustained else tc_peak), 4),
                         "frac_of_burst": round(gate / tc_peak, 4), "peak_source": peak_src,
                         "kernel": "gemm_tc_kernel on gate_up 5120x55296, inside the prefill loop"},
            "burst": {"achieved": round(gate_burst, 1), "peak": tc_peak, "unit": "TFLOP/s",
                      "frac": round(gate_burst / tc_peak, 4),
                      "how": "gate_up 5120x55296 at M=4096 timed alone (3 calls after an idle pause), "
                             "before the prefill loop"},
            "layer_frac_of_peak": round(tflops / world / tc_peak, 4),
        },
        "e2e": {"value": round(e2e_val, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "per step: pinned-host X -> device, one w4a16_gemv_batch call (the stack's 256 "
                       "products) through the Python binding, outputs -> pinned host"},
        "sweep": sweep_summary(sweep),
        "gpu_launches": launches,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="skip the per-config timing sweep")
    ap.add_argument("--clock-log", default=None, help="keep the raw nvidia-smi clock samples in this CSV file")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())

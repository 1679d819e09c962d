"""Benchmark: invariant GEMM TFLOP/s (headline) and selected-token logprob
tokens/s on one GB300, with roofline fractions, the float64 oracle timed on
the host cores, and an end-to-end number through the C ABI with host buffers.

Step (the timed unit): the three dense projection GEMMs of an 8B-class
decoder at M = 4096 tokens -- (K, N) in {(4096, 4096), (4096, 12288),
(12288, 4096)} -- through iso_gemm with an 8-leaf contract.  Inputs are
resident in HBM; L2 is flushed before every step, outside the per-step
CUDA-event window: a 256 MiB write evicts every input line, then a 256 MiB
read of another buffer writes the dirty lines back, so the step starts with
neither its inputs nor dirty data in the 129 MB L2.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same step on its own batch (data
parallel replicas, no collective on the data path; weak scaling); timing is
the max over ranks.  ``--impl reference`` times the float64 CPU oracle (the
only reference implementation this project has) on a bounded sample of the
same workload on rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

SHAPES = [(4096, 4096), (4096, 12288), (12288, 4096)]  # (K, N)
M_TOKENS = 4096
LEAVES = 8
# row chunks of each shape in the end-to-end pipeline, in order.  Measured on GB300: equal chunks
# 1 -> 705, 2 -> 762-781, 4 -> 735, 8 -> 555 TFLOP/s; smaller first and last chunks (1024 or 512
# rows) 702-758.
E2E_SPLITS = [[2048, 2048], [2048, 2048], [2048, 2048]]
METRIC = "invariant GEMM TFLOP/s & logprob tokens/s on 1 GB300; % of roofline; bitwise checks"
WORKLOAD = ("dense projection GEMMs of an 8B-class decoder: M=4096 tokens, (K,N) in "
            "{(4096,4096),(4096,12288),(12288,4096)}, bf16 in / fp32 accumulate / bf16 out, 8 contiguous K-leaves, "
            "balanced-tree combine")
LP_T, LP_H, LP_V = 4096, 4096, 151936


def bench_config(world):
    """The workload description both arms print (the same keys and values)."""
    return dict(workload=WORKLOAD, global_batch=M_TOKENS * world, parallelism=f"replicas{world}",
                l2="flushed before every step (256 MiB write, then a 256 MiB read of another buffer so L2 holds no "
                   "dirty lines; outside the event window)", leaves=LEAVES)


def rnd(x, sig=5):
    """Round every float of a nested structure to `sig` significant digits (a short JSON line)."""
    if isinstance(x, float):
        return float(f"{x:.{sig}g}")
    if isinstance(x, dict):
        return {k: rnd(v, sig) for k, v in x.items()}
    if isinstance(x, (list, tuple)):
        return [rnd(v, sig) for v in x]
    return x


def step_flops(M=M_TOKENS):
    return sum(2.0 * M * K * N for K, N in SHAPES)


def max_over_ranks(x: float, world: int, device) -> float:
    """Max of a per-rank scalar over all ranks (the job's time is its slowest rank)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, units_per_rank: float, ms_max: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return world * units_per_rank / (ms_max * 1e-3)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), tc=float(d["bf16_tflops"]), tc_sus=float(d["bf16_tflops_sustained"]),
                    src="measured")
    return dict(hbm=6800.0, tc=1900.0, tc_sus=1700.0, src="fallback")


# the sources whose change invalidates committed traffic figures: the GEMM engine and the host
# code that picks its schedule (pairs, stage depth, raster groups)
ENGINE_SOURCES = ("gemm_tcgen05.cu", "iso_ptx.cuh", "iso_internal.h", "capi.cu")


def kernel_source_hash():
    """Hash of the engine sources' code: comments and blank lines do not count (no string
    literal in these files holds a comment marker), so a comment edit keeps the figures."""
    h = hashlib.sha256()
    for f in ENGINE_SOURCES:
        text = open(os.path.join(ROOT, "parallelism_invariant_logprob_gb300", "csrc", f)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for line in text.splitlines():
            code = line.split("//", 1)[0].rstrip()
            if code:
                h.update(code.encode() + b"\n")
    return h.hexdigest()[:16]


def committed_traffic(kernel_key):
    """DRAM bytes per launch from a committed ncu summary, only if the kernel
    source has not changed since it was captured."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(kernel_key)
    if not d or d.get("source_hash") != kernel_source_hash():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 8:
                self.rows.append(parts)

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["nvidia-smi unavailable"])
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm = [float(r[0]) for r in self.rows if r[0].replace(".", "").isdigit()]
        mx = [float(r[1]) for r in self.rows if r[1].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in self.rows for i in range(4) if r[4 + i].lower() == "active"})
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return dict(sm_mhz=statistics.median(loaded) if loaded else None, sm_max_mhz=max(mx) if mx else None,
                    reasons=reasons, samples=len(self.rows))


# ----------------------------------------------------------------- CPU oracle
def oracle_gemm_sample(rows, seed=1):
    """Time the oracle on `rows` rows of each projection; returns (flops, seconds, cores)."""
    import numpy as np
    import torch
    import oracle
    from parallelism_invariant_logprob_gb300 import inputs
    oracle._load()
    flops, secs = 0.0, 0.0
    for K, N in SHAPES:
        A, Bm = inputs.gemm_inputs(rows, K, N, seed=seed)
        Ab = A.view(torch.int16).numpy().view(np.uint16)
        Bb = Bm.view(torch.int16).numpy().view(np.uint16)
        t0 = time.perf_counter()
        oracle.gemm_root(Ab, Bb, LEAVES)
        secs += time.perf_counter() - t0
        flops += 2.0 * rows * K * N
    return flops, secs, os.cpu_count() or 1


def cpu_baseline(target_s=10.0):
    f, s, cores = oracle_gemm_sample(4)
    rows = max(4, min(512, int(4 * target_s / max(s, 1e-3))))
    f, s, cores = oracle_gemm_sample(rows)
    return dict(value=f / s / 1e12, unit="TFLOP/s", cores=cores, kind="oracle",
                sample=f"float64 oracle (leaf tree, 8 leaves) on {rows} rows of each of the 3 projection shapes "
                       f"(full K and N), {s:.1f} s; value = flops / time")


def run_reference(args, rank, world):
    if rank != 0:
        return
    times, vals = [], []
    rows = None
    for i in range(args.warmup + args.steps):
        if rows is None:
            f, s, cores = oracle_gemm_sample(4)
            rows = max(4, min(256, int(4 * 6.0 / max(s, 1e-3))))
        f, s, cores = oracle_gemm_sample(rows)
        if i >= args.warmup:
            times.append(s)
            vals.append(f / s / 1e12)
    v = statistics.mean(vals)
    sample = (f"float64 oracle on {rows} of the {M_TOKENS} rows of each projection per step (full K, N); "
              f"value = flops of that sample / its time")
    line = dict(impl="reference", metric=METRIC, value=v, unit="TFLOP/s", n_gpus=world, steps=args.steps,
                warmup=args.warmup, ms_per_step=1e3 * statistics.mean(times), higher_is_better=True,
                scaling="weak", vs_baseline=None, dtype="f64", data="synthetic",
                config=bench_config(world),
                cpu_baseline=dict(value=v, unit="TFLOP/s", cores=os.cpu_count() or 1, kind="oracle", sample=sample),
                e2e=dict(value=v, unit="TFLOP/s", h2d_bytes_per_step=0, d2h_bytes_per_step=0))
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- GPU arm
def run_ours(args, rank, world):
    import torch
    import torch.distributed as dist
    from parallelism_invariant_logprob_gb300 import binding as B
    from parallelism_invariant_logprob_gb300 import inputs

    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    c = B.Contract(LEAVES)
    stream = torch.cuda.current_stream()
    peaks = load_peaks()

    # resident inputs (one batch per rank)
    Xs, Ws, Cs = [], [], []
    for i, (K, N) in enumerate(SHAPES):
        X, W = inputs.gemm_inputs(M_TOKENS, K, N, seed=100 + 10 * rank + i, device=dev)
        Xs.append(X)
        Ws.append(W)
        Cs.append(torch.empty(M_TOKENS, N, dtype=torch.bfloat16, device=dev))
    flush = L2Flush(dev)

    def step(ev=None):
        for i in range(len(SHAPES)):
            if ev is not None:
                ev[i][0].record(stream)
            B.gemm(c, Xs[i], Ws[i], out=Cs[i], stream=stream)
            if ev is not None:
                ev[i][1].record(stream)

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    assert B.last_device_status(c) == B.ISO_OK

    per_step_ms, launch_ms = [], [[] for _ in SHAPES]
    sampler = ClockSampler(dev.index)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    wall0 = time.perf_counter()
    for _ in range(args.steps):
        flush()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in SHAPES]
        step(ev)
        torch.cuda.synchronize()
        per_step_ms.append(ev[0][0].elapsed_time(ev[-1][1]))
        for i in range(len(SHAPES)):
            launch_ms[i].append(ev[i][0].elapsed_time(ev[i][1]))
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    assert B.last_device_status(c) == B.ISO_OK

    ms = max_over_ranks(statistics.mean(per_step_ms), world, dev)
    value = job_throughput(world, step_flops(), ms) / 1e12

    # roofline of the dominant kernel (the leaf-tree GEMM): algorithmic flops / its launch time
    kern_s = sum(sum(l) for l in launch_ms) * 1e-3
    achieved = args.steps * step_flops() / kern_s / 1e12
    traffic = committed_traffic("iso_leaf_tree_gemm_kernel<EPI_BF16>/M4096")
    roofline = dict(bound="tensor", achieved=achieved, peak=peaks["tc"], unit="TFLOP/s", frac=achieved / peaks["tc"],
                    traffic=traffic, peak_kind=f"bf16 dense burst, {peaks['src']}",
                    per_shape_tflops={f"{K}x{N}": 2.0 * M_TOKENS * K * N / (statistics.mean(launch_ms[i]) * 1e-3) / 1e12
                                      for i, (K, N) in enumerate(SHAPES)})

    # end to end through the C ABI with host buffers: H2D of the step's activations, D2H of its
    # outputs, pipelined over three streams in the row chunks of E2E_SPLITS: the next
    # chunk's activations upload while the GEMM of the current chunk runs, and each chunk's
    # outputs download as soon as its GEMM is done, so both copy directions and the tensor cores
    # work at once and only the last chunk's GEMM and download follow the last upload.  A row's
    # bits do not depend on the rows launched with it, so the chunks give the same bits as one
    # launch per shape (checked below against the device-resident results).
    ref_c = [Cc.clone() for Cc in Cs]  # the device-resident results of the same inputs
    pinned_x = [X.cpu().pin_memory() for X in Xs]
    pinned_c = [torch.empty(Cc.shape, dtype=Cc.dtype, pin_memory=True) for Cc in Cs]
    h2d = sum(x.numel() * 2 for x in pinned_x)
    d2h = sum(x.numel() * 2 for x in pinned_c)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    e2e_ms = []
    for it in range(args.warmup + args.steps):
        flush()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in)
        for i in range(len(SHAPES)):
            r1 = 0
            for rows in E2E_SPLITS[i]:
                r0, r1 = r1, r1 + rows
                with torch.cuda.stream(s_in):
                    Xs[i][r0:r1].copy_(pinned_x[i][r0:r1], non_blocking=True)
                landed = torch.cuda.Event()
                landed.record(s_in)
                stream.wait_event(landed)
                B.gemm(c, Xs[i][r0:r1], Ws[i], out=Cs[i][r0:r1], stream=stream)
                done = torch.cuda.Event()
                done.record(stream)
                s_out.wait_event(done)
                with torch.cuda.stream(s_out):
                    pinned_c[i][r0:r1].copy_(Cs[i][r0:r1], non_blocking=True)
        s_out.wait_stream(s_in)
        e1.record(s_out)
        torch.cuda.synchronize()
        if it >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    for i in range(len(SHAPES)):  # what came back to the host is the device-resident result
        assert torch.equal(pinned_c[i].view(torch.int16), ref_c[i].cpu().view(torch.int16))
    e2e_t = max_over_ranks(statistics.mean(e2e_ms), world, dev)
    e2e = dict(value=job_throughput(world, step_flops(), e2e_t) / 1e12, unit="TFLOP/s", h2d_bytes_per_step=h2d,
               d2h_bytes_per_step=d2h)

    extra = {}
    if not args.skip_secondary:
        extra = secondary(c, dev, stream, peaks, rank)

    if rank == 0:
        config = bench_config(world)
        config["contract_digest"] = c.digest.hex()[:16]
        line = dict(metric=METRIC, value=value, unit="TFLOP/s", n_gpus=world, steps=args.steps, warmup=args.warmup,
                    ms_per_step=ms, higher_is_better=True, scaling="weak", vs_baseline=None, dtype="bf16",
                    data="synthetic", config=config, roofline=roofline, e2e=e2e, gpu_launches=args.steps * len(SHAPES),
                    clocks=clocks, wall_s_timed_region=wall)
        if world == 1 and not args.skip_cpu:
            line["cpu_baseline"] = cpu_baseline()
        if extra:
            if args.details:
                with open(args.details, "w") as f:
                    json.dump(extra, f, indent=1)
            line["secondary"] = secondary_summary(extra)
            bw = dict(extra["bitwise"])
            bw["e2e_host_results_vs_resident"] = 0  # asserted above: the host copies equal the resident results
            line["bitwise"] = dict(mismatching_elements_total=sum(bw.values()), checks=len(bw), detail=bw)
            line["logprob"] = logprob_summary(extra["logprob"])  # last: the end of the line is what logs keep
        print(json.dumps(rnd(line)), flush=True)


def secondary_summary(x):
    """The secondary measurements in a few keys (full figures: --details)."""
    g = x["gemm_sweep"]
    small = {f"M{M}_{K}x{N}": g[f"M{M}_K{K}_N{N}"]["ws_hbm_frac"] for K, N in SHAPES for M in (1, 64)}
    small_stream = {f"M{M}_{K}x{N}": g[f"M{M}_K{K}_N{N}"]["stream_hbm_frac"] for K, N in SHAPES for M in (1, 64)}
    at = x["attention"]
    return dict(gemm_small_m_hbm_frac=small, gemm_small_m_back_to_back_hbm_frac=small_stream,
                overhead_vs_cublas_M4096={f"{K}x{N}": g[f"M4096_K{K}_N{N}"]["overhead_vs_cublas"] for K, N in SHAPES},
                rmsnorm_hbm_frac=x["rmsnorm"]["roofline_frac"],
                attention=dict(prefill_tc_frac=at["roofline_frac"], decode_hbm_frac=at["decode"]["roofline_frac"]),
                moe=dict(ms=x["moe"]["ms"], tflops=x["moe"]["tflops"], tc_frac=x["moe"]["roofline_frac"]),
                diagnostics_ms=x["diagnostics"]["ms"], config1_us=x["config1"]["us"],
                rollout=dict(tokens_per_s=x["rollout"]["tokens_per_s"], tc_frac=x["rollout"]["roofline_frac"]))


def logprob_summary(lp):
    vp = lp["vocab_parallel"]
    return dict(workload=lp["workload"], tokens_per_s=lp["tokens_per_s"], ms=lp["ms"], tflops=lp["tflops"],
                roofline_frac=lp["roofline_frac"], bound=lp["bound"],
                T1=dict(tokens_per_s=lp["T1"]["tokens_per_s"], hbm_frac=lp["T1"]["roofline_frac"]),
                T64=dict(tokens_per_s=lp["T64"]["tokens_per_s"], hbm_frac=lp["T64"]["roofline_frac"]),
                vocab_parallel_same_bits=all(v["same_bits_as_single_call"] for v in vp.values()))


def run_tp(args, rank, world):
    """Row-parallel TP step (--parallel tp): the same three M = 4096 projections with K split over
    the N ranks (rank r owns the contiguous leaves of its K slice): each rank's leaf partial, an
    all-gather of the fp32 subtree roots (transport only) and the tree combine on every rank.
    Total work is fixed, so scaling is strong; value = the step's flops / the slowest rank's time."""
    import torch
    import torch.distributed as dist
    from parallelism_invariant_logprob_gb300 import binding as B
    from parallelism_invariant_logprob_gb300 import exchange, inputs
    dev = torch.device("cuda", int(os.environ.get("LOCAL_RANK", "0")))
    torch.cuda.set_device(dev)
    c = B.Contract(LEAVES)
    ops = exchange.LibraryOps(c, stream=torch.cuda.current_stream())
    group = dist.group.WORLD if world > 1 else None
    As, Bs = [], []
    for i, (K, N) in enumerate(SHAPES):
        X, W = inputs.gemm_inputs(M_TOKENS, K, N, seed=100 + i, device=dev)
        Kl = K // world
        As.append(X[:, rank * Kl:(rank + 1) * Kl].contiguous())
        Bs.append(W[rank * Kl:(rank + 1) * Kl].contiguous())
        del X, W
    flush = L2Flush(dev)

    def step():
        for i in range(len(SHAPES)):
            if world > 1:
                exchange.row_parallel_gemm(As[i], Bs[i], ops, group)
            else:
                B.tree_combine(c, B.gemm_leaf_partial(c, 0, 1, As[i], Bs[i])[None])

    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize()
    ts = []
    sampler = ClockSampler(dev.index)
    sampler.start()
    for _ in range(args.steps):
        flush()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        step()
        e1.record()
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    clocks = sampler.stop()
    assert B.last_device_status(c) == B.ISO_OK
    ms = max_over_ranks(statistics.mean(ts), world, dev)
    if rank == 0:
        config = bench_config(world)
        config.update(parallelism=f"tp{world}", global_batch=M_TOKENS,
                      exchange="all-gather of fp32 subtree roots (transport only), then the tree combine")
        line = dict(metric=METRIC, value=step_flops() / (ms * 1e-3) / 1e12, unit="TFLOP/s", n_gpus=world,
                    steps=args.steps, warmup=args.warmup, ms_per_step=ms, higher_is_better=True, scaling="strong",
                    vs_baseline=None, dtype="bf16", data="synthetic", config=config, clocks=clocks,
                    gpu_launches=args.steps * len(SHAPES) * 2)
        print(json.dumps(rnd(line)), flush=True)


def mismatches(a, b) -> int:
    """Elements whose bits differ (bf16 / fp32 / int tensors of the same shape)."""
    import torch
    if a.dtype in (torch.bfloat16, torch.float16):
        a, b = a.view(torch.int16), b.view(torch.int16)
    elif a.dtype == torch.float32:
        a, b = a.view(torch.int32), b.view(torch.int32)
    return int((a != b).sum().item())


def config1_and_rollout(c, dev, stream, peaks, flush):
    """Config 1 (A [32 x 2048] x B [2048 x 512], 4 leaves): time per call and its bitwise checks
    (rows alone and in sub-batches of 1 / 7 / 32, leaf partials + combine for R = 1, 2, 4).
    Config 5 (the packed rollout batch, 64 sequences of ~U[1, 8192] tokens, 259,611 rows):
    iso_rmsnorm + iso_selected_logprob over the packed prefill, and sampled tokens as one-token
    decode calls, which must give the prefill's bits."""
    import torch
    from parallelism_invariant_logprob_gb300 import binding as B
    from parallelism_invariant_logprob_gb300 import inputs
    out, bits = {}, {}
    c4 = B.Contract(4)
    A, Bm = inputs.gemm_inputs(32, 2048, 512, seed=0, device=dev)
    C = B.gemm(c4, A, Bm)
    t = time_call(lambda: B.gemm(c4, A, Bm, out=C, stream=stream), 20, 3, stream)
    rows = 0
    for M in (1, 7, 32):
        for r0 in range(0, 32 - M + 1, max(1, M)):
            rows += mismatches(B.gemm(c4, A[r0:r0 + M].contiguous(), Bm), C[r0:r0 + M])
    tp = 0
    for R in (1, 2, 4):
        Kl = 2048 // R
        S = torch.stack([B.gemm_leaf_partial(c4, r, R, A[:, r * Kl:(r + 1) * Kl].contiguous(), Bm[r * Kl:(r + 1) * Kl])
                         for r in range(R)])
        tp += mismatches(B.tree_combine(c4, S), C)
    out["config1"] = dict(workload="A [32 x 2048] x B [2048 x 512], 4 leaves", us=t * 1e3,
                          tflops=2.0 * 32 * 2048 * 512 / (t * 1e-3) / 1e12)
    bits["config1_rows_m1_m7_m32"] = rows
    bits["config1_partial_combine_r1_r2_r4"] = tp
    # config 5
    H, V = 4096, 151936
    lens = inputs.sequence_lengths(64, 8192, seed=4)
    total = sum(lens)
    states = inputs.normal_bf16((total, H), 1.0, seed=5, device=dev)
    _, gamma = inputs.rmsnorm_inputs(1, H, seed=6)
    gamma = gamma.to(dev)
    W = inputs.normal_bf16((H, V), 0.02, seed=7, device=dev)
    ids = inputs.uniform_ids(total, V, seed=8, device=dev)
    h = torch.empty_like(states)
    lp = torch.empty(total, dtype=torch.float32, device=dev)
    ws = torch.empty(B.selected_logprob_workspace(c, total, V), dtype=torch.uint8, device=dev)

    def prefill():
        B.rmsnorm(c, states, gamma, 1e-6, out=h, stream=stream)
        B.selected_logprob(c, h, W, ids, out=lp, ws=ws, stream=stream)
    tp5 = time_call(prefill, 3, 1, stream)
    g = torch.Generator().manual_seed(9)
    sample = torch.randperm(total, generator=g)[:256].tolist()
    ws1 = torch.empty(B.selected_logprob_workspace(c, 1, V), dtype=torch.uint8, device=dev)
    h1 = torch.empty(1, H, dtype=torch.bfloat16, device=dev)
    dec = torch.empty(len(sample), 4, dtype=torch.float32, device=dev)
    for i, t_ in enumerate(sample):
        B.rmsnorm(c, states[t_:t_ + 1], gamma, 1e-6, out=h1, stream=stream)
        B.selected_logprob(c, h1, W, ids[t_:t_ + 1], out=dec[i, :1], ws=ws1, stream=stream)
    bits["rollout_decode_vs_prefill_256_tokens"] = mismatches(dec[:, 0].contiguous(), lp[torch.tensor(sample, device=dev)])
    fl = 2.0 * total * H * V
    out["rollout"] = dict(workload=f"64 packed sequences, {total} tokens: iso_rmsnorm + iso_selected_logprob, H=4096, "
                                   f"V=151936", ms=tp5, tokens_per_s=total / (tp5 * 1e-3),
                          tflops=fl / (tp5 * 1e-3) / 1e12, roofline_frac=fl / (peaks["tc"] * 1e12) / (tp5 * 1e-3))
    del states, h, W, ws
    return out, bits


class L2Flush:
    """Called before a timed call: a 256 MiB write evicts every line of the inputs from the
    129 MB L2, then a 256 MiB read of a second buffer evicts the write's dirty lines, so their
    write-back to HBM happens here, outside the event window, and not inside the timed kernel."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(64 << 20, dtype=torch.float32, device=dev)
        self.r = torch.ones(64 << 20, dtype=torch.float32, device=dev)
        self.acc = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        import torch
        self.w.zero_()
        torch.sum(self.r, dim=0, out=self.acc)


def time_call(fn, iters, warm, stream, flush=None):
    import torch
    for _ in range(warm):
        if flush is not None:
            flush()
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(iters):
        if flush is not None:
            flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.mean(ts)


def stream_call(fn, args, stream, flush, reps=4, trials=3):
    """Per-call time (ms) of fn(a) issued back to back over the argument list `args` (weight
    copies whose total is larger than L2, so every call streams its weights from HBM): the
    decode-loop cost, where one call's launch and prologue overlap the previous call's tail.
    Best of `trials` runs of reps x len(args) calls, each run after an L2 flush."""
    import torch
    for a in args:
        fn(a)
    torch.cuda.synchronize()
    best = float("inf")
    for _ in range(trials):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        n = reps * len(args)
        e0.record(stream)
        for i in range(n):
            fn(args[i % len(args)])
        e1.record(stream)
        torch.cuda.synchronize()
        best = min(best, e0.elapsed_time(e1) / n)
    return best


def secondary(c, dev, stream, peaks, rank):
    """Logprob (config 3), small-M GEMMs, simulated-TP partial+combine, RMSNorm,
    MoE layer and a non-invariant cuBLAS reference for the invariance overhead."""
    import torch
    from parallelism_invariant_logprob_gb300 import binding as B
    from parallelism_invariant_logprob_gb300 import inputs
    out = {}
    bits = {}
    flush = L2Flush(dev)

    # selected-token logprob, T = 4096, H = 4096, V = 151936; the hidden states are RMS-normalised
    # rows (iso_rmsnorm with unit gamma over N(0,1) rows, before the timed region)
    h, W, ids = logprob_workload(c, dev)
    lp_out = torch.empty(LP_T, dtype=torch.float32, device=dev)
    ws = torch.empty(B.selected_logprob_workspace(c, LP_T, LP_V), dtype=torch.uint8, device=dev)
    t = time_call(lambda: B.selected_logprob(c, h, W, ids, out=lp_out, ws=ws, stream=stream), 5, 2, stream)
    fl = 2.0 * LP_T * LP_H * LP_V
    byt = 2.0 * LP_H * LP_V + 2.0 * LP_T * LP_H + 8.0 * LP_T
    ideal = max(fl / (peaks["tc"] * 1e12), byt / (peaks["hbm"] * 1e9))
    out["logprob"] = dict(workload="T=4096, H=4096 (RMS-normalised rows), V=151936, 8 leaves, 63 chunks",
                          tokens_per_s=LP_T / (t * 1e-3), ms=t, tflops=fl / (t * 1e-3) / 1e12,
                          roofline_frac=ideal / (t * 1e-3), bound="tensor")
    for T in (1, 64):
        hT, idT = h[:T].contiguous(), ids[:T].contiguous()
        wsT = torch.empty(B.selected_logprob_workspace(c, T, LP_V), dtype=torch.uint8, device=dev)
        oT = torch.empty(T, dtype=torch.float32, device=dev)
        tt = time_call(lambda: B.selected_logprob(c, hT, W, idT, out=oT, ws=wsT, stream=stream), 5, 2, stream, flush)
        byt = 2.0 * LP_H * LP_V + 2.0 * T * LP_H + 8.0 * T
        out["logprob"][f"T{T}"] = dict(ms=tt, tokens_per_s=T / (tt * 1e-3), hbm_gbs=byt / (tt * 1e-3) / 1e9,
                                       roofline_frac=byt / (peaks["hbm"] * 1e9) / (tt * 1e-3), bound="hbm")
    # RMSNorm + logprob at T = 4096: the separate stages against the fused A prologue (same bits)
    xr, gr = inputs.rmsnorm_inputs(LP_T, LP_H, seed=12, device=dev)
    hn = torch.empty_like(xr)
    ws_f = torch.empty(B.rmsnorm_selected_logprob_workspace(c, LP_T, LP_V), dtype=torch.uint8, device=dev)

    def separate():
        B.rmsnorm(c, xr, gr, 1e-6, out=hn, stream=stream)
        B.selected_logprob(c, hn, W, ids, out=lp_out, ws=ws, stream=stream)
    t_sep = time_call(separate, 5, 2, stream, flush)
    t_fused = time_call(lambda: B.rmsnorm_selected_logprob(c, xr, gr, 1e-6, W, ids, out=lp_out, ws=ws_f, stream=stream),
                        5, 2, stream, flush)
    out["logprob"]["rmsnorm_fused"] = dict(workload="iso_rmsnorm + iso_selected_logprob vs iso_rmsnorm_selected_logprob, "
                                                    "T=4096, H=4096, V=151936", ms_separate=t_sep, ms_fused=t_fused)
    # vocab-parallel logprob: R chunk-aligned vocabulary shards (one per simulated rank, each timed
    # on its own shard of W), then the combine over the rank-ordered statistics; one rank's time is
    # its partial, the job's the slowest partial plus the combine
    vp = {}
    chunk_cols = 19 * 128
    for R in (2, 4):
        v0s = [int(round(LP_V * r / R / chunk_cols)) * chunk_cols for r in range(R)]
        bounds = v0s + [LP_V]
        parts, stats, zs = [], [], []
        for r in range(R):
            v0, v1 = bounds[r], bounds[r + 1]
            Wr = W[:, v0:v1]
            ws_r = torch.empty(max(int(c.lib.iso_selected_logprob_partial_workspace(c.handle, LP_T, v1 - v0)), 16),
                               dtype=torch.uint8, device=dev)
            s_r, z_r = B.selected_logprob_partial(c, h, Wr, ids, LP_V, v0, ws=ws_r, stream=stream)
            parts.append(time_call(lambda: B.selected_logprob_partial(c, h, Wr, ids, LP_V, v0, stats_r=s_r, zsel_r=z_r,
                                                                       ws=ws_r, stream=stream), 3, 1, stream, flush))
            stats.append(s_r)
            zs.append(z_r)
        st_all, z_all = torch.cat(stats, 0), torch.stack(zs)
        t_comb = time_call(lambda: B.selected_logprob_combine(c, v0s, st_all, z_all, ids, LP_V, out=lp_out, stream=stream),
                           5, 2, stream, flush)
        vp_bad = mismatches(lp_out, B.selected_logprob(c, h, W, ids))
        bits[f"vocab_parallel_R{R}"] = vp_bad
        vp[f"R{R}"] = dict(shard_v0=v0s, ms_partial_max=max(parts), ms_partial_min=min(parts), ms_combine=t_comb,
                           ms_single_call_over_R=t / R, same_bits_as_single_call=vp_bad == 0)
    out["logprob"]["vocab_parallel"] = vp
    del h, W, ids, ws, xr, hn, ws_f

    # GEMM at small M (weight-streaming, HBM-bound) and the cuBLAS non-invariant reference
    gm = {}
    for K, N in SHAPES:
        X, Wt = inputs.gemm_inputs(M_TOKENS, K, N, seed=5, device=dev)
        for M in (1, 8, 64, 512, 4096):
            Xm = X[:M].contiguous()
            Cm = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
            tt = time_call(lambda: B.gemm(c, Xm, Wt, out=Cm, stream=stream), 5, 2, stream, flush)
            tb = time_call(lambda: torch.matmul(Xm, Wt, out=Cm), 5, 2, stream, flush)
            byt = 2.0 * (M * K + K * N + M * N)
            gm[f"M{M}_K{K}_N{N}"] = dict(ms=tt, tflops=2.0 * M * K * N / (tt * 1e-3) / 1e12,
                                         hbm_gbs=byt / (tt * 1e-3) / 1e9, cublas_ms=tb,
                                         overhead_vs_cublas=tt / tb)
            if M <= 128:  # iso_gemm_ws: the same bits, leaf groups spread over more SMs
                wsg = torch.empty(max(B.gemm_workspace(c, M, N, K), 16), dtype=torch.uint8, device=dev)
                tw = time_call(lambda: B.gemm_ws(c, Xm, Wt, out=Cm, ws=wsg, stream=stream), 5, 2, stream, flush)
                gm[f"M{M}_K{K}_N{N}"].update(ws_ms=tw, ws_hbm_gbs=byt / (tw * 1e-3) / 1e9,
                                             ws_hbm_frac=byt / (tw * 1e-3) / 1e9 / peaks["hbm"],
                                             ws_overhead_vs_cublas=tw / tb)
                # back to back over rotating weight copies (> 300 MB in all): the decode loop
                copies = [Wt] + [inputs.gemm_inputs(1, K, N, seed=50 + j, device=dev)[1]
                                 for j in range(max(3, -(-300_000_000 // (2 * K * N))) - 1)]
                ts = stream_call(lambda W_: B.gemm(c, Xm, W_, out=Cm, stream=stream), copies, stream, flush)
                tsb = stream_call(lambda W_: torch.matmul(Xm, W_, out=Cm), copies, stream, flush)
                gm[f"M{M}_K{K}_N{N}"].update(stream_ms=ts, stream_hbm_frac=byt / (ts * 1e-3) / 1e9 / peaks["hbm"],
                                             stream_cublas_ms=tsb,
                                             stream_cublas_hbm_frac=byt / (tsb * 1e-3) / 1e9 / peaks["hbm"],
                                             weight_copies=len(copies))
                del copies
        # simulated TP: R ranks' partials + combine at M = 4096
        for R in (2, 8):
            Kl = K // R
            Xr = [X[:, r * Kl:(r + 1) * Kl].contiguous() for r in range(R)]
            Wr = [Wt[r * Kl:(r + 1) * Kl] for r in range(R)]
            S = torch.empty(R, M_TOKENS, N, dtype=torch.float32, device=dev)
            Cc = torch.empty(M_TOKENS, N, dtype=torch.bfloat16, device=dev)

            def tp():
                for r in range(R):
                    B.gemm_leaf_partial(c, r, R, Xr[r], Wr[r], out=S[r], stream=stream)
                B.tree_combine(c, S, out=Cc, stream=stream)
            tt = time_call(tp, 3, 1, stream, flush)
            gm[f"TP{R}_M4096_K{K}_N{N}"] = dict(ms=tt, tflops=2.0 * M_TOKENS * K * N / (tt * 1e-3) / 1e12)
            full = B.gemm(c, X, Wt)
            bits[f"tp{R}_partials_vs_single_{K}x{N}"] = mismatches(Cc, full)
            if R == 2:  # rows alone and in a 7-row batch against the same rows of the 4096-row product
                bits[f"rows_m1_m7_vs_m4096_{K}x{N}"] = (
                    sum(mismatches(B.gemm(c, X[r:r + 1].contiguous(), Wt), full[r:r + 1]) for r in (0, 2047, 4095)) +
                    mismatches(B.gemm(c, X[100:107].contiguous(), Wt), full[100:107]))
        del X, Wt
    out["gemm_sweep"] = gm

    # RMSNorm, T = 262144 x 4096 (the packed-prefill size)
    x, g = inputs.rmsnorm_inputs(262144, 4096, seed=4, device=dev)
    y = torch.empty_like(x)
    tt = time_call(lambda: B.rmsnorm(c, x, g, 1e-6, out=y, stream=stream), 5, 2, stream)
    byt = 4.0 * 262144 * 4096 + 2 * 4096
    out["rmsnorm"] = dict(workload="T=262144, H=4096", ms=tt, hbm_gbs=byt / (tt * 1e-3) / 1e9,
                          roofline_frac=byt / (peaks["hbm"] * 1e9) / (tt * 1e-3), bound="hbm")
    del x, y

    # mismatch diagnostics over a packed rollout batch: 64 sequences, lengths ~ U[1, 8192] (seed 4)
    g = torch.Generator().manual_seed(4)
    lens = torch.randint(1, 8193, (64,), generator=g)
    offs = torch.cat([torch.zeros(1, dtype=torch.int64), torch.cumsum(lens, 0)]).to(torch.int32).to(dev)
    n = int(lens.sum())
    lp_r = (-torch.abs(torch.randn(n, generator=g)) * 2).to(dev)
    lp_t = lp_r + (torch.rand(n, generator=g) < 0.5).to(dev) * torch.randn(n, generator=g).to(dev) * 1e-3
    dg = B.mismatch_diagnostics(c, lp_t, lp_r, offs, stream=stream)
    tt = time_call(lambda: B.mismatch_diagnostics(c, lp_t, lp_r, offs, stream=stream, out=dg), 5, 2, stream, flush)
    byt = 16.0 * n + 4.0 * 65 + 33.0 * 64  # 2 fp32 in + 2 fp32 out per token; offsets; per-sequence outputs
    # bound by FP64 arithmetic (one block per sequence; this part has ~2 FP64 ops per clock per SM),
    # not by its 16 bytes per token of traffic, so no HBM fraction is claimed
    out["diagnostics"] = dict(workload=f"64 packed sequences, {n} tokens", ms=tt, tokens_per_s=n / (tt * 1e-3),
                              hbm_gbs=byt / (tt * 1e-3) / 1e9, bound="fp64")

    out["attention"] = attention_measure(c, dev, stream, peaks, flush)
    bits["attention_decode_vs_prefill_64_rows"] = out["attention"]["decode_vs_prefill_mismatches"]

    # MoE expert layer: T=8192, H=2048, E=128, F=768, k=8
    T, H, E, F, k = 8192, 2048, 128, 768, 8
    xm, W1, W2, logits = inputs.moe_inputs(T, H, E, F, seed=3, device=dev)
    ids_m, w_m = B.moe_route(c, logits, k)
    om = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    wsm = torch.empty(B.grouped_gemm_moe_workspace(c, T, E, k, H, F), dtype=torch.uint8, device=dev)
    tt = time_call(lambda: B.grouped_gemm_moe(c, xm, ids_m, w_m, W1, W2, out=om, ws=wsm, stream=stream), 10, 3, stream,
                   flush)
    fl = 2.0 * T * k * (H * 2 * F + F * H)
    out["moe"] = dict(workload="T=8192, H=2048, E=128, F=768, k=8", ms=tt, tflops=fl / (tt * 1e-3) / 1e12,
                      roofline_frac=fl / (peaks["tc"] * 1e12) / (tt * 1e-3))
    moe_base = om.clone()
    bits["moe_partitions_p2_p8_random"] = sum(
        mismatches(B.grouped_gemm_moe(c, xm, ids_m, w_m, W1, W2, expert_partition=part, ws=wsm, stream=stream), moe_base)
        for part in ([e * 2 // E for e in range(E)], [e * 8 // E for e in range(E)],
                     inputs.random_partition(E, 4, seed=7).tolist()))
    # expert parallelism: R ranks own contiguous expert sets; a rank's time is its partial (the slot
    # rows of its experts), the job's the slowest partial plus the combine after the exchange
    ep = {}
    ys = torch.empty(T * k, H, dtype=torch.bfloat16, device=dev)
    ws_p = torch.empty(B.moe_experts_partial_workspace(c, T, E, k, H, F), dtype=torch.uint8, device=dev)
    for R in (2, 4):
        parts = []
        for r in range(R):
            mask = [e * R // E == r for e in range(E)]
            parts.append(time_call(lambda: B.moe_experts_partial(c, xm, ids_m, W1, W2, mask, y_slots=ys, ws=ws_p,
                                                                  stream=stream), 5, 2, stream, flush))
        t_comb = time_call(lambda: B.moe_combine(c, ys.view(T, k, H), w_m, out=om, stream=stream), 5, 2, stream, flush)
        ep_bad = mismatches(om, B.grouped_gemm_moe(c, xm, ids_m, w_m, W1, W2, ws=wsm, stream=stream))
        bits[f"expert_parallel_R{R}"] = ep_bad
        ep[f"R{R}"] = dict(ms_partial_max=max(parts), ms_partial_min=min(parts), ms_combine=t_comb,
                           ms_layer_over_R=tt / R, same_bits_as_layer=ep_bad == 0)
    out["moe"]["expert_parallel"] = ep
    del xm, W1, W2, wsm, ys, ws_p
    extra, bits5 = config1_and_rollout(c, dev, stream, peaks, flush)
    out.update(extra)
    bits.update(bits5)
    out["bitwise"] = bits
    return out


def logprob_workload(c, dev):
    """Selected-token logprob inputs: h = iso_rmsnorm(x, unit gamma) of x ~ N(0,1) [4096 x 4096]
    (the final norm's output, as the LM head sees it), W ~ N(0, 0.02^2) [4096 x 151936], ids
    uniform in [0, 151936)."""
    import torch
    from parallelism_invariant_logprob_gb300 import binding as B
    from parallelism_invariant_logprob_gb300 import inputs
    x, W, ids = inputs.logprob_inputs(LP_T, LP_H, LP_V, seed=2, device=dev)
    h = B.rmsnorm(c, x, torch.ones(LP_H, dtype=torch.bfloat16, device=dev), 1e-6)
    torch.cuda.synchronize()
    return h, W, ids


ATT_HQ, ATT_HKV, ATT_D = 32, 8, 128  # 8B-class decoder: 32 query heads over 8 KV heads


def attention_workload(dev, small=False):
    """Causal attention over the packed rollout batch (64 sequences, lengths ~ U[1, 8192],
    seed 4), or 8 sequences of 2048 tokens (small)."""
    from parallelism_invariant_logprob_gb300 import inputs
    lens = [2048] * 8 if small else inputs.sequence_lengths(64, 8192, seed=4)
    Q, K, V, qs, ks, p0 = inputs.attention_inputs(lens, [0] * len(lens), ATT_HQ, ATT_HKV, ATT_D, seed=6, device=dev)
    return lens, Q, K, V, qs, ks, p0


def attention_flops(lens):
    # 2 d flops for q.k and 2 d for p.v per (row, visible key) pair, per query head
    return 4.0 * ATT_D * ATT_HQ * sum(L * (L + 1) // 2 for L in lens)


def attention_measure(c, dev, stream, peaks, flush):
    """Packed prefill over the rollout batch, and one decode step per sequence (its last
    position, reading its whole KV cache)."""
    import math
    import torch
    from parallelism_invariant_logprob_gb300 import binding as B
    lens, Q, K, V, qs, ks, p0 = attention_workload(dev)
    scale = 1.0 / math.sqrt(ATT_D)
    o = torch.empty_like(Q)
    lse = torch.empty(Q.shape[0], ATT_HQ, dtype=torch.float32, device=dev)
    mq = max(lens)
    tt = time_call(lambda: B.attention(c, Q, K, V, qs, ks, p0, scale, max_q_rows=mq, out=o, lse=lse, stream=stream),
                   3, 1, stream)
    fl = attention_flops(lens)
    r = dict(workload=f"causal prefill, 64 packed sequences ({sum(lens)} tokens), {ATT_HQ} query / {ATT_HKV} KV "
                      f"heads, d {ATT_D}", ms=tt, tflops=fl / (tt * 1e-3) / 1e12,
             roofline_frac=fl / (peaks["tc"] * 1e12) / (tt * 1e-3), bound="tensor")
    # decode: the last row of each sequence
    last = (qs[1:] - 1).long()
    Qd = Q[last].contiguous()
    dq = torch.arange(len(lens) + 1, dtype=torch.int32, device=dev)
    dpos = torch.tensor([L - 1 for L in lens], dtype=torch.int32, device=dev)
    od = torch.empty_like(Qd)
    ld = torch.empty(len(lens), ATT_HQ, dtype=torch.float32, device=dev)
    td = time_call(lambda: B.attention(c, Qd, K, V, dq, ks, dpos, scale, max_q_rows=1, out=od, lse=ld, stream=stream),
                   5, 2, stream, flush)
    byt = 2.0 * 2 * ATT_HKV * ATT_D * sum(lens) + 2.0 * 2 * len(lens) * ATT_HQ * ATT_D
    r["decode_vs_prefill_mismatches"] = mismatches(od, o[last]) + mismatches(ld, lse[last])
    r["decode"] = dict(workload=f"one row per sequence at its last position, {len(lens)} sequences", ms=td,
                       hbm_gbs=byt / (td * 1e-3) / 1e9, roofline_frac=byt / (peaks["hbm"] * 1e9) / (td * 1e-3),
                       bound="hbm")
    return r


def profile_target(target: str, calls: int):
    """Run one workload `calls` times with no timing output (the program ncu profiles)."""
    import torch
    from parallelism_invariant_logprob_gb300 import binding as B
    from parallelism_invariant_logprob_gb300 import inputs
    dev = torch.device("cuda", 0)
    c = B.Contract(LEAVES)
    if target == "gemm":
        X, W = inputs.gemm_inputs(M_TOKENS, 4096, 12288, seed=100, device=dev)
        C = torch.empty(M_TOKENS, 12288, dtype=torch.bfloat16, device=dev)
        fn = lambda: B.gemm(c, X, W, out=C)
    elif target == "gemm_m1":  # a decode-size GEMM: one row, 4096 x 4096 (leaf groups on clusters)
        X, W = inputs.gemm_inputs(1, 4096, 4096, seed=100, device=dev)
        C = torch.empty(1, 4096, dtype=torch.bfloat16, device=dev)
        fn = lambda: B.gemm(c, X, W, out=C)
    elif target == "logprob":
        h, W, ids = logprob_workload(c, dev)
        out = torch.empty(LP_T, dtype=torch.float32, device=dev)
        ws = torch.empty(B.selected_logprob_workspace(c, LP_T, LP_V), dtype=torch.uint8, device=dev)
        fn = lambda: B.selected_logprob(c, h, W, ids, out=out, ws=ws)
    elif target == "moe":
        T, H, E, F, k = 8192, 2048, 128, 768, 8
        x, W1, W2, logits = inputs.moe_inputs(T, H, E, F, seed=3, device=dev)
        ids, w = B.moe_route(c, logits, k)
        om = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
        wsm = torch.empty(B.grouped_gemm_moe_workspace(c, T, E, k, H, F), dtype=torch.uint8, device=dev)
        fn = lambda: B.grouped_gemm_moe(c, x, ids, w, W1, W2, out=om, ws=wsm)
    elif target in ("attention", "attention_small"):
        import math
        lens, Q, K, V, qs, ks, p0 = attention_workload(dev, small=target == "attention_small")
        o = torch.empty_like(Q)
        lse = torch.empty(Q.shape[0], ATT_HQ, dtype=torch.float32, device=dev)
        fn = lambda: B.attention(c, Q, K, V, qs, ks, p0, 1.0 / math.sqrt(ATT_D), max_q_rows=max(lens), out=o, lse=lse)
    elif target == "attention_decode":  # one row per sequence of the rollout batch at its last position
        import math
        lens, Q, K, V, qs, ks, p0 = attention_workload(dev)
        Qd = Q[(qs[1:] - 1).long()].contiguous()
        del Q  # the packed queries are not needed for the decode rows
        dq = torch.arange(len(lens) + 1, dtype=torch.int32, device=dev)
        dpos = torch.tensor([L - 1 for L in lens], dtype=torch.int32, device=dev)
        od = torch.empty_like(Qd)
        ld = torch.empty(len(lens), ATT_HQ, dtype=torch.float32, device=dev)
        fn = lambda: B.attention(c, Qd, K, V, dq, ks, dpos, 1.0 / math.sqrt(ATT_D), max_q_rows=1, out=od, lse=ld)
    elif target == "diagnostics":
        gen = torch.Generator().manual_seed(4)
        lens = torch.randint(1, 8193, (64,), generator=gen)
        offs = torch.cat([torch.zeros(1, dtype=torch.int64), torch.cumsum(lens, 0)]).to(torch.int32).to(dev)
        n = int(lens.sum())
        lp_r = (-torch.abs(torch.randn(n, generator=gen)) * 2).to(dev)
        lp_t = lp_r + (torch.rand(n, generator=gen) < 0.5).to(dev) * torch.randn(n, generator=gen).to(dev) * 1e-3
        dg = B.mismatch_diagnostics(c, lp_t, lp_r, offs)
        fn = lambda: B.mismatch_diagnostics(c, lp_t, lp_r, offs, out=dg)
    elif target == "rmsnorm":
        x, g = inputs.rmsnorm_inputs(262144, 4096, seed=4, device=dev)
        y = torch.empty_like(x)
        fn = lambda: B.rmsnorm(c, x, g, 1e-6, out=y)
    else:
        raise SystemExit(f"unknown profile target {target}")
    for _ in range(calls):
        fn()
    torch.cuda.synchronize()
    assert B.last_device_status(c) == B.ISO_OK


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--skip-secondary", action="store_true")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--details", default=None, help="write the full secondary measurements to this JSON file")
    ap.add_argument("--parallel", default="dp", choices=["dp", "tp"],
                    help="dp: data-parallel replicas (the default step); tp: row-parallel TP over K-leaves")
    ap.add_argument("--profile-target", choices=["gemm", "gemm_m1", "logprob", "moe", "rmsnorm", "attention",
                                                     "attention_small", "diagnostics", "attention_decode"],
                    help="run one workload --steps times without timing (for ncu) and exit")
    args = ap.parse_args()
    if args.profile_target:
        profile_target(args.profile_target, args.steps)
        return
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    try:
        if args.parallel == "tp":
            run_tp(args, rank, world)
        else:
            run_ours(args, rank, world)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()

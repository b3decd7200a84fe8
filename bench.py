#!/usr/bin/env python
"""Benchmark: the 8B-shaped ternary linear stack on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one pass of the whole hot path over one batch: all 252
projection linears of a 36-layer, Qwen3-8B-shaped decoder (hidden 4096,
q/o 4096x4096, k/v 1024x4096, gate/up 12288x4096, down 4096x12288), as 144
dependent launches (q/k/v and gate/up grouped) replayed from a CUDA graph
with programmatic dependent launch, on seeded synthetic weights with the
pages' code statistics.  The headline is N = 1 decode in mode A (bf16
activations, fp32 accumulation); beside it: the N = 8 speculative-verify
batch (modes A and B), the same pass as one persistent chain launch, the
0.6B-shaped stack, a single 2048 x 1024 linear, the int8 output head with
its fused argmax, and the N = 512 prefill.

Prints ONE JSON line (rank 0).  Under torchrun each rank runs an
independent replica (the path has no exchange step); value is the sum of the
ranks' tokens/s over the max-over-ranks time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "8B-shape ternary linears: tokens/s at N=1 and N=8; HBM GB/s as % of B300 peak"
WORKLOAD = ("8B-shaped ternary linear stack: 36 layers x 7 projections (252 matrices, "
            "q/o 4096x4096, k/v 1024x4096, gate/up 12288x4096, down 4096x12288), N=1 decode, "
            "mode A (bf16 activations, fp32 accumulate, fp32 out)")
L2_BYTES = 126 * 1024 * 1024


def peaks():
    """(HBM GB/s, kind, bf16 TFLOP/s burst, kind) from MEASURED_PEAKS.json.
    The prefill pass is timed over a few replays of ~13 ms, not seconds, so
    its denominator is the burst figure."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        hbm, hk = float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        d, hbm, hk = {}, 6400.0, "fallback"
    try:
        bf, bk = float(d["bf16_tflops"]), "measured (bf16_tflops, burst)"
    except (KeyError, ValueError):
        bf, bk = 1800.0, "fallback (burst)"
    return hbm, hk, bf, bk


# ---------------------------------------------------------------- clocks
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]
        return False

    def summary(self):
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


def measured_traffic(alg_per_launch, record="tl_mma_kernel_traffic.txt"):
    """DRAM bytes per launch of the decode kernel: the ncu-measured bytes per
    algorithmic byte (profiles/<record>) times this run's algorithmic bytes
    per launch; None when the record is missing or the kernels' device code
    changed since it was captured."""
    import hashlib
    here = os.path.dirname(os.path.abspath(__file__))
    rec = os.path.join(here, "profiles", record)
    src = os.path.join(here, "bit_matvec_ternary_b300", "csrc", "tl_kernels.cu")
    try:
        kv = {}
        for line in open(rec):
            line = line.strip()
            if line and not line.startswith("#") and "=" in line:
                k, v = line.split("=", 1)
                kv[k] = v
        text = open(src).read()
        device = text[:text.index("// ------------------------------------------------------------------ host side")]
        if hashlib.sha256(device.encode()).hexdigest() != kv["device_source_sha256"]:
            return None
        ratio = (int(kv["dram_bytes_read"]) + int(kv["dram_bytes_write"])) / int(kv["algorithmic_bytes"])
        return ratio * alg_per_launch
    except (OSError, KeyError, ValueError):
        return None


# ---------------------------------------------------------------- timing
def time_graph(stack, steps, warmup, torch):
    g = stack.graph
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        g.replay()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def time_chain(chain, steps, warmup, torch):
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        chain.run()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        chain.run()
    end.record(stream)
    torch.cuda.synchronize()
    if chain.status() != 0:
        raise RuntimeError(f"chain reported device status {chain.status()}")
    return start.elapsed_time(end) / steps


def time_e2e(stack, steps, warmup, torch):
    """Per step: pinned host -> device copies of all inputs, the pass, and
    device -> host copies of all outputs, inside the timed region -- one
    replay of the stack's graph with its host copies (``capture_e2e``: each
    layer's inputs copied in ahead of it and its outputs copied out after it,
    on two copy streams beside the launches)."""
    stream = torch.cuda.current_stream()
    hx = torch.empty(stack.X_flat.shape, dtype=stack.X_flat.dtype, pin_memory=True)
    hx.copy_(stack.X_flat.cpu())
    hy = torch.empty(stack.Y_flat.shape, dtype=stack.Y_flat.dtype, pin_memory=True)
    g = stack.capture_e2e(hx, hy)

    def step():
        g.replay()

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for _ in range(steps):
        step()
    end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps, stack.input_bytes(), stack.output_bytes()


# ---------------------------------------------------------------- oracle legs
class OracleSample:
    """Layer 0's seven linears packed for the CPU oracle; run() times passes
    over them and extrapolates to the whole 252-linear stack."""

    def __init__(self, host, shape, N):
        from oracle import oracle as O
        from bit_matvec_ternary_b300 import synth
        self.O, self.shape, self.N = O, shape, N
        self.cores = O.host_cores()
        self.packed = {}
        for p in synth.PROJ_ORDER:
            W, scale = host[(0, p)]
            P = O.pack(W)
            self.packed[p] = (P, scale, O.rowsum(P, W.shape[0], W.shape[1]), W.shape)
        shp = shape.linear_shapes()
        self.xs = {p: synth.activations(N, shp[p][1], seed=424242 + i)
                   for i, p in enumerate(synth.PROJ_ORDER)}
        self.order = synth.PROJ_ORDER

    def run(self, seconds, mode=0):
        O = self.O
        per_layer = self.shape.ternary_weights_per_layer()
        done, t0 = 0, time.perf_counter()
        while True:
            for p in self.order:
                P, scale, rs, (M, K) = self.packed[p]
                if mode == 0:
                    O.linear_a_mt(P, scale, M, K, self.xs[p], nthreads=self.cores)
                else:
                    Q, s, z = O.quant(self.xs[p])
                    O.linear_b_mt(P, scale, rs, M, K, Q, s, z, nthreads=self.cores)
            done += per_layer
            el = time.perf_counter() - t0
            if el >= seconds:
                break
        passes = done / self.shape.ternary_weights()
        desc = (f"layer 0's 7 linears x{done // per_layer} ({done / 1e9:.2f}e9 weights), "
                f"N={self.N}, mode {'A' if mode == 0 else 'B'}, extrapolated to "
                f"{len(self.order) * self.shape.layers} linears")
        return self.N * passes / el, desc


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle on the host cores (rank 0 only)."""
    if rank != 0:
        return None
    from bit_matvec_ternary_b300 import synth
    shape = synth.NEUTRINO_8B
    host = {}
    for p in synth.PROJ_ORDER:
        M, K = shape.linear_shapes()[p]
        seed = synth.matrix_seed(0, 0, p)
        host[(0, p)] = (synth.ternary(M, K, synth.zero_fraction(shape, 0, p), seed),
                        synth.scales(M, seed))
    sampler = OracleSample(host, shape, 1)
    cores = sampler.cores
    sample_s, per_token = [], []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        v, desc = sampler.run(seconds=0.0)
        el = time.perf_counter() - t0
        if i >= args.warmup:
            sample_s.append(el)                # one layer's 7 linears, measured
            per_token.append(1.0 / v)          # seconds per token, extrapolated x36
    value = 1.0 / (sum(per_token) / len(per_token))
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * sum(sample_s) / len(sample_s), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": 1, "seq_len": 1,
                       "parallelism": "none (host threads)",
                       "step": "each timed step runs layer 0's 7 linears (1/36 of the stack) on "
                               "the oracle; ms_per_step is that measured time, and value "
                               "extrapolates it to the 36-layer stack (x36)"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": "each step: " + desc},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def flush_l2(torch, buf):
    buf.zero_()


def _graph_us(torch, body, reps, replays=5):
    """Median device time of one replay of a CUDA graph of `reps` calls of
    `body`, in microseconds (events on the launching stream)."""
    stream = torch.cuda.current_stream()
    cs = torch.cuda.Stream()
    cs.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cs):
        for _ in range(reps):
            body()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    t = []
    for _ in range(replays):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        t.append(e0.elapsed_time(e1) * 1e3)
    return statistics.median(t)


def _cold_us(torch, call, flush, reps=20):
    """Launch-to-launch microseconds of `call` with L2 flushed before it and
    no host time inside: a graph of (256 MiB write, call) pairs less a graph
    of the writes alone, per pair."""
    both = _graph_us(torch, lambda: (flush_l2(torch, flush), call()), reps)
    alone = _graph_us(torch, lambda: flush_l2(torch, flush), reps)
    return (both - alone) / reps


def _launch_times(torch, call, flush, reps=50, cold_reps=20):
    """(warm us, cold us) per launch: `reps` launches replayed as one CUDA
    graph, L2-warm; and `_cold_us` (L2 flushed before each launch)."""
    for _ in range(5):
        call()
    torch.cuda.synchronize()
    warm = _graph_us(torch, call, reps) / reps
    return warm, _cold_us(torch, call, flush, cold_reps)


def bench_neighbours(args, torch, tl, hbm_peak):
    """The rows beside the ternary linears, at the 8B shapes, one and eight
    tokens: the block-scale linear (12288 x 4096, one scale per row and
    128-column block, seeded normal float weights ternarised by absmean) and
    the fused RMSNorm + quantisation (hidden 4096) and SwiGLU + quantisation
    (12288).  Per launch: warm (a graph of 50 launches) and cold (L2 flushed)
    microseconds; GB/s and the HBM fraction from the cold time and the
    algorithmic bytes (inputs once, outputs once)."""
    import numpy as np
    from bit_matvec_ternary_b300 import synth
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")

    def bf16(a):
        return torch.from_numpy(synth.to_bf16_bits(a.astype(np.float32)).view(np.int16)).view(
            torch.bfloat16).cuda()

    def line(warm, cold, alg):
        return {"warm_us": warm, "cold_us": cold, "algorithmic_bytes": alg,
                "cold_gbs": alg / (cold * 1e3), "cold_frac_of_hbm": alg / (cold * 1e3) / hbm_peak}

    out = {}
    rng = np.random.default_rng(7)
    M, K = 12288, 4096
    bw = tl.BlockScaledWeight.from_float(rng.standard_normal((M, K), dtype=np.float32) * 0.02)
    KB = (K + 127) // 128
    bs = {"shape": "12288x4096, fp32 scale per (row, 128-column block), mode A, fp32 out"}
    for N in (1, 8):
        x = bf16(rng.standard_normal((N, K)))
        y = torch.empty((N, M), dtype=torch.float32, device="cuda")
        warm, cold = _launch_times(torch, lambda: tl.tl_linear_blockscale(bw, x, out=y), flush)
        bs[f"n{N}"] = line(warm, cold, tl.tl_packed_bytes(M, K) + 4 * M * KB + 2 * N * K + 4 * N * M)
    out["blockscale_linear"] = bs
    del bw
    D, F = 4096, 12288
    rq = {"shape": "RMSNorm over 4096 then per-token int8 quantisation (bf16 and int8 out)"}
    sq = {"shape": "silu(gate) * up over 12288 then per-token int8 quantisation (bf16 and int8 out)"}
    gamma = bf16(rng.uniform(0.8, 1.2, D))
    for N in (1, 8):
        x = bf16(rng.standard_normal((N, D)))
        warm, cold = _launch_times(torch, lambda: tl.tl_rmsnorm_quant(x, gamma), flush)
        rq[f"n{N}"] = line(warm, cold, 2 * N * D + 2 * D + 2 * N * D + N * D + 8 * N)
        gt, ut = bf16(rng.standard_normal((N, F))), bf16(rng.standard_normal((N, F)))
        warm, cold = _launch_times(torch, lambda: tl.tl_swiglu_quant(gt, ut), flush)
        sq[f"n{N}"] = line(warm, cold, 4 * N * F + 2 * N * F + N * F + 8 * N)
    out["rmsnorm_quant"] = rq
    out["swiglu_quant"] = sq
    return out


def bench_single_linear(args, torch, tl, hbm_peak, cpu):
    """A single 2048 x 1024 ternary linear at one token, modes A and B:
    launch-to-launch latency (back to back, L2-warm: 200 launches replayed
    as one CUDA graph, so no host launch cost is in it; the same 200 calls
    from the Python loop are reported beside it) and, with a 256 MiB buffer
    written between timed launches to flush L2, cold GB/s."""
    import numpy as np
    from bit_matvec_ternary_b300 import synth
    M, K = 2048, 1024
    W = synth.ternary(M, K, 0.626, 0)
    scale = synth.scales(M, 0)
    w = tl.TernaryWeight.from_int8(W, scale)
    x = synth.activations(1, K, seed=0)
    xt = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).cuda()
    q, s, z = tl.tl_quantize_act(xt)
    ws = tl.make_workspace([[w]], 1)
    y = torch.empty((1, M), dtype=torch.float32, device="cuda")
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    out = {"shape": "2048x1024, N=1, seed 0"}
    for mode, name in ((tl.TL_MODE_BF16, "mode_a"), (tl.TL_MODE_I8, "mode_b")):
        if mode == tl.TL_MODE_BF16:
            call = lambda: tl.tl_linear(w, xt, out=y, workspace=ws)
        else:
            call = lambda: tl.tl_linear(w, q, s, z, out=y, mode=mode, workspace=ws)
        for _ in range(20):
            call()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 200
        e0.record(stream)
        for _ in range(reps):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
        host_us = e0.elapsed_time(e1) * 1e3 / reps
        cs = torch.cuda.Stream()
        cs.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cs):
            for _ in range(reps):
                call()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        lat_us = e0.elapsed_time(e1) * 1e3 / reps
        cold_us = _cold_us(torch, call, flush)
        alg = tl.tl_packed_bytes(M, K) + 4 * M + 2 * K + 4 * M + (4 * M + 8 if mode else 0)
        out[name] = {"latency_us": lat_us, "host_loop_us": host_us, "cold_us": cold_us,
                     "algorithmic_bytes": alg,
                     "cold_gbs": alg / (cold_us / 1e6) / 1e9,
                     "cold_frac_of_hbm": alg / (cold_us / 1e6) / 1e9 / hbm_peak}
    if cpu:
        from oracle import oracle as O
        P = O.pack(W)
        rs = O.rowsum(P, M, K)
        Qr, sr, zr = O.quant(x)
        for name, fn in (("oracle_mode_a", lambda nt: O.linear_a_mt(P, scale, M, K, x, nthreads=nt)),
                         ("oracle_mode_b", lambda nt: O.linear_b_mt(P, scale, rs, M, K, Qr, sr, zr,
                                                                     nthreads=nt))):
            res = {}
            for label, nt in (("single_thread_ms", 1), ("all_cores_ms", O.host_cores())):
                t = []
                for _ in range(5):
                    t0 = time.perf_counter()
                    fn(nt)
                    t.append((time.perf_counter() - t0) * 1e3)
                res[label] = statistics.median(t)
            res["cores"] = O.host_cores()
            out[name] = res
    return out


def bench_stack_line(shape, N, mode, args, torch, tl, hbm_peak, weights=None, **kw):
    from bit_matvec_ternary_b300.stack import LinearStack
    st = LinearStack(shape, N=N, mode=mode, out_dtype=tl.TL_OUT_F32, weights=weights, **kw)
    st.capture()
    ms = time_graph(st, args.steps, args.warmup, torch)
    a = st.algorithmic_bytes()
    line = {"tokens_s": N / (ms / 1e3), "ms_per_step": ms, "algorithmic_bytes": a,
            "gbs": a / (ms / 1e3) / 1e9, "frac_of_hbm": a / (ms / 1e3) / 1e9 / hbm_peak,
            "launches_per_step": st.launches_per_step}
    del st
    torch.cuda.empty_cache()
    return line


def bench_head(args, torch, tl, hbm_peak):
    """The int8 output head (151,936 x 4,096, one scale per row) with its
    fused argmax, at one and eight tokens; seeded synthetic table."""
    V, D = 151_936, 4096
    g = torch.Generator(device="cuda")
    g.manual_seed(1234)
    H = torch.randint(-128, 128, (V, D), dtype=torch.int8, device="cuda", generator=g)
    scale = torch.rand(V, device="cuda", generator=g) * 0.045 + 0.005
    head = tl.Head(H, scale)
    out = {}
    from bit_matvec_ternary_b300 import synth
    import numpy as np
    for N in (1, 8):
        x = synth.activations(N, D, seed=55, outlier_frac=0.01)
        xt = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).cuda()
        Q, s, z = tl.tl_quantize_act(xt)
        tok = torch.empty(N, dtype=torch.int32, device="cuda")
        best = torch.empty(N, dtype=torch.float32, device="cuda")
        stream = torch.cuda.current_stream()
        for _ in range(args.warmup):
            head.argmax(Q, s, z, token=tok, best=best)
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            head.argmax(Q, s, z, token=tok, best=best)
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        alg = V * D + 4 * V + N * D + 8 * N + 8 * N
        out[f"n{N}"] = {"us": ms * 1e3, "algorithmic_bytes": alg,
                        "gbs": alg / (ms / 1e3) / 1e9,
                        "frac_of_hbm": alg / (ms / 1e3) / 1e9 / hbm_peak,
                        "tokens_s": N / (ms / 1e3),
                        "kernel": "tl_head_kernel" if N <= 2 else "tl_head_mma_kernel"}
    out["shape"] = f"int8 {V}x{D}, fp32 scale per row, argmax fused, logits not written"
    return out


# ---------------------------------------------------------------- main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-n8", action="store_true", help="skip the N=8 lines")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle leg")
    ap.add_argument("--no-prefill", action="store_true", help="skip the N=512 prefill line")
    ap.add_argument("--no-head", action="store_true", help="skip the int8 head lines")
    ap.add_argument("--no-small", action="store_true",
                    help="skip the 0.6B stack and single-linear lines")
    ap.add_argument("--layers", type=int, default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        out = run_reference(args, rank, world)
        if out is not None:
            print(json.dumps(out), flush=True)
        return

    import torch
    import torch.distributed as dist
    from bit_matvec_ternary_b300 import build as tlbuild
    tlbuild.build()
    from bit_matvec_ternary_b300 import synth, tl
    from bit_matvec_ternary_b300.stack import LinearStack, StackWeights

    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    shape = synth.NEUTRINO_8B
    hbm_peak, peak_kind, bf16_peak, bf16_kind = peaks()

    # ---- N = 1, mode A: the headline
    t_gen = time.perf_counter()
    weights = StackWeights(shape, keep_host=(0,) if rank == 0 else (), layers=args.layers)
    t_gen = time.perf_counter() - t_gen
    stack = LinearStack(shape, N=1, mode=tl.TL_MODE_BF16, out_dtype=tl.TL_OUT_F32,
                        weights=weights)
    stack.capture()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        ms = time_graph(stack, args.steps, args.warmup, torch)
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
    clocks = clk.summary()
    t = torch.tensor([ms], device="cuda")
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms_max = float(t.item())
    tok_s = world * 1.0 / (ms_max / 1e3)
    alg = stack.algorithmic_bytes()
    gbs = alg / (ms_max / 1e3) / 1e9
    launches = stack.launches_per_step

    ms_e2e, h2d, d2h = time_e2e(stack, args.steps, args.warmup, torch)
    e2e = {"value": world / (ms_e2e / 1e3), "unit": "tokens/s", "ms_per_step": ms_e2e,
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
           "how": "per step: one replay of a graph holding the 144 C-ABI launches and the host "
                  "copies: each layer's inputs copied in from pinned host memory ahead of it "
                  "and its outputs copied out to pinned host memory after it, on two copy "
                  "streams beside the launches (all 144 inputs in, all 252 outputs out)"}
    # the same pass as one persistent chain launch (tl_chain_run), for comparison
    ms_chain = time_chain(stack.chain(), args.steps, args.warmup, torch)
    chain_line = {"ms_per_step": ms_chain, "tokens_s": 1.0 / (ms_chain / 1e3),
                  "launches_per_step": 1, "frac_of_hbm": alg / (ms_chain / 1e3) / 1e9 / hbm_peak,
                  "kernel": "tl_chain_kernel"}

    cpu = None
    host0 = stack.host                      # layer 0's matrices, for the oracle samples
    if rank == 0 and not args.no_cpu:
        sampler = OracleSample(stack.host, shape, 1)
        v, desc = sampler.run(seconds=10.0)
        cpu = {"value": v, "unit": "tokens/s", "cores": sampler.cores, "kind": "oracle",
               "sample": desc}
    del stack
    torch.cuda.empty_cache()

    extra = {}
    if not args.no_n8:
        # mode B at eight tokens: the quantisation inside each linear launch
        # (TL_MODE_I8_FUSED), with the two-launch form (a quantiser launch
        # before each linear launch) and its chain beside it
        for mode, name in ((tl.TL_MODE_BF16, "n8_mode_a"), (tl.TL_MODE_I8_FUSED, "n8_mode_b")):
            st8 = LinearStack(shape, N=8, mode=mode, out_dtype=tl.TL_OUT_F32, outlier_frac=0.01,
                              weights=weights)
            st8.capture()
            ms8 = time_graph(st8, args.steps, args.warmup, torch)
            a8 = st8.algorithmic_bytes()
            extra[name] = {"tokens_s": 8 / (ms8 / 1e3), "ms_per_step": ms8,
                           "algorithmic_bytes": a8, "gbs": a8 / (ms8 / 1e3) / 1e9,
                           "frac_of_hbm": a8 / (ms8 / 1e3) / 1e9 / hbm_peak,
                           "launches_per_step": st8.launches_per_step}
            if mode == tl.TL_MODE_I8_FUSED:
                del st8
                torch.cuda.empty_cache()
                extra[name]["two_launch"] = bench_stack_line(shape, 8, tl.TL_MODE_I8, args, torch,
                                                             tl, hbm_peak, weights=weights,
                                                             outlier_frac=0.01)
                st8 = LinearStack(shape, N=8, mode=tl.TL_MODE_I8, out_dtype=tl.TL_OUT_F32,
                                  outlier_frac=0.01, weights=weights)
            ms8c = time_chain(st8.chain(), args.steps, args.warmup, torch)
            extra[name]["chain"] = {"tokens_s": 8 / (ms8c / 1e3), "ms_per_step": ms8c,
                                    "frac_of_hbm": a8 / (ms8c / 1e3) / 1e9 / hbm_peak}
            del st8
            torch.cuda.empty_cache()
            if rank == 0 and not args.no_cpu:
                # the oracle on the same eight tokens' work (a bounded sample)
                s8 = OracleSample(host0, shape, 8)
                v8, d8 = s8.run(seconds=3.0, mode=0 if mode == tl.TL_MODE_BF16 else 1)
                extra[name]["cpu_oracle"] = {"value": v8, "unit": "tokens/s", "cores": s8.cores,
                                             "kind": "oracle", "sample": d8}

    # N = 1 in mode B: quantisation inside each linear launch, and the
    # two-launch form (a quantiser launch in front of every linear launch)
    extra["n1_mode_b"] = bench_stack_line(shape, 1, tl.TL_MODE_I8_FUSED, args, torch, tl,
                                          hbm_peak, weights=weights)
    extra["n1_mode_b"]["two_launch"] = bench_stack_line(shape, 1, tl.TL_MODE_I8, args, torch, tl,
                                                        hbm_peak, weights=weights)
    if not args.no_head:
        extra["head_argmax"] = bench_head(args, torch, tl, hbm_peak)
        torch.cuda.empty_cache()
    if not args.no_small:
        # the 0.6B-shaped stack (28 layers, hidden 1024), unit-RMS inputs
        extra["stack_06b_n1"] = bench_stack_line(synth.NEUTRINO_06B, 1, tl.TL_MODE_BF16, args,
                                                 torch, tl, hbm_peak, unit_rms=True)
        if rank == 0 and not args.no_cpu:
            # the oracle on layer 0 of the 0.6B-shaped stack (same seeds)
            sh6, host6 = synth.NEUTRINO_06B, {}
            for p in synth.PROJ_ORDER:
                M6, K6 = sh6.linear_shapes()[p]
                seed6 = synth.matrix_seed(0, 0, p)
                host6[(0, p)] = (synth.ternary(M6, K6, synth.zero_fraction(sh6, 0, p), seed6),
                                 synth.scales(M6, seed6))
            s6 = OracleSample(host6, sh6, 1)
            v6, d6 = s6.run(seconds=2.0)
            extra["stack_06b_n1"]["cpu_oracle"] = {"value": v6, "unit": "tokens/s",
                                                   "cores": s6.cores, "kind": "oracle",
                                                   "sample": d6}
        extra["single_linear_2048x1024"] = bench_single_linear(
            args, torch, tl, hbm_peak, cpu=rank == 0 and not args.no_cpu)
        extra.update(bench_neighbours(args, torch, tl, hbm_peak))
        torch.cuda.empty_cache()

    if not args.no_prefill:
        # prefill-sized batch: 512 tokens, int8 symmetric per-token activations,
        # bf16 out, every linear on the tcgen05 kernel; the quantiser writes the
        # integers as bf16 for it (TL_MODE_I8_FUSED: two launches per linear
        # group), with the three-launch form (quantiser, int8 -> bf16, linear)
        # beside it
        flops = 2.0 * shape.ternary_weights_per_layer() * (args.layers or shape.layers) * 512
        lines = {}
        for mode in (tl.TL_MODE_I8_FUSED, tl.TL_MODE_I8):
            stp = LinearStack(shape, N=512, mode=mode, out_dtype=tl.TL_OUT_BF16,
                              symmetric=True, weights=weights)
            stp.capture()
            msp = time_graph(stp, max(3, args.steps // 4), args.warmup, torch)
            lines[mode] = (msp, stp.launches_per_step + 4 * stp.layers)
            del stp
            torch.cuda.empty_cache()
        msp, nl = lines[tl.TL_MODE_I8_FUSED]
        tflops = flops / (msp / 1e3) / 1e12
        ms3, nl3 = lines[tl.TL_MODE_I8]
        extra["prefill_n512"] = {
            "tokens_s": 512 / (msp / 1e3), "ms_per_step": msp, "flops_per_step": flops,
            "mode": "B (int8 symmetric per-token, values fed to the tensor cores as exact bf16)",
            "out": "bf16",
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": bf16_peak,
                         "unit": "TFLOP/s", "frac": tflops / bf16_peak,
                         "peak_kind": bf16_kind, "kernel": "tl_prefill_kernel"},
            "launches_per_step": nl,
            "three_launch": {"tokens_s": 512 / (ms3 / 1e3), "ms_per_step": ms3,
                             "launches_per_step": nl3}}

    if rank == 0:
        out = {
            "metric": METRIC, "value": tok_s, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": 1, "seq_len": 1,
                       "parallelism": f"replicas x{world}" if world > 1 else "none",
                       "layers": args.layers or shape.layers,
                       "setup_s": round(t_gen, 1),
                       "l2": f"inputs larger than L2: {alg / 1e9:.3f} GB streamed per step vs "
                             f"{L2_BYTES / 2**20:.0f} MiB L2; no flush"},
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": gbs / hbm_peak, "traffic": measured_traffic(alg / launches),
                         "traffic_note": "bytes per launch: ncu DRAM bytes per algorithmic byte "
                                         "of one gate+up launch, times this step's mean "
                                         "algorithmic bytes per launch",
                         "kernel": "tl_mma_kernel",
                         "peak_kind": peak_kind + " (MEASURED_PEAKS.json hbm_gbs)",
                         "algorithmic_bytes_per_step": alg, "launches_per_step": launches,
                         "avg_launch_us": ms_max * 1e3 / launches},
            "chain": chain_line,
            "e2e": e2e,
            "gpu_launches": launches * args.steps,
            "clocks": clocks,
            "cpu_baseline": cpu,
        }
        out.update(extra)
        print(json.dumps(out), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

"""Throughput of the chunked test-time-training memory scan on GB300.

One step = one ttm_*_fwd call over the whole workload (every step of the scan:
loads, coefficients, scores, errors, reads, state carry, final state).
Default workload: Titans long context, B=1 H=16 T=131072 d=128 chunk 64, bf16
inputs (2.2 GB of inputs, larger than L2, so no flush is needed between steps).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload ID] [--impl ours|reference]

Prints one JSON line (rank 0).  With N > 1 (torchrun) every rank runs the same
workload on its own GPU with no communication on the data path (the scan's
sequences are independent), so scaling is weak; only the timing uses a
barrier and a max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import ttm_inputs as wl  # noqa: E402

METRIC = "memory-scan tokens/s (B·H·T per sec) on 1 GB300; % of roofline"
UNIT = "tokens/s"
DEFAULT_WORKLOAD = 4
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


# ----------------------------------------------------------------------------
# algorithmic work (what the chunked method must move and compute)
# ----------------------------------------------------------------------------

def algorithmic(w: wl.Workload) -> dict:
    """Bytes and FLOPs per token-head and per call.

    Bytes: q, k, v read and z written in the input dtype, the gates read (4 B
    each), the initial state read and the final state written once per (b, h).
    FLOPs: linear memory W.K, W.Q and the state update (6 d^2), Titans adds S.Q
    and the S update (10 d^2), plus 4 b d for the chunk's score and correction
    contractions; the 2-layer memory 22 hidden d + 2 b (2 d + 2 hidden).
    """
    es = 2 if w.dtype == "bf16" else 4
    d, b = w.d, w.chunk
    gates = 4 * (1 + (w.eta[0] != "zero") + (w.alpha[0] != "zero"))
    per_tok = 4 * d * es + gates
    seqs, nb0 = w.B * w.H, (1 if w.w0_shared else w.B) * w.H
    if w.kind == "mlp":
        state = 2 * w.hidden * d * 4                     # W1 and W2 of one sequence
        state_bytes = nb0 * state + seqs * 2 * state     # read W1_0, W2_0; write W1, W2, S1, S2
        flop_tok = 22 * w.hidden * d + 2 * b * (2 * d + 2 * w.hidden)
    else:
        state = d * d * 4
        state_bytes = nb0 * state + seqs * state * (2 if w.kind == "titans" else 1)
        flop_tok = (10 if w.kind == "titans" else 6) * d * d + 4 * b * d
    total_bytes = w.tokens * per_tok + state_bytes
    return dict(bytes_per_token=per_tok, flop_per_token=flop_tok, bytes=total_bytes,
                flops=w.tokens * flop_tok)


def load_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return {"hbm_gbs": float(j["hbm_gbs"]), "bf16_tflops": float(j["bf16_tflops"])}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def roof(flops: float, nbytes: float, kernel_s: float, fp32_kernel: bool) -> dict:
    """The roofline of the scan's target: t_roof is the slower of the
    algorithmic bytes at the measured HBM copy bandwidth and the algorithmic
    FLOPs at the measured dense bf16 tensor peak, whatever unit the kernel
    computes on; frac = t_roof / measured time.  A kernel that computes on the
    fp32 CUDA cores also reports its fraction of the fp32 FMA peak, as a
    secondary figure only."""
    peaks, src = load_peaks()
    t_hbm = nbytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = flops / (peaks["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        r = {"bound": "hbm", "achieved": nbytes / kernel_s / 1e9, "peak": peaks["hbm_gbs"],
             "unit": "GB/s"}
    else:
        r = {"bound": "tensor", "achieved": flops / kernel_s / 1e12,
             "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    r["frac"] = r["achieved"] / r["peak"]
    r["t_roof_s"] = max(t_hbm, t_tc)
    r["peak_source"] = src
    if fp32_kernel:
        alu = fp32_alu_peak_tflops(2070.0)
        r["fp32_alu"] = {"achieved": flops / kernel_s / 1e12, "peak": alu, "unit": "TFLOP/s",
                         "frac": flops / kernel_s / 1e12 / alu,
                         "peak_source": "derived: 152 SMs x 128 fp32 lanes x 2 x 2070 MHz"}
    r["algorithmic_bytes"] = nbytes
    r["algorithmic_flops"] = flops
    return r


def roofline(w: wl.Workload, kernel_s: float, kernel_name: str) -> dict:
    a = algorithmic(w)
    r = roof(a["flops"], a["bytes"], kernel_s, kernel_name.endswith("_simt"))
    r["kernel"] = kernel_name
    r["traffic"] = profiled_traffic(kernel_name, w)
    return r


def kernel_source_digest(kernel_name: str) -> str:
    src = {"linear_simt": ["scan_simt.cu"], "mlp_simt": ["scan_simt.cu", "scan_mlp_simt.cu", "scan_mlp_cluster.cu"],
           "linear_tc": ["scan_linear_tc.cu"], "mlp_tc": ["scan_mlp_tc.cu"],
           "linear_seq": ["scan_linear_seq.cu"],
           "linear_step": ["step.cu"], "dgd_tc": ["scan_dgd_tc.cu"],
           "bwd_tc": ["scan_linear_tc.cu", "scan_bwd_tc.cu"]}.get(kernel_name)
    if not src:
        return ""
    h = hashlib.sha256()
    try:
        for name in src:
            with open(os.path.join(ROOT, "test_neural_memory_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
        return h.hexdigest()[:16]
    except OSError:
        return ""


def profiled_traffic(kernel_name: str, w):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel source changed since the counters were taken.  `w` is a workload,
    or the key of a decode configuration ("decode_n1", ...)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            j = json.load(f)
    except (OSError, ValueError):
        return None
    e = j.get(f"{kernel_name}/{w}" if isinstance(w, str) else f"{kernel_name}/workload{w.id}")
    if not e or e.get("source_sha256_16") != kernel_source_digest(kernel_name):
        return None
    return e.get("dram_bytes_per_launch")


# ----------------------------------------------------------------------------
# decode step (--mode decode): n tokens per sequence per call, state resident
# ----------------------------------------------------------------------------

DECODE = dict(B=64, H=16, d=128, chunk=64)


def decode_algorithmic(B, H, d, chunk, n, es=2) -> dict:
    """Bytes one call must move: the state W, S and the chunk snapshot read
    once, W and S written once, the snapshot written once per chunk; q, k, v
    read and z written in the input dtype; three 4-byte gates per token."""
    state = d * d * 4
    per_seq = 3 * state + 2 * state + state * n / chunk + n * (4 * d * es + 12)
    return {"bytes": B * H * per_seq, "flops": B * H * n * 6 * d * d}


def run_decode(args, rank, world, dev):
    import test_neural_memory_gb300 as ttm

    c = DECODE
    n = args.decode_tokens
    B, H, d, chunk = c["B"], c["H"], c["d"], c["chunk"]
    name = f"titans decode step B{B} H{H} d{d} chunk {chunk}, {n} token(s) per call, bf16"
    w, inp = wl.generate_custom(kind="titans", dtype="bf16", B=B, H=H, T=n, d=d, chunk=chunk,
                                seed=1234)
    stream = torch.cuda.current_stream(dev)
    dd = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    W = dd["W0"].clone()
    S = torch.zeros_like(W)
    Wc = torch.empty_like(W)
    z = torch.empty_like(dd["v"])
    pos = [0]

    def step():
        _, _, pos[0] = ttm.titans_step(dd["q"], dd["k"], dd["v"], dd["theta"], W, chunk, pos[0],
                                       eta=dd["eta"], alpha=dd["alpha"], S=S, Wc=Wc, z=z,
                                       stream=stream)

    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak:
        step()
        torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    launches0 = ttm.launch_count()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.steps):
        step()
    g1.record(stream)
    torch.cuda.synchronize(dev)
    launches = ttm.launch_count() - launches0
    barrier(world)
    clocks = sampler.stop()
    ms = max_over_ranks(g0.elapsed_time(g1), world, dev) / args.steps
    status = ttm.device_status()
    if status != ttm.OK:
        raise RuntimeError(f"device status {ttm.status_str(status)}")

    a = decode_algorithmic(B, H, d, chunk, n)
    peaks, src = load_peaks()
    achieved = a["bytes"] / (ms / 1e3) / 1e9
    tokens = B * H * n
    # end to end: each call's token inputs go host -> device, its outputs z back
    host = {k: (None if v is None else v.pin_memory()) for k, v in inp.items() if k != "W0"}
    hz = torch.empty(z.shape, dtype=z.dtype, pin_memory=True)
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)

    def e2e_step():
        for k, v in host.items():
            if v is not None:
                dd[k].copy_(v, non_blocking=True)
        step()
        hz.copy_(z, non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ems = max_over_ranks(e0.elapsed_time(e1), world, dev) / args.steps
    line = {
        "metric": "decode-step tokens/s (B·H sequences x tokens per call) on 1 GB300; % of roofline",
        "value": tokens * world / (ms / 1e3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, "B": B, "H": H, "d": d, "chunk": chunk,
                   "tokens_per_call": n, "kind": "titans-step",
                   "parallelism": f"replicas{world}" if world > 1 else "single-gpu",
                   "l2": "state larger than L2 (no flush needed)"
                   if a["bytes"] > 129e6 else "L2 not flushed: state fits in L2",
                   "kernel": "linear_step"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                     "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"], "peak_source": src,
                     "kernel": "linear_step", "algorithmic_bytes": a["bytes"],
                     "algorithmic_flops": a["flops"],
                     "traffic": profiled_traffic("linear_step", f"decode_n{n}")},
        "e2e": {"value": tokens * world / (ems / 1e3), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": hz.numel() * hz.element_size(),
                "steps": args.steps, "ms_per_step": ems},
        "gpu_launches": launches, "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_decode_sample(B, H, d, chunk, args.cpu_seconds)
    return line


def oracle_decode_sample(B, H, d, chunk, seconds) -> dict:
    """The float64 oracle's token loop on a bounded sample of sequences: the
    same per-token work as a decode step (one gradient step and one read)."""
    import oracle
    seqs, T = 16, 64
    w, inp = wl.generate_custom(kind="titans", dtype="bf16", B=1, H=seqs, T=T, d=d, chunk=chunk,
                                seed=1234)
    f = lambda t: None if t is None else t.double().numpy()
    t0 = time.perf_counter()
    reps = 0
    while True:
        r = oracle.linear_primal(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["theta"]),
                                 f(inp["W0"]), chunk, eta=f(inp["eta"]), alpha=f(inp["alpha"]))
        reps += 1
        el = time.perf_counter() - t0
        if el > min(seconds, 5.0):
            break
    return {"value": seqs * T * reps / el, "unit": "tokens/s", "cores": r["threads"],
            "kind": "oracle", "seconds": el,
            "sample": f"{seqs} sequences x {T} tokens (d={d}), token loop, float64, x{reps}"}


# ----------------------------------------------------------------------------
# gradient of the scan (--mode bwd): one ttm_titans_bwd call per step
# ----------------------------------------------------------------------------

def fp32_alu_peak_tflops(sm_mhz: float) -> float:
    """Dense fp32 FMA rate of the CUDA cores: 152 SMs x 128 fp32 lanes x 2 FLOP
    per FMA x the SM clock."""
    return 152 * 128 * 2 * sm_mhz * 1e6 / 1e12


def bwd_algorithmic(w: wl.Workload) -> dict:
    """FLOPs and bytes of one gradient call, per token-head: the forward scan
    that rebuilds the chunk-start states (10 d^2 + 4 b d) plus the chunk-form
    backward products evaluated once (22 d^2 + 8 b d: the errors, the end-state
    adjoints applied to the keys, the state-adjoint update, W^T dz, S^T dz and
    the three key-gradient products, each 2 d^2; the masked b x b score and
    error products, 8 b d).  Bytes: q, k, v, dz read and dq, dk, dv written in
    the input dtype, three gates read and their gradients written."""
    es = 2 if w.dtype == "bf16" else 4
    d, b = w.d, w.chunk
    flop_tok = 32 * d * d + 12 * b * d
    byte_tok = 7 * d * es + 2 * 12
    return {"flops": w.tokens * flop_tok, "bytes": w.tokens * byte_tok,
            "flop_per_token": flop_tok, "bytes_per_token": byte_tok}


def run_bwd(args, rank, world, dev):
    import test_neural_memory_gb300 as ttm

    w = workload_of(args)
    if w.kind == "mlp":
        raise SystemExit("--mode bwd covers the linear / Titans memory")
    inp = wl.generate(w)
    adj = wl.generate_adjoints(w.B, w.H, w.T, w.d, w.d, dtype=w.dtype, seed=4321,
                               with_S=w.kind == "titans")
    stream = torch.cuda.current_stream(dev)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    a = {k: (None if v is None else v.to(dev)) for k, v in adj.items()}
    ws_bytes = ttm.lib().ttm_titans_bwd_workspace_size(w.B, w.H, w.T, w.d, w.d, w.chunk,
                                                       1 if w.dtype == "bf16" else 0,
                                                       int(w.w0_shared))
    ws = torch.empty(int(ws_bytes), dtype=torch.uint8, device=dev)
    out = ttm.titans_bwd(d["q"], d["k"], d["v"], d["theta"], d["W0"], w.chunk, a["dz"],
                         eta=d["eta"], alpha=d["alpha"], dW=a["dW"], dS=a["dS"],
                         w0_shared=w.w0_shared, workspace=ws, stream=stream)

    def step(dd=d, aa=a, oo=out):
        ttm.titans_bwd(dd["q"], dd["k"], dd["v"], dd["theta"], dd["W0"], w.chunk, aa["dz"],
                       eta=dd["eta"], alpha=dd["alpha"], dW=aa["dW"], dS=aa["dS"],
                       w0_shared=w.w0_shared, workspace=ws, out=oo, stream=stream)

    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak:
        step()
        torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    launches0 = ttm.launch_count()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.steps):
        step()
    g1.record(stream)
    torch.cuda.synchronize(dev)
    launches = ttm.launch_count() - launches0
    barrier(world)
    clocks = sampler.stop()
    ms = max_over_ranks(g0.elapsed_time(g1), world, dev) / args.steps
    status = ttm.device_status()
    if status != ttm.OK:
        raise RuntimeError(f"device status {ttm.status_str(status)}")

    # end to end: inputs and adjoints host -> device, every gradient back
    host_in = {k: v.pin_memory() for k, v in {**inp, **adj}.items() if v is not None}
    dev_in = {k: torch.empty_like(v, device=dev) for k, v in host_in.items()}
    host_out = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                for k, v in out.items() if v is not None}
    din = {k: dev_in.get(k) for k in inp}
    ain = {k: dev_in.get(k) for k in adj}
    out2 = {k: (None if v is None else torch.empty_like(v)) for k, v in out.items()}

    def e2e_step():
        for k, v in host_in.items():
            dev_in[k].copy_(v, non_blocking=True)
        step(din, ain, out2)
        for k, v in host_out.items():
            v.copy_(out2[k], non_blocking=True)

    e2e = None
    if args.e2e_steps > 0:
        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        ems = max_over_ranks(e0.elapsed_time(e1), world, dev) / args.e2e_steps
        e2e = {"value": w.tokens * world / (ems / 1e3), "unit": UNIT,
               "h2d_bytes_per_step": sum(v.numel() * v.element_size() for v in host_in.values()),
               "d2h_bytes_per_step": sum(v.numel() * v.element_size() for v in host_out.values()),
               "steps": args.e2e_steps, "ms_per_step": ems}

    alg = bwd_algorithmic(w)
    kern = ttm.last_kernel()  # bwd_tc: chain and local passes on tcgen05; bwd_simt: all fp32
    label = ("linear_bwd (chain, local pass: tcgen05; scores from the forward scan)"
             if kern == "bwd_tc" else "linear_bwd (all passes fp32)")
    line = {
        "metric": "gradient tokens/s (ttm_titans_bwd: dq, dk, dv, gates, W0) on 1 GB300",
        "value": w.tokens * world / (ms / 1e3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": w.name + " (gradient)", "B": w.B, "H": w.H, "T": w.T, "d": w.d,
                   "chunk": w.chunk, "kind": w.kind,
                   "parallelism": f"replicas{world}" if world > 1 else "single-gpu",
                   "l2": "inputs larger than L2 (no flush needed)", "kernel": kern,
                   "workspace_bytes": int(ws_bytes)},
        "roofline": dict(roof(alg["flops"], alg["bytes"], ms / 1e3, kern == "bwd_simt"),
                         kernel=label,
                         traffic=(profiled_traffic(kern, f"bwd_workload{w.id}")
                                  if kern == "bwd_tc" and not args.T else None)),
        "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_bwd_sample(w, inp, adj, args.cpu_seconds)
    return line


def oracle_bwd_sample(w, inp, adj, seconds) -> dict:
    """The float64 oracle's gradient on every (b, h) but only the first T_s tokens."""
    import oracle
    f = lambda t, T_s: None if t is None else t[:, :, :T_s].double().numpy()
    T_s = min(w.T, 2 * w.chunk)
    t0 = time.perf_counter()
    while True:
        r = oracle.linear_primal_bwd(f(inp["q"], T_s), f(inp["k"], T_s), f(inp["v"], T_s),
                                     f(inp["theta"], T_s), inp["W0"].double().numpy(), w.chunk,
                                     f(adj["dz"], T_s), eta=f(inp["eta"], T_s),
                                     alpha=f(inp["alpha"], T_s),
                                     dW=None if adj["dW"] is None else adj["dW"].double().numpy(),
                                     dS=None if adj["dS"] is None else adj["dS"].double().numpy(),
                                     shared_over_batch=w.w0_shared)
        dt = time.perf_counter() - t0
        if dt > seconds / 4 or T_s >= w.T:
            break
        T_s = min(w.T, T_s * 2)
        t0 = time.perf_counter()
    tokens = w.B * w.H * T_s
    return {"value": tokens / dt, "unit": UNIT, "cores": int(r["threads"]), "kind": "oracle",
            "seconds": dt, "sample": f"all {w.B * w.H} (b,h) sequences, first {T_s} of {w.T} "
                                     f"tokens each, float64 reverse mode, {r['threads']} threads"}


# ----------------------------------------------------------------------------
# DGD memory scan (--mode dgd): one ttm_dgd_fwd call per step
# ----------------------------------------------------------------------------

def run_dgd(args, rank, world, dev):
    import test_neural_memory_gb300 as ttm

    w = workload_of(args)
    inp = wl.generate(w)
    gates = wl.generate_dgd_gates(w.B, w.H, w.T, seed=77)
    stream = torch.cuda.current_stream(dev)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    g = {k: v.to(dev) for k, v in gates.items()}
    z = torch.empty_like(d["v"])
    W = torch.empty((w.B, w.H, w.d, w.d), dtype=torch.float32, device=dev)

    def step():
        ttm.dgd_fwd(d["q"], d["k"], d["v"], g["eta"], g["alpha"], d["W0"], w.chunk,
                    w0_shared=w.w0_shared, z=z, W_out=W, stream=stream)

    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak:
        step()
        torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    launches0 = ttm.launch_count()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.steps):
        step()
    g1.record(stream)
    torch.cuda.synchronize(dev)
    launches = ttm.launch_count() - launches0
    barrier(world)
    clocks = sampler.stop()
    ms = max_over_ranks(g0.elapsed_time(g1), world, dev) / args.steps
    if ttm.device_status() != ttm.OK:
        raise RuntimeError("device status")
    kernel = ttm.last_kernel()
    es = 2 if w.dtype == "bf16" else 4
    byte_tok = 4 * w.d * es + 8                     # q, k, v, z and the two gates
    state = w.d * w.d * 4
    nbytes = w.tokens * byte_tok + w.B * w.H * 2 * state
    # chunk form per token: [Q; K] W^T, A~N R0 and Y R0, plus the pre-pass's
    # scores [Q; K] K^T, A~N and Y = K^T diag(r) N per 64-token chunk
    dk = dv = w.d
    c = 64
    flops_tok = (4 * dk * dv + 2 * c * dv + 2 * dk * dv +
                 (2 * 2 * c * c * dk + 2 * c * c * c + 2 * dk * c * c) / c)
    rl = roof(flops_tok * w.tokens, nbytes, ms / 1e3, kernel == "dgd_step")
    rl.update({"kernel": kernel,
               "traffic": profiled_traffic(kernel, f"dgd_workload{w.id}") if not args.T else None})
    line = {
        "metric": "DGD-memory scan tokens/s (ttm_dgd_fwd) on 1 GB300",
        "value": w.tokens * world / (ms / 1e3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": w.name + " (DGD update)", "B": w.B, "H": w.H, "T": w.T,
                   "d": w.d, "chunk": w.chunk, "kind": "dgd",
                   "parallelism": f"replicas{world}" if world > 1 else "single-gpu",
                   "l2": "inputs larger than L2 (no flush needed)", "kernel": kernel},
        "roofline": rl,
        "e2e": None, "gpu_launches": launches, "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        T_s = min(w.T, 2048)
        f = lambda t: t[:, :, :T_s].double().numpy()
        t0 = time.perf_counter()
        r = oracle.dgd_primal(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(gates["eta"]),
                              f(gates["alpha"]), inp["W0"].double().numpy(), w.chunk,
                              shared_over_batch=w.w0_shared)
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": w.B * w.H * T_s / dt, "unit": UNIT,
                                "cores": int(r["threads"]), "kind": "oracle", "seconds": dt,
                                "sample": f"all {w.B * w.H} sequences, first {T_s} tokens"}
    return line


# ----------------------------------------------------------------------------
# LMM layer (--mode layer): one ttm_lmm_layer_fwd call per step
# ----------------------------------------------------------------------------

def run_layer(args, rank, world, dev):
    import test_neural_memory_gb300 as ttm

    w = workload_of(args)
    B, T, Hh, d = w.B, w.T, w.H, w.d
    D = Hh * d
    p = wl.generate_lmm(B, T, Hh, d, conv_k=4, seed=99)
    dp = {k: v.to(dev) for k, v in p.items()}
    stream = torch.cuda.current_stream(dev)
    n_ws = int(ttm.lib().ttm_lmm_layer_workspace_size(B, T, Hh, d, w.chunk, 1))
    ws = torch.empty(n_ws, dtype=torch.uint8, device=dev)
    y = torch.empty_like(dp["x"])
    Wout = torch.empty((B, Hh, d, d), dtype=torch.float32, device=dev)
    Sout = torch.empty_like(Wout)

    def step():
        ttm.lmm_layer_fwd(dp["x"], dp["W_in"], dp["conv_w"], dp["rms_w"], dp["W_o"], 0.1,
                          dp["W0"], w.chunk, y=y, W_out=Wout, S_out=Sout, workspace=ws,
                          stream=stream)

    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak:
        step()
        torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    launches0 = ttm.launch_count()
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.steps):
        step()
    g1.record(stream)
    torch.cuda.synchronize(dev)
    launches = ttm.launch_count() - launches0
    barrier(world)
    clocks = sampler.stop()
    ms = max_over_ranks(g0.elapsed_time(g1), world, dev) / args.steps
    if ttm.device_status() != ttm.OK:
        raise RuntimeError("device status")
    P = 4 * D + 3 * Hh
    gemm_flops = 2 * B * T * D * (P + D)
    scan_flops = algorithmic(w)["flops"]
    flops = gemm_flops + scan_flops
    peaks, src = load_peaks()
    achieved = flops / (ms / 1e3) / 1e12
    line = {
        "metric": "LMM-layer tokens/s (ttm_lmm_layer_fwd: projections, conv, scan, output) on 1 GB300",
        "value": B * T * world / (ms / 1e3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic, random-init weights",
        "config": {"workload": f"LMM layer B{B} T{T} H{Hh} d{d} (D={D}) chunk {w.chunk} conv 4",
                   "B": B, "T": T, "H": Hh, "d": d, "chunk": w.chunk,
                   "parallelism": f"replicas{world}" if world > 1 else "single-gpu",
                   "l2": "inputs larger than L2 (no flush needed)", "kernel": "lmm layer"},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                     "peak_source": src, "kernel": "lmm layer (whole call)",
                     "algorithmic_flops": flops, "gemm_flops": gemm_flops,
                     "scan_flops": scan_flops, "traffic": None},
        "e2e": None, "gpu_launches": launches, "clocks": clocks,
    }
    return line


# ----------------------------------------------------------------------------
# clocks sampled while the GPU is under load
# ----------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.rows: list[list[str]] = []
        self.proc = None
        self.uuid = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            self.uuid = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if self.uuid:
            cmd.insert(1, f"--id={self.uuid if self.uuid.startswith('GPU-') else 'GPU-' + self.uuid}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=5)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            if len(r) < 8:
                continue
            try:
                sm.append(float(r[0]))
                smax.append(float(r[1]))
            except ValueError:
                continue
            for n, val in zip(names, r[4:8]):
                if val.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def call_fn(w: wl.Workload, d: dict, outs: dict, stream):
    import test_neural_memory_gb300 as ttm
    if w.kind == "linear":
        return lambda: ttm.linear_fwd(d["q"], d["k"], d["v"], d["theta"], d["W0"], w.chunk,
                                      w0_shared=w.w0_shared, z=outs["z"], W_out=outs["W"],
                                      workspace=outs["ws"], stream=stream)
    if w.kind == "titans":
        return lambda: ttm.titans_fwd(d["q"], d["k"], d["v"], d["theta"], d["W0"], w.chunk,
                                      eta=d["eta"], alpha=d["alpha"], w0_shared=w.w0_shared,
                                      z=outs["z"], W_out=outs["W"], S_out=outs["S"],
                                      workspace=outs["ws"], stream=stream)
    return lambda: ttm.mlp_fwd(d["q"], d["k"], d["v"], d["theta"], d["W1_0"], d["W2_0"],
                               w.chunk, eta=d["eta"], alpha=d["alpha"], w0_shared=w.w0_shared,
                               z=outs["z"], W1_out=outs["W1"], W2_out=outs["W2"],
                               S1_out=outs["S1"], S2_out=outs["S2"], stream=stream)


def alloc_outputs(w: wl.Workload, dev, pin=False) -> dict:
    es = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    mk = lambda shape, dt=torch.float32: torch.empty(shape, dtype=dt, device=dev,
                                                     pin_memory=pin)
    o = {"z": mk((w.B, w.H, w.T, w.d), es)}
    if w.kind == "mlp":
        o.update(W1=mk((w.B, w.H, w.hidden, w.d)), W2=mk((w.B, w.H, w.d, w.hidden)),
                 S1=mk((w.B, w.H, w.hidden, w.d)), S2=mk((w.B, w.H, w.d, w.hidden)))
    else:
        import test_neural_memory_gb300 as ttm
        o["W"] = mk((w.B, w.H, w.d, w.d))
        o["S"] = mk((w.B, w.H, w.d, w.d)) if w.kind == "titans" else None
        # scratch for the per-chunk coefficients (device only; not an output)
        nbytes = ttm.linear_workspace_size(w.B, w.H, w.T, w.d, w.d, w.chunk,
                                           ttm.BF16 if w.dtype == "bf16" else ttm.F32)
        o["ws"] = (torch.empty(nbytes, dtype=torch.uint8, device=dev if not pin else "cuda")
                   if nbytes else None)
    return o


def oracle_sample(w: wl.Workload, inp: dict, T_s: int, keep: dict | None = None) -> dict:
    """Time the float64 oracle, as it stands, on every (b, h) of the workload
    but only its first T_s tokens.  If `keep` is a dict, the oracle's reads z
    of those tokens are stored in keep["z"] (for the parity figures)."""
    import oracle
    f = lambda t: None if t is None else t[:, :, :T_s].double().numpy()
    t0 = time.perf_counter()
    if w.kind == "mlp":
        r = oracle.mlp_primal(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["theta"]),
                              inp["W1_0"].double().numpy(), inp["W2_0"].double().numpy(),
                              w.chunk, eta=f(inp["eta"]), alpha=f(inp["alpha"]),
                              shared_over_batch=w.w0_shared)
    else:
        r = oracle.linear_primal(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["theta"]),
                                 inp["W0"].double().numpy(), w.chunk, eta=f(inp["eta"]),
                                 alpha=f(inp["alpha"]), shared_over_batch=w.w0_shared)
    dt = time.perf_counter() - t0
    if keep is not None:
        keep["z"] = r["z"]
    tokens = w.B * w.H * min(T_s, w.T)
    return {"value": tokens / dt, "unit": UNIT, "cores": int(r["threads"]), "kind": "oracle",
            "seconds": dt,
            "sample": f"all {w.B * w.H} (b,h) sequences, first {min(T_s, w.T)} of {w.T} tokens "
                      f"each ({tokens} token-heads), float64, {r['threads']} threads"}


def oracle_tokens_for(w: wl.Workload, seconds: float) -> int:
    """Tokens per sequence that keep the oracle near `seconds` on this host,
    from a short calibration run."""
    inp = wl.generate(w.shrink(T=min(w.T, 256)))
    probe = oracle_sample(w.shrink(T=min(w.T, 256)), inp, 256)
    per_tok = probe["seconds"] / min(w.T, 256)
    T_s = int(max(w.chunk, min(w.T, seconds / max(per_tok, 1e-9))))
    return max(w.chunk, (T_s // w.chunk) * w.chunk) if T_s >= w.chunk else T_s


def run_ours(args, rank, world, dev):
    import test_neural_memory_gb300 as ttm

    w_full = workload_of(args)
    inp = wl.generate(w_full)
    if args.shard == "bh":
        lo, hi = shard_bh(w_full.B, w_full.H, rank, world)
        w, inp = shard_inputs(w_full, inp, lo, hi)
    else:
        w = w_full
    stream = torch.cuda.current_stream(dev)
    d = {k: (None if v is None else v.to(dev)) for k, v in inp.items()}
    outs = alloc_outputs(w, dev)
    step = call_fn(w, d, outs, stream)

    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    kernel_name = ttm.last_kernel()
    # keep the GPU busy ~1 s before the timed region so the clock record has samples
    t_soak = time.perf_counter()
    while time.perf_counter() - t_soak < args.soak:
        step()
        torch.cuda.synchronize(dev)
    barrier(world)
    torch.cuda.synchronize(dev)
    launches0 = ttm.launch_count()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for a, b in ev:
        a.record(stream)
        step()
        b.record(stream)
    g1.record(stream)
    torch.cuda.synchronize(dev)
    launches = ttm.launch_count() - launches0
    barrier(world)
    clocks = sampler.stop()
    total_ms = g0.elapsed_time(g1)
    kern_ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps
    total_ms = max_over_ranks(total_ms, world, dev)
    kern_ms = max_over_ranks(kern_ms, world, dev)
    status = ttm.device_status()
    if status != ttm.OK:
        raise RuntimeError(f"device status {ttm.status_str(status)}")

    # end to end through the public API with host buffers
    e2e = run_e2e(args, w, inp, dev, stream, world) if args.e2e_steps > 0 else None

    sharded = args.shard == "bh"
    job_tokens = w_full.tokens if sharded else w.tokens * world
    value = job_tokens * args.steps / (total_ms / 1e3)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "strong" if sharded else "weak", "vs_baseline": None, "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": w_full.name, "B": w_full.B, "H": w_full.H, "T": w.T, "d": w.d,
                   "chunk": w.chunk, "kind": w.kind, "hidden": w.hidden or None,
                   "parallelism": (f"bh-shard{world}" if sharded else
                                   (f"replicas{world}" if world > 1 else "single-gpu")),
                   "l2": "inputs larger than L2 (no flush needed)"
                   if algorithmic(w)["bytes"] > 129e6 else "L2 not flushed: inputs fit in L2",
                   "kernel": kernel_name},
        "roofline": roofline(w, kern_ms / 1e3, kernel_name),
        "e2e": e2e, "gpu_launches": launches, "clocks": clocks,
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        T_s = oracle_tokens_for(w, args.cpu_seconds)
        keep = {}
        line["cpu_baseline"] = oracle_sample(w, inp, T_s, keep)
        line["parity"] = parity_of(outs["z"][:, :, :T_s], keep["z"], w.dtype)
    return line


def parity_of(z_gpu, z_ref, dtype: str) -> dict:
    """The GPU reads of the timed call against the oracle's on the tokens the
    CPU baseline ran (a prefix of every sequence: the scan is causal, so the
    full-length call's first tokens are exactly the oracle's case).  Normwise
    max|gpu - oracle| / max|oracle| is the pass criterion; the elementwise
    error with a 1e-6 max floor is reported beside it."""
    import numpy as np
    g = z_gpu.detach().double().cpu().numpy()
    r = np.asarray(z_ref, dtype=np.float64)
    scale = float(np.abs(r).max()) if r.size else 0.0
    diff = np.abs(g - r)
    normwise = float(diff.max() / scale) if scale > 0 else float(diff.max(initial=0.0))
    elem = float((diff / (np.abs(r) + 1e-6 * scale)).max()) if scale > 0 else normwise
    tol = 2e-2 if dtype == "bf16" else 1e-4
    return {"output": "z", "tokens_checked": int(r.shape[0] * r.shape[1] * r.shape[2]),
            "normwise": normwise, "elementwise_floor_1e-6": elem, "tol_normwise": tol,
            "pass": normwise <= tol}


E2E_SEGMENT = 8192   # tokens per segment of the host-buffer scan


def run_e2e(args, w, inp, dev, stream, world):
    """Same metric through the public API with pinned host inputs: every step
    copies its inputs host->device and reads the outputs back.  The linear /
    Titans scan uses its host-buffer entry point (ttm_titans_fwd_host), which
    overlaps the copies of one segment with the scan of the next; the 2-layer
    memory copies everything in, scans, and copies everything out."""
    if w.kind != "mlp":
        return run_e2e_host(args, w, inp, dev, stream, world)
    host = {k: (None if v is None else v.pin_memory()) for k, v in inp.items()}
    dbuf = {k: (None if v is None else torch.empty_like(v, device=dev)) for k, v in inp.items()}
    outs = alloc_outputs(w, dev)
    hout = {k: (None if v is None or k == "ws" else
                torch.empty(v.shape, dtype=v.dtype, pin_memory=True)) for k, v in outs.items()}
    step = call_fn(w, dbuf, outs, stream)
    h2d = sum(v.numel() * v.element_size() for v in host.values() if v is not None)
    d2h = sum(v.numel() * v.element_size() for v in hout.values() if v is not None)

    def one():
        for k, v in host.items():
            if v is not None:
                dbuf[k].copy_(v, non_blocking=True)
        step()
        for k, v in outs.items():
            if hout.get(k) is not None:
                hout[k].copy_(v, non_blocking=True)

    for _ in range(max(1, min(args.warmup, 3))):
        one()
    torch.cuda.synchronize(dev)
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = args.e2e_steps
    a.record(stream)
    for _ in range(n):
        one()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(a.elapsed_time(b), world, dev)
    return {"value": w.tokens * world * n / (ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "ms_per_step": ms / n}


def run_e2e_host(args, w, inp, dev, stream, world):
    import test_neural_memory_gb300 as ttm
    h = {k: (None if v is None else v.contiguous().pin_memory()) for k, v in inp.items()}
    outs = alloc_outputs(w, "cpu", pin=True)
    seg = min(E2E_SEGMENT, (w.T + w.chunk - 1) // w.chunk * w.chunk)
    seg = max(w.chunk, seg // w.chunk * w.chunk)
    need = ttm.titans_fwd_host_workspace_size(w.B, w.H, w.T, w.d, w.d, w.chunk,
                                              ttm.BF16 if w.dtype == "bf16" else ttm.F32, seg)
    ws = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    titans = w.kind == "titans"

    def one():
        ttm.titans_fwd_host(h["q"], h["k"], h["v"], h["theta"], h["W0"], w.chunk,
                            eta=h["eta"] if titans else None, alpha=h["alpha"] if titans else None,
                            w0_shared=w.w0_shared, z=outs["z"], W_out=outs["W"],
                            S_out=outs["S"] if titans else None, want_S=titans,
                            seg_tokens=seg, workspace=ws, device=dev, stream=stream)

    h2d = sum(v.numel() * v.element_size() for k, v in h.items()
              if v is not None and (titans or k not in ("eta", "alpha")))
    d2h = sum(v.numel() * v.element_size() for k, v in outs.items()
              if v is not None and k != "ws")
    for _ in range(max(1, min(args.warmup, 3))):
        one()
    torch.cuda.synchronize(dev)
    barrier(world)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n = args.e2e_steps
    a.record(stream)
    for _ in range(n):
        one()
    b.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(a.elapsed_time(b), world, dev)
    return {"value": w.tokens * world * n / (ms / 1e3), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": n,
            "ms_per_step": ms / n, "api": f"ttm_titans_fwd_host, {seg}-token segments"}


# ----------------------------------------------------------------------------
# reference arm: the float64 oracle on the host cores
# ----------------------------------------------------------------------------

def workload_of(args) -> wl.Workload:
    """The named workload, optionally with a shorter sequence (profiling runs)."""
    w = wl.WORKLOADS[args.workload]
    if args.T:
        w = w.shrink(T=args.T, name=f"{w.name} (T shortened to {args.T})")
    return w


def run_reference(args):
    w = workload_of(args)
    per_step = max(0.5, args.reference_seconds / max(1, args.steps + args.warmup))
    T_s = oracle_tokens_for(w, per_step)
    inp = wl.generate(w.shrink(T=T_s))
    for _ in range(args.warmup):
        oracle_sample(w, inp, T_s)
    times = []
    last = None
    for _ in range(args.steps):
        last = oracle_sample(w, inp, T_s)
        times.append(last["seconds"])
    tokens = w.B * w.H * T_s
    value = tokens * len(times) / sum(times)
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * sum(times) / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "T": w.T, "d": w.d,
                   "chunk": w.chunk, "kind": w.kind, "hidden": w.hidden or None,
                   "sample_tokens_per_sequence": T_s},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": last["cores"], "kind": "oracle",
                         "sample": last["sample"]},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


# ----------------------------------------------------------------------------

def shard_bh(B: int, H: int, rank: int, world: int) -> tuple[int, int]:
    """The (b, h) sequences of rank `rank` under --shard bh: a contiguous,
    balanced range [lo, hi) of the flat unit index b * H + h.  The sequences
    are independent, so each rank scans its own with no exchange."""
    n = B * H
    base, extra = divmod(n, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def shard_inputs(w: wl.Workload, inp: dict, lo: int, hi: int) -> tuple[wl.Workload, dict]:
    """Inputs of units lo..hi-1 as one batch row of hi - lo heads: q, k, v and
    gates [1, n, T, .], the initial memory of each unit gathered to [1, n, ...]
    (a shared initial memory is expanded per unit)."""
    n = hi - lo
    flat = lambda t: None if t is None else t.reshape(w.B * w.H, *t.shape[2:])[lo:hi].unsqueeze(0)
    out = {k: flat(inp[k]) for k in ("q", "k", "v", "theta", "eta", "alpha")}
    heads = torch.arange(lo, hi) % w.H
    batch = torch.arange(lo, hi) // w.H
    for k in ("W0", "W1_0", "W2_0"):
        if k in inp:
            t = inp[k]
            out[k] = (t[0, heads] if w.w0_shared else t[batch, heads]).unsqueeze(0).contiguous()
    out = {k: (None if v is None else v.contiguous()) for k, v in out.items()}
    return w.shrink(B=1, H=n, w0_shared=False), out


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(x: float, world: int, dev) -> float:
    if world == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, choices=sorted(wl.WORKLOADS))
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--soak", type=float, default=1.0, help="seconds of untimed load before timing")
    ap.add_argument("--e2e-steps", type=int, default=5, help="0 skips the end-to-end leg")
    ap.add_argument("--T", type=int, default=0,
                    help="shorten the sequence (profiling only; the metric line says so)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--reference-seconds", type=float, default=120.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--mode", choices=["scan", "decode", "bwd", "dgd", "layer"], default="scan",
                    help="decode: the streaming decode step; bwd: the scan's gradient; "
                         "dgd: the DGD-memory scan; layer: the LMM layer")
    ap.add_argument("--decode-tokens", type=int, default=1, help="tokens per decode call")
    ap.add_argument("--shard", choices=["none", "bh"], default="none",
                    help="bh: split the workload's (b, h) sequences over the ranks "
                         "(strong scaling, no exchange); none: one replica per rank")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    import test_neural_memory_gb300 as ttm
    ttm.build()
    runner = {"scan": run_ours, "decode": run_decode, "bwd": run_bwd, "dgd": run_dgd,
              "layer": run_layer}[args.mode]
    line = runner(args, rank, world, dev)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

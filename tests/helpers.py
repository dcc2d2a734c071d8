"""Shared test plumbing: run the GPU library and the oracle on the same inputs
and compare them with the tolerance rule of the scan's parity bar.

Tolerance rule: for each output tensor, max|gpu - oracle| / max|oracle| must
stay below 1e-4 when q, k, v are fp32 and 2e-2 when they are bf16 (fp32
accumulation in both cases).  The elementwise error with a 1e-6 max floor is
reported next to it.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = {"f32": 1e-4, "bf16": 2e-2}


def max_rel(gpu, ref) -> float:
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.abs(ref).max() if ref.size else 0.0
    if ref.size == 0:
        return 0.0
    if scale == 0.0:
        return float(np.abs(gpu).max())
    return float(np.abs(gpu - ref).max() / scale)


def max_rel_elem(gpu, ref, floor=1e-6) -> float:
    """Elementwise relative error with an absolute floor of floor * max|ref|:
    max over elements of |gpu - ref| / (|ref| + floor * max|ref|).  Reported
    next to the normwise bound; it is large wherever an output is tiny next to
    the tensor's largest entry, so it is not the pass criterion."""
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if ref.size == 0:
        return 0.0
    scale = np.abs(ref).max()
    den = np.abs(ref) + floor * scale
    if scale == 0.0:
        return float(np.abs(gpu).max())
    return float((np.abs(gpu - ref) / den).max())


def to_dev(inp: dict, device="cuda") -> dict:
    return {k: (None if v is None else v.to(device)) for k, v in inp.items()}


def f64(t):
    return None if t is None else t.detach().double().cpu().numpy()


def run_linear_gpu(w, inp, kind=None, device="cuda", S0=None):
    import test_neural_memory_gb300 as ttm
    kind = kind or w.kind
    d = to_dev(inp, device)
    if kind == "linear":
        z, W = ttm.linear_fwd(d["q"], d["k"], d["v"], d["theta"], d["W0"], w.chunk,
                              w0_shared=w.w0_shared)
        S = None
    else:
        S0d = None if S0 is None else S0.to(device)
        z, W, S = ttm.titans_fwd(d["q"], d["k"], d["v"], d["theta"], d["W0"], w.chunk,
                                 eta=d["eta"], alpha=d["alpha"], S0=S0d, w0_shared=w.w0_shared)
    torch.cuda.synchronize()
    return dict(z=z, W=W, S=S, kernel=ttm.last_kernel())


def run_linear_oracle(w, inp, heads=None, S0=None):
    """Oracle on every (b, h) or on the listed head indices only (all batch rows)."""
    sel = slice(None) if heads is None else list(heads)
    pick = lambda t: None if t is None else f64(t)[:, sel]
    W0 = f64(inp["W0"])[:, sel]
    r = oracle.linear_primal(pick(inp["q"]), pick(inp["k"]), pick(inp["v"]), pick(inp["theta"]),
                             W0, w.chunk, eta=pick(inp["eta"]), alpha=pick(inp["alpha"]),
                             S0=None if S0 is None else f64(S0)[:, sel],
                             shared_over_batch=w.w0_shared)
    return r


def run_mlp_gpu(w, inp, device="cuda", S1_0=None, S2_0=None):
    import test_neural_memory_gb300 as ttm
    d = to_dev(inp, device)
    dev = lambda t: None if t is None else t.to(device=device, dtype=torch.float32).contiguous()
    z, W1, W2, S1, S2 = ttm.mlp_fwd(d["q"], d["k"], d["v"], d["theta"], d["W1_0"], d["W2_0"],
                                    w.chunk, eta=d["eta"], alpha=d["alpha"],
                                    S1_0=dev(S1_0), S2_0=dev(S2_0), w0_shared=w.w0_shared)
    torch.cuda.synchronize()
    return dict(z=z, W1=W1, W2=W2, S1=S1, S2=S2, kernel=ttm.last_kernel())


def run_mlp_oracle(w, inp, heads=None, S1_0=None, S2_0=None):
    sel = slice(None) if heads is None else list(heads)
    pick = lambda t: None if t is None else f64(t)[:, sel]
    return oracle.mlp_primal(pick(inp["q"]), pick(inp["k"]), pick(inp["v"]), pick(inp["theta"]),
                             pick(inp["W1_0"]), pick(inp["W2_0"]), w.chunk, eta=pick(inp["eta"]),
                             alpha=pick(inp["alpha"]), S1_0=pick(S1_0), S2_0=pick(S2_0),
                             shared_over_batch=w.w0_shared)


def compare(gpu: dict, ref: dict, names, tol, heads=None) -> dict:
    """Normwise check per output tensor (the pass criterion); the elementwise
    error with a 1e-6 max floor is reported alongside in the failure message."""
    errs, elem = {}, {}
    for n in names:
        g = f64(gpu[n])
        if heads is not None:
            g = g[:, list(heads)]
        errs[n] = max_rel(g, ref[n])
        elem[n] = max_rel_elem(g, ref[n])
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, (f"parity failed (tol {tol}): normwise {errs}; "
                     f"elementwise (1e-6 max floor) {elem}")
    return errs

"""Failure detection without a GPU fault.

- Host side: the test hooks validate their arguments, and an injected launch
  failure (TTM_DBG_FAIL_CALLS) comes back through the binding as a TTMError
  with TTM_ERR_CUDA, after which calls succeed again.
- Device side: a bounded wait of the tensor-core scan is made to run out (a
  chunk whose barrier is announced 16 bytes more than is copied, so the wait
  can never complete) under a short wait limit; the call returns, the device
  status word reports TTM_ERR_TIMEOUT once, and the next call is correct.  The
  same for the chain pass of the tensor-core gradient.
- Non-finite data: a step size far above the pages' stability bound
  ("TTT layers 与 fast weights" §1.2, eq (12): 0 < theta |k|^2 < 1 in this
  scale) makes the memory grow by ~300x per chunk; the scan must neither hang
  nor invent finite numbers: its reads are finite wherever the float64 oracle's
  are well inside the fp32 range and non-finite wherever the oracle's exceed it.
"""
import time

import numpy as np
import pytest
import torch

import test_neural_memory_gb300 as ttm
import ttm_inputs as wl
from tests import helpers as H

gpu = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _reset_hooks():
    ttm.build()
    yield
    for opt, val in (("wait_cycles", 0), ("stall_chunk", -1), ("fail_calls", 0)):
        ttm.lib().ttm_debug_set(ttm.DEBUG[opt], val)


def test_debug_hooks_validate_their_arguments():
    L = ttm.lib()
    assert L.ttm_debug_set(99, 0) == ttm.ERR_INVALID_ARG
    assert L.ttm_debug_set(ttm.DEBUG["wait_cycles"], -5) == ttm.ERR_INVALID_ARG
    assert L.ttm_debug_set(ttm.DEBUG["stall_chunk"], -2) == ttm.ERR_INVALID_ARG
    assert L.ttm_debug_set(ttm.DEBUG["fail_calls"], -1) == ttm.ERR_INVALID_ARG
    for opt, val in (("wait_cycles", 1000), ("stall_chunk", 3), ("fail_calls", 2)):
        assert L.ttm_debug_set(ttm.DEBUG[opt], val) == ttm.OK
    with pytest.raises(ttm.TTMError) as e:
        ttm.debug_set("wait_cycles", -1)
    assert e.value.code == ttm.ERR_INVALID_ARG


def _small_titans(seed=7, T=256, d=64):
    w, inp = wl.generate_custom(kind="titans", dtype="bf16", B=1, H=2, T=T, d=d, chunk=64,
                                seed=seed)
    return w, inp, H.to_dev(inp)


def _titans(w, d):
    return ttm.titans_fwd(d["q"], d["k"], d["v"], d["theta"], d["W0"], w.chunk, eta=d["eta"],
                          alpha=d["alpha"])


@gpu
def test_injected_launch_failure_reaches_the_caller():
    w, inp, d = _small_titans()
    ttm.debug_set("fail_calls", 1)
    with pytest.raises(ttm.TTMError) as e:
        _titans(w, d)
    assert e.value.code == ttm.ERR_CUDA
    z, W, S = _titans(w, d)            # the hook is used up: this one runs
    torch.cuda.synchronize()
    ref = H.run_linear_oracle(w, inp)
    H.compare({"z": z, "W": W, "S": S}, ref, ["z", "W", "S"], H.TOL["bf16"])
    assert ttm.device_status() == ttm.OK


@gpu
def test_bounded_wait_runs_out_and_the_next_call_is_correct():
    w, inp, d = _small_titans()
    assert ttm.device_status() == ttm.OK
    with ttm.kernel_policy("tc"):
        ttm.debug_set("wait_cycles", 20_000_000)     # ~10 ms at 2 GHz
        ttm.debug_set("stall_chunk", 1)
        t0 = time.perf_counter()
        _titans(w, d)
        assert ttm.last_kernel() == "linear_tc"
        status = ttm.device_status()                 # synchronises
        elapsed = time.perf_counter() - t0
        assert status == ttm.ERR_TIMEOUT, ttm.status_str(status)
        assert elapsed < 30.0
        assert ttm.device_status() == ttm.OK         # the query cleared it
        ttm.debug_set("wait_cycles", 0)
        z, W, S = _titans(w, d)
        torch.cuda.synchronize()
        assert ttm.last_kernel() == "linear_tc"
    assert ttm.device_status() == ttm.OK
    ref = H.run_linear_oracle(w, inp)
    H.compare({"z": z, "W": W, "S": S}, ref, ["z", "W", "S"], H.TOL["bf16"])


@gpu
def test_gradient_chain_bounded_wait_runs_out_and_the_next_call_is_correct():
    # the tensor-core chain's loader announces 16 bytes more than it copies for
    # its third chunk: that stage's waits run out, every role of the chain
    # unwinds in lockstep, the status word reports TTM_ERR_TIMEOUT once, and the
    # next gradient matches the oracle
    from tests.test_bwd import check, run_bwd
    T = 6 * 64 + 9
    w, inp = wl.generate_custom(kind="titans", dtype="bf16", B=1, H=2, T=T, d=64, chunk=64,
                                seed=31)
    adj = wl.generate_adjoints(1, 2, T, 64, 64, dtype="bf16", seed=32, with_S=True)
    d, a = H.to_dev(inp), H.to_dev(adj)
    assert ttm.device_status() == ttm.OK
    ttm.debug_set("wait_cycles", 20_000_000)     # ~10 ms at 2 GHz
    ttm.debug_set("stall_chunk", 2)
    t0 = time.perf_counter()
    ttm.titans_bwd(d["q"], d["k"], d["v"], d["theta"], d["W0"], 64, a["dz"], eta=d.get("eta"),
                   alpha=d.get("alpha"), dW=a["dW"], dS=a["dS"])
    assert ttm.last_kernel() == "bwd_tc"
    status = ttm.device_status()                 # synchronises
    elapsed = time.perf_counter() - t0
    assert status == ttm.ERR_TIMEOUT, ttm.status_str(status)
    assert elapsed < 30.0
    assert ttm.device_status() == ttm.OK         # the query cleared it
    ttm.debug_set("wait_cycles", 0)
    g, r, names = run_bwd("titans", "bf16", B=1, Hh=2, T=T, d=64, chunk=64, seed=31, S0=True)
    assert ttm.last_kernel() == "bwd_tc"
    check(g, r, names, H.TOL["bf16"])
    assert ttm.device_status() == ttm.OK


FP32_MAX = float(np.finfo(np.float32).max)


@gpu
@pytest.mark.parametrize("dtype,kernel", [("f32", "linear_simt"), ("bf16", "linear_tc")])
def test_unstable_step_size_gives_non_finite_where_the_oracle_overflows_fp32(dtype, kernel):
    nch = 24
    w, inp = wl.generate_custom(kind="linear", dtype=dtype, B=1, H=2, T=64 * nch, d=64,
                                chunk=64, seed=5)
    inp["theta"] = torch.full_like(inp["theta"], 100.0)
    d = H.to_dev(inp)
    z, W = ttm.linear_fwd(d["q"], d["k"], d["v"], d["theta"], d["W0"], w.chunk)
    torch.cuda.synchronize()
    assert ttm.last_kernel() == kernel
    assert ttm.device_status() == ttm.OK
    ref = H.run_linear_oracle(w, inp)
    zr, zg = ref["z"], H.f64(z)
    mag = np.abs(zr).max(axis=-1)                       # per token, float64
    finite_g = np.isfinite(zg).all(axis=-1)
    assert np.isfinite(zr).all()                        # float64 still holds it
    assert (mag > FP32_MAX).any() and (mag < 1e30).any()
    # well inside the fp32 range: finite; beyond it: never a finite number
    assert finite_g[mag < 1e30].all()
    assert not finite_g[mag > FP32_MAX].any()
    # the first chunk is an ordinary scan of large but representable values
    tol = H.TOL[dtype]
    assert H.max_rel(zg[:, :, :64], zr[:, :, :64]) <= tol
    # the final memory lies beyond the fp32 range in float64
    assert np.abs(ref["W"]).max() > FP32_MAX
    assert not np.isfinite(H.f64(W)).all()

"""ttm_titans_fwd_host: the scan with every tensor in host memory, streamed
through the device in segments of whole chunks (the chunk form restarts from
whatever state the previous chunk left, "TTT layers 与 fast weights" eq (6)).

Host-side checks run without a GPU; the parity cases compare the streamed
result with the oracle on the same seeded inputs, and with the device-buffer
entry point at full size."""
import ctypes

import pytest
import torch

import oracle  # noqa: F401  (test infrastructure only)
import test_neural_memory_gb300 as ttm
import ttm_inputs as wl
from tests import helpers as H

INVALID = ttm.ERR_INVALID_ARG
gpu = pytest.mark.gpu


def _no_gpu_reachable() -> bool:
    ttm.build()
    return ttm.cuda_device_count() == 0 and not torch.cuda.is_available()


host_only = pytest.mark.skipif(not _no_gpu_reachable(),
                               reason="passes fake addresses; host-only")


@pytest.fixture(scope="module")
def L():
    ttm.build()
    return ttm.lib()


def test_workspace_size_rules(L):
    size = ttm.titans_fwd_host_workspace_size
    assert size(1, 2, 1000, 64, 64, 64, "bf16", 100) == 0          # not whole chunks
    assert size(1, 2, 1000, 64, 64, 64, "bf16", 32) == 0           # shorter than a chunk
    a = size(1, 2, 1000, 64, 64, 64, "bf16", 256)
    b = size(1, 2, 1000, 64, 64, 64, "bf16", 512)
    assert 0 < a < b
    # segments never exceed the (chunk-rounded) sequence
    assert size(1, 2, 100, 64, 64, 64, "bf16", 8192) == size(1, 2, 100, 64, 64, 64, "bf16", 128)
    assert size(1, 2, 0, 64, 64, 64, "f32", 64) > 0


@host_only
def test_rejects_malformed_before_any_copy(L):
    p = lambda i: ctypes.c_void_p((1 << 20) * (i + 1))
    ws = ctypes.c_void_p(1 << 30)

    def call(T=1000, chunk=64, seg=256, wsb=1 << 40, W0=p(4), workspace=ws, theta=p(3)):
        return L.ttm_titans_fwd_host(1, 2, T, 64, 64, chunk, ttm.BF16, p(0), p(1), p(2), None,
                                     theta, None, W0, None, 0, p(5), p(6), None, seg, workspace,
                                     wsb, None)
    assert call(seg=100) == INVALID
    assert call(seg=0) == INVALID
    assert call(chunk=0) == INVALID
    assert call(W0=None) == INVALID
    assert call(theta=None) == INVALID
    assert call(workspace=None) == INVALID
    assert call(workspace=ctypes.c_void_p((1 << 30) + 16)) == INVALID   # not 256-byte aligned
    assert call(wsb=1024) == INVALID                                      # short workspace


def _pinned(inp):
    return {k: (None if v is None else v.contiguous().pin_memory()) for k, v in inp.items()}


def _host_run(w, inp, seg, S0=None, want_S=True):
    h = _pinned(inp)
    z, W, S = ttm.titans_fwd_host(h["q"], h["k"], h["v"], h["theta"], h["W0"], w.chunk,
                                  eta=h["eta"], alpha=h["alpha"],
                                  S0=None if S0 is None else S0.contiguous().pin_memory(),
                                  w0_shared=w.w0_shared, seg_tokens=seg, want_S=want_S)
    torch.cuda.synchronize()
    return dict(z=z, W=W, S=S)


CASES = [
    # (kind, dtype, B, H, T, d, chunk, seg, shared)
    ("titans", "bf16", 2, 2, 1000, 64, 64, 256, False),    # tensor-core scan, ragged last segment
    ("titans", "f32", 1, 3, 333, 32, 16, 64, False),       # CUDA-core scan, ragged last chunk
    ("titans", "bf16", 2, 1, 700, 128, 64, 192, True),     # W0 shared over the batch
    ("linear", "f32", 1, 2, 130, 16, 8, 24, False),        # no momentum, no forgetting
]


@gpu
@pytest.mark.parametrize("case", range(len(CASES)))
def test_streamed_matches_oracle(case):
    kind, dt, B, Hh, T, d, chunk, seg, shared = CASES[case]
    w, inp = wl.generate_custom(kind="titans" if kind == "titans" else "linear", B=B, H=Hh, T=T,
                                d=d, chunk=chunk, dtype=dt, w0_shared=shared, seed=300 + case)
    if kind == "linear":
        inp = dict(inp, eta=None, alpha=None)
    g = _host_run(w, inp, seg)
    ref = H.run_linear_oracle(w, inp)
    names = ["z", "W"] + (["S"] if kind == "titans" else [])
    H.compare(g, ref, names, H.TOL[dt])


@gpu
def test_streamed_with_initial_momentum_and_empty_sequence():
    w, inp = wl.generate_custom(kind="titans", B=1, H=2, T=200, d=64, chunk=64, dtype="bf16",
                                seed=311)
    S0 = 0.01 * torch.randn(1, 2, 64, 64, generator=torch.Generator().manual_seed(5))
    g = _host_run(w, inp, 128, S0=S0)
    ref = H.run_linear_oracle(w, inp, S0=S0)
    H.compare(g, ref, ["z", "W", "S"], H.TOL["bf16"])
    # T = 0: the state passes through unchanged
    empty = {k: (None if v is None else (v[:, :, :0] if v.dim() >= 3 and k != "W0" else v))
             for k, v in inp.items()}
    w0 = wl.Workload(0, "custom", "titans", 1, 2, 0, 64, 64, "bf16", w.theta, w.eta, w.alpha,
                     w.w0, False, 0)
    g0 = _host_run(w0, empty, 64, S0=S0)
    assert torch.equal(g0["W"], inp["W0"].float()) and torch.equal(g0["S"], S0.float())


@gpu
def test_streamed_full_long_workload_matches_device_call():
    """Titans long-context workload (B=1 H=16 T=131072 d=128 chunk 64, bf16) in
    segments of 8192 tokens against the device-buffer call on the same inputs;
    the streamed result differs only where a segment starts (errors taken
    directly from the carried state instead of through the recursion)."""
    w = wl.WORKLOADS[4]
    inp = wl.generate(w)
    g = _host_run(w, inp, 8192)
    dev = H.run_linear_gpu(w, inp)
    for n in ("z", "W", "S"):
        err = H.max_rel(H.f64(g[n]), H.f64(dev[n]))
        assert err < 2e-2, (n, err)

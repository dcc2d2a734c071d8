"""ttm_titans_fwd_noalloc: the scan for callers that cannot allocate device memory.

Such a caller only has its inputs and outputs and may not call cudaMalloc, so
it cannot hand ttm_titans_fwd the workspace its tensor-core path needs; the
no-alloc entry point takes that scratch from a fixed 16 MiB block inside the
library instead.  These tests call it through the C ABI and check that two
calls in a row give what ttm_titans_fwd gives on the same inputs (bit for bit:
both run the same kernels on the same inputs, so any difference would be a
scratch mix-up), that the shape really goes through the scratch-using
tensor-core kernel, and that a call needing more scratch than the block holds
is refused.
"""
import ctypes

import pytest
import torch

import ttm_inputs as wl
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    import test_neural_memory_gb300 as ttm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ttm.build()
    lib = ttm.lib()
    i, p = ctypes.c_int, ctypes.c_void_p
    lib.ttm_titans_fwd_noalloc.argtypes = [i] * 7 + [p] * 6 + [p, p, i, p, p, p, p]
    lib.ttm_titans_fwd_noalloc.restype = i
    return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(L, w, d, S0=None):
    B, Hh, T, dk = d["q"].shape
    z = torch.empty_like(d["v"])
    W = torch.empty((B, Hh, dk, dk), dtype=torch.float32, device="cuda")
    S = torch.empty_like(W)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.ttm_titans_fwd_noalloc(B, Hh, T, dk, dk, w.chunk, 1, _ptr(d["q"]), _ptr(d["k"]),
                                  _ptr(d["v"]), _ptr(d["eta"]), _ptr(d["theta"]),
                                  _ptr(d["alpha"]), _ptr(d["W0"]), _ptr(S0), 0, _ptr(z),
                                  _ptr(W), _ptr(S), stream)
    return rc, z, W, S


def test_noalloc_matches_titans_fwd_twice(L):
    import test_neural_memory_gb300 as ttm
    for seed in (31, 32):     # two calls in a row on the shared scratch
        w, inp = wl.generate_custom(kind="titans", dtype="bf16", B=2, H=4, T=1000, d=128,
                                    chunk=64, seed=seed)
        d = H.to_dev(inp)
        S0 = 0.01 * torch.randn((w.B, w.H, w.d, w.d), device="cuda")
        # the shape needs scratch, so the block inside the library is in use
        assert ttm.linear_workspace_size(w.B, w.H, w.T, w.d, w.d, w.chunk, ttm.BF16) > 0
        rc, z, W, S = _noalloc(L, w, d, S0)
        torch.cuda.synchronize()
        assert rc == ttm.OK, ttm.status_str(rc)
        assert ttm.last_kernel() == "linear_tc"
        z_ref, W_ref, S_ref = ttm.titans_fwd(d["q"], d["k"], d["v"], d["theta"], d["W0"],
                                             w.chunk, eta=d["eta"], alpha=d["alpha"], S0=S0)
        torch.cuda.synchronize()
        assert ttm.last_kernel() == "linear_tc"
        for a, b in ((z, z_ref), (W, W_ref), (S, S_ref)):
            assert H.max_rel(H.f64(a), H.f64(b)) <= H.TOL["bf16"]
            assert torch.equal(a, b)
    assert ttm.device_status() == ttm.OK


def test_noalloc_refuses_more_than_its_scratch(L):
    import test_neural_memory_gb300 as ttm
    # 16 sequences x 64 chunks x 17424 bytes = 17.8 MB > 16 MiB: refused on the
    # host.  The buffers are real and full-sized all the same, so that a call
    # that got through by mistake would stay inside memory it owns.
    tok = lambda: torch.zeros((1, 16, 4096, 128), dtype=torch.bfloat16, device="cuda")
    st = lambda: torch.zeros((1, 16, 128, 128), dtype=torch.float32, device="cuda")
    q, k, v, z = tok(), tok(), tok(), tok()
    theta = torch.zeros((1, 16, 4096), dtype=torch.float32, device="cuda")
    W0, W = st(), st()
    with ttm.kernel_policy("auto"):
        rc = L.ttm_titans_fwd_noalloc(1, 16, 4096, 128, 128, 64, 1, _ptr(q), _ptr(k), _ptr(v),
                                      None, _ptr(theta), None, _ptr(W0), None, 0, _ptr(z),
                                      _ptr(W), None, None)
    torch.cuda.synchronize()
    assert rc == ttm.ERR_UNSUPPORTED

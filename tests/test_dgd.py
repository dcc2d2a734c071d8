"""GPU parity of the DGD memory ("Nested Learning" §8.1 eq (88) with the eq (93)
objective, chunk-wise per §8.2): the scan ttm_dgd_fwd and the decode step
ttm_dgd_step against the float64 oracle on the same seeded inputs.  Tolerance
per output tensor: max|gpu - oracle| / max|oracle| below 1e-4 for fp32
inputs and 2e-2 for bf16 inputs."""
import pytest
import torch

import oracle
import ttm_inputs as wl
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import test_neural_memory_gb300 as ttm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ttm.build()
    yield
    assert ttm.device_status() == ttm.OK


def make(dtype, B, Hh, T, d, dv=None, seed=0, shared=False):
    w, inp = wl.generate_custom(kind="linear", dtype=dtype, B=B, H=Hh, T=T, d=d, chunk=1,
                                seed=seed, w0_shared=shared)
    if dv is not None:
        g = torch.Generator().manual_seed(seed + 3)
        inp["v"] = torch.randn((B, Hh, T, dv), generator=g).to(inp["q"].dtype)
        inp["W0"] = 0.02 * torch.randn((1 if shared else B, Hh, dv, d), generator=g)
    inp.update(wl.generate_dgd_gates(B, Hh, T, seed=seed + 5))
    return inp


def oracle_run(inp, chunk, shared=False):
    f = H.f64
    return oracle.dgd_primal(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["eta"]),
                             f(inp["alpha"]), f(inp["W0"]), chunk, shared_over_batch=shared)


def gpu_run(inp, chunk, shared=False):
    import test_neural_memory_gb300 as ttm
    d = H.to_dev(inp)
    z, W = ttm.dgd_fwd(d["q"], d["k"], d["v"], d["eta"], d["alpha"], d["W0"], chunk,
                       w0_shared=shared)
    torch.cuda.synchronize()
    return dict(z=z, W=W)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_scan_ragged_chunks(dtype):
    inp = make(dtype, B=2, Hh=2, T=150, d=64, seed=1)
    H.compare(gpu_run(inp, 64), oracle_run(inp, 64), ["z", "W"], H.TOL[dtype])


def test_scan_shared_initial_memory():
    inp = make("f32", B=3, Hh=2, T=40, d=32, seed=2, shared=True)
    H.compare(gpu_run(inp, 16, shared=True), oracle_run(inp, 16, shared=True), ["z", "W"],
              H.TOL["f32"])


def test_scan_rectangular_and_chunk_one():
    inp = make("f32", B=1, Hh=2, T=33, d=32, dv=48, seed=3)
    H.compare(gpu_run(inp, 16), oracle_run(inp, 16), ["z", "W"], H.TOL["f32"])
    H.compare(gpu_run(inp, 1), oracle_run(inp, 1), ["z", "W"], H.TOL["f32"])


@pytest.mark.parametrize("d", [16, 128, 512])
def test_scan_widths(d):
    inp = make("f32", B=1, Hh=1, T=40, d=d, seed=4)
    H.compare(gpu_run(inp, 8), oracle_run(inp, 8), ["z", "W"], H.TOL["f32"])


def test_scan_many_rows_block_sizes():
    """10 240 rows of d = 128: the four-rows-per-warp kernel in blocks of 8 warps."""
    inp = make("bf16", B=8, Hh=10, T=24, d=128, seed=7)
    H.compare(gpu_run(inp, 8), oracle_run(inp, 8), ["z", "W"], H.TOL["bf16"])


def test_scan_in_place_and_empty():
    import test_neural_memory_gb300 as ttm
    inp = make("f32", B=2, Hh=1, T=20, d=32, seed=6)
    d = H.to_dev(inp)
    W = d["W0"].clone()
    z, W2 = ttm.dgd_fwd(d["q"], d["k"], d["v"], d["eta"], d["alpha"], W, 8, W_out=W)
    torch.cuda.synchronize()
    H.compare(dict(z=z, W=W), oracle_run(inp, 8), ["z", "W"], H.TOL["f32"])
    e = make("f32", B=2, Hh=1, T=0, d=32, seed=7)
    de = H.to_dev(e)
    _, W0out = ttm.dgd_fwd(de["q"], de["k"], de["v"], de["eta"], de["alpha"], de["W0"], 8)
    torch.cuda.synchronize()
    assert torch.equal(W0out.cpu(), e["W0"])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prefill_then_decode(dtype):
    import test_neural_memory_gb300 as ttm
    T0, calls, chunk = 128, [1, 5, 64, 3, 1], 64
    inp = make(dtype, B=2, Hh=2, T=T0 + sum(calls), d=64, seed=8)
    d = H.to_dev(inp)
    part = lambda x, t0, t1: x[:, :, t0:t1].contiguous()
    z0, W = ttm.dgd_fwd(*(part(d[n], 0, T0) for n in ("q", "k", "v", "eta", "alpha")), d["W0"],
                        chunk)
    zs, Wc, pos, t = [z0], None, 0, T0
    for n in calls:
        z, Wc, pos = ttm.dgd_step(*(part(d[x], t, t + n) for x in ("q", "k", "v", "eta", "alpha")),
                                  W, chunk, pos, Wc=Wc)
        zs.append(z)
        t += n
    torch.cuda.synchronize()
    H.compare(dict(z=torch.cat(zs, dim=2), W=W), oracle_run(inp, chunk), ["z", "W"],
              H.TOL[dtype])

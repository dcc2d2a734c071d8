"""GPU parity of the DGD memory ("Nested Learning" §8.1 eq (88) with the eq (93)
objective, chunk-wise per §8.2): the scan ttm_dgd_fwd (the fp32 token loop and
the tensor-core chunk form) and the decode step ttm_dgd_step against the
float64 oracle on the same seeded inputs.  Tolerance per output tensor:
max|gpu - oracle| / max|oracle| below 1e-4 for fp32 inputs and 2e-2 for bf16
inputs."""
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


def gpu_run(inp, chunk, shared=False, policy="auto", kernel=None):
    import test_neural_memory_gb300 as ttm
    d = H.to_dev(inp)
    with ttm.kernel_policy(policy):
        z, W = ttm.dgd_fwd(d["q"], d["k"], d["v"], d["eta"], d["alpha"], d["W0"], chunk,
                           w0_shared=shared)
        torch.cuda.synchronize()
        if kernel is not None:
            assert ttm.last_kernel() == kernel
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


# ---------------------------------------------------------------- chunk form
# Tensor-core path (bf16, d_k = d_v in {64, 128}, chunk 64) under the "tc"
# policy, so a shape it does not take fails instead of running elsewhere.

TC_CASES = [
    dict(B=1, Hh=1, T=1),            # one token
    dict(B=1, Hh=2, T=64),           # exactly one chunk
    dict(B=2, Hh=1, T=65),           # one token into the second chunk
    dict(B=2, Hh=3, T=1000),         # many chunks, ragged last chunk (40 tokens)
]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("case", range(len(TC_CASES)))
def test_chunk_form_shapes(d, case):
    c = TC_CASES[case]
    inp = make("bf16", B=c["B"], Hh=c["Hh"], T=c["T"], d=d, seed=40 + case)
    H.compare(gpu_run(inp, 64, policy="tc", kernel="dgd_tc"), oracle_run(inp, 64), ["z", "W"],
              H.TOL["bf16"])


def test_chunk_form_shared_initial_memory():
    inp = make("bf16", B=3, Hh=2, T=300, d=128, seed=50, shared=True)
    H.compare(gpu_run(inp, 64, shared=True, policy="tc", kernel="dgd_tc"),
              oracle_run(inp, 64, shared=True), ["z", "W"], H.TOL["bf16"])


def test_chunk_form_in_place_and_no_retention_decay():
    """alpha = 1 (nothing forgotten) and W_out = W0 in place."""
    import test_neural_memory_gb300 as ttm
    inp = make("bf16", B=2, Hh=2, T=200, d=64, seed=51)
    inp["alpha"] = torch.ones_like(inp["alpha"])
    ref = oracle_run(inp, 64)
    d = H.to_dev(inp)
    W = d["W0"].clone()
    with ttm.kernel_policy("tc"):
        z, W2 = ttm.dgd_fwd(d["q"], d["k"], d["v"], d["eta"], d["alpha"], W, 64, W_out=W)
        torch.cuda.synchronize()
        assert ttm.last_kernel() == "dgd_tc"
    assert W2.data_ptr() == W.data_ptr()
    H.compare(dict(z=z, W=W), ref, ["z", "W"], H.TOL["bf16"])


def test_chunk_form_matches_token_loop():
    """The chunk form and the fp32 token loop agree to bf16-operand precision."""
    inp = make("bf16", B=1, Hh=4, T=2000, d=128, seed=52)
    a = gpu_run(inp, 64, policy="tc", kernel="dgd_tc")
    b = gpu_run(inp, 64, policy="simt", kernel="dgd_step")
    for n in ("z", "W"):
        assert H.max_rel(H.f64(a[n]), H.f64(b[n])) < H.TOL["bf16"], n


def test_chunk_form_long_context_workload():
    """The long-context shape (B1 H16 T131072 d128, bf16, chunk 64) with the DGD
    gates of the bench: the automatic choice is the chunk form; z and W of two
    heads against the oracle."""
    w = wl.WORKLOADS[4]
    inp = wl.generate(w)
    inp.update(wl.generate_dgd_gates(w.B, w.H, w.T, seed=77))
    out = gpu_run(inp, w.chunk, kernel="dgd_tc")
    heads = [0, 9]
    sub = {n: inp[n][:, heads] for n in ("q", "k", "v", "eta", "alpha", "W0")}
    ref = oracle_run(sub, w.chunk)
    H.compare({n: out[n][:, heads] for n in ("z", "W")}, ref, ["z", "W"], H.TOL["bf16"])

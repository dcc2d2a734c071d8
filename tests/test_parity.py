"""GPU parity: every entry point against the float64 oracle on the same seeded
inputs, on shrunk shapes with ragged tails and edge cases, and on the five
full-size workloads (full-size runs compare whole heads, chosen so the oracle
finishes in seconds)."""
import numpy as np
import pytest
import torch

import ttm_inputs as wl
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import test_neural_memory_gb300 as ttm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ttm.build()
    ttm.lib()
    yield
    assert ttm.device_status() == ttm.OK


def _linear_case(kind, policy="auto", **kw):
    import test_neural_memory_gb300 as ttm
    w, inp = wl.generate_custom(kind=kind, **kw)
    S0 = None
    if kind == "titans" and kw.get("seed", 0) % 2 == 1:
        S0 = 0.01 * torch.randn((1 if w.w0_shared else w.B, w.H, w.d, w.d))
    with ttm.kernel_policy(policy):
        g = H.run_linear_gpu(w, inp, S0=S0)
    ref = H.run_linear_oracle(w, inp, S0=S0)
    names = ["z", "W"] + (["S"] if kind == "titans" else [])
    errs = H.compare(g, ref, names, H.TOL[w.dtype])
    return g["kernel"], errs


SHRUNK = [
    # ragged T with several chunks
    dict(B=1, H=2, T=100, d=64, chunk=16),
    # T shorter than one chunk
    dict(B=1, H=1, T=37, d=64, chunk=64),
    # one token per chunk (delta rule)
    dict(B=1, H=1, T=33, d=64, chunk=1),
    # chunk longer than the kernel's on-chip token block, ragged tail
    dict(B=1, H=1, T=150, d=64, chunk=48),
    # several sequences, d = 128
    dict(B=2, H=3, T=70, d=128, chunk=64),
    # single token
    dict(B=1, H=1, T=1, d=64, chunk=16),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", ["linear", "titans"])
@pytest.mark.parametrize("case", range(len(SHRUNK)))
def test_linear_shrunk(kind, dtype, case):
    kernel, errs = _linear_case(kind, dtype=dtype, seed=case, **SHRUNK[case])
    assert kernel.startswith("linear")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_linear_shared_initial_state(dtype):
    _linear_case("linear", dtype=dtype, B=3, H=2, T=90, d=64, chunk=16, w0_shared=True, seed=4)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_titans_nonzero_momentum_state(dtype):
    _linear_case("titans", dtype=dtype, B=2, H=1, T=130, d=64, chunk=64, seed=5)


def test_simt_policy_matches_oracle_bf16():
    kernel, _ = _linear_case("titans", policy="simt", dtype="bf16", B=1, H=2, T=200, d=128,
                             chunk=64, seed=6)
    assert kernel == "linear_simt"


def test_rectangular_memory():
    import test_neural_memory_gb300 as ttm
    g = torch.Generator().manual_seed(3)
    B, Hh, T, dk, dv, chunk = 1, 2, 77, 64, 48, 16
    q = torch.nn.functional.normalize(torch.randn(B, Hh, T, dk, generator=g), dim=-1)
    k = torch.nn.functional.normalize(torch.randn(B, Hh, T, dk, generator=g), dim=-1)
    v = torch.randn(B, Hh, T, dv, generator=g)
    th = 0.1 * torch.sigmoid(torch.randn(B, Hh, T, generator=g))
    et = 0.8 + 0.2 * torch.sigmoid(torch.randn(B, Hh, T, generator=g))
    al = 0.05 * torch.sigmoid(torch.randn(B, Hh, T, generator=g))
    W0 = 0.02 * torch.randn(B, Hh, dv, dk, generator=g)
    c = lambda t: t.cuda()
    z, W, S = ttm.titans_fwd(c(q), c(k), c(v), c(th), c(W0), chunk, eta=c(et), alpha=c(al))
    import oracle
    r = oracle.linear_primal(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                             th.double().numpy(), W0.double().numpy(), chunk,
                             eta=et.double().numpy(), alpha=al.double().numpy())
    for n, t in (("z", z), ("W", W), ("S", S)):
        assert H.max_rel(H.f64(t), r[n]) < H.TOL["f32"], n


def test_empty_sequence_copies_initial_state():
    import test_neural_memory_gb300 as ttm
    W0 = torch.randn(2, 3, 64, 64, device="cuda")
    S0 = torch.randn(2, 3, 64, 64, device="cuda")
    e = torch.empty(2, 3, 0, 64, device="cuda")
    th = torch.empty(2, 3, 0, device="cuda")
    z, W, S = ttm.titans_fwd(e, e.clone(), e.clone(), th, W0, 16, S0=S0)
    torch.cuda.synchronize()
    assert z.numel() == 0 and torch.equal(W, W0) and torch.equal(S, S0)


def test_in_place_state_update():
    import test_neural_memory_gb300 as ttm
    w, inp = wl.generate_custom(kind="titans", dtype="bf16", B=1, H=2, T=64, d=64, chunk=16,
                                seed=8)
    d = H.to_dev(inp)
    z1, W1, S1 = ttm.titans_fwd(d["q"], d["k"], d["v"], d["theta"], d["W0"], 16,
                                eta=d["eta"], alpha=d["alpha"])
    Wbuf = d["W0"].clone()
    z2, W2, _ = ttm.titans_fwd(d["q"], d["k"], d["v"], d["theta"], Wbuf, 16, eta=d["eta"],
                               alpha=d["alpha"], W_out=Wbuf)
    torch.cuda.synchronize()
    assert torch.equal(W2, W1) and torch.equal(z1, z2)


def test_split_call_continuation():
    """Passing a call's final (W, S) to a second call equals one call when the
    split falls on a chunk boundary."""
    import test_neural_memory_gb300 as ttm
    w, inp = wl.generate_custom(kind="titans", dtype="f32", B=1, H=2, T=96, d=64, chunk=16,
                                seed=9)
    d = H.to_dev(inp)
    z, W, S = ttm.titans_fwd(d["q"], d["k"], d["v"], d["theta"], d["W0"], 16, eta=d["eta"],
                             alpha=d["alpha"])
    cut = 48
    part = lambda t, a, b: t[:, :, a:b].contiguous()
    za, Wa, Sa = ttm.titans_fwd(*(part(d[n], 0, cut) for n in ("q", "k", "v", "theta")),
                                d["W0"], 16, eta=part(d["eta"], 0, cut),
                                alpha=part(d["alpha"], 0, cut))
    zb, Wb, Sb = ttm.titans_fwd(*(part(d[n], cut, 96) for n in ("q", "k", "v", "theta")),
                                Wa, 16, eta=part(d["eta"], cut, 96),
                                alpha=part(d["alpha"], cut, 96), S0=Sa)
    torch.cuda.synchronize()
    assert H.max_rel(H.f64(torch.cat([za, zb], dim=2)), H.f64(z)) < 1e-5
    assert H.max_rel(H.f64(Wb), H.f64(W)) < 1e-5 and H.max_rel(H.f64(Sb), H.f64(S)) < 1e-5


# ---------------------------------------------------------------- MLP memory

MLP_SHRUNK = [
    dict(B=1, H=2, T=50, d=64, hidden=256, chunk=16),
    dict(B=1, H=1, T=21, d=64, hidden=256, chunk=1),
    dict(B=2, H=1, T=40, d=32, hidden=128, chunk=8),
    dict(B=1, H=2, T=75, d=128, hidden=64, chunk=32),
    dict(B=1, H=1, T=19, d=16, hidden=24, chunk=5),
    # two-CTA cluster kernel: d = 128, hidden = 128, ragged last chunk
    dict(B=1, H=2, T=45, d=128, hidden=128, chunk=12),
    # d = 8: the one-token-per-lane kernel
    dict(B=1, H=1, T=23, d=8, hidden=32, chunk=4),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", range(len(MLP_SHRUNK)))
def test_mlp_shrunk(dtype, case):
    w, inp = wl.generate_custom(kind="mlp", dtype=dtype, seed=20 + case, **MLP_SHRUNK[case])
    g = H.run_mlp_gpu(w, inp)
    ref = H.run_mlp_oracle(w, inp)
    H.compare(g, ref, ["z", "W1", "W2", "S1", "S2"], H.TOL[dtype])


# ------------------------------------------------------ full-size workloads

def _full_linear(wid, heads):
    w = wl.WORKLOADS[wid]
    inp = wl.generate(w)
    g = H.run_linear_gpu(w, inp)
    ref = H.run_linear_oracle(w, inp, heads=heads)
    names = ["z", "W"] + (["S"] if w.kind == "titans" else [])
    return g["kernel"], H.compare(g, ref, names, H.TOL[w.dtype], heads=heads)


def test_full_workload_1():
    _full_linear(1, None)


def test_full_workload_2():
    _full_linear(2, None)


def test_full_workload_3():
    _full_linear(3, [0, 7, 11])


def test_full_workload_4():
    _full_linear(4, [0, 9, 15])


def test_full_workload_5():
    w = wl.WORKLOADS[5]
    inp = wl.generate(w)
    g = H.run_mlp_gpu(w, inp)
    heads = [0, 13]
    ref = H.run_mlp_oracle(w, inp, heads=heads)
    H.compare(g, ref, ["z", "W1", "W2", "S1", "S2"], H.TOL[w.dtype], heads=heads)

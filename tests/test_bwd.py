"""GPU parity of the scan's gradient (ttm_titans_bwd / ttm_linear_bwd) against
the float64 oracle's reverse-mode gradient on the same seeded inputs and
adjoints.  Tolerance per output tensor: max|gpu - oracle| / max|oracle| below
1e-4 for fp32 inputs and 2e-2 for bf16 inputs (the scan's parity bar)."""
import numpy as np
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


def run_bwd(kind, dtype, B, Hh, T, d, chunk, dv=None, seed=0, shared=False, adj_final=True,
            S0=False, theta=None):
    """Gradient on the GPU and in the oracle; returns (gpu dict, oracle dict, names)."""
    import test_neural_memory_gb300 as ttm
    kw = dict(kind=kind, dtype=dtype, B=B, H=Hh, T=T, d=d, chunk=chunk, seed=seed,
              w0_shared=shared)
    if theta is not None:
        kw["theta"] = theta
    w, inp = wl.generate_custom(**kw)
    dk = d
    if dv is not None:   # rectangular memory: v and W0 with dv rows
        g = torch.Generator().manual_seed(seed + 7)
        inp["v"] = torch.randn((B, Hh, T, dv), generator=g).to(inp["q"].dtype)
        inp["W0"] = 0.02 * torch.randn((1 if shared else B, Hh, dv, dk), generator=g)
    dvv = inp["v"].shape[-1]
    titans = kind == "titans"
    if S0:
        g = torch.Generator().manual_seed(seed + 9)
        inp["S0"] = 0.01 * torch.randn(tuple(inp["W0"].shape), generator=g)
    adj = wl.generate_adjoints(B, Hh, T, dk, dvv, dtype=dtype, seed=seed + 11, with_S=titans)
    if not adj_final:
        adj["dW"] = None
        adj["dS"] = None
    d_ = H.to_dev(inp)
    a_ = H.to_dev(adj)
    g = ttm.titans_bwd(d_["q"], d_["k"], d_["v"], d_["theta"], d_["W0"], chunk, a_["dz"],
                       eta=d_.get("eta"), alpha=d_.get("alpha"), S0=d_.get("S0"),
                       dW=a_["dW"], dS=a_["dS"], w0_shared=shared)
    torch.cuda.synchronize()
    f = H.f64
    r = oracle.linear_primal_bwd(f(inp["q"]), f(inp["k"]), f(inp["v"]), f(inp["theta"]),
                                 f(inp["W0"]), chunk, f(adj["dz"]), eta=f(inp.get("eta")),
                                 alpha=f(inp.get("alpha")), S0=f(inp.get("S0")),
                                 dW=f(adj["dW"]), dS=f(adj["dS"]), shared_over_batch=shared)
    names = ["dq", "dk", "dv", "dtheta", "dW0", "dS0"]
    if inp.get("eta") is not None:
        names.append("deta")
    if inp.get("alpha") is not None:
        names.append("dalpha")
    return g, r, names


def check(g, r, names, tol):
    errs = {n: H.max_rel(H.f64(g[n]), r[n]) for n in names}
    bad = {n: e for n, e in errs.items() if not e <= tol}
    assert not bad, f"gradient parity failed (tol {tol}): {errs}"
    return errs


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_titans_ragged_chunks(dtype):
    # three chunks of 64: two full and a ragged tail of 22 tokens
    g, r, names = run_bwd("titans", dtype, B=2, Hh=2, T=150, d=64, chunk=64, seed=1, S0=True)
    check(g, r, names, H.TOL[dtype])


def test_titans_full_width_d128():
    # d = 128: eight 16-row tiles in the local pass, sixteen 8-row chain slices
    g, r, names = run_bwd("titans", "f32", B=1, Hh=2, T=130, d=128, chunk=64, seed=2)
    check(g, r, names, H.TOL["f32"])


def test_linear_rectangular_memory():
    g, r, names = run_bwd("linear", "f32", B=2, Hh=1, T=70, d=32, dv=48, chunk=16, seed=3)
    check(g, r, names, H.TOL["f32"])


def test_shared_initial_memory_sums_over_batch():
    g, r, names = run_bwd("titans", "f32", B=3, Hh=2, T=40, d=32, chunk=16, seed=4, shared=True)
    assert tuple(g["dW0"].shape) == (1, 2, 32, 32)
    check(g, r, names, H.TOL["f32"])


def test_delta_rule_chunk_one():
    g, r, names = run_bwd("linear", "f32", B=1, Hh=2, T=9, d=16, chunk=1, seed=5)
    check(g, r, names, H.TOL["f32"])


def test_only_output_adjoints():
    # no adjoint on the final state: the gradient flows from the reads alone
    g, r, names = run_bwd("titans", "f32", B=1, Hh=1, T=100, d=64, chunk=32, seed=6,
                          adj_final=False)
    check(g, r, names, H.TOL["f32"])


def test_chunk_not_a_power_of_two():
    g, r, names = run_bwd("titans", "bf16", B=1, Hh=3, T=77, d=96, chunk=24, seed=8)
    check(g, r, names, H.TOL["bf16"])


def test_empty_sequence_passes_the_final_adjoint_through():
    import test_neural_memory_gb300 as ttm
    for shared in (False, True):
        w, inp = wl.generate_custom(kind="titans", dtype="f32", B=2, H=2, T=0, d=16, chunk=4,
                                    w0_shared=shared)
        adj = wl.generate_adjoints(2, 2, 0, 16, 16, seed=3)
        d_, a_ = H.to_dev(inp), H.to_dev(adj)
        g = ttm.titans_bwd(d_["q"], d_["k"], d_["v"], d_["theta"], d_["W0"], 4, a_["dz"],
                           eta=d_["eta"], alpha=d_["alpha"], dW=a_["dW"], dS=a_["dS"],
                           w0_shared=shared)
        torch.cuda.synchronize()
        want_W = adj["dW"].sum(0, keepdim=True) if shared else adj["dW"]
        want_S = adj["dS"].sum(0, keepdim=True) if shared else adj["dS"]
        assert torch.allclose(g["dW0"].cpu(), want_W, atol=1e-6)
        assert torch.allclose(g["dS0"].cpu(), want_S, atol=1e-6)


@pytest.mark.parametrize("chunk,d", [(128, 64), (16, 256)])
def test_unsupported_shapes_are_refused(chunk, d):
    import test_neural_memory_gb300 as ttm
    w, inp = wl.generate_custom(kind="titans", dtype="f32", B=1, H=1, T=8, d=d, chunk=chunk)
    adj = wl.generate_adjoints(1, 1, 8, d, d, seed=1)
    d_, a_ = H.to_dev(inp), H.to_dev(adj)
    with pytest.raises(ttm.TTMError) as e:
        ttm.titans_bwd(d_["q"], d_["k"], d_["v"], d_["theta"], d_["W0"], chunk, a_["dz"],
                       eta=d_["eta"], alpha=d_["alpha"], dW=a_["dW"], dS=a_["dS"])
    assert e.value.code == ttm.ERR_UNSUPPORTED


def test_narrow_key_long_chunk():
    # dk = 16 < chunk = 64: the gate-gradient tables outgrow the q / k buffers
    g, r, names = run_bwd("titans", "bf16", B=1, Hh=2, T=100, d=16, chunk=64, seed=9)
    check(g, r, names, H.TOL["bf16"])


@pytest.mark.parametrize("policy", ["auto", "simt"])
def test_bf16_d128_both_checkpoint_scans(policy):
    # bf16, d = 128, chunk 64: the tensor-core scan writes the chunk-start
    # states under the automatic policy, the CUDA-core scan under "simt"
    import test_neural_memory_gb300 as ttm
    with ttm.kernel_policy(policy):
        g, r, names = run_bwd("titans", "bf16", B=1, Hh=2, T=200, d=128, chunk=64, seed=10,
                              S0=True)
    check(g, r, names, H.TOL["bf16"])


# ------------------------------------------ tensor-core chain and local passes
# bf16, d_k = d_v in {64, 128}, chunk 64: under the automatic policy the chain
# (the state adjoint at every chunk end) and the local pass (dq, dk, dv and the
# gate gradients) run on the tensor cores.

@pytest.mark.parametrize("kind,d,T,seed", [("titans", 64, 130, 20), ("titans", 128, 64, 21),
                                            ("linear", 128, 200, 22), ("titans", 128, 1, 23),
                                            ("titans", 128, 100, 27)])
def test_tensor_core_local_pass(kind, d, T, seed):
    import test_neural_memory_gb300 as ttm
    with ttm.kernel_policy("auto"):
        g, r, names = run_bwd(kind, "bf16", B=2, Hh=2, T=T, d=d, chunk=64, seed=seed,
                              S0=(kind == "titans"))
        assert ttm.last_kernel() == "bwd_tc"
    check(g, r, names, H.TOL["bf16"])


@pytest.mark.parametrize("d", [64, 128])
def test_tensor_core_chain_many_chunks(d):
    # thirteen chunks, the last one ragged: the chain's two-stage input ring
    # wraps its phases several times and carries the adjoint through all of them
    import test_neural_memory_gb300 as ttm
    with ttm.kernel_policy("auto"):
        g, r, names = run_bwd("titans", "bf16", B=1, Hh=2, T=12 * 64 + 5, d=d, chunk=64,
                              seed=26 + d, S0=True)
        assert ttm.last_kernel() == "bwd_tc"
    check(g, r, names, H.TOL["bf16"])


def test_tensor_core_local_pass_shared_memory_and_no_final_adjoint():
    import test_neural_memory_gb300 as ttm
    with ttm.kernel_policy("auto"):
        g, r, names = run_bwd("titans", "bf16", B=3, Hh=2, T=150, d=128, chunk=64, seed=24,
                              shared=True, adj_final=False)
        assert ttm.last_kernel() == "bwd_tc"
    check(g, r, names, H.TOL["bf16"])


def test_tensor_core_and_cuda_core_gradients_agree():
    import test_neural_memory_gb300 as ttm
    out = {}
    for policy, kern in (("auto", "bwd_tc"), ("simt", "bwd_simt")):
        with ttm.kernel_policy(policy):
            g, r, names = run_bwd("titans", "bf16", B=1, Hh=4, T=640, d=128, chunk=64, seed=25)
            assert ttm.last_kernel() == kern
        out[policy] = g
    for n in names:
        if out["auto"][n] is None:
            continue
        assert H.max_rel(H.f64(out["auto"][n]), H.f64(out["simt"][n])) < H.TOL["bf16"], n

"""GPU parity of the tensor-core (tcgen05 + TMA) linear / Titans kernel.

The kernel policy is forced to "tc", so a shape the tensor-core kernel does
not take fails instead of silently running on the CUDA-core kernel."""
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
    yield
    assert ttm.device_status() == ttm.OK


def run_case(kind, S0_scale=0.0, **kw):
    import test_neural_memory_gb300 as ttm
    w, inp = wl.generate_custom(kind=kind, dtype="bf16", chunk=64, **kw)
    S0 = None
    if S0_scale:
        g = torch.Generator().manual_seed(99)
        S0 = S0_scale * torch.randn((1 if w.w0_shared else w.B, w.H, w.d, w.d), generator=g)
    with ttm.kernel_policy("tc"):
        g_out = H.run_linear_gpu(w, inp, S0=S0)
    assert g_out["kernel"] == "linear_tc"
    ref = H.run_linear_oracle(w, inp, S0=S0)
    names = ["z", "W"] + (["S"] if kind == "titans" else [])
    return H.compare(g_out, ref, names, H.TOL["bf16"])


TC_CASES = [
    dict(B=1, H=1, T=1, d=64),          # one token
    dict(B=1, H=1, T=63, d=64),         # shorter than a chunk
    dict(B=1, H=1, T=64, d=128),        # exactly one chunk
    dict(B=1, H=2, T=65, d=128),        # one token into the second chunk
    dict(B=2, H=2, T=200, d=64),        # ragged tail, several sequences
    dict(B=1, H=3, T=500, d=128),       # many chunks
]


@pytest.mark.parametrize("kind", ["titans", "linear"])
@pytest.mark.parametrize("case", range(len(TC_CASES)))
def test_tc_shapes(kind, case):
    run_case(kind, seed=100 + case, **TC_CASES[case])


def test_tc_nonzero_momentum_state():
    run_case("titans", S0_scale=0.05, B=2, H=1, T=300, d=128, seed=7)


def test_tc_shared_initial_state():
    run_case("linear", B=3, H=2, T=150, d=64, w0_shared=True, seed=8)


def test_tc_matches_simt():
    """Both kernels on the same inputs agree to bf16-operand precision."""
    import test_neural_memory_gb300 as ttm
    w, inp = wl.generate_custom(kind="titans", dtype="bf16", B=1, H=4, T=1000, d=128, chunk=64,
                                seed=9)
    with ttm.kernel_policy("tc"):
        a = H.run_linear_gpu(w, inp)
    with ttm.kernel_policy("simt"):
        b = H.run_linear_gpu(w, inp)
    assert a["kernel"] == "linear_tc" and b["kernel"] == "linear_simt"
    for n in ("z", "W", "S"):
        assert H.max_rel(H.f64(a[n]), H.f64(b[n])) < H.TOL["bf16"], n


def test_tc_rejects_what_it_does_not_cover():
    import test_neural_memory_gb300 as ttm
    w, inp = wl.generate_custom(kind="titans", dtype="f32", B=1, H=1, T=64, d=64, chunk=64)
    with ttm.kernel_policy("tc"), pytest.raises(ttm.TTMError) as e:
        H.run_linear_gpu(w, inp)
    assert e.value.code == ttm.ERR_UNSUPPORTED

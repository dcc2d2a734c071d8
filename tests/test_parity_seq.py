"""GPU parity of the tensor-core scan with one CTA per sequence (d = 64,
gradient points every 16 or 32 tokens inside 64-token tiles; "TTT layers 与
fast weights" §1.1 eqs (6)-(9), mini-batch b = 16).

Every case runs under the "tc" policy, so a shape the kernel does not take
fails instead of running on the CUDA-core kernel, and checks that the
sequence kernel is the one that ran.  Cases span several tiles with a ragged
last tile, one token, a tile boundary inside a sub-chunk count, shared and
per-sequence initial memory, momentum and forgetting with an initial
momentum, and the TTT-Linear 125M-layer workload at full size on sampled
heads."""
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


def run_case(kind, chunk, S0_scale=0.0, **kw):
    import test_neural_memory_gb300 as ttm
    w, inp = wl.generate_custom(kind=kind, dtype="bf16", chunk=chunk, d=64, **kw)
    S0 = None
    if S0_scale:
        g = torch.Generator().manual_seed(77)
        S0 = S0_scale * torch.randn((1 if w.w0_shared else w.B, w.H, w.d, w.d), generator=g)
    with ttm.kernel_policy("tc"):
        out = H.run_linear_gpu(w, inp, S0=S0)
    assert out["kernel"] == "linear_seq"
    ref = H.run_linear_oracle(w, inp, S0=S0)
    names = ["z", "W"] + (["S"] if kind == "titans" else [])
    return H.compare(out, ref, names, H.TOL["bf16"])


CASES = [
    dict(B=1, H=1, T=1),            # one token
    dict(B=1, H=1, T=17),           # one sub-chunk and one token
    dict(B=1, H=2, T=64),           # exactly one tile
    dict(B=2, H=1, T=65),           # one token into the second tile
    dict(B=2, H=3, T=1000),         # many tiles, ragged last tile (40 tokens)
]


@pytest.mark.parametrize("chunk", [16, 32])
@pytest.mark.parametrize("kind", ["linear", "titans"])
@pytest.mark.parametrize("case", range(len(CASES)))
def test_seq_shapes(kind, chunk, case):
    run_case(kind, chunk, seed=300 + case, **CASES[case])


def test_seq_shared_initial_memory():
    run_case("linear", 16, B=4, H=2, T=300, w0_shared=True, seed=11)


@pytest.mark.parametrize("chunk", [16, 32])
def test_seq_titans_initial_momentum(chunk):
    run_case("titans", chunk, S0_scale=0.05, B=2, H=2, T=450, seed=12)


def test_seq_titans_without_gates_returns_the_last_step():
    # eta = alpha = 0 through the Titans entry point: S is the last token's step
    run_case("titans", 16, B=1, H=2, T=130, eta=("zero",), alpha=("zero",), seed=13)


def test_chunk_64_stays_on_the_row_slice_kernel():
    import test_neural_memory_gb300 as ttm
    w, inp = wl.generate_custom(kind="linear", dtype="bf16", chunk=64, d=64, B=1, H=1, T=128)
    with ttm.kernel_policy("tc"):
        out = H.run_linear_gpu(w, inp)
    assert out["kernel"] == "linear_tc"


def test_seq_matches_simt():
    """The sequence kernel and the fp32 CUDA-core kernel agree to bf16-operand
    precision on the same inputs."""
    import test_neural_memory_gb300 as ttm
    w, inp = wl.generate_custom(kind="titans", dtype="bf16", B=1, H=4, T=2000, d=64, chunk=16,
                                seed=14)
    with ttm.kernel_policy("tc"):
        a = H.run_linear_gpu(w, inp)
    with ttm.kernel_policy("simt"):
        b = H.run_linear_gpu(w, inp)
    assert a["kernel"] == "linear_seq" and b["kernel"] == "linear_simt"
    for n in ("z", "W", "S"):
        assert H.max_rel(H.f64(a[n]), H.f64(b[n])) < H.TOL["bf16"], n


def test_seq_full_workload_3():
    """TTT-Linear at the 125M-layer shape (B8 H12 T8192 d64, chunk 16, W0 shared
    over the batch): the automatic choice is the sequence kernel; z and W of
    three heads (every batch row) against the oracle."""
    w = wl.WORKLOADS[3]
    inp = wl.generate(w)
    out = H.run_linear_gpu(w, inp)
    assert out["kernel"] == "linear_seq"
    heads = [0, 5, 11]
    ref = H.run_linear_oracle(w, inp, heads=heads)
    H.compare(out, ref, ["z", "W"], H.TOL["bf16"], heads=heads)

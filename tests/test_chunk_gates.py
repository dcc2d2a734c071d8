"""GPU parity of the Titans scan with chunk-level gates ("论文速览 | Titans" §4.6:
theta, eta, alpha shared by the tokens of a chunk).  The per-chunk call must
give exactly what the per-token call gives on the same gates repeated over
each chunk's tokens, and both must match the float64 oracle."""
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


def expand(g, T, chunk):
    return None if g is None else g.repeat_interleave(chunk, dim=-1)[..., :T].contiguous()


@pytest.mark.parametrize("dtype,d,chunk,T,policy", [
    ("bf16", 128, 64, 300, "auto"),    # tensor-core scan: ragged last chunk
    ("bf16", 64, 64, 130, "simt"),
    ("f32", 64, 16, 70, "auto"),       # CUDA-core scan
    ("f32", 32, 40, 100, "auto"),      # chunks longer than its 32-token block
])
def test_chunk_gates_match_repeated_token_gates(dtype, d, chunk, T, policy):
    import test_neural_memory_gb300 as ttm
    B, Hh = 2, 2
    nch = (T + chunk - 1) // chunk
    w, inp = wl.generate_custom(kind="titans", dtype=dtype, B=B, H=Hh, T=T, d=d, chunk=chunk,
                                seed=3)
    cg = wl.generate_chunk_gates(B, Hh, nch, seed=4)
    tok = {k: expand(v, T, chunk) for k, v in cg.items()}
    d_ = H.to_dev(inp)
    c_ = H.to_dev(cg)
    t_ = H.to_dev(tok)
    with ttm.kernel_policy(policy):
        z1, W1, S1 = ttm.titans_fwd_chunk_gates(d_["q"], d_["k"], d_["v"], c_["theta"],
                                                d_["W0"], chunk, eta=c_["eta"],
                                                alpha=c_["alpha"])
        z2, W2, S2 = ttm.titans_fwd(d_["q"], d_["k"], d_["v"], t_["theta"], d_["W0"], chunk,
                                    eta=t_["eta"], alpha=t_["alpha"])
    torch.cuda.synchronize()
    assert torch.equal(z1, z2) and torch.equal(W1, W2) and torch.equal(S1, S2)
    ref_inp = dict(inp, **tok)
    ref = H.run_linear_oracle(w, ref_inp)
    H.compare(dict(z=z1, W=W1, S=S1), ref, ["z", "W", "S"], H.TOL[dtype])

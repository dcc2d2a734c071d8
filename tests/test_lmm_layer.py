"""GPU parity of the LMM layer (ttm_lmm_layer_fwd: the memory as a standalone
sequence layer, "论文速览 | Titans" §6.4, §7.1-§7.3) against the float64
oracle, which rounds to bf16 at the points where the GPU layer stores bf16.
Tolerance 2e-2 per tensor (bf16 activations), on y, on the layer's own
contribution y - x, and on the final memory."""
import numpy as np
import pytest
import torch

import ttm_inputs as wl
from oracle import lmm
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


@pytest.mark.parametrize("B,T,Hh,d,chunk,conv_k", [
    (2, 150, 2, 64, 64, 4),     # tensor-core scan, ragged last chunk
    (1, 70, 3, 32, 16, 3),      # CUDA-core scan
    (1, 64, 2, 128, 64, 1),     # no conv taps beyond the current token
])
def test_layer_matches_oracle(B, T, Hh, d, chunk, conv_k):
    import test_neural_memory_gb300 as ttm
    p = wl.generate_lmm(B, T, Hh, d, conv_k=conv_k, seed=B * 100 + T)
    s = 0.1
    dev = H.to_dev(p)
    y, W, S = ttm.lmm_layer_fwd(dev["x"], dev["W_in"], dev["conv_w"], dev["rms_w"], dev["W_o"],
                                s, dev["W0"], chunk)
    torch.cuda.synchronize()
    f = H.f64
    r = lmm.lmm_layer(f(p["x"]), f(p["W_in"]), f(p["conv_w"]), f(p["rms_w"]), f(p["W_o"]), s,
                      f(p["W0"]), chunk, Hh, round_bf16=True)
    x = f(p["x"])
    errs = {"y": H.max_rel(f(y), r["y"]), "y-x": H.max_rel(f(y) - x, r["y"] - x),
            "W": H.max_rel(f(W), r["W"]), "S": H.max_rel(f(S), r["S"])}
    assert all(e <= H.TOL["bf16"] for e in errs.values()), errs

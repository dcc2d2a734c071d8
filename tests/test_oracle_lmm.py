"""Pins of the float64 LMM-layer oracle (oracle/lmm.py) to facts outside
itself.  CPU only."""
import numpy as np
import scipy.special
import torch

from oracle import lmm


def _params(rng, D, H, K=4, scale=0.05):
    P = 4 * D + 3 * H
    return dict(W_in=scale * rng.standard_normal((D, P)),
                conv_w=rng.standard_normal((3, D, K)) / K,
                rms_w=1.0 + 0.1 * rng.standard_normal(D // H),
                W_o=scale * rng.standard_normal((D, D)))


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    a = rng.standard_normal(10000) * 10.0 ** rng.integers(-5, 5, 10000)
    ref = torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    assert np.array_equal(lmm._bf16(a), ref)


def test_activations_match_library():
    x = np.linspace(-20, 20, 401)
    assert np.allclose(lmm.sigmoid(x), scipy.special.expit(x), rtol=1e-15, atol=0)
    assert np.allclose(lmm.silu(x), x * scipy.special.expit(x), rtol=1e-15, atol=1e-300)


def test_causal_conv_taps():
    rng = np.random.default_rng(1)
    u = rng.standard_normal((2, 7, 5))
    w = np.zeros((5, 4))
    w[:, 3] = 1.0                                # the current token only
    assert np.array_equal(lmm.causal_conv(u, w), u)
    w = np.zeros((5, 4))
    w[:, 1] = 1.0                                # two tokens back
    ref = np.zeros_like(u)
    ref[:, 2:] = u[:, :-2]
    assert np.array_equal(lmm.causal_conv(u, w), ref)
    w = rng.standard_normal((5, 4))              # brute force
    ref = np.zeros_like(u)
    for t in range(7):
        for j in range(4):
            s = t - 3 + j
            if s >= 0:
                ref[:, t] += w[:, j] * u[:, s]
    assert np.allclose(lmm.causal_conv(u, w), ref, atol=1e-14)


def test_zero_output_projection_is_the_residual():
    rng = np.random.default_rng(2)
    B, T, H, d = 2, 9, 2, 4
    p = _params(rng, H * d, H)
    p["W_o"] = np.zeros_like(p["W_o"])
    x = rng.standard_normal((B, T, H * d))
    r = lmm.lmm_layer(x, p["W_in"], p["conv_w"], p["rms_w"], p["W_o"], 0.1,
                      0.02 * rng.standard_normal((1, H, d, d)), 4, H)
    assert np.array_equal(r["y"], x)
    assert np.allclose(np.linalg.norm(r["q"], axis=-1), 1.0)
    assert np.allclose(np.linalg.norm(r["k"], axis=-1), 1.0)


def test_one_token_from_empty_memory_closed_form():
    """T = 1, W0 = 0: S_1 = 2 theta v k^T, W_1 = S_1, so z = 2 theta (k . q) v."""
    rng = np.random.default_rng(3)
    B, H, d = 1, 2, 4
    D = H * d
    p = _params(rng, D, H)
    x = rng.standard_normal((B, 1, D))
    s = 0.3
    r = lmm.lmm_layer(x, p["W_in"], p["conv_w"], p["rms_w"], p["W_o"], s,
                      np.zeros((1, H, d, d)), 4, H)
    proj = x[0, 0] @ p["W_in"]
    y = x[0, 0].copy()
    o = np.zeros(D)
    for h in range(H):
        sl = slice(h * d, (h + 1) * d)
        # only the current tap of the conv sees a token
        qh = lmm.silu(p["conv_w"][0, sl, -1] * proj[sl])
        kh = lmm.silu(p["conv_w"][1, sl, -1] * proj[D:2 * D][sl])
        vh = lmm.silu(p["conv_w"][2, sl, -1] * proj[2 * D:3 * D][sl])
        qh, kh = qh / np.linalg.norm(qh), kh / np.linalg.norm(kh)
        th = s * lmm.sigmoid(proj[4 * D + h])
        z = 2 * th * (kh @ qh) * vh
        o[sl] = z / np.sqrt(np.mean(z * z) + 1e-6) * p["rms_w"] * proj[3 * D:4 * D][sl]
    y += o @ p["W_o"]
    assert np.allclose(r["y"][0, 0], y, atol=1e-12)

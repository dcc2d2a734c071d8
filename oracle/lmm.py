"""LMM layer (the neural memory used on its own as a sequence layer), float64
numpy.  TEST INFRASTRUCTURE ONLY: the reference that the GPU layer is compared
against; the GPU library never imports it.

The layer follows "论文速览 | Titans" §6.4 (LMM: the memory as a standalone
sequence model) and §7.1-§7.3 (SiLU after the q, k, v projections, l2
normalisation of q and k, a short depthwise convolution after the
projections, residual connections, normalisation and linear gating before the
output projection).  The pages leave the exact wiring open; the plainest
reading taken here, per token t of a sequence x [T, D] with D = H d:

    p      = x W_in                                  (one projection: q | k | v | g | gate logits)
    u_c    = sum_j conv_w[c, j] p[t - (K-1) + j, c]  (causal depthwise conv of width K
                                                      on the q, k, v channels)
    q, k, v = SiLU(u) per channel; q, k l2-normalised per head
    theta  = s sigmoid(logit_theta), eta = sigmoid(logit_eta), alpha = sigmoid(logit_alpha)
    z      = Titans memory scan of (q, k, v) per head         (oracle.linear_primal)
    o      = RMSNorm_head(z) * rms_w * g                       (linear gate g = p's g columns)
    y      = x + o W_o                                         (residual)

`round_bf16` (optional) rounds the tensors that the GPU layer stores in bf16
(projection output, q / k / v, z, o) at the same points, so that the parity
test compares like with like; the arithmetic between those points stays
float64.
"""
from __future__ import annotations

import numpy as np

from . import linear_primal


def _bf16(a):
    """Round float64 values to the nearest bf16 (ties to even) and back."""
    f = np.asarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    rounded = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return rounded.astype(np.uint32).view(np.float32).astype(np.float64)


def silu(x):
    return x / (1.0 + np.exp(-x))


def sigmoid(x):
    return 1.0 / (1.0 + np.exp(-x))


def split_projection(p, H, d):
    """Columns of the input projection: q | k | v | g (D each) then theta, eta,
    alpha logits (H each)."""
    D = H * d
    return (p[..., :D], p[..., D:2 * D], p[..., 2 * D:3 * D], p[..., 3 * D:4 * D],
            p[..., 4 * D:4 * D + H], p[..., 4 * D + H:4 * D + 2 * H],
            p[..., 4 * D + 2 * H:4 * D + 3 * H])


def causal_conv(u, w):
    """u [B, T, C], w [C, K]: out[t, c] = sum_j w[c, j] u[t - (K-1) + j, c]
    (taps before the sequence start read zero)."""
    B, T, C = u.shape
    K = w.shape[1]
    out = np.zeros_like(u)
    for j in range(K):
        shift = K - 1 - j
        if shift >= T:
            continue
        out[:, shift:, :] += w[None, None, :, j] * u[:, :T - shift, :]
    return out


def lmm_layer(x, W_in, conv_w, rms_w, W_o, theta_scale, W0, chunk, H, w0_shared=True,
              round_bf16=False, eps=1e-6):
    """x [B, T, D]; W_in [D, 4D + 3H]; conv_w [3, D, K]; rms_w [d]; W_o [D, D];
    W0 [1 or B, H, d, d].  Returns dict(y, W, S, q, k, v, theta, eta, alpha, z, o)."""
    rnd = _bf16 if round_bf16 else (lambda a: a)
    x = np.asarray(x, dtype=np.float64)
    B, T, D = x.shape
    d = D // H
    p = rnd(x @ np.asarray(W_in, dtype=np.float64))
    pq, pk, pv, g, lt, le, la = split_projection(p, H, d)
    heads = lambda a: a.reshape(B, T, H, d).transpose(0, 2, 1, 3)     # [B, H, T, d]
    q = silu(causal_conv(pq, conv_w[0]))
    k = silu(causal_conv(pk, conv_w[1]))
    v = silu(causal_conv(pv, conv_w[2]))
    q, k, v = heads(q), heads(k), heads(v)
    q = q / np.maximum(np.linalg.norm(q, axis=-1, keepdims=True), eps)
    k = k / np.maximum(np.linalg.norm(k, axis=-1, keepdims=True), eps)
    q, k, v = rnd(q), rnd(k), rnd(v)
    gates = lambda a: a.transpose(0, 2, 1)                              # [B, H, T]
    theta = theta_scale * sigmoid(gates(lt))
    eta = sigmoid(gates(le))
    alpha = sigmoid(gates(la))
    r = linear_primal(q, k, v, theta, W0, chunk, eta=eta, alpha=alpha,
                      shared_over_batch=w0_shared)
    z = rnd(r["z"])                                                     # [B, H, T, d]
    ms = np.mean(z * z, axis=-1, keepdims=True)
    zn = z / np.sqrt(ms + eps) * np.asarray(rms_w, dtype=np.float64)
    o = rnd(zn.transpose(0, 2, 1, 3).reshape(B, T, D) * g)
    y = x + o @ np.asarray(W_o, dtype=np.float64)
    return dict(y=y, W=r["W"], S=r["S"], q=q, k=k, v=v, theta=theta, eta=eta, alpha=alpha,
                z=z, o=o)

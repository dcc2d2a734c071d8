"""Matrix ("dual") form of the linear / Titans scan in float64 PyTorch, so
that automatic differentiation can give its gradient.

TEST INFRASTRUCTURE ONLY: an independent route to the gradient that the
reverse-mode token loop in ``ttm_oracle.c`` computes by hand.  The pages ask
for exactly this check: run the token loop and the dual form in double
precision on small chunks and compare the gradients of the slow parameters,
the rates and W0 entry by entry ("TTT layers 与 fast weights" §1.2, on forward
and backward equivalence of the dual form).

The chunk algebra is that of ``dual.py`` ("TTT layers 与 fast weights" §1.1,
eqs (7)-(9); momentum and decay unrolled as in "论文速览 | Titans" §4.3 and
§4.5): inside a chunk that starts from (W, S), for local tokens s <= t

    W_t = beta_t W + c_t S - sum_{s<=t} theta_s w(s,t) grad_s
    S_t = P_t S - sum_{s<=t} theta_s mom(s->t) grad_s,   grad_s = 2 (W k_s - v_s) k_s^T

with the coefficients formed by explicit products of the gates.  Every
operation is a differentiable torch op on float64 CPU tensors.
"""
from __future__ import annotations

import torch


def _prod(x: torch.Tensor, lo: int, hi: int) -> torch.Tensor:
    """prod_{j=lo..hi} x[j]; 1 when the range is empty."""
    if hi < lo:
        return torch.ones((), dtype=x.dtype)
    return torch.prod(x[lo:hi + 1])


def _coefficients(theta, eta, alpha):
    n = theta.shape[0]
    keep = 1.0 - alpha
    beta = torch.stack([_prod(keep, 0, t) for t in range(n)])
    P = torch.stack([_prod(eta, 0, t) for t in range(n)])
    c = torch.stack([sum(_prod(keep, r + 1, t) * P[r] for r in range(t + 1)) for t in range(n)])
    C = [[None] * n for _ in range(n)]
    Pm = [[None] * n for _ in range(n)]
    zero = torch.zeros((), dtype=theta.dtype)
    for t in range(n):
        for s in range(n):
            if s > t:
                C[t][s] = zero
                Pm[t][s] = zero
                continue
            w = sum(_prod(keep, r + 1, t) * _prod(eta, s + 1, r) for r in range(s, t + 1))
            C[t][s] = theta[s] * w
            Pm[t][s] = theta[s] * _prod(eta, s + 1, t)
    C = torch.stack([torch.stack(row) for row in C])
    Pm = torch.stack([torch.stack(row) for row in Pm])
    return beta, P, c, C, Pm


def linear_dual_torch(q, k, v, theta, W0, chunk, eta=None, alpha=None, S0=None):
    """One (b, h) sequence: q, k [T,dk], v [T,dv], gates [T], W0 / S0 [dv,dk]
    (float64 tensors, any of them may require grad).  Returns z [T,dv], W, S."""
    T = q.shape[0]
    eta = torch.zeros(T, dtype=torch.float64) if eta is None else eta
    alpha = torch.zeros(T, dtype=torch.float64) if alpha is None else alpha
    W = W0
    S = torch.zeros_like(W0) if S0 is None else S0
    zs = []
    for c0 in range(0, T, chunk):
        c1 = min(c0 + chunk, T)
        K, Q, V = k[c0:c1], q[c0:c1], v[c0:c1]
        beta, P, c, C, Pm = _coefficients(theta[c0:c1], eta[c0:c1], alpha[c0:c1])
        E = W @ K.T - V.T                        # errors at the chunk-start state, [dv, n]
        A = torch.tril(Q @ K.T) * C              # causal (inclusive) scores times coefficients
        zs.append(beta[:, None] * (Q @ W.T) + c[:, None] * (Q @ S.T) - 2.0 * A @ E.T)
        W, S = (beta[-1] * W + c[-1] * S - 2.0 * (E * C[-1]) @ K,
                P[-1] * S - 2.0 * (E * Pm[-1]) @ K)
    return torch.cat(zs, dim=0), W, S

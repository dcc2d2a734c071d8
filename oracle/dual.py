"""Matrix ("dual") form of the chunked memory scan, float64 numpy.

TEST INFRASTRUCTURE ONLY: used to cross-check the token loop in
``ttm_oracle.c`` (primal form == dual form), never by the GPU library.

Within one chunk every gradient is taken at the chunk-start state, so the
writes of the whole chunk can be gathered into matrix products instead of
materialising a state per token ("TTT layers 与 fast weights", §1.1, eqs (7)
to (9)).  With momentum and forgetting, unrolling the two linear recurrences
inside the chunk gives, for local tokens s <= t,

    decay(r -> t) = prod_{j=r+1..t} (1 - alpha_j)       ("论文速览 | Titans" §4.3)
    mom(s -> r)   = prod_{j=s+1..r} eta_j               ("论文速览 | Titans" §4.5)
    W_t = beta_t W_0 + c_t S_0 - sum_{s<=t} theta_s w(s,t) grad_s
    S_t = P_t S_0 - sum_{s<=t} theta_s mom(s -> t) grad_s

with beta_t = prod_{j<=t}(1-alpha_j), P_t = prod_{j<=t} eta_j,
c_t = sum_{r<=t} decay(r->t) P_r and w(s,t) = sum_{r=s..t} decay(r->t) mom(s->r).
The coefficients are formed here by explicit products (slow, obvious), not by
the recurrences a kernel would use.
"""
from __future__ import annotations

import math

import numpy as np


def _prod(x, lo, hi):
    """prod_{j=lo..hi} x[j]; 1 when the range is empty."""
    p = 1.0
    for j in range(lo, hi + 1):
        p *= x[j]
    return p


def chunk_coefficients(theta, eta, alpha):
    """beta[t], P[t], c[t], C[t,s] = theta_s w(s,t), Pm[t,s] = theta_s mom(s->t) (s<=t)."""
    n = len(theta)
    keep = 1.0 - np.asarray(alpha, dtype=np.float64)
    eta = np.asarray(eta, dtype=np.float64)
    beta = np.array([_prod(keep, 0, t) for t in range(n)])
    P = np.array([_prod(eta, 0, t) for t in range(n)])
    c = np.array([sum(_prod(keep, r + 1, t) * P[r] for r in range(t + 1)) for t in range(n)])
    C = np.zeros((n, n))
    Pm = np.zeros((n, n))
    for t in range(n):
        for s in range(t + 1):
            w = sum(_prod(keep, r + 1, t) * _prod(eta, s + 1, r) for r in range(s, t + 1))
            C[t, s] = theta[s] * w
            Pm[t, s] = theta[s] * _prod(eta, s + 1, t)
    return beta, P, c, C, Pm


def linear_dual(q, k, v, theta, W0, chunk, eta=None, alpha=None, S0=None):
    """One (b, h) sequence: q, k [T,dk], v [T,dv], gates [T], W0/S0 [dv,dk]."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    T = q.shape[0]
    theta = np.asarray(theta, dtype=np.float64)
    eta = np.zeros(T) if eta is None else np.asarray(eta, dtype=np.float64)
    alpha = np.zeros(T) if alpha is None else np.asarray(alpha, dtype=np.float64)
    W = np.array(W0, dtype=np.float64)
    S = np.zeros_like(W) if S0 is None else np.array(S0, dtype=np.float64)
    z = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, chunk):
        sl = slice(c0, min(c0 + chunk, T))
        K, Q, V = k[sl], q[sl], v[sl]
        beta, P, c, C, Pm = chunk_coefficients(theta[sl], eta[sl], alpha[sl])
        E = W @ K.T - V.T                      # errors at the chunk-start state, [dv, n]
        A = np.tril(Q @ K.T) * C               # causal (inclusive) scores times coefficients
        z[sl] = beta[:, None] * (Q @ W.T) + c[:, None] * (Q @ S.T) - 2.0 * A @ E.T
        W, S = (beta[-1] * W + c[-1] * S - 2.0 * (E * C[-1]) @ K,
                P[-1] * S - 2.0 * (E * Pm[-1]) @ K)
    return z, W, S


def _gelu(x):
    return 0.5 * x * (1.0 + np.vectorize(math.erf)(x / math.sqrt(2.0)))


def _gelu_grad(x):
    Phi = 0.5 * (1.0 + np.vectorize(math.erf)(x / math.sqrt(2.0)))
    return Phi + x * np.exp(-0.5 * x * x) / math.sqrt(2.0 * math.pi)


def mlp_dual(q, k, v, theta, W1_0, W2_0, chunk, eta=None, alpha=None, S1_0=None, S2_0=None):
    """One (b, h) sequence of the 2-layer memory f(x) = W2 GELU(W1 x) in matrix form."""
    q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
    T = q.shape[0]
    theta = np.asarray(theta, dtype=np.float64)
    eta = np.zeros(T) if eta is None else np.asarray(eta, dtype=np.float64)
    alpha = np.zeros(T) if alpha is None else np.asarray(alpha, dtype=np.float64)
    W1 = np.array(W1_0, dtype=np.float64)
    W2 = np.array(W2_0, dtype=np.float64)
    S1 = np.zeros_like(W1) if S1_0 is None else np.array(S1_0, dtype=np.float64)
    S2 = np.zeros_like(W2) if S2_0 is None else np.array(S2_0, dtype=np.float64)
    z = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, chunk):
        sl = slice(c0, min(c0 + chunk, T))
        K, Q, V = k[sl], q[sl], v[sl]
        beta, P, c, C, Pm = chunk_coefficients(theta[sl], eta[sl], alpha[sl])
        Hk = K @ W1.T                                   # [n, hidden]
        Ak = _gelu(Hk)
        E = 2.0 * (Ak @ W2.T - V)                       # [n, d]  output-side error
        D1 = (E @ W2) * _gelu_grad(Hk)                  # [n, hidden]  hidden-side error
        mask = np.tril(np.ones((len(K), len(K))))
        Hq = (beta[:, None] * (Q @ W1.T) + c[:, None] * (Q @ S1.T)
              - (mask * C * (Q @ K.T)) @ D1)
        Aq = _gelu(Hq)
        z[sl] = (beta[:, None] * (Aq @ W2.T) + c[:, None] * (Aq @ S2.T)
                 - (mask * C * (Aq @ Ak.T)) @ E)
        W1, S1 = (beta[-1] * W1 + c[-1] * S1 - (D1 * C[-1][:, None]).T @ K,
                  P[-1] * S1 - (D1 * Pm[-1][:, None]).T @ K)
        W2, S2 = (beta[-1] * W2 + c[-1] * S2 - (E * C[-1][:, None]).T @ Ak,
                  P[-1] * S2 - (E * Pm[-1][:, None]).T @ Ak)
    return z, W1, W2, S1, S2

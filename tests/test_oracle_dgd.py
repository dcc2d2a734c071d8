"""Pins of the float64 DGD oracle ("Nested Learning" §8.1 eq (88) with the
matrix memory and L2 objective of eq (93), chunk-wise as in §8.2, read as eq
(86) prints it: y_t = M_{t-1} q_t, before the token's own write) to facts
outside itself.  CPU only.

- Two hand-worked examples of eq (93) (a scalar memory at chunk 1 and 2, and
  a 2x2 memory) fix the update, the gradient point and the read position; a
  read after the write gives different numbers for both.
- Chunk 1 with retention 1 is the online delta rule toward v / 2 with step
  2 eta, i.e. the already pinned linear oracle with theta = eta and targets
  v / 2, whose read after token t-1 is the DGD read of token t.
- Orthonormal keys decouple the k k^T term: every M_{t-1} k_t is the snapshot's
  M_c k_t times the retention so far, so the chunk has a closed form.
- The chunk form: with w_t = -eta_t (M_{t-1} k_t + M_c k_t - v_t), M_t is
  gamma_t M_c + sum_{s<=t} (gamma_t / gamma_s) w_s k_s^T, and the w_t solve a unit
  lower-triangular system in the key products k_s . k_t (solved here by a
  library routine), which must give the token loop's outputs.
"""
import numpy as np
import pytest
import scipy.linalg

import oracle


def _dgd(q, k, v, eta, alpha, W0, chunk):
    r = oracle.dgd_primal(q[None, None], k[None, None], v[None, None], eta[None, None],
                          alpha[None, None], W0[None, None], chunk)
    return r["z"][0, 0], r["W"][0, 0]


def test_hand_worked_examples(golden):
    g = golden("p3_dgd_read_before_write.json")
    sc = g["scalar"]
    a = lambda x: np.asarray(x, dtype=np.float64)
    for chunk in (1, 2):
        z, W = _dgd(a(sc["q"])[:, None], a(sc["k"])[:, None], a(sc["v"])[:, None], a(sc["eta"]),
                    a(sc["alpha"]), a([[sc["M0"]]]), chunk)
        want = sc[f"chunk_{chunk}"]
        assert np.allclose(z[:, 0], want["z"], atol=1e-14)
        assert np.allclose(W[0, 0], want["M_final"], atol=1e-14)
        assert not np.allclose(z[:, 0], sc["read_after_write_would_give"])
    m = g["matrix"]
    z, W = _dgd(a(m["q"]), a(m["k"]), a(m["v"]), a(m["eta"]), a(m["alpha"]), a(m["M0"]),
                m["chunk"])
    assert np.allclose(z, m["z"], atol=1e-14)
    assert np.allclose(W, m["M_final"], atol=1e-14)
    assert not np.allclose(z, m["read_after_write_would_give"])
    z1, W1 = _dgd(a(m["q"])[:1], a(m["k"])[:1], a(m["v"])[:1], a(m["eta"])[:1],
                  a(m["alpha"])[:1], a(m["M0"]), m["chunk"])
    assert np.allclose(W1, m["M1"], atol=1e-14)


def test_chunk_one_unit_retention_is_the_linear_delta_rule():
    rng = np.random.default_rng(1)
    T, dk, dv = 17, 5, 3
    q, k = rng.standard_normal((T, dk)), rng.standard_normal((T, dk)) / np.sqrt(dk)
    v = rng.standard_normal((T, dv))
    eta = rng.uniform(0.05, 0.3, T)
    W0 = rng.standard_normal((dv, dk))
    z, W = _dgd(q, k, v, eta, np.ones(T), W0, 1)
    # the linear oracle reads after each write: its read after token t-1 with
    # the query of token t is the DGD read of token t
    q_next = np.concatenate([q[1:], q[:1]])
    r = oracle.linear_primal(q_next[None, None], k[None, None], (v / 2)[None, None],
                             eta[None, None], W0[None, None], 1)
    assert np.allclose(z[0], W0 @ q[0], atol=1e-12)
    assert np.allclose(z[1:], r["z"][0, 0][:-1], atol=1e-12)
    assert np.allclose(W, r["W"][0, 0], atol=1e-12)


def test_orthonormal_keys_closed_form():
    rng = np.random.default_rng(2)
    dk, dv = 6, 4
    n = dk                                        # one chunk of dk orthonormal keys
    Qk, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    k = Qk.T                                      # rows orthonormal
    q = rng.standard_normal((n, dk))
    v = rng.standard_normal((n, dv))
    eta = rng.uniform(0.1, 0.4, n)
    alpha = rng.uniform(0.7, 1.0, n)
    Mc = rng.standard_normal((dv, dk))
    z, W = _dgd(q, k, v, eta, alpha, Mc, n)
    g = np.cumprod(alpha)                         # gamma_t = prod_{r<=t} alpha_r
    gprev = np.concatenate([[1.0], g[:-1]])
    # w_t = -eta_t (gamma_{t-1} Mc k_t + Mc k_t - v_t): no coupling between orthogonal keys
    w = -eta[:, None] * ((gprev[:, None] + 1.0) * (k @ Mc.T) - v)
    M_end = g[-1] * Mc + sum((g[-1] / g[s]) * np.outer(w[s], k[s]) for s in range(n))
    assert np.allclose(W, M_end, atol=1e-12)
    for t in range(n):
        # the read of token t sees the memory before its write (step t - 1)
        Mprev = gprev[t] * Mc + sum((gprev[t] / g[s]) * np.outer(w[s], k[s]) for s in range(t))
        assert np.allclose(z[t], Mprev @ q[t], atol=1e-12)


@pytest.mark.parametrize("T,chunk", [(23, 8), (16, 16), (9, 4)])
def test_chunk_form_with_triangular_solve(T, chunk):
    rng = np.random.default_rng(T * 100 + chunk)
    dk, dv = 5, 3
    q, k = rng.standard_normal((T, dk)), rng.standard_normal((T, dk)) / np.sqrt(dk)
    v = rng.standard_normal((T, dv))
    eta = rng.uniform(0.05, 0.3, T)
    alpha = rng.uniform(0.6, 1.0, T)
    W0 = rng.standard_normal((dv, dk))
    z, W = _dgd(q, k, v, eta, alpha, W0, chunk)
    M = W0.copy()
    zs = []
    for c0 in range(0, T, chunk):
        sl = slice(c0, min(T, c0 + chunk))
        K, Q, V, et, al = k[sl], q[sl], v[sl], eta[sl], alpha[sl]
        n = K.shape[0]
        g = np.cumprod(al)
        gprev = np.concatenate([[1.0], g[:-1]])
        KK = K @ K.T
        Lm = np.zeros((n, n))
        for t in range(n):
            for s in range(t):
                Lm[t, s] = et[t] * (gprev[t] / g[s]) * KK[s, t]
        R = -et[:, None] * (gprev[:, None] * (K @ M.T) + (K @ M.T) - V)
        Wv = scipy.linalg.solve_triangular(np.eye(n) + Lm, R, lower=True, unit_diagonal=True)
        D = np.tril(gprev[:, None] / g[None, :], -1)   # gamma_{t-1} / gamma_s for s < t
        zs.append(gprev[:, None] * (Q @ M.T) + (D * (Q @ K.T)) @ Wv)
        M = g[-1] * M + ((g[-1] / g)[:, None] * Wv).T @ K
    assert np.allclose(z, np.concatenate(zs), atol=1e-11)
    assert np.allclose(W, M, atol=1e-11)


def test_shared_initial_memory():
    rng = np.random.default_rng(4)
    B, H, T, d = 2, 2, 7, 3
    q, k, v = (rng.standard_normal((B, H, T, d)) for _ in range(3))
    eta, alpha = rng.uniform(0.1, 0.3, (B, H, T)), rng.uniform(0.8, 1.0, (B, H, T))
    W0 = rng.standard_normal((1, H, d, d))
    r = oracle.dgd_primal(q, k, v, eta, alpha, W0, 3, shared_over_batch=True)
    r2 = oracle.dgd_primal(q, k, v, eta, alpha, np.repeat(W0, B, axis=0), 3)
    assert np.array_equal(r["z"], r2["z"]) and np.array_equal(r["W"], r2["W"])


@pytest.mark.parametrize("T", [150, 64, 1])
def test_operator_form_of_the_tensor_core_scan(T):
    """The form the tensor-core kernels apply, restated here in float64: per chunk
    of 64 (the last one padded with alpha = 1, eta = 0 and zero rows), with
    R[t][s] = prod_{s<tau<t} alpha_tau built by products (no division), a_{t-1}
    the retention up to t - 1 and r_s = prod_{tau>s} alpha_tau:
      L = eta_t R (K K^T) (strictly lower), N = (I + L)^-1,
      A~N = (R o Q K^T) N, Y = K^T diag(r) N,
      R0 = diag(eta (a_- + 1)) K W_c^T - diag(eta) V,
      Z = diag(a_-) Q W_c^T - A~N R0,  W_end^T = a_{n-1} W_c^T - Y R0.
    It must give the token loop's reads and final memory."""
    rng = np.random.default_rng(T + 7)
    dk, dv, C = 6, 4, 64
    q, k = rng.standard_normal((T, dk)), rng.standard_normal((T, dk)) / np.sqrt(dk)
    v = rng.standard_normal((T, dv))
    eta = rng.uniform(0.02, 0.2, T)
    alpha = rng.uniform(0.85, 1.0, T)
    W0 = rng.standard_normal((dv, dk))
    z, W = _dgd(q, k, v, eta, alpha, W0, C)
    Wt = W0.T.copy()
    zs = []
    for c0 in range(0, T, C):
        n = min(C, T - c0)
        Q, K, V = (np.zeros((C, x.shape[1])) for x in (q, k, v))
        Q[:n], K[:n], V[:n] = q[c0:c0 + n], k[c0:c0 + n], v[c0:c0 + n]
        et, al = np.zeros(C), np.ones(C)
        et[:n], al[:n] = eta[c0:c0 + n], alpha[c0:c0 + n]
        R = np.zeros((C, C))
        for t in range(C):
            p = 1.0
            for s in range(t - 1, -1, -1):       # walk down from the diagonal
                R[t, s] = p
                p *= al[s]
        a_prev = np.ones(C)
        for t in range(1, C):
            a_prev[t] = a_prev[t - 1] * al[t - 1]
        r = np.ones(C)
        for s in range(C - 2, -1, -1):
            r[s] = r[s + 1] * al[s + 1]
        a_end = a_prev[-1] * al[-1]
        L = et[:, None] * R * (K @ K.T)
        N = np.linalg.inv(np.eye(C) + L)
        AN = (R * (Q @ K.T)) @ N
        Y = (K.T * r[None, :]) @ N
        R0 = (et * (a_prev + 1.0))[:, None] * (K @ Wt) - et[:, None] * V
        zs.append((a_prev[:, None] * (Q @ Wt) - AN @ R0)[:n])
        Wt = a_end * Wt - Y @ R0
    assert np.allclose(z, np.concatenate(zs), atol=1e-11)
    assert np.allclose(W, Wt.T, atol=1e-11)

"""Pins of the float64 oracle to facts outside itself.

Every check here is CPU-only.  The values come from the pages' worked examples
(``tests/golden/*.json``, each citing its page and section), from closed forms
the pages state, from library routines (torch autograd, math.erf) and from
invariants of the mathematics.  Together they are meant to catch a dropped
term, a wrong sign or factor, a transposed operand, a wrong chunk boundary or
a read taken before the write.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import dual


def lin(k, v, theta, chunk, q=None, W0=None, eta=None, alpha=None, S0=None):
    """Run the oracle on one (b, h) sequence given as [T, d] arrays."""
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    if k.ndim == 1:
        k = k[:, None]
    if v.ndim == 1:
        v = v[:, None]
    T, dk = k.shape
    dv = v.shape[1]
    q = k if q is None else np.asarray(q, dtype=np.float64).reshape(T, dk)
    theta = np.broadcast_to(np.asarray(theta, dtype=np.float64), (T,))
    W0 = np.zeros((dv, dk)) if W0 is None else np.asarray(W0, dtype=np.float64).reshape(dv, dk)
    ex = lambda a: None if a is None else np.broadcast_to(np.asarray(a, np.float64), (T,))[None, None]
    S0 = None if S0 is None else np.asarray(S0, dtype=np.float64).reshape(1, 1, dv, dk)
    r = oracle.linear_primal(q[None, None], k[None, None], v[None, None], theta[None, None],
                             W0[None, None], chunk, eta=ex(eta), alpha=ex(alpha), S0=S0)
    return r["z"][0, 0], r["W"][0, 0], r["S"][0, 0]


# ---------------------------------------------------------------- page pins

def test_p1_two_token_chunk(golden):
    g = golden("p1_two_token_chunk.json")
    z1, W1, _ = lin(g["k"], g["v"], g["theta"], 1, q=g["q"])
    assert np.allclose(z1[:, 0], g["online_b1"]["reads"], atol=1e-14)
    assert np.isclose(W1[0, 0], g["online_b1"]["final_w"], atol=1e-14)
    z2, W2, _ = lin(g["k"], g["v"], g["theta"], 2, q=g["q"])
    assert np.allclose(z2[:, 0], g["chunk_b2"]["reads"], atol=1e-14)
    assert np.isclose(W2[0, 0], g["chunk_b2"]["final_w"], atol=1e-14)


def test_p2_delta_rule_2d(golden):
    g = golden("p2_delta_rule_2d.json")
    z, W, _ = lin(g["k"], g["v"], g["theta"], 1, q=g["q"])
    assert np.allclose(z, g["b1"]["reads"], atol=1e-14)
    assert np.allclose(W, g["b1"]["W2"], atol=1e-14)
    _, W1, _ = lin(g["k"][:1], g["v"][:1], g["theta"], 1, q=g["q"][:1])
    assert np.allclose(W1, g["b1"]["W1"], atol=1e-14)
    z, W, _ = lin(g["k"], g["v"], g["theta"], 2, q=g["q"])
    assert np.allclose(W, g["b2"]["W2"], atol=1e-14)
    assert np.allclose(z[1], g["b2"]["read_token2"], atol=1e-14)


def test_p2_eq11_error_recurrence(golden):
    g = golden("p2_eq11_error_recurrence.json")
    for case in g["cases"]:
        n = len(case["u"])
        z, _, _ = lin(np.ones(n), np.ones(n), case["theta"], 1)
        assert np.allclose(z[:, 0], case["u"], atol=1e-12), case


def test_p1_delta_correction(golden):
    g = golden("p1_delta_correction.json")
    z, W, _ = lin([g["k"]], [g["v"]], g["theta"], 1, q=[g["k"]], W0=g["W0"])
    assert np.allclose(W.T, g["page_W_new_row_convention"], atol=1e-14)
    assert np.allclose(z[0], g["reads"]["key_1_0"], atol=1e-14)
    assert np.allclose(W @ np.array([0.0, 1.0]), g["reads"]["key_0_1"], atol=1e-14)


def test_p2_interference(golden):
    g = golden("p2_interference.json")
    k1 = g["k"][0]
    z, _, _ = lin(g["k"], g["v"], g["theta"], 1, q=[k1, k1])
    assert np.allclose(z[1], g["W2_k1"], atol=1e-14)
    _, W1, _ = lin(g["k"][:1], g["v"][:1], g["theta"], 1)
    assert np.allclose(W1 @ np.array(g["k"][1]), g["W1_k2"], atol=1e-14)
    assert np.allclose(np.array(g["v"][1]) - W1 @ np.array(g["k"][1]), g["residual_2"], atol=1e-14)


def test_p1_titans_scalar(golden):
    g = golden("p1_titans_scalar.json")
    theta = g["step_half_loss"] / 2.0
    v = g["W_prev"] * 1.0 - g["g_half_loss"]       # half-loss gradient (W k - v) k with k = 1
    z, W, S = lin([1.0], [v], theta, 1, q=[1.0], W0=[[g["W_prev"]]], eta=g["mu"],
                  alpha=g["alpha"], S0=[[g["U_prev"]]])
    assert np.isclose(S[0, 0], g["U_new"], atol=1e-14)
    assert np.isclose(W[0, 0], g["W_new"], atol=1e-14)
    assert np.isclose(z[0, 0], g["W_new"], atol=1e-14)


def test_p1_linear_attention(golden):
    g = golden("p1_linear_attention.json")
    q = [g["q"], g["q"]]
    z, W, _ = lin(g["k"], g["v"], g["theta"], 2, q=q)
    assert np.allclose(z[1], g["read"], atol=1e-14)
    assert np.allclose(W.T, g["S2_row_convention"], atol=1e-14)


def test_p2_end_to_end_scalar(golden):
    for c in golden("p2_end_to_end_scalar.json")["cases"]:
        z, W, _ = lin([1.0], [2.0], c["eta_half_loss"] / 2.0, 1, q=[1.0], W0=[[c["w0"]]])
        assert np.isclose(W[0, 0], c["w1"], atol=1e-14)


def test_eq7_eq9_single_chunk_closed_form():
    """'TTT layers 与 fast weights' eqs (7)-(9): identity views (q = k = v = x), one chunk."""
    rng = np.random.default_rng(7)
    b, d, eta = 9, 5, 0.07
    X = rng.standard_normal((d, b))            # columns are tokens, as on the page
    W0 = rng.standard_normal((d, d))
    z, W, _ = lin(X.T, X.T, eta, b, q=X.T, W0=W0)
    resid = W0 @ X - X
    Wb = W0 - 2 * eta * resid @ X.T                                     # eq (7)
    Z = W0 @ X - 2 * eta * resid @ np.triu(X.T @ X)                     # eqs (8), (9)
    assert np.allclose(W, Wb, atol=1e-12)
    assert np.allclose(z.T, Z, atol=1e-12)


# ------------------------------------------------------------- self-checks

def _rand_seq(rng, T, dk, dv):
    k = rng.standard_normal((T, dk)); k /= np.linalg.norm(k, axis=1, keepdims=True)
    q = rng.standard_normal((T, dk)); q /= np.linalg.norm(q, axis=1, keepdims=True)
    v = rng.standard_normal((T, dv))
    return q, k, v


def test_selfcheck_a_delta_rule():
    """b = 1 equals the delta rule S_t = S_{t-1}(I - beta k k^T) + beta v k^T with beta = 2 theta
    ('TTT layers 与 fast weights' eq (5) and the DeltaNet comparison after it)."""
    rng = np.random.default_rng(1)
    T, dk, dv = 23, 6, 4
    q, k, v = _rand_seq(rng, T, dk, dv)
    theta = 0.3 * rng.random(T)
    W0 = rng.standard_normal((dv, dk))
    z, W, _ = lin(k, v, theta, 1, q=q, W0=W0)
    M = W0.copy()
    for t in range(T):
        beta = 2 * theta[t]
        M = M @ (np.eye(dk) - beta * np.outer(k[t], k[t])) + beta * np.outer(v[t], k[t])
        assert np.allclose(z[t], M @ q[t], atol=1e-12)
    assert np.allclose(W, M, atol=1e-12)


def test_selfcheck_b_zero_momentum_is_minibatch_gd():
    """eta = alpha = 0 reduces Titans to plain mini-batch GD ('TTT layers 与 fast weights' eq (6)
    with G_t taken at the end of the previous mini-batch)."""
    rng = np.random.default_rng(2)
    T, dk, dv, b = 37, 5, 3, 8
    q, k, v = _rand_seq(rng, T, dk, dv)
    theta = 0.2 * rng.random(T)
    W0 = rng.standard_normal((dv, dk))
    z0, W_0, _ = lin(k, v, theta, b, q=q, W0=W0, eta=np.zeros(T), alpha=np.zeros(T),
                     S0=rng.standard_normal((dv, dk)))
    z1, W_1, _ = lin(k, v, theta, b, q=q, W0=W0)
    assert np.allclose(z0, z1, atol=1e-13) and np.allclose(W_0, W_1, atol=1e-13)
    # eq (6): W_t = W_{t'} - sum over the chunk so far of theta_s G_s, G_s at W_{t'}
    W = W0.copy()
    for c0 in range(0, T, b):
        Wt = W.copy()
        acc = np.zeros_like(W)
        for t in range(c0, min(c0 + b, T)):
            acc += theta[t] * 2 * np.outer(Wt @ k[t] - v[t], k[t])
            assert np.allclose(z0[t], (Wt - acc) @ q[t], atol=1e-12)
        W = Wt - acc
    assert np.allclose(W_0, W, atol=1e-12)


@pytest.mark.parametrize("chunk", [1, 4, 7, 16])
def test_selfcheck_c_dual_equals_primal_linear(chunk):
    rng = np.random.default_rng(3 + chunk)
    T, dk, dv = 45, 6, 5                       # 45 is not a multiple of 4, 7 or 16
    q, k, v = _rand_seq(rng, T, dk, dv)
    theta = 0.1 * rng.random(T)
    eta = 0.8 + 0.2 * rng.random(T)
    alpha = 0.05 * rng.random(T)
    W0 = 0.3 * rng.standard_normal((dv, dk))
    S0 = 0.1 * rng.standard_normal((dv, dk))
    zp, Wp, Sp = lin(k, v, theta, chunk, q=q, W0=W0, eta=eta, alpha=alpha, S0=S0)
    zd, Wd, Sd = dual.linear_dual(q, k, v, theta, W0, chunk, eta=eta, alpha=alpha, S0=S0)
    assert np.allclose(zp, zd, atol=1e-13)
    assert np.allclose(Wp, Wd, atol=1e-13)
    assert np.allclose(Sp, Sd, atol=1e-13)


@pytest.mark.parametrize("chunk", [1, 3, 8])
def test_selfcheck_c_dual_equals_primal_mlp(chunk):
    rng = np.random.default_rng(11 + chunk)
    T, d, hid = 19, 4, 7
    q, k, v = _rand_seq(rng, T, d, d)
    theta = 0.05 * rng.random(T)
    eta = 0.9 * np.ones(T) - 0.1 * rng.random(T)
    alpha = 0.02 * rng.random(T)
    W1 = 0.5 * rng.standard_normal((hid, d))
    W2 = 0.5 * rng.standard_normal((d, hid))
    S1 = 0.1 * rng.standard_normal((hid, d))
    S2 = 0.1 * rng.standard_normal((d, hid))
    r = oracle.mlp_primal(q[None, None], k[None, None], v[None, None], theta[None, None],
                          W1[None, None], W2[None, None], chunk, eta=eta[None, None],
                          alpha=alpha[None, None], S1_0=S1[None, None], S2_0=S2[None, None])
    zd, W1d, W2d, S1d, S2d = dual.mlp_dual(q, k, v, theta, W1, W2, chunk, eta=eta, alpha=alpha,
                                           S1_0=S1, S2_0=S2)
    assert np.allclose(r["z"][0, 0], zd, atol=1e-13)
    for a, b_ in ((r["W1"], W1d), (r["W2"], W2d), (r["S1"], S1d), (r["S2"], S2d)):
        assert np.allclose(a[0, 0], b_, atol=1e-13)


def test_selfcheck_d_mlp_gradient_finite_differences():
    """Analytic inner gradients against central differences at several step sizes
    ('TTT layers 与 fast weights' §1.2, advice on multi-scale finite-difference checks)."""
    rng = np.random.default_rng(5)
    d, hid = 3, 5
    W1 = rng.standard_normal((hid, d))
    W2 = rng.standard_normal((d, hid))
    k = rng.standard_normal(d)
    v = rng.standard_normal(d)
    g1, g2 = oracle.mlp_grad(W1, W2, k, v)
    best = []
    for eps in (1e-3, 1e-4, 1e-5, 1e-6):
        n1 = np.zeros_like(W1)
        n2 = np.zeros_like(W2)
        for idx in np.ndindex(W1.shape):
            P, M = W1.copy(), W1.copy(); P[idx] += eps; M[idx] -= eps
            n1[idx] = (oracle.mlp_loss(P, W2, k, v) - oracle.mlp_loss(M, W2, k, v)) / (2 * eps)
        for idx in np.ndindex(W2.shape):
            P, M = W2.copy(), W2.copy(); P[idx] += eps; M[idx] -= eps
            n2[idx] = (oracle.mlp_loss(W1, P, k, v) - oracle.mlp_loss(W1, M, k, v)) / (2 * eps)
        best.append(max(np.abs(n1 - g1).max(), np.abs(n2 - g2).max()))
    assert min(best) < 1e-8, best
    assert best[0] > best[1] or best[0] < 1e-8            # error falls with eps at first


def test_selfcheck_d_mlp_gradient_autograd():
    """The same gradients from torch autograd with its exact GELU."""
    rng = np.random.default_rng(6)
    d, hid = 4, 6
    W1 = torch.tensor(rng.standard_normal((hid, d)), requires_grad=True)
    W2 = torch.tensor(rng.standard_normal((d, hid)), requires_grad=True)
    k = torch.tensor(rng.standard_normal(d))
    v = torch.tensor(rng.standard_normal(d))
    loss = ((W2 @ torch.nn.functional.gelu(W1 @ k) - v) ** 2).sum()
    loss.backward()
    g1, g2 = oracle.mlp_grad(W1.detach().numpy(), W2.detach().numpy(), k.numpy(), v.numpy())
    assert np.allclose(g1, W1.grad.numpy(), atol=1e-12)
    assert np.allclose(g2, W2.grad.numpy(), atol=1e-12)
    assert math.isclose(oracle.mlp_loss(W1.detach().numpy(), W2.detach().numpy(), k.numpy(),
                                        v.numpy()), loss.item(), rel_tol=1e-13)


def _autograd_scan(q, k, v, theta, eta, alpha, chunk, f, params):
    """Token loop whose gradients come from torch autograd, not from a formula."""
    W = [p.clone() for p in params]
    S = [torch.zeros_like(p) for p in params]
    zs = []
    for t in range(q.shape[0]):
        if t % chunk == 0:
            Wc = [w.clone() for w in W]
        P = [w.clone().requires_grad_(True) for w in Wc]
        ((f(P, k[t]) - v[t]) ** 2).sum().backward()
        for i in range(len(W)):
            S[i] = eta[t] * S[i] - theta[t] * P[i].grad
            W[i] = (1 - alpha[t]) * W[i] + S[i]
        zs.append(f(W, q[t]).detach())
    return torch.stack(zs), W, S


def test_linear_oracle_against_autograd_scan():
    rng = np.random.default_rng(8)
    T, d, chunk = 14, 3, 4
    q, k, v = (torch.tensor(x) for x in _rand_seq(rng, T, d, d))
    theta, eta, alpha = (torch.tensor(x) for x in
                         (0.2 * rng.random(T), 0.9 * rng.random(T), 0.1 * rng.random(T)))
    W0 = torch.tensor(rng.standard_normal((d, d)))
    z, W, S = _autograd_scan(q, k, v, theta, eta, alpha, chunk, lambda P, x: P[0] @ x, [W0])
    zo, Wo, So = lin(k.numpy(), v.numpy(), theta.numpy(), chunk, q=q.numpy(), W0=W0.numpy(),
                     eta=eta.numpy(), alpha=alpha.numpy())
    assert np.allclose(zo, z.numpy(), atol=1e-12)
    assert np.allclose(Wo, W[0].numpy(), atol=1e-12) and np.allclose(So, S[0].numpy(), atol=1e-12)


def test_mlp_oracle_against_autograd_scan():
    rng = np.random.default_rng(9)
    T, d, hid, chunk = 11, 3, 5, 3
    q, k, v = (torch.tensor(x) for x in _rand_seq(rng, T, d, d))
    theta, eta, alpha = (torch.tensor(x) for x in
                         (0.2 * rng.random(T), 0.9 * rng.random(T), 0.1 * rng.random(T)))
    W1 = torch.tensor(rng.standard_normal((hid, d)))
    W2 = torch.tensor(rng.standard_normal((d, hid)))
    f = lambda P, x: P[1] @ torch.nn.functional.gelu(P[0] @ x)
    z, W, S = _autograd_scan(q, k, v, theta, eta, alpha, chunk, f, [W1, W2])
    r = oracle.mlp_primal(q.numpy()[None, None], k.numpy()[None, None], v.numpy()[None, None],
                          theta.numpy()[None, None], W1.numpy()[None, None],
                          W2.numpy()[None, None], chunk, eta=eta.numpy()[None, None],
                          alpha=alpha.numpy()[None, None])
    assert np.allclose(r["z"][0, 0], z.numpy(), atol=1e-12)
    assert np.allclose(r["W1"][0, 0], W[0].numpy(), atol=1e-12)
    assert np.allclose(r["W2"][0, 0], W[1].numpy(), atol=1e-12)
    assert np.allclose(r["S1"][0, 0], S[0].numpy(), atol=1e-12)
    assert np.allclose(r["S2"][0, 0], S[1].numpy(), atol=1e-12)


def test_gelu_against_erf_and_differences():
    for x in (-3.0, -1.2, -0.3, 0.0, 0.4, 1.7, 5.0):
        assert math.isclose(oracle.gelu(x), 0.5 * x * (1 + math.erf(x / math.sqrt(2))),
                            rel_tol=1e-15, abs_tol=1e-300)
        h = 1e-5
        fd = (oracle.gelu(x + h) - oracle.gelu(x - h)) / (2 * h)
        assert abs(fd - oracle.gelu_grad(x)) < 1e-9
    assert math.isclose(oracle.gelu(1.0), torch.nn.functional.gelu(torch.tensor(1.0,
                        dtype=torch.float64)).item(), rel_tol=1e-15)


# -------------------------------------------------------------- invariants

def _titans_case(seed, T=29, dk=5, dv=4):
    rng = np.random.default_rng(seed)
    q, k, v = _rand_seq(rng, T, dk, dv)
    return dict(q=q, k=k, v=v, theta=0.15 * rng.random(T), eta=0.7 + 0.3 * rng.random(T),
                alpha=0.1 * rng.random(T), W0=rng.standard_normal((dv, dk)),
                S0=rng.standard_normal((dv, dk))), rng


def _run(c, chunk, **over):
    c = {**c, **over}
    return lin(c["k"], c["v"], c["theta"], chunk, q=c["q"], W0=c["W0"], eta=c["eta"],
               alpha=c["alpha"], S0=c["S0"])


def test_I1_superposition():
    c, rng = _titans_case(20)
    c2, _ = _titans_case(21)
    a, b = 0.7, -1.3
    mix = dict(W0=a * c["W0"] + b * c2["W0"], S0=a * c["S0"] + b * c2["S0"],
               v=a * c["v"] + b * c2["v"])
    r1 = _run(c, 6)
    r2 = _run(c, 6, W0=c2["W0"], S0=c2["S0"], v=c2["v"])
    rm = _run(c, 6, **mix)
    for x1, x2, xm in zip(r1, r2, rm):
        assert np.allclose(a * x1 + b * x2, xm, atol=1e-12)


def test_I2_row_permutation():
    c, rng = _titans_case(22)
    perm = rng.permutation(c["v"].shape[1])
    r = _run(c, 5)
    rp = _run(c, 5, W0=c["W0"][perm], S0=c["S0"][perm], v=c["v"][:, perm])
    assert np.allclose(r[0][:, perm], rp[0], atol=1e-13)
    assert np.allclose(r[1][perm], rp[1], atol=1e-13)
    assert np.allclose(r[2][perm], rp[2], atol=1e-13)


def test_I3_sequence_independence():
    rng = np.random.default_rng(23)
    B, H, T, d = 2, 3, 17, 4
    q = rng.standard_normal((B, H, T, d)); k = rng.standard_normal((B, H, T, d))
    v = rng.standard_normal((B, H, T, d)); th = 0.1 * rng.random((B, H, T))
    et = 0.9 * rng.random((B, H, T)); al = 0.1 * rng.random((B, H, T))
    W0 = rng.standard_normal((1, H, d, d))
    r = oracle.linear_primal(q, k, v, th, W0, 5, eta=et, alpha=al, shared_over_batch=True)
    for b in range(B):
        for h in range(H):
            z, W, S = lin(k[b, h], v[b, h], th[b, h], 5, q=q[b, h], W0=W0[0, h], eta=et[b, h],
                          alpha=al[b, h])
            assert np.array_equal(z, r["z"][b, h]) and np.array_equal(W, r["W"][b, h])
            assert np.array_equal(S, r["S"][b, h])


def test_I4_consistent_memory_is_a_fixed_point():
    rng = np.random.default_rng(24)
    T, d = 21, 5
    q, k, _ = _rand_seq(rng, T, d, d)
    W0 = rng.standard_normal((d, d))
    v = k @ W0.T
    z, W, _ = lin(k, v, 0.3 * rng.random(T), 4, q=q, W0=W0)
    assert np.allclose(W, W0, atol=1e-13)
    assert np.allclose(z, q @ W0.T, atol=1e-13)


@pytest.mark.parametrize("T1", [12, 13])
def test_I5_split_call_continuation(T1):
    c, _ = _titans_case(25, T=30)
    chunk = 4
    z, W, S = _run(c, chunk)
    first = {key: (c[key][:T1] if key in ("q", "k", "v", "theta", "eta", "alpha") else c[key])
             for key in c}
    second = {key: (c[key][T1:] if key in ("q", "k", "v", "theta", "eta", "alpha") else c[key])
              for key in c}
    za, Wa, Sa = _run(first, chunk)
    zb, Wb, Sb = _run(second, chunk, W0=Wa, S0=Sa)
    same = np.allclose(np.concatenate([za, zb]), z, atol=1e-12) and np.allclose(Wb, W, atol=1e-12)
    # continuation is exact only when the split falls on a chunk boundary
    assert same == (T1 % chunk == 0)


def test_I6_zero_step_closed_form():
    """theta = 0 leaves only decay and momentum: W_T = beta_T W0 + (sum_r beta_T/beta_r P_r) S0
    ('论文速览 | Titans' §4.3 unrolled form)."""
    c, _ = _titans_case(26)
    T = len(c["theta"])
    z, W, S = _run(c, 7, theta=np.zeros(T))
    keep = 1 - c["alpha"]
    beta_T = np.prod(keep)
    P = np.cumprod(c["eta"])
    coef = sum(np.prod(keep[r + 1:]) * P[r] for r in range(T))
    assert np.allclose(W, beta_T * c["W0"] + coef * c["S0"], atol=1e-13)
    assert np.allclose(S, P[-1] * c["S0"], atol=1e-13)


def test_shared_initial_state_over_batch():
    rng = np.random.default_rng(27)
    B, H, T, d = 3, 2, 9, 3
    q = rng.standard_normal((B, H, T, d)); k = rng.standard_normal((B, H, T, d))
    v = rng.standard_normal((B, H, T, d)); th = 0.1 * rng.random((B, H, T))
    W0 = rng.standard_normal((1, H, d, d))
    a = oracle.linear_primal(q, k, v, th, W0, 4, shared_over_batch=True)
    b = oracle.linear_primal(q, k, v, th, np.repeat(W0, B, axis=0), 4)
    assert np.array_equal(a["z"], b["z"]) and np.array_equal(a["W"], b["W"])


def test_empty_sequence_returns_initial_state():
    W0 = np.arange(4.0).reshape(1, 1, 2, 2)
    r = oracle.linear_primal(np.zeros((1, 1, 0, 2)), np.zeros((1, 1, 0, 2)),
                             np.zeros((1, 1, 0, 2)), np.zeros((1, 1, 0)), W0, 3)
    assert r["z"].shape == (1, 1, 0, 2) and np.array_equal(r["W"], W0)

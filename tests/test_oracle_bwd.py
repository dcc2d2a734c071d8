"""Pins of the float64 oracle's gradient (reverse mode through the token loop)
to facts outside itself.  CPU only.

- Central finite differences of the forward oracle at several step sizes, the
  check the pages prescribe for outer gradients ("TTT layers 与 fast weights"
  §1.2: perturb a slow parameter both ways, re-run the whole inner loop, and
  watch the difference converge over several scales).
- The gradient of an independent dual-form restatement by torch autograd, in
  float64 (the same passage: token loop and dual form must agree on the
  gradients of the slow parameters, the rates and W0, entry by entry).
- The pages' worked scalar examples of outer gradients (tests/golden).
- Closed forms: the derivative of a one-token read, and linearity in dz.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.dual_grad import linear_dual_torch


def _problem(rng, B=1, H=1, T=7, dk=3, dv=3, titans=True, s0=True, scale=0.3):
    q, k = (rng.standard_normal((B, H, T, dk)) for _ in range(2))
    v = rng.standard_normal((B, H, T, dv))
    p = dict(q=q, k=k, v=v, theta=rng.uniform(0.05, 0.2, (B, H, T)),
             W0=scale * rng.standard_normal((B, H, dv, dk)))
    if titans:
        p["eta"] = rng.uniform(0.5, 0.95, (B, H, T))
        p["alpha"] = rng.uniform(0.0, 0.1, (B, H, T))
        if s0:
            p["S0"] = 0.1 * rng.standard_normal((B, H, dv, dk))
    adj = dict(dz=rng.standard_normal((B, H, T, dv)), dW=rng.standard_normal((B, H, dv, dk)),
               dS=rng.standard_normal((B, H, dv, dk)) if titans else None)
    return p, adj


def _loss(p, adj, chunk, shared=False):
    r = oracle.linear_primal(p["q"], p["k"], p["v"], p["theta"], p["W0"], chunk,
                             eta=p.get("eta"), alpha=p.get("alpha"), S0=p.get("S0"),
                             shared_over_batch=shared, threads=1)
    L = float((r["z"] * adj["dz"]).sum() + (r["W"] * adj["dW"]).sum())
    if adj["dS"] is not None:
        L += float((r["S"] * adj["dS"]).sum())
    return L


def _grad(p, adj, chunk, shared=False):
    return oracle.linear_primal_bwd(p["q"], p["k"], p["v"], p["theta"], p["W0"], chunk,
                                    adj["dz"], eta=p.get("eta"), alpha=p.get("alpha"),
                                    S0=p.get("S0"), dW=adj["dW"], dS=adj["dS"],
                                    shared_over_batch=shared, threads=1)


GRAD_OF = {"q": "dq", "k": "dk", "v": "dv", "theta": "dtheta", "eta": "deta",
           "alpha": "dalpha", "W0": "dW0", "S0": "dS0"}


def _central(p, adj, chunk, name, h, shared=False, idxs=None):
    x = p[name]
    idxs = list(np.ndindex(x.shape)) if idxs is None else idxs
    out = {}
    for idx in idxs:
        for sgn in (1, -1):
            pp = dict(p)
            pp[name] = x.copy()
            pp[name][idx] += sgn * h
            out.setdefault(idx, []).append(_loss(pp, adj, chunk, shared))
    return {i: (a - b) / (2 * h) for i, (a, b) in out.items()}


@pytest.mark.parametrize("case", ["titans_ragged", "linear", "rect_two_chunks", "shared_w0"])
def test_gradient_matches_central_differences(case):
    rng = np.random.default_rng(
        {"titans_ragged": 1, "linear": 2, "rect_two_chunks": 3, "shared_w0": 4}[case])
    shared = False
    if case == "titans_ragged":
        p, adj = _problem(rng, T=7, dk=3, dv=3)
        chunk = 3                       # chunks of 3, 3 and a ragged 1
    elif case == "linear":
        p, adj = _problem(rng, T=6, dk=3, dv=2, titans=False)
        chunk = 4
    elif case == "rect_two_chunks":
        p, adj = _problem(rng, T=8, dk=4, dv=2, s0=False)
        chunk = 4
    else:
        p, adj = _problem(rng, B=2, T=5, dk=2, dv=3)
        p["W0"] = p["W0"][:1]
        p["S0"] = p["S0"][:1]
        chunk, shared = 2, True
    g = _grad(p, adj, chunk, shared)
    for name in [n for n in GRAD_OF if n in p]:
        fd = _central(p, adj, chunk, name, 1e-6, shared)
        got = np.array([g[GRAD_OF[name]][i] for i in fd])
        ref = np.array(list(fd.values()))
        scale = max(np.abs(ref).max(), 1e-12)
        assert np.abs(got - ref).max() / scale < 1e-7, name


def test_difference_quotients_converge_at_second_order():
    """Along a random direction through a whole input tensor, the central
    difference approaches the directional derivative like h^2 over several
    step sizes.  (With every other entry held fixed the loss is a polynomial of
    degree <= 2 in any single entry, since the update is affine in the state
    and each gate enters one token's update once, so a single-entry central
    difference is already exact; a whole-tensor direction is not.)"""
    rng = np.random.default_rng(3)
    p, adj = _problem(rng, T=9, dk=3, dv=3)
    g = _grad(p, adj, 4)
    for name in ("k", "theta", "eta", "alpha"):
        d = rng.standard_normal(p[name].shape)
        exact = float((g[GRAD_OF[name]] * d).sum())
        errs = []
        for h in (4e-2, 4e-3, 4e-4):
            Ls = []
            for sgn in (1, -1):
                pp = dict(p)
                pp[name] = p[name] + sgn * h * d
                Ls.append(_loss(pp, adj, 4))
            errs.append(abs((Ls[0] - Ls[1]) / (2 * h) - exact))
        assert errs[0] > 1e-9 * abs(exact), (name, errs)     # the direction is not quadratic
        assert errs[1] < errs[0] / 50 and errs[2] < errs[1] / 50, (name, errs)


def test_gradient_equals_autograd_of_dual_form():
    rng = np.random.default_rng(11)
    T, dk, dv, chunk = 13, 4, 3, 5
    p, adj = _problem(rng, T=T, dk=dk, dv=dv)
    g = _grad(p, adj, chunk)
    t = {n: torch.tensor(x[0, 0], dtype=torch.float64, requires_grad=True) for n, x in p.items()}
    z, W, S = linear_dual_torch(t["q"], t["k"], t["v"], t["theta"], t["W0"], chunk,
                                eta=t["eta"], alpha=t["alpha"], S0=t["S0"])
    L = ((z * torch.tensor(adj["dz"][0, 0])).sum() + (W * torch.tensor(adj["dW"][0, 0])).sum()
         + (S * torch.tensor(adj["dS"][0, 0])).sum())
    L.backward()
    for n, x in t.items():
        ref = x.grad.numpy()
        got = g[GRAD_OF[n]][0, 0]
        assert np.abs(got - ref).max() <= 1e-11 * max(1.0, np.abs(ref).max()), n


def test_gradient_is_linear_in_the_adjoints():
    rng = np.random.default_rng(5)
    p, a1 = _problem(rng, T=6, dk=2, dv=2)
    _, a2 = _problem(rng, T=6, dk=2, dv=2)
    mix = {k: (None if a1[k] is None else 2.0 * a1[k] - 3.0 * a2[k]) for k in a1}
    g1, g2, gm = _grad(p, a1, 4), _grad(p, a2, 4), _grad(p, mix, 4)
    for k in GRAD_OF.values():
        assert np.allclose(gm[k], 2.0 * g1[k] - 3.0 * g2[k], atol=1e-12)


def test_one_token_closed_form():
    """One token from W0, L = dz . z with z = W1 q, W1 = (1-a) W0 + S1,
    S1 = eta S0 - 2 theta (W0 k - v) k^T: every derivative written out."""
    rng = np.random.default_rng(9)
    dk, dv = 3, 2
    k, q = rng.standard_normal(dk), rng.standard_normal(dk)
    v, dz = rng.standard_normal(dv), rng.standard_normal(dv)
    W0, S0 = rng.standard_normal((dv, dk)), rng.standard_normal((dv, dk))
    th, et, al = 0.3, 0.7, 0.2
    e = W0 @ k - v
    S1 = et * S0 - 2 * th * np.outer(e, k)
    W1 = (1 - al) * W0 + S1
    g = oracle.linear_primal_bwd(q[None, None, None], k[None, None, None], v[None, None, None],
                                 np.full((1, 1, 1), th), W0[None, None], 1,
                                 dz[None, None, None], eta=np.full((1, 1, 1), et),
                                 alpha=np.full((1, 1, 1), al), S0=S0[None, None])
    # dz^T W1 q with W1 = (1-al) W0 + et S0 - 2 th e k^T and e = W0 k - v
    assert np.allclose(g["dq"][0, 0, 0], W1.T @ dz, atol=1e-13)
    assert np.isclose(g["dalpha"][0, 0, 0], -dz @ W0 @ q, atol=1e-13)
    assert np.isclose(g["deta"][0, 0, 0], dz @ S0 @ q, atol=1e-13)
    assert np.isclose(g["dtheta"][0, 0, 0], -2 * (dz @ e) * (k @ q), atol=1e-13)
    assert np.allclose(g["dv"][0, 0, 0], 2 * th * (k @ q) * dz, atol=1e-13)
    dk_ref = -2 * th * ((dz @ e) * q + (k @ q) * (W0.T @ dz))
    assert np.allclose(g["dk"][0, 0, 0], dk_ref, atol=1e-13)
    dW0_ref = (1 - al) * np.outer(dz, q) - 2 * th * (k @ q) * np.outer(dz, k)
    assert np.allclose(g["dW0"][0, 0], dW0_ref, atol=1e-13)
    assert np.allclose(g["dS0"][0, 0], et * np.outer(dz, q), atol=1e-13)


def _scalar_grad(theta, w0, k, v, q, dz, eta=None, alpha=None):
    one = lambda x: np.full((1, 1, 1), float(x))
    r = oracle.linear_primal(one(q)[..., None], one(k)[..., None], one(v)[..., None], one(theta),
                             np.full((1, 1, 1, 1), w0), 1)
    g = oracle.linear_primal_bwd(one(q)[..., None], one(k)[..., None], one(v)[..., None],
                                 one(theta), np.full((1, 1, 1, 1), w0), 1,
                                 np.full((1, 1, 1, 1), float(dz)))
    return r, g


def test_p1_outer_gradient_through_the_target(golden):
    g = golden("p1_outer_gradient_target.json")
    for c in g["cases"]:
        r, gr = _scalar_grad(g["theta"], g["W0"], g["k"], c["beta"], g["q"], 1.0)
        assert np.isclose(r["z"][0, 0, 0, 0], c["read"], atol=1e-14)
        assert np.isclose(gr["dv"][0, 0, 0, 0], g["dread_dbeta"], atol=1e-14)


def test_p2_second_order_gradient_of_the_key(golden):
    g = golden("p2_outer_gradient_key.json")
    r, _ = _scalar_grad(g["theta"], g["w0"], g["k"], g["v"], g["q"], 1.0)
    z = r["z"][0, 0, 0, 0]
    assert np.isclose(r["W"][0, 0, 0, 0], g["w1"], atol=1e-14)
    assert np.isclose(z - g["y"], g["outer_residual"], atol=1e-14)
    _, gr = _scalar_grad(g["theta"], g["w0"], g["k"], g["v"], g["q"], z - g["y"])
    # the read's query is a separate input (q = 1), so dL/dk is the page's
    # second-order term alone
    assert np.isclose(gr["dk"][0, 0, 0, 0], g["dL_dk"], atol=1e-14)
    _, g1 = _scalar_grad(g["theta"], g["w0"], g["k"], g["v"], g["q"], 1.0)
    assert np.isclose(g1["dk"][0, 0, 0, 0], g["dw1_dk"], atol=1e-14)


def test_p2_end_to_end_outer_gradients(golden):
    g = golden("p2_end_to_end_scalar.json")
    y = g["outer_target"]
    for c in g["cases"]:
        theta = c["eta_half_loss"] / 2.0
        r, _ = _scalar_grad(theta, c["w0"], 1.0, 2.0, 1.0, 1.0)
        w1 = r["W"][0, 0, 0, 0]
        assert np.isclose(w1, c["w1"], atol=1e-14)
        _, gr = _scalar_grad(theta, c["w0"], 1.0, 2.0, 1.0, w1 - y)
        assert np.isclose(gr["dW0"][0, 0, 0, 0], c["dL_dw0"], atol=1e-14)
        assert np.isclose(gr["dtheta"][0, 0, 0] / 2.0, c["dL_deta_half_loss"], atol=1e-14)
    # the page's closed forms away from its printed case
    for w0, eta_h in ((0.5, 0.3), (-1.0, 0.8)):
        r, _ = _scalar_grad(eta_h / 2.0, w0, 1.0, 2.0, 1.0, 1.0)
        w1 = r["W"][0, 0, 0, 0]
        assert np.isclose(w1, (1 - eta_h) * w0 + 2 * eta_h, atol=1e-14)
        _, gr = _scalar_grad(eta_h / 2.0, w0, 1.0, 2.0, 1.0, w1 - y)
        assert np.isclose(gr["dW0"][0, 0, 0, 0], (w1 - y) * (1 - eta_h), atol=1e-14)
        assert np.isclose(gr["dtheta"][0, 0, 0] / 2.0, (w1 - y) * (2 - w0), atol=1e-14)

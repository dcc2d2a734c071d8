"""Seeded synthetic inputs for the memory scan (shared by tests, smoke and bench).

This module holds none of the scan's arithmetic: it only draws the tensors a
call consumes.  The pages train on text corpora that are not available here;
these draws stand in for the projected views such a model would produce.

Recipe (every workload):
  * a CPU ``torch.Generator`` seeded with ``seed`` (default 1000 + workload id);
  * draw order: q, k, v, then the gate normals (theta, eta, alpha, for those
    gates that are drawn), then the initial memory (W0, or W1 then W2);
  * q, k ~ N(0, 1), L2-normalised per token in float32, then cast to the
    workload dtype; v ~ N(0, 1) cast likewise;
  * theta_t = s * sigmoid(N(0,1)); eta_t = 0.8 + 0.2 * sigmoid(N(0,1));
    alpha_t = 0.05 * sigmoid(N(0,1)); constant gates are full [B,H,T] arrays;
  * initial memory ~ N(0, 0.02^2) unless the workload fixes it to zero.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class Workload:
    id: int
    name: str
    kind: str              # "linear" (TTT-Linear), "titans" (momentum + forgetting), "mlp"
    B: int
    H: int
    T: int
    d: int                 # d_k = d_v (and the MLP's input/output width)
    chunk: int
    dtype: str             # "f32" or "bf16": dtype of q, k, v and z
    theta: tuple           # ("sigmoid", s) or ("const", value)
    eta: tuple = ("zero",)     # ("zero",), ("const", v) or ("titans",)
    alpha: tuple = ("zero",)   # ("zero",), ("const", v) or ("titans",)
    w0: str = "normal"     # "normal" or "zero"
    w0_shared: bool = False
    hidden: int = 0        # MLP hidden width (0 for linear memory)
    notes: str = field(default="", compare=False)

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.T

    def shrink(self, **kw) -> "Workload":
        return replace(self, **kw)


WORKLOADS = {
    1: Workload(1, "ttt-linear tiny B1 H2 T256 d64 b16 f32", "linear", 1, 2, 256, 64, 16, "f32",
                ("const", 0.1)),
    2: Workload(2, "titans linear B2 H8 T4096 d64 b64 bf16", "titans", 2, 8, 4096, 64, 64, "bf16",
                ("sigmoid", 0.1), ("titans",), ("titans",), w0="zero"),
    3: Workload(3, "ttt-linear 125M-layer B8 H12 T8192 d64 b16 bf16", "linear", 8, 12, 8192, 64,
                16, "bf16", ("sigmoid", 0.05), w0_shared=True),
    4: Workload(4, "titans long-context B1 H16 T131072 d128 b64 bf16", "titans", 1, 16, 131072,
                128, 64, "bf16", ("sigmoid", 0.1), ("titans",), ("titans",),
                notes="initial W0 ~ N(0, 0.02^2), S0 = 0"),
    5: Workload(5, "mlp memory B4 H16 T16384 d64 hidden256 b16 bf16", "mlp", 4, 16, 16384, 64,
                16, "bf16", ("sigmoid", 0.02), ("const", 0.9), ("const", 0.01), hidden=256),
}


def _torch_dtype(name: str):
    return {"f32": torch.float32, "bf16": torch.bfloat16}[name]


def _gate(spec, g, shape, default=None):
    kind = spec[0]
    if kind == "zero":
        return default
    if kind == "const":
        return torch.full(shape, float(spec[1]), dtype=torch.float32)
    if kind == "sigmoid":
        return float(spec[1]) * torch.sigmoid(torch.randn(shape, generator=g))
    if kind == "titans-eta":
        return 0.8 + 0.2 * torch.sigmoid(torch.randn(shape, generator=g))
    if kind == "titans-alpha":
        return 0.05 * torch.sigmoid(torch.randn(shape, generator=g))
    raise ValueError(spec)


def generate(w: Workload, seed: int | None = None) -> dict:
    """CPU tensors for one call: q, k, v (w.dtype), theta/eta/alpha (f32 or None),
    W0 [B|1,H,d,d] (linear) or W1_0 [B,H,hidden,d], W2_0 [B,H,d,hidden] (mlp)."""
    g = torch.Generator().manual_seed(1000 + w.id if seed is None else seed)
    B, H, T, d = w.B, w.H, w.T, w.d
    dt = _torch_dtype(w.dtype)
    q = torch.randn((B, H, T, d), generator=g)
    k = torch.randn((B, H, T, d), generator=g)
    v = torch.randn((B, H, T, d), generator=g)
    q = q / q.norm(dim=-1, keepdim=True)
    k = k / k.norm(dim=-1, keepdim=True)
    out = {"q": q.to(dt).contiguous(), "k": k.to(dt).contiguous(), "v": v.to(dt).contiguous()}
    del q, k, v
    shape = (B, H, T)
    out["theta"] = _gate(w.theta, g, shape)
    eta_spec = ("titans-eta",) if w.eta[0] == "titans" else w.eta
    alpha_spec = ("titans-alpha",) if w.alpha[0] == "titans" else w.alpha
    out["eta"] = _gate(eta_spec, g, shape)
    out["alpha"] = _gate(alpha_spec, g, shape)
    nb = 1 if w.w0_shared else B
    if w.kind == "mlp":
        hs = (nb, H, w.hidden, d)
        out["W1_0"] = 0.02 * torch.randn(hs, generator=g)
        out["W2_0"] = 0.02 * torch.randn((nb, H, d, w.hidden), generator=g)
    elif w.w0 == "zero":
        out["W0"] = torch.zeros((nb, H, d, d))
    else:
        out["W0"] = 0.02 * torch.randn((nb, H, d, d), generator=g)
    return out


def generate_custom(kind="titans", B=1, H=2, T=100, d=64, chunk=16, dtype="f32", hidden=0,
                    theta=("sigmoid", 0.1), eta=None, alpha=None, w0="normal",
                    w0_shared=False, seed=0):
    """Inputs for a shrunk or edge-case variant; gates default to the workload kind's."""
    if eta is None:
        eta = ("titans",) if kind == "titans" else (("const", 0.9) if kind == "mlp" else ("zero",))
    if alpha is None:
        alpha = ("titans",) if kind == "titans" else (("const", 0.01) if kind == "mlp" else ("zero",))
    w = Workload(0, "custom", kind, B, H, T, d, chunk, dtype, theta, eta, alpha, w0, w0_shared,
                 hidden)
    return w, generate(w, seed=seed)


def generate_adjoints(B, H, T, dk, dv, dtype="f32", seed=0, with_S=True) -> dict:
    """Seeded adjoints of a scan's outputs for gradient checks: dz ~ N(0, 1) in
    the workload dtype ([B,H,T,dv]), dW and dS ~ N(0, 1) fp32 ([B,H,dv,dk]; dS
    None unless with_S).  Drawn in that order from a CPU generator."""
    g = torch.Generator().manual_seed(seed)
    dz = torch.randn((B, H, T, dv), generator=g).to(_torch_dtype(dtype))
    dW = torch.randn((B, H, dv, dk), generator=g)
    dS = torch.randn((B, H, dv, dk), generator=g) if with_S else None
    return dict(dz=dz, dW=dW, dS=dS)


def generate_dgd_gates(B, H, T, seed=0) -> dict:
    """Seeded gates of the DGD memory: step eta_t = 0.1 sigmoid(N(0,1)) and
    retention alpha_t = 0.9 + 0.1 sigmoid(N(0,1)), [B,H,T] fp32, drawn in that
    order from a CPU generator.  With L2-normalised keys the factor
    (alpha I - eta k k^T) then stays a contraction."""
    g = torch.Generator().manual_seed(seed)
    eta = 0.1 * torch.sigmoid(torch.randn((B, H, T), generator=g))
    alpha = 0.9 + 0.1 * torch.sigmoid(torch.randn((B, H, T), generator=g))
    return dict(eta=eta, alpha=alpha)


def generate_chunk_gates(B, H, nch, theta_scale=0.1, seed=0) -> dict:
    """Seeded chunk-level gates with the Titans recipe, one value per (sequence,
    chunk): theta = s sigmoid(N(0,1)), eta = 0.8 + 0.2 sigmoid(N(0,1)),
    alpha = 0.05 sigmoid(N(0,1)), [B,H,nch] fp32, drawn in that order."""
    g = torch.Generator().manual_seed(seed)
    theta = theta_scale * torch.sigmoid(torch.randn((B, H, nch), generator=g))
    eta = 0.8 + 0.2 * torch.sigmoid(torch.randn((B, H, nch), generator=g))
    alpha = 0.05 * torch.sigmoid(torch.randn((B, H, nch), generator=g))
    return dict(theta=theta, eta=eta, alpha=alpha)


def generate_lmm(B, T, H, d, conv_k=4, seed=0) -> dict:
    """Seeded input and random-init parameters of the LMM layer, drawn in this
    order from a CPU generator: x ~ N(0,1) [B,T,D] bf16; W_in ~ N(0, 0.05^2)
    [D, 4D+3H] bf16; conv_w ~ N(0,1)/conv_k [3,D,conv_k]; rms_w = 1 + 0.1 N(0,1)
    [d]; W_o ~ N(0, 0.05^2) [D,D] bf16; W0 ~ N(0, 0.02^2) [1,H,d,d] (shared)."""
    g = torch.Generator().manual_seed(seed)
    D = H * d
    x = torch.randn((B, T, D), generator=g).to(torch.bfloat16)
    W_in = (0.05 * torch.randn((D, 4 * D + 3 * H), generator=g)).to(torch.bfloat16)
    conv_w = torch.randn((3, D, conv_k), generator=g) / conv_k
    rms_w = 1.0 + 0.1 * torch.randn((d,), generator=g)
    W_o = (0.05 * torch.randn((D, D), generator=g)).to(torch.bfloat16)
    W0 = 0.02 * torch.randn((1, H, d, d), generator=g)
    return dict(x=x, W_in=W_in, conv_w=conv_w, rms_w=rms_w, W_o=W_o, W0=W0)

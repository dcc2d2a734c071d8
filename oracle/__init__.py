"""Float64 CPU oracle for the chunked test-time-training memory scan.

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's
CPU-baseline leg are the only callers.  The GPU library never imports this
package and this package never imports the GPU library: the two share no code.

``ttm_oracle.c`` holds the token-by-token recurrence (see its header for the
passages it follows).  This module compiles it with the system C compiler on
first use and wraps it with ctypes; ``dual.py`` holds an independent
matrix-form restatement used only to cross-check the token loop.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ttm_oracle.c")
_LIB = os.path.join(_HERE, "_build", "libttm_oracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile the C oracle (plain -O2, no target-specific flags)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            os.makedirs(os.path.dirname(_LIB), exist_ok=True)
            tmp = _LIB + f".{os.getpid()}.tmp"
            subprocess.run(["gcc", "-O2", "-std=c11", "-D_GNU_SOURCE", "-fPIC", "-shared",
                            _SRC, "-o", tmp, "-lm", "-lpthread"], check=True)
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i, d = ctypes.c_int, _dp
        lib.oracle_linear_primal.argtypes = [i, i, i, i, i, i, d, d, d, d, d, d, d, d, i,
                                             d, d, d, i]
        lib.oracle_linear_primal.restype = i
        lib.oracle_linear_primal_bwd.argtypes = [i, i, i, i, i, i, d, d, d, d, d, d, d, d, i,
                                                 d, d, d, d, d, d, d, d, d, d, d, i]
        lib.oracle_linear_primal_bwd.restype = i
        lib.oracle_dgd_primal.argtypes = [i, i, i, i, i, i, d, d, d, d, d, d, i, d, d, i]
        lib.oracle_dgd_primal.restype = i
        lib.oracle_mlp_primal.argtypes = [i, i, i, i, i, i, d, d, d, d, d, d, d, d, d, d, i,
                                          d, d, d, d, d, i]
        lib.oracle_mlp_primal.restype = i
        lib.oracle_mlp_grad.argtypes = [i, i, d, d, d, d, d, d]
        lib.oracle_mlp_grad.restype = None
        lib.oracle_mlp_loss.argtypes = [i, i, d, d, d, d]
        lib.oracle_mlp_loss.restype = ctypes.c_double
        lib.oracle_gelu.argtypes = [ctypes.c_double]
        lib.oracle_gelu.restype = ctypes.c_double
        lib.oracle_gelu_grad.argtypes = [ctypes.c_double]
        lib.oracle_gelu_grad.restype = ctypes.c_double
        _lib = lib
    return _lib


def _f64(x, shape=None):
    if x is None:
        return None
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    if shape is not None:
        a = a.reshape(shape)
    return a


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


class Result(dict):
    """Outputs of one oracle run plus the number of threads it used."""


def linear_primal(q, k, v, theta, W0, chunk, eta=None, alpha=None, S0=None,
                  shared_over_batch=False, threads=0) -> Result:
    """Token-by-token linear / Titans memory scan in float64.

    q, k: [B,H,T,dk]; v: [B,H,T,dv]; theta/eta/alpha: [B,H,T] (eta, alpha None = 0);
    W0 (and S0): [B,H,dv,dk] or [1,H,dv,dk] when shared_over_batch.
    Returns z [B,H,T,dv], W [B,H,dv,dk], S [B,H,dv,dk] and the thread count.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    theta = _f64(theta, (B, H, T))
    eta = _f64(eta, (B, H, T)) if eta is not None else None
    alpha = _f64(alpha, (B, H, T)) if alpha is not None else None
    nb = 1 if shared_over_batch else B
    W0 = _f64(W0, (nb, H, dv, dk))
    S0 = _f64(S0, (nb, H, dv, dk)) if S0 is not None else None
    z = np.zeros((B, H, T, dv))
    W = np.zeros((B, H, dv, dk))
    S = np.zeros((B, H, dv, dk))
    used = _load().oracle_linear_primal(B, H, T, dk, dv, int(chunk), _ptr(q), _ptr(k), _ptr(v),
                                        _ptr(eta), _ptr(theta), _ptr(alpha), _ptr(W0), _ptr(S0),
                                        int(bool(shared_over_batch)), _ptr(z), _ptr(W), _ptr(S),
                                        int(threads))
    if used < 0:
        raise ValueError("oracle_linear_primal rejected its arguments")
    return Result(z=z, W=W, S=S, threads=used)


def linear_primal_bwd(q, k, v, theta, W0, chunk, dz, eta=None, alpha=None, S0=None, dW=None,
                      dS=None, shared_over_batch=False, threads=0) -> Result:
    """Gradient of the linear / Titans memory scan in float64, by reverse mode
    through the token loop of `linear_primal`.

    For the outer loss L with dL/dz = dz [B,H,T,dv], dL/dW_T = dW and
    dL/dS_T = dS ([B,H,dv,dk] or None = 0), returns dq, dk [B,H,T,dk],
    dv [B,H,T,dv], dtheta [B,H,T], deta / dalpha [B,H,T] (None when the gate
    is None), dW0 / dS0 shaped like W0 (summed over the batch when W0 is
    shared) and the thread count.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    theta = _f64(theta, (B, H, T))
    eta = _f64(eta, (B, H, T)) if eta is not None else None
    alpha = _f64(alpha, (B, H, T)) if alpha is not None else None
    nb = 1 if shared_over_batch else B
    W0 = _f64(W0, (nb, H, dv, dk))
    S0 = _f64(S0, (nb, H, dv, dk)) if S0 is not None else None
    dz = _f64(dz, (B, H, T, dv))
    dW = _f64(dW, (B, H, dv, dk)) if dW is not None else None
    dS = _f64(dS, (B, H, dv, dk)) if dS is not None else None
    out = dict(dq=np.zeros((B, H, T, dk)), dk=np.zeros((B, H, T, dk)),
               dv=np.zeros((B, H, T, dv)), dtheta=np.zeros((B, H, T)),
               deta=np.zeros((B, H, T)) if eta is not None else None,
               dalpha=np.zeros((B, H, T)) if alpha is not None else None,
               dW0=np.zeros((B, H, dv, dk)), dS0=np.zeros((B, H, dv, dk)))
    o = out
    used = _load().oracle_linear_primal_bwd(
        B, H, T, dk, dv, int(chunk), _ptr(q), _ptr(k), _ptr(v), _ptr(eta), _ptr(theta),
        _ptr(alpha), _ptr(W0), _ptr(S0), int(bool(shared_over_batch)), _ptr(dz), _ptr(dW),
        _ptr(dS), _ptr(o["dq"]), _ptr(o["dk"]), _ptr(o["dv"]), _ptr(o["deta"]),
        _ptr(o["dtheta"]), _ptr(o["dalpha"]), _ptr(o["dW0"]), _ptr(o["dS0"]), int(threads))
    if used < 0:
        raise ValueError("oracle_linear_primal_bwd rejected its arguments")
    if shared_over_batch:
        o["dW0"] = o["dW0"].sum(axis=0, keepdims=True)
        o["dS0"] = o["dS0"].sum(axis=0, keepdims=True)
    return Result(**o, threads=used)


def dgd_primal(q, k, v, eta, alpha, W0, chunk, shared_over_batch=False, threads=0) -> Result:
    """DGD memory scan in float64: M_t = M_{t-1}(alpha_t I - eta_t k k^T)
    - eta_t (Mc k - v) k^T, read z_t = M_{t-1} q_t before the token's write
    ("Nested Learning" eq (86); see ttm_oracle.c).
    q, k: [B,H,T,dk]; v: [B,H,T,dv]; eta (step), alpha (retention): [B,H,T];
    W0: [B|1,H,dv,dk].  Returns z, W and the thread count."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    eta = _f64(eta, (B, H, T))
    alpha = _f64(alpha, (B, H, T))
    W0 = _f64(W0, (1 if shared_over_batch else B, H, dv, dk))
    z = np.zeros((B, H, T, dv))
    W = np.zeros((B, H, dv, dk))
    used = _load().oracle_dgd_primal(B, H, T, dk, dv, int(chunk), _ptr(q), _ptr(k), _ptr(v),
                                     _ptr(eta), _ptr(alpha), _ptr(W0),
                                     int(bool(shared_over_batch)), _ptr(z), _ptr(W), int(threads))
    if used < 0:
        raise ValueError("oracle_dgd_primal rejected its arguments")
    return Result(z=z, W=W, threads=used)


def mlp_primal(q, k, v, theta, W1_0, W2_0, chunk, eta=None, alpha=None, S1_0=None, S2_0=None,
               shared_over_batch=False, threads=0) -> Result:
    """Token-by-token deep-memory scan, f(x) = W2 GELU(W1 x), in float64.

    q, k, v: [B,H,T,d]; W1_0: [B|1,H,hidden,d]; W2_0: [B|1,H,d,hidden].
    Returns z, W1, W2, S1, S2 and the thread count.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, d = q.shape
    nb = 1 if shared_over_batch else B
    W1_0 = _f64(W1_0)
    hidden = W1_0.shape[-2]
    W1_0 = W1_0.reshape(nb, H, hidden, d)
    W2_0 = _f64(W2_0, (nb, H, d, hidden))
    S1_0 = _f64(S1_0, (nb, H, hidden, d)) if S1_0 is not None else None
    S2_0 = _f64(S2_0, (nb, H, d, hidden)) if S2_0 is not None else None
    theta = _f64(theta, (B, H, T))
    eta = _f64(eta, (B, H, T)) if eta is not None else None
    alpha = _f64(alpha, (B, H, T)) if alpha is not None else None
    z = np.zeros((B, H, T, d))
    W1 = np.zeros((B, H, hidden, d))
    W2 = np.zeros((B, H, d, hidden))
    S1 = np.zeros((B, H, hidden, d))
    S2 = np.zeros((B, H, d, hidden))
    used = _load().oracle_mlp_primal(B, H, T, d, hidden, int(chunk), _ptr(q), _ptr(k), _ptr(v),
                                     _ptr(eta), _ptr(theta), _ptr(alpha), _ptr(W1_0), _ptr(W2_0),
                                     _ptr(S1_0), _ptr(S2_0), int(bool(shared_over_batch)),
                                     _ptr(z), _ptr(W1), _ptr(W2), _ptr(S1), _ptr(S2), int(threads))
    if used < 0:
        raise ValueError("oracle_mlp_primal rejected its arguments")
    return Result(z=z, W1=W1, W2=W2, S1=S1, S2=S2, threads=used)


def mlp_grad(W1, W2, k, v):
    """(dl/dW1, dl/dW2) of l = ||W2 GELU(W1 k) - v||^2 for one token."""
    W1, W2, k, v = _f64(W1), _f64(W2), _f64(k), _f64(v)
    hidden, d = W1.shape
    g1 = np.zeros_like(W1)
    g2 = np.zeros_like(W2)
    _load().oracle_mlp_grad(d, hidden, _ptr(W1), _ptr(W2), _ptr(k), _ptr(v), _ptr(g1), _ptr(g2))
    return g1, g2


def mlp_loss(W1, W2, k, v) -> float:
    W1, W2, k, v = _f64(W1), _f64(W2), _f64(k), _f64(v)
    hidden, d = W1.shape
    return _load().oracle_mlp_loss(d, hidden, _ptr(W1), _ptr(W2), _ptr(k), _ptr(v))


def gelu(x: float) -> float:
    return _load().oracle_gelu(float(x))


def gelu_grad(x: float) -> float:
    return _load().oracle_gelu_grad(float(x))

"""Thin Python binding of libttm.so, the GB300 chunked test-time-training memory scan.

Argument marshalling only: every step of the scan runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (PyTorch supplies device memory and
streams); outputs are allocated here when not given.  There is no CPU
fallback: if the library is missing the calls raise.

    z, W = linear_fwd(q, k, v, theta, W0, chunk)
    z, W, S = titans_fwd(q, k, v, theta, W0, chunk, eta=eta, alpha=alpha)
    z, W1, W2, S1, S2 = mlp_fwd(q, k, v, theta, W1_0, W2_0, chunk, eta=eta, alpha=alpha)
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import re

from ._build import LIB, ROOT, build  # noqa: F401  (build is part of the public surface)

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT = range(5)
F32, BF16 = 0, 1
POLICY = {"auto": 0, "simt": 1, "tc": 2}
KERNEL_NAMES = {0: "none", 1: "linear_simt", 2: "mlp_simt", 3: "linear_tc", 4: "mlp_tc",
                5: "linear_seq", 6: "dgd_step", 7: "dgd_tc", 8: "bwd_simt", 9: "bwd_tc"}

_lib = None


class TTMError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_str(code)} (status {code})")


def lib() -> ctypes.CDLL:
    """The loaded libttm.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is missing; build it with "
                               "`python -m test_neural_memory_gb300._build`")
        L = ctypes.CDLL(LIB)
        i, p = ctypes.c_int, ctypes.c_void_p
        sz = ctypes.c_size_t
        L.ttm_linear_fwd.argtypes = [i] * 7 + [p] * 6 + [p, i, p, p, p, sz, p]
        L.ttm_titans_fwd.argtypes = [i] * 7 + [p] * 6 + [p, p, i, p, p, p, p, sz, p]
        L.ttm_linear_workspace_size.argtypes = [i] * 7
        L.ttm_linear_workspace_size.restype = sz
        L.ttm_mlp_fwd.argtypes = [i] * 7 + [p] * 6 + [p] * 4 + [i] + [p] * 5 + [p]
        L.ttm_mlp_gelu.argtypes = [p, p, p, i, p]
        L.ttm_titans_step.argtypes = [i] * 8 + [p] * 6 + [p] * 4 + [p]
        L.ttm_linear_step.argtypes = [i] * 8 + [p] * 4 + [p] * 3 + [p]
        L.ttm_dgd_fwd.argtypes = [i] * 7 + [p] * 5 + [p, i, p, p, p, sz, p]
        L.ttm_dgd_workspace_size.argtypes = [i] * 7
        L.ttm_dgd_workspace_size.restype = sz
        L.ttm_lmm_layer_workspace_size.argtypes = [i] * 6
        L.ttm_lmm_layer_workspace_size.restype = sz
        L.ttm_lmm_layer_fwd.argtypes = ([i] * 6 + [p] * 5 + [ctypes.c_float, p, i, p, p, p, p, sz,
                                                              p])
        L.ttm_titans_fwd_chunk_gates.argtypes = [i] * 7 + [p] * 6 + [p, p, i, p, p, p, p, sz, p]
        L.ttm_titans_fwd_host_workspace_size.argtypes = [i] * 8
        L.ttm_titans_fwd_host_workspace_size.restype = sz
        L.ttm_titans_fwd_host.argtypes = [i] * 7 + [p] * 6 + [p, p, i, p, p, p, i, p, sz, p]
        L.ttm_dgd_step.argtypes = [i] * 8 + [p] * 5 + [p, p, p, p]
        L.ttm_titans_bwd_workspace_size.argtypes = [i] * 8
        L.ttm_titans_bwd_workspace_size.restype = sz
        L.ttm_titans_bwd.argtypes = ([i] * 7 + [p] * 6 + [p, p, i] + [p] * 3 + [p] * 3 +
                                     [p] * 5 + [p, sz, p])
        L.ttm_linear_bwd.argtypes = [i] * 7 + [p] * 4 + [p, i] + [p] * 7 + [p, sz, p]
        L.ttm_mlp_gelu.restype = i
        for f in (L.ttm_linear_fwd, L.ttm_titans_fwd, L.ttm_mlp_fwd):
            f.restype = i
        L.ttm_status_str.argtypes = [i]
        L.ttm_status_str.restype = ctypes.c_char_p
        L.ttm_set_kernel_policy.argtypes = [i]
        L.ttm_set_kernel_policy.restype = i
        L.ttm_last_kernel.restype = i
        L.ttm_device_status.restype = i
        L.ttm_cuda_device_count.restype = i
        L.ttm_debug_set.argtypes = [i, ctypes.c_longlong]
        L.ttm_debug_set.restype = i
        L.ttm_launch_count.restype = ctypes.c_ulonglong
        _lib = L
    return _lib


def declared_symbols() -> list[str]:
    """Function names declared in include/ttm.h (the ABI this binding wraps)."""
    with open(os.path.join(ROOT, "include", "ttm.h")) as f:
        text = f.read()
    return re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(ttm_\w+)\s*\(", text, flags=re.M)


def status_str(code: int) -> str:
    return lib().ttm_status_str(int(code)).decode()


def set_kernel_policy(policy: str) -> str:
    old = lib().ttm_set_kernel_policy(POLICY[policy])
    return {v: k for k, v in POLICY.items()}[old]


@contextlib.contextmanager
def kernel_policy(policy: str):
    old = set_kernel_policy(policy)
    try:
        yield
    finally:
        set_kernel_policy(old)


def last_kernel() -> str:
    return KERNEL_NAMES.get(lib().ttm_last_kernel(), "unknown")


def launch_count() -> int:
    """Kernels enqueued by this process through the library so far."""
    return int(lib().ttm_launch_count())


def device_status() -> int:
    return lib().ttm_device_status()


DEBUG = {"wait_cycles": 1, "stall_chunk": 2, "fail_calls": 3}


def debug_set(option: str, value: int) -> None:
    """Failure-detection test hooks of the library (see ttm_debug_set)."""
    _check(lib().ttm_debug_set(DEBUG[option], int(value)), "ttm_debug_set")


def cuda_device_count() -> int:
    """CUDA devices the library's own runtime can reach (0 without a GPU)."""
    return int(lib().ttm_cuda_device_count())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return F32
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"q/k/v must be float32 or bfloat16, got {t.dtype}")


def _stream(t, stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code: int, what: str):
    if code != OK:
        raise TTMError(code, what)


def linear_workspace_size(B, H, T, dk, dv, chunk, dtype_code) -> int:
    """Workspace bytes the linear / Titans scan needs under the current policy."""
    return int(lib().ttm_linear_workspace_size(B, H, T, dk, dv, int(chunk), dtype_code))


def alloc_workspace(q, v, chunk):
    """A device workspace (uint8 tensor) sized for this call, or None."""
    import torch
    B, H, T, dk = q.shape
    n = linear_workspace_size(B, H, T, dk, v.shape[-1], chunk, _dtype_code(q))
    return torch.empty(n, dtype=torch.uint8, device=q.device) if n else None


def _ws(workspace):
    if workspace is None:
        return None, 0
    return _ptr(workspace), workspace.numel() * workspace.element_size()


def linear_fwd(q, k, v, theta, W0, chunk, *, w0_shared=False, z=None, W_out=None,
               workspace=None, stream=None):
    """TTT-Linear scan.  q, k: [B,H,T,dk]; v: [B,H,T,dv]; theta: [B,H,T] fp32;
    W0: [B|1,H,dv,dk] fp32.  Returns (z, W_out)."""
    import torch
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    z = torch.empty_like(v) if z is None else z
    W_out = torch.empty((B, H, dv, dk), dtype=torch.float32, device=q.device) if W_out is None else W_out
    if workspace is None:
        workspace = alloc_workspace(q, v, chunk)
    wp, wb = _ws(workspace)
    _check(lib().ttm_linear_fwd(B, H, T, dk, dv, int(chunk), _dtype_code(q), _ptr(q), _ptr(k),
                                _ptr(v), None, _ptr(theta), None, _ptr(W0), int(bool(w0_shared)),
                                _ptr(z), _ptr(W_out), wp, wb, _stream(q, stream)),
           "ttm_linear_fwd")
    return z, W_out


def titans_fwd(q, k, v, theta, W0, chunk, *, eta=None, alpha=None, S0=None, w0_shared=False,
               z=None, W_out=None, S_out=None, want_S=True, workspace=None, stream=None):
    """Titans linear-memory scan with momentum (eta) and forgetting (alpha).
    Returns (z, W_out, S_out); S_out is None when want_S is False."""
    import torch
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    z = torch.empty_like(v) if z is None else z
    shape = (B, H, dv, dk)
    W_out = torch.empty(shape, dtype=torch.float32, device=q.device) if W_out is None else W_out
    if S_out is None and want_S:
        S_out = torch.empty(shape, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(q, v, chunk)
    wp, wb = _ws(workspace)
    _check(lib().ttm_titans_fwd(B, H, T, dk, dv, int(chunk), _dtype_code(q), _ptr(q), _ptr(k),
                                _ptr(v), _ptr(eta), _ptr(theta), _ptr(alpha), _ptr(W0), _ptr(S0),
                                int(bool(w0_shared)), _ptr(z), _ptr(W_out), _ptr(S_out), wp, wb,
                                _stream(q, stream)), "ttm_titans_fwd")
    return z, W_out, S_out


def titans_fwd_host_workspace_size(B, H, T, dk, dv, chunk, dtype, seg_tokens) -> int:
    """Device bytes ttm_titans_fwd_host needs (0 for rejected arguments)."""
    code = BF16 if dtype in ("bf16", BF16) else F32
    return int(lib().ttm_titans_fwd_host_workspace_size(B, H, T, dk, dv, int(chunk), code,
                                                        int(seg_tokens)))


def titans_fwd_host(q, k, v, theta, W0, chunk, *, eta=None, alpha=None, S0=None,
                    w0_shared=False, z=None, W_out=None, S_out=None, want_S=True,
                    seg_tokens=8192, workspace=None, device=None, stream=None):
    """ttm_titans_fwd_host: q, k, v, gates, W0, S0 and the outputs are CPU tensors
    (page-locked for full copy bandwidth); the sequence is streamed through
    `device` in segments of `seg_tokens` tokens.  The outputs are complete once
    `stream` (default: the device's current stream) has been synchronised.
    Returns (z, W_out, S_out)."""
    import torch
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    pin = lambda shape, dt: torch.empty(shape, dtype=dt, pin_memory=True)
    z = pin(v.shape, v.dtype) if z is None else z
    shape = (B, H, dv, dk)
    W_out = pin(shape, torch.float32) if W_out is None else W_out
    if S_out is None and want_S:
        S_out = pin(shape, torch.float32)
    need = titans_fwd_host_workspace_size(B, H, T, dk, dv, chunk, _dtype_code(q), seg_tokens)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    s = torch.cuda.current_stream(dev) if stream is None else stream
    _check(lib().ttm_titans_fwd_host(B, H, T, dk, dv, int(chunk), _dtype_code(q), _ptr(q),
                                     _ptr(k), _ptr(v), _ptr(eta), _ptr(theta), _ptr(alpha),
                                     _ptr(W0), _ptr(S0), int(bool(w0_shared)), _ptr(z),
                                     _ptr(W_out), _ptr(S_out), int(seg_tokens),
                                     ctypes.c_void_p(workspace.data_ptr()),
                                     workspace.numel() * workspace.element_size(),
                                     ctypes.c_void_p(s.cuda_stream)), "ttm_titans_fwd_host")
    return z, W_out, S_out


def titans_fwd_chunk_gates(q, k, v, theta, W0, chunk, *, eta=None, alpha=None, S0=None,
                           w0_shared=False, z=None, W_out=None, S_out=None, workspace=None,
                           stream=None):
    """Titans scan with one gate value per (sequence, chunk): theta / eta / alpha are
    [B,H,ceil(T/chunk)] fp32.  Returns (z, W_out, S_out)."""
    import torch
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    z = torch.empty_like(v) if z is None else z
    shape = (B, H, dv, dk)
    W_out = torch.empty(shape, dtype=torch.float32, device=q.device) if W_out is None else W_out
    S_out = torch.empty(shape, dtype=torch.float32, device=q.device) if S_out is None else S_out
    if workspace is None:
        workspace = alloc_workspace(q, v, chunk)
    wp, wb = _ws(workspace)
    _check(lib().ttm_titans_fwd_chunk_gates(B, H, T, dk, dv, int(chunk), _dtype_code(q), _ptr(q),
                                            _ptr(k), _ptr(v), _ptr(eta), _ptr(theta), _ptr(alpha),
                                            _ptr(W0), _ptr(S0), int(bool(w0_shared)), _ptr(z),
                                            _ptr(W_out), _ptr(S_out), wp, wb, _stream(q, stream)),
           "ttm_titans_fwd_chunk_gates")
    return z, W_out, S_out


def titans_step(q, k, v, theta, W, chunk, pos, *, eta=None, alpha=None, S=None, Wc=None,
                z=None, stream=None):
    """Decode step: continues every sequence by n tokens (q, k: [B,H,n,dk]; v: [B,H,n,dv];
    gates [B,H,n]) from the state W (and momentum S) at position `pos` of the current
    chunk.  W, S, Wc ([B,H,dv,dk] fp32) are updated in place; Wc is allocated when None
    (allowed only at pos == 0).  Returns (z, Wc, new_pos)."""
    import torch
    B, H, n, dk = q.shape
    dv = v.shape[-1]
    z = torch.empty_like(v) if z is None else z
    if Wc is None:
        if pos != 0:
            raise TTMError(ERR_INVALID_ARG, "titans_step (Wc is required in mid-chunk)")
        Wc = torch.empty_like(W)
    _check(lib().ttm_titans_step(B, H, n, dk, dv, int(chunk), int(pos), _dtype_code(q), _ptr(q),
                                 _ptr(k), _ptr(v), _ptr(eta), _ptr(theta), _ptr(alpha), _ptr(W),
                                 _ptr(S), _ptr(Wc), _ptr(z), _stream(q, stream)),
           "ttm_titans_step")
    return z, Wc, (pos + n) % chunk


def dgd_workspace_size(B, H, T, dk, dv, chunk, dtype_code) -> int:
    """Workspace bytes the DGD scan needs under the current policy."""
    return int(lib().ttm_dgd_workspace_size(B, H, T, dk, dv, int(chunk), dtype_code))


def dgd_fwd(q, k, v, eta, alpha, W0, chunk, *, w0_shared=False, z=None, W_out=None,
            workspace=None, stream=None):
    """DGD memory scan ("Nested Learning" eqs (88), (93)): eta is the step and alpha the
    retention factor ([B,H,T] fp32).  W0: [B|1,H,dv,dk] fp32.  The workspace the
    tensor-core path needs is allocated here unless given.  Returns (z, W_out)."""
    import torch
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    z = torch.empty_like(v) if z is None else z
    W_out = (torch.empty((B, H, dv, dk), dtype=torch.float32, device=q.device)
             if W_out is None else W_out)
    if workspace is None:
        n = dgd_workspace_size(B, H, T, dk, dv, chunk, _dtype_code(q))
        workspace = torch.empty(n, dtype=torch.uint8, device=q.device) if n else None
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(lib().ttm_dgd_fwd(B, H, T, dk, dv, int(chunk), _dtype_code(q), _ptr(q), _ptr(k),
                             _ptr(v), _ptr(eta), _ptr(alpha), _ptr(W0), int(bool(w0_shared)),
                             _ptr(z), _ptr(W_out), _ptr(workspace), wsb, _stream(q, stream)),
           "ttm_dgd_fwd")
    return z, W_out


def dgd_step(q, k, v, eta, alpha, W, chunk, pos, *, Wc=None, z=None, stream=None):
    """DGD decode step: as titans_step, with the DGD update.  Returns (z, Wc, new_pos)."""
    import torch
    B, H, n, dk = q.shape
    dv = v.shape[-1]
    z = torch.empty_like(v) if z is None else z
    if Wc is None:
        if pos != 0:
            raise TTMError(ERR_INVALID_ARG, "dgd_step (Wc is required in mid-chunk)")
        Wc = torch.empty_like(W)
    _check(lib().ttm_dgd_step(B, H, n, dk, dv, int(chunk), int(pos), _dtype_code(q), _ptr(q),
                              _ptr(k), _ptr(v), _ptr(eta), _ptr(alpha), _ptr(W), _ptr(Wc),
                              _ptr(z), _stream(q, stream)), "ttm_dgd_step")
    return z, Wc, (pos + n) % chunk


def lmm_layer_fwd(x, W_in, conv_w, rms_w, W_o, theta_scale, W0, chunk, *, w0_shared=True,
                  y=None, W_out=None, S_out=None, workspace=None, stream=None):
    """LMM layer (memory as a standalone sequence layer): x [B,T,H*d] bf16 -> y; see
    ttm_lmm_layer_fwd for the wiring.  H is read from W0 ([1|B,H,d,d]).  Returns
    (y, W_out, S_out)."""
    import torch
    B, T, D = x.shape
    H, d = W0.shape[1], W0.shape[-1]
    conv_k = conv_w.shape[-1]
    y = torch.empty_like(x) if y is None else y
    shape = (B, H, d, d)
    W_out = torch.empty(shape, dtype=torch.float32, device=x.device) if W_out is None else W_out
    S_out = torch.empty(shape, dtype=torch.float32, device=x.device) if S_out is None else S_out
    if workspace is None:
        n = int(lib().ttm_lmm_layer_workspace_size(B, T, H, d, int(chunk), int(bool(w0_shared))))
        if n == 0:
            raise TTMError(ERR_UNSUPPORTED, "ttm_lmm_layer_workspace_size")
        workspace = torch.empty(n, dtype=torch.uint8, device=x.device)
    wp, wb = _ws(workspace)
    _check(lib().ttm_lmm_layer_fwd(B, T, H, d, int(chunk), conv_k, _ptr(x), _ptr(W_in),
                                   _ptr(conv_w), _ptr(rms_w), _ptr(W_o), float(theta_scale),
                                   _ptr(W0), int(bool(w0_shared)), _ptr(y), _ptr(W_out),
                                   _ptr(S_out), wp, wb, _stream(x, stream)), "ttm_lmm_layer_fwd")
    return y, W_out, S_out


def titans_bwd(q, k, v, theta, W0, chunk, dz, *, eta=None, alpha=None, S0=None, dW=None,
               dS=None, w0_shared=False, want_gates=True, want_dS0=True, workspace=None,
               out=None, stream=None):
    """Gradient of the Titans (or, with eta = alpha = None, TTT-Linear) scan for the
    adjoints dz ([B,H,T,dv], dtype of v), dW / dS ([B,H,dv,dk] fp32 or None).
    Returns a dict with dq, dk, dv (dtype of q), dtheta, deta, dalpha ([B,H,T] fp32;
    deta / dalpha None when the gate is None or want_gates is False), dW0, dS0 (shaped
    like W0; dS0 None when want_dS0 is False).  `out` may hold preallocated tensors for
    any of these keys."""
    import torch
    B, H, T, dk = q.shape
    dv = v.shape[-1]
    dev = q.device
    f32 = lambda shape: torch.empty(shape, dtype=torch.float32, device=dev)
    out = out or {}
    pick = lambda key, make: out[key] if out.get(key) is not None else make()
    has_eta, has_alpha = eta is not None and want_gates, alpha is not None and want_gates
    g = dict(dq=pick("dq", lambda: torch.empty_like(q)),
             dk=pick("dk", lambda: torch.empty_like(k)),
             dv=pick("dv", lambda: torch.empty_like(v)),
             dtheta=pick("dtheta", lambda: f32((B, H, T))),
             deta=pick("deta", lambda: f32((B, H, T))) if has_eta else None,
             dalpha=pick("dalpha", lambda: f32((B, H, T))) if has_alpha else None,
             dW0=pick("dW0", lambda: f32(tuple(W0.shape))),
             dS0=pick("dS0", lambda: f32(tuple(W0.shape))) if want_dS0 else None)
    if workspace is None:
        n = int(lib().ttm_titans_bwd_workspace_size(B, H, T, dk, dv, int(chunk), _dtype_code(q),
                                                    int(bool(w0_shared))))
        if n == 0 and T > 0:
            raise TTMError(ERR_UNSUPPORTED, "ttm_titans_bwd_workspace_size")
        workspace = torch.empty(n, dtype=torch.uint8, device=dev) if n else None
    wp, wb = _ws(workspace)
    _check(lib().ttm_titans_bwd(B, H, T, dk, dv, int(chunk), _dtype_code(q), _ptr(q), _ptr(k),
                                _ptr(v), _ptr(eta), _ptr(theta), _ptr(alpha), _ptr(W0), _ptr(S0),
                                int(bool(w0_shared)), _ptr(dz), _ptr(dW), _ptr(dS), _ptr(g["dq"]),
                                _ptr(g["dk"]), _ptr(g["dv"]), _ptr(g["deta"]), _ptr(g["dtheta"]),
                                _ptr(g["dalpha"]), _ptr(g["dW0"]), _ptr(g["dS0"]), wp, wb,
                                _stream(q, stream)), "ttm_titans_bwd")
    return g


def mlp_fwd(q, k, v, theta, W1_0, W2_0, chunk, *, eta=None, alpha=None, S1_0=None, S2_0=None,
            w0_shared=False, z=None, W1_out=None, W2_out=None, S1_out=None, S2_out=None,
            want_S=True, stream=None):
    """Deep-memory scan, f(x) = W2 GELU(W1 x).  W1_0: [B|1,H,hidden,d], W2_0: [B|1,H,d,hidden].
    Returns (z, W1, W2, S1, S2)."""
    import torch
    B, H, T, d = q.shape
    hidden = W1_0.shape[-2]
    dev = q.device
    z = torch.empty_like(v) if z is None else z
    mk = lambda s: torch.empty(s, dtype=torch.float32, device=dev)
    W1_out = mk((B, H, hidden, d)) if W1_out is None else W1_out
    W2_out = mk((B, H, d, hidden)) if W2_out is None else W2_out
    if want_S or eta is not None:
        S1_out = mk((B, H, hidden, d)) if S1_out is None else S1_out
        S2_out = mk((B, H, d, hidden)) if S2_out is None else S2_out
    _check(lib().ttm_mlp_fwd(B, H, T, d, hidden, int(chunk), _dtype_code(q), _ptr(q), _ptr(k),
                             _ptr(v), _ptr(eta), _ptr(theta), _ptr(alpha), _ptr(W1_0),
                             _ptr(W2_0), _ptr(S1_0), _ptr(S2_0), int(bool(w0_shared)), _ptr(z),
                             _ptr(W1_out), _ptr(W2_out), _ptr(S1_out), _ptr(S2_out),
                             _stream(q, stream)), "ttm_mlp_fwd")
    return z, W1_out, W2_out, S1_out, S2_out


def mlp_gelu(x, *, want_grad=True, stream=None):
    """GELU(x) and GELU'(x) of a float32 CUDA tensor, as the 2-layer memory kernel
    evaluates them on the device.  Returns (y, dy) (dy None unless want_grad)."""
    import torch
    if x.dtype != torch.float32 or not x.is_cuda:
        raise TTMError(ERR_INVALID_ARG, "mlp_gelu (expects a float32 CUDA tensor)")
    x = x.contiguous()
    y = torch.empty_like(x)
    dy = torch.empty_like(x) if want_grad else None
    _check(lib().ttm_mlp_gelu(_ptr(x), _ptr(y), _ptr(dy), x.numel(), _stream(x, stream)),
           "ttm_mlp_gelu")
    return y, dy

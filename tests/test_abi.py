"""The C ABI without a GPU: the library loads, exports what include/ttm.h
declares, and rejects malformed calls on the host before touching CUDA."""
import ctypes

import pytest
import torch

import test_neural_memory_gb300 as ttm

INVALID, UNSUPPORTED, CUDA = ttm.ERR_INVALID_ARG, ttm.ERR_UNSUPPORTED, ttm.ERR_CUDA


@pytest.fixture(scope="module")
def L():
    ttm.build()
    return ttm.lib()


def test_exports_every_declared_symbol(L):
    names = ttm.declared_symbols()
    assert {"ttm_linear_fwd", "ttm_titans_fwd", "ttm_mlp_fwd", "ttm_status_str"} <= set(names)
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    for code in range(5):
        assert ttm.status_str(code) and ttm.status_str(code) != "unknown status"
    assert ttm.status_str(99) == "unknown status"


def test_policy_round_trip(L):
    assert ttm.set_kernel_policy("simt") == "auto"
    assert ttm.set_kernel_policy("tc") == "simt"
    assert ttm.set_kernel_policy("auto") == "tc"
    assert L.ttm_set_kernel_policy(7) == -1
    assert ttm.set_kernel_policy("auto") == "auto"


# Fake device addresses: validation must reject every call that gets them
# before any use, and no test hands them to a call that would pass validation.
# Tests that pass them run only where the library's own runtime reaches no
# GPU (torch may not see a device that the statically linked runtime does).
A = 1 << 20


def _no_gpu_reachable() -> bool:
    ttm.build()
    return ttm.cuda_device_count() == 0 and not torch.cuda.is_available()


host_only = pytest.mark.skipif(not _no_gpu_reachable(),
                               reason="passes fake device addresses; host-only")


def P(i, misalign=0):
    return ctypes.c_void_p(A * (i + 1) + misalign)


def lin_call(L, B=1, H=1, T=8, dk=64, dv=64, chunk=4, dt=1, q=P(0), k=P(1), v=P(2), eta=None,
             theta=P(3), alpha=None, W0=P(4), shared=0, z=P(5), W=P(6), ws=None, wsb=0):
    return L.ttm_linear_fwd(B, H, T, dk, dv, chunk, dt, q, k, v, eta, theta, alpha, W0, shared,
                            z, W, ws, wsb, None)


@host_only
def test_linear_rejects_malformed(L):
    assert lin_call(L, B=0) == INVALID
    assert lin_call(L, T=-1) == INVALID
    assert lin_call(L, chunk=0) == INVALID
    assert lin_call(L, dt=5) == INVALID
    assert lin_call(L, dk=12) == INVALID          # bf16 rows must be multiples of 8
    assert lin_call(L, dt=0, dk=6) == INVALID     # fp32 rows must be multiples of 4
    assert lin_call(L, W0=None) == INVALID
    assert lin_call(L, theta=None) == INVALID
    assert lin_call(L, q=P(0, 8)) == INVALID      # not 16-byte aligned
    assert lin_call(L, eta=P(7)) == INVALID       # TTT-Linear has no momentum
    assert lin_call(L, alpha=P(7)) == INVALID
    assert lin_call(L, z=P(0)) == INVALID         # output overlaps an input
    assert lin_call(L, W=P(4), shared=1) == INVALID   # in place only when not shared


@host_only
def test_titans_and_mlp_reject_malformed(L):
    r = L.ttm_titans_fwd(1, 1, 8, 64, 64, 4, 1, P(0), P(1), P(2), P(3), P(4), P(5), P(6),
                         P(7), 0, P(8), P(9), P(9), None, 0, None)
    assert r == INVALID                            # S_out == W_out
    r = L.ttm_mlp_fwd(1, 1, 8, 64, 256, 4, 1, P(0), P(1), P(2), P(3), P(4), None, P(5), P(6),
                      None, None, 0, P(8), P(9), P(10), None, None, None)
    assert r == INVALID                            # eta given without S outputs
    r = L.ttm_mlp_fwd(1, 1, 8, 64, 256, 4, 1, P(0), P(1), P(2), None, P(4), None, P(5), P(6),
                      None, None, 0, P(8), P(9), P(10), P(11), None, None)
    assert r == INVALID                            # S1_out without S2_out
    r = L.ttm_mlp_fwd(1, 1, 8, 60, 256, 4, 1, P(0), P(1), P(2), None, P(4), None, P(5), P(6),
                      None, None, 0, P(8), P(9), P(10), None, None, None)
    assert r == INVALID                            # d not a multiple of 8


@host_only
def test_tc_policy_reports_unsupported_on_host(L):
    with ttm.kernel_policy("tc"):
        # fp32 inputs never run on the tensor-core kernel
        assert lin_call(L, dt=0) == UNSUPPORTED


@host_only
def test_workspace_size_and_checks(L):
    # tensor-core shapes need one 17424-byte record per (sequence, 64-token chunk)
    with ttm.kernel_policy("tc"):
        assert L.ttm_linear_workspace_size(2, 3, 130, 128, 128, 64, 1) == 2 * 3 * 3 * 17424
        assert L.ttm_linear_workspace_size(1, 1, 64, 64, 64, 64, 0) == 0   # fp32: rejected
        # a tensor-core call without (enough) workspace is malformed
        assert lin_call(L, T=64, chunk=64) == INVALID
        assert lin_call(L, T=64, chunk=64, ws=P(9), wsb=100) == INVALID
        # workspace overlapping an input
        assert lin_call(L, T=64, chunk=64, ws=P(0), wsb=17424) == INVALID
    with ttm.kernel_policy("simt"):
        assert L.ttm_linear_workspace_size(2, 3, 130, 128, 128, 64, 1) == 0


@host_only
def test_no_device_is_reported_without_any_address(L):
    # with no reachable device the library's own queries fail cleanly: the
    # device count is 0 and the status query reports a CUDA error
    assert L.ttm_cuda_device_count() == 0
    assert ttm.device_status() == CUDA


def test_python_layer_raises(L):
    with pytest.raises(ttm.TTMError) as e:
        ttm._check(INVALID, "ttm_linear_fwd")
    assert e.value.code == INVALID


def step_call(L, B=1, H=1, n=1, dk=64, dv=64, chunk=4, pos=0, dt=1, q=P(0), k=P(1), v=P(2),
              eta=None, theta=P(3), alpha=None, W=P(4), S=None, Wc=P(5), z=P(6)):
    return L.ttm_titans_step(B, H, n, dk, dv, chunk, pos, dt, q, k, v, eta, theta, alpha, W, S,
                             Wc, z, None)


@host_only
def test_step_rejects_malformed(L):
    assert step_call(L, n=0) == INVALID
    assert step_call(L, pos=-1) == INVALID
    assert step_call(L, pos=4) == INVALID              # position must be inside the chunk
    assert step_call(L, chunk=0) == INVALID
    assert step_call(L, theta=None) == INVALID
    assert step_call(L, Wc=None) == INVALID
    assert step_call(L, eta=P(7)) == INVALID            # momentum without its state
    assert step_call(L, dk=12) == INVALID
    assert step_call(L, W=P(1)) == INVALID              # state overlaps an input
    assert step_call(L, Wc=P(4)) == INVALID             # outputs overlap each other
    assert step_call(L, q=P(0, 8)) == INVALID           # misaligned
    assert step_call(L, dk=520) == UNSUPPORTED          # one warp per row holds <= 512 columns
    assert L.ttm_linear_step(1, 1, 1, 64, 64, 4, 5, 1, P(0), P(1), P(2), P(3), P(4), P(5),
                             P(6), None) == INVALID


def bwd_call(L, B=1, H=1, T=8, dk=64, dv=64, chunk=4, dt=1, q=P(0), k=P(1), v=P(2), eta=None,
             theta=P(3), alpha=None, W0=P(4), S0=None, shared=0, dz=P(5), dW=None, dS=None,
             dq=P(10), dk_=P(11), dv_=P(12), deta=None, dtheta=P(13), dalpha=None, dW0=P(14),
             dS0=None, ws=P(20), wsb=1 << 30):
    return L.ttm_titans_bwd(B, H, T, dk, dv, chunk, dt, q, k, v, eta, theta, alpha, W0, S0,
                            shared, dz, dW, dS, dq, dk_, dv_, deta, dtheta, dalpha, dW0, dS0, ws,
                            wsb, None)


@host_only
def test_bwd_rejects_malformed(L):
    assert bwd_call(L, chunk=0) == INVALID
    assert bwd_call(L, dz=None) == INVALID
    assert bwd_call(L, dtheta=None) == INVALID
    assert bwd_call(L, deta=P(15)) == INVALID                   # no eta, no deta
    assert bwd_call(L, dalpha=P(15)) == INVALID
    assert bwd_call(L, dq=P(0)) == INVALID                      # output overlaps an input
    assert bwd_call(L, dk_=P(10)) == INVALID                    # outputs overlap each other
    assert bwd_call(L, dW0=P(20)) == INVALID                    # output inside the workspace
    assert bwd_call(L, q=P(0, 8)) == INVALID                    # misaligned
    assert bwd_call(L, wsb=1024) == INVALID                     # workspace too small
    assert bwd_call(L, ws=None, wsb=0) == INVALID
    assert bwd_call(L, chunk=128) == UNSUPPORTED                # chunk above 64
    assert bwd_call(L, dk=256) == UNSUPPORTED                   # key wider than 128
    assert L.ttm_titans_bwd_workspace_size(1, 1, 8, 64, 64, 128, 1, 0) == 0


@host_only
def test_bwd_workspace_size(L):
    # state and adjoint per chunk boundary (4 x dv x dk fp32) plus a record of
    # bc^2 + 4 bc + 1 floats rounded up to 4; shared W0 adds per-sequence partials
    per_chunk = 4 * 64 * 64 * 4 + ((64 * 64 + 4 * 64 + 1 + 3) // 4 * 4) * 4
    with ttm.kernel_policy("simt"):
        assert L.ttm_titans_bwd_workspace_size(2, 3, 130, 64, 64, 64, 1, 0) == 2 * 3 * 3 * per_chunk
        assert (L.ttm_titans_bwd_workspace_size(2, 3, 130, 64, 64, 64, 1, 1) ==
                2 * 3 * 3 * per_chunk + 2 * 3 * 2 * 64 * 64 * 4)
    # where the tensor-core scan writes the checkpoints, its 17424-byte records come on top
    with ttm.kernel_policy("auto"):
        assert (L.ttm_titans_bwd_workspace_size(2, 3, 130, 64, 64, 64, 1, 0) ==
                2 * 3 * 3 * per_chunk + 2 * 3 * 3 * 17424)
        assert (L.ttm_titans_bwd_workspace_size(2, 3, 130, 64, 64, 64, 0, 0) ==
                2 * 3 * 3 * per_chunk)                         # fp32: CUDA-core forward



def dgd_call(L, B=1, H=1, T=8, dk=64, dv=64, chunk=64, dt=1, q=P(0), k=P(1), v=P(2), eta=P(3),
             alpha=P(4), W0=P(5), shared=0, z=P(6), W=P(7), ws=None, wsb=0):
    return L.ttm_dgd_fwd(B, H, T, dk, dv, chunk, dt, q, k, v, eta, alpha, W0, shared, z, W, ws,
                         wsb, None)


@host_only
def test_dgd_workspace_size_and_checks(L):
    # chunk form: per (sequence, 64-token chunk) A~N (64 rows) and K^T diag(r) N (dk rows)
    # of 128 bytes each, then 1024 bytes of vectors
    with ttm.kernel_policy("auto"):
        assert L.ttm_dgd_workspace_size(2, 3, 130, 128, 128, 64, 1) == 2 * 3 * 3 * (8192 + 16384 + 1024)
        assert L.ttm_dgd_workspace_size(1, 2, 64, 64, 64, 64, 1) == 2 * (8192 + 8192 + 1024)
        assert L.ttm_dgd_workspace_size(1, 1, 64, 64, 64, 64, 0) == 0     # fp32: token loop
        assert L.ttm_dgd_workspace_size(1, 1, 64, 64, 64, 32, 1) == 0     # chunk 32: token loop
        assert L.ttm_dgd_workspace_size(1, 1, 64, 96, 96, 64, 1) == 0     # d 96: token loop
        assert L.ttm_dgd_workspace_size(1, 1, 0, 64, 64, 64, 1) == 0
        # the chunk form without (enough) workspace is malformed; so is overlap
        assert dgd_call(L) == INVALID
        assert dgd_call(L, ws=P(9), wsb=100) == INVALID
        assert dgd_call(L, ws=P(0), wsb=1 << 20) == INVALID
        assert dgd_call(L, ws=P(9, 8), wsb=1 << 20) == INVALID           # misaligned
    with ttm.kernel_policy("simt"):
        assert L.ttm_dgd_workspace_size(2, 3, 130, 128, 128, 64, 1) == 0
    with ttm.kernel_policy("tc"):
        assert dgd_call(L, dt=0) == UNSUPPORTED                         # fp32 never on tensor cores
        assert dgd_call(L, chunk=16) == UNSUPPORTED

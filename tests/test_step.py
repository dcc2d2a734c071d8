"""GPU parity of the streaming decode step (ttm_titans_step / ttm_linear_step)
against the float64 token-loop oracle.

A sequence is prefilled by the chunked scan (or not at all) and then continued
token by token in calls of irregular sizes, so calls start in mid-chunk and
cross chunk boundaries; the concatenated outputs and the final state must
match the oracle run over the whole sequence in one go."""
import pytest
import torch

import ttm_inputs as wl
from tests import helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import test_neural_memory_gb300 as ttm
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    ttm.build()
    yield
    assert ttm.device_status() == ttm.OK


def _part(x, t0, t1):
    return None if x is None else x[:, :, t0:t1].contiguous()


def run_decode(kind, dtype, T0, calls, chunk, d=64, dv=None, B=2, Hh=2, seed=0, theta=None):
    """Prefill T0 tokens with the chunked scan, then decode sum(calls) tokens;
    returns (gpu dict, oracle dict)."""
    import test_neural_memory_gb300 as ttm
    T = T0 + sum(calls)
    kw = dict(kind=kind, dtype=dtype, B=B, H=Hh, T=T, d=d, chunk=chunk, seed=seed)
    if theta is not None:
        kw["theta"] = theta
    w, inp = wl.generate_custom(**kw)
    if dv is not None:   # rectangular memory: replace v with dv columns
        g = torch.Generator().manual_seed(seed + 1)
        v = torch.randn((B, Hh, T, dv), generator=g)
        inp["v"] = v.to(inp["q"].dtype)
        inp["W0"] = 0.02 * torch.randn((B, Hh, dv, d), generator=g)
    dev = H.to_dev(inp)
    dvv = dev["v"].shape[-1]
    titans = kind == "titans"
    zs = []
    if T0 > 0:
        z0, W, S = ttm.titans_fwd(*(_part(dev[n], 0, T0) for n in ("q", "k", "v", "theta")),
                                  dev["W0"], chunk, eta=_part(dev["eta"], 0, T0),
                                  alpha=_part(dev["alpha"], 0, T0))
        zs.append(z0)
        assert T0 % chunk == 0
    else:
        W = dev["W0"].clone()
        S = torch.zeros_like(W)
    if not titans:
        S = None
    Wc, pos, t = None, 0, T0
    for n in calls:
        z, Wc, pos = ttm.titans_step(*(_part(dev[x], t, t + n) for x in ("q", "k", "v", "theta")),
                                     W, chunk, pos, eta=_part(dev["eta"], t, t + n),
                                     alpha=_part(dev["alpha"], t, t + n), S=S, Wc=Wc)
        zs.append(z)
        t += n
    torch.cuda.synchronize()
    gpu = dict(z=torch.cat(zs, dim=2), W=W, S=S if S is not None else torch.zeros_like(W))
    ref = H.run_linear_oracle(w, inp)
    assert gpu["z"].shape[-1] == dvv
    return gpu, ref


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_prefill_then_decode_titans(dtype):
    gpu, ref = run_decode("titans", dtype, T0=192, calls=[1, 1, 5, 64, 6], chunk=64, seed=41)
    H.compare(gpu, ref, ["z", "W", "S"], H.TOL[dtype])


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_decode_from_scratch_crossing_chunks(dtype):
    gpu, ref = run_decode("titans", dtype, T0=0, calls=[1, 3, 60, 2, 84], chunk=16, seed=42)
    H.compare(gpu, ref, ["z", "W", "S"], H.TOL[dtype])


def test_linear_decode_no_momentum():
    gpu, ref = run_decode("linear", "f32", T0=32, calls=[7, 9, 16, 1], chunk=16, seed=43)
    H.compare(gpu, ref, ["z", "W"], H.TOL["f32"])


def test_delta_rule_chunk_one():
    # chunk 1: every token opens a chunk, i.e. the online delta rule
    gpu, ref = run_decode("linear", "f32", T0=0, calls=[5, 1, 10], chunk=1, seed=44)
    H.compare(gpu, ref, ["z", "W"], H.TOL["f32"])


@pytest.mark.parametrize("d,dv", [(16, 8), (16, 12), (512, 32), (96, 64), (128, 128), (128, 24)])
def test_decode_widths(d, dv):
    # dk below one warp, the widest row, and a width that is not a power of two
    gpu, ref = run_decode("titans", "f32", T0=0, calls=[3, 20, 1], chunk=8, d=d, dv=dv, B=1,
                          Hh=2, seed=45, theta=("sigmoid", 0.02))
    H.compare(gpu, ref, ["z", "W", "S"], H.TOL["f32"])


@pytest.mark.parametrize("dtype,B,Hh", [("bf16", 8, 10), ("f32", 4, 10)])
def test_decode_many_rows_block_sizes(dtype, B, Hh):
    """Enough rows that the four-rows-per-warp kernel takes blocks of 8 warps
    (10 240 rows) or 4 warps (5 120 rows) instead of 2."""
    gpu, ref = run_decode("titans", dtype, T0=0, calls=[3, 9, 1], chunk=8, d=128, B=B, Hh=Hh,
                          seed=46, theta=("sigmoid", 0.02))
    H.compare(gpu, ref, ["z", "W", "S"], H.TOL[dtype])


def test_decode_rejects_mid_chunk_without_snapshot():
    import test_neural_memory_gb300 as ttm
    w, inp = wl.generate_custom(kind="titans", dtype="f32", B=1, H=1, T=2, d=64, chunk=4, seed=1)
    d = H.to_dev(inp)
    with pytest.raises(ttm.TTMError):
        ttm.titans_step(d["q"], d["k"], d["v"], d["theta"], d["W0"].clone(), 4, 1,
                        eta=d["eta"], alpha=d["alpha"], S=torch.zeros_like(d["W0"]))

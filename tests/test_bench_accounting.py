"""bench.py's roofline accounting, recomputed by hand from the workload shapes:
the algorithmic bytes and FLOPs every reported fraction divides by, and the
roof each kind of kernel is measured against."""
import bench
import ttm_inputs as wl


def test_titans_long_context_bytes_and_flops():
    w = wl.WORKLOADS[4]                      # B1 H16 T131072 d128 chunk 64, bf16
    assert (w.B, w.H, w.T, w.d, w.chunk, w.dtype) == (1, 16, 131072, 128, 64, "bf16")
    a = bench.algorithmic(w)
    tok = 1 * 16 * 131072
    per_tok = 4 * 128 * 2 + 3 * 4            # q, k, v, z in bf16; theta, eta, alpha in fp32
    state = 128 * 128 * 4
    assert a["bytes_per_token"] == per_tok
    # W0 read once per head; W and S written once per sequence
    assert a["bytes"] == tok * per_tok + 16 * state + 16 * 2 * state
    assert a["flops"] == tok * (10 * 128 * 128 + 4 * 64 * 128)
    assert abs(a["bytes"] / 1e9 - 2.1758) < 1e-3 and abs(a["flops"] / 1e9 - 412.3) < 0.1


def test_mlp_workload_flops():
    w = wl.WORKLOADS[5]                      # B4 H16 T16384 d64 hidden 256 chunk 16
    a = bench.algorithmic(w)
    per_tok = 22 * 256 * 64 + 2 * 16 * (2 * 64 + 2 * 256)
    assert a["flops"] == 4 * 16 * 16384 * per_tok
    assert abs(a["flops"] / 1e9 - 399.43) < 0.01


def test_roof_is_the_slower_of_hbm_and_bf16_for_every_kernel():
    peaks, _ = bench.load_peaks()
    w4, w5 = wl.WORKLOADS[4], wl.WORKLOADS[5]
    a4, a5 = bench.algorithmic(w4), bench.algorithmic(w5)
    r = bench.roofline(w4, 2.445e-3, "linear_tc")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert abs(r["achieved"] - a4["bytes"] / 2.445e-3 / 1e9) < 1e-6
    t_roof = max(a4["bytes"] / (peaks["hbm_gbs"] * 1e9), a4["flops"] / (peaks["bf16_tflops"] * 1e12))
    assert abs(r["frac"] - t_roof / 2.445e-3) < 1e-12
    # a CUDA-core kernel is measured against the same roof: for the 2-layer
    # memory that is the bf16 tensor peak (399.4 GFLOP / 1909.9 TFLOP/s = 209 us)
    r = bench.roofline(w5, 24.15e-3, "mlp_simt")
    assert r["bound"] == "tensor" and r["peak"] == peaks["bf16_tflops"]
    t_roof = a5["flops"] / (peaks["bf16_tflops"] * 1e12)
    assert abs(r["t_roof_s"] - t_roof) < 1e-15 and abs(r["frac"] - t_roof / 24.15e-3) < 1e-12
    # its fraction of the fp32 FMA pipe is only a secondary field
    alu = r["fp32_alu"]
    assert abs(alu["peak"] - 152 * 128 * 2 * 2070e6 / 1e12) < 1e-9
    assert abs(alu["frac"] - a5["flops"] / 24.15e-3 / 1e12 / alu["peak"]) < 1e-12
    r = bench.roofline(w5, 5.53e-3, "mlp_tc")
    assert r["bound"] == "tensor" and "fp32_alu" not in r


def test_fp32_alu_peak():
    assert abs(bench.fp32_alu_peak_tflops(2070.0) - 80.54784) < 1e-9

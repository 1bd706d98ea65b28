"""Host arithmetic of the bench line: the per-kernel floors and bounds, the
chained launches' algorithmic sums, and the expert-size histogram that the
bucket sweep reports beside the skewed workload."""
import importlib.util
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_mod2", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    argv = sys.argv
    try:
        sys.argv = ["bench.py"]
        spec.loader.exec_module(mod)
    finally:
        sys.argv = argv
    return mod


SHAPE = {"T": 4096, "H": 2048, "E": 128, "k": 8, "F": 768}
PEAKS = {"hbm_gbs": 6775.3, "bf16_tflops": 1900.5, "bf16_tflops_sustained": 1691.5}


def test_chained_launches_sum_their_two_gemms():
    b = _bench()
    algo = b.algorithmic(SHAPE)
    for chain, (m1, m2) in (("gemm_ffn_fwd", ("gemm_fc1_fwd", "gemm_fc2_fwd")),
                            ("gemm_ffn_dgrad", ("gemm_fc2_dgrad", "gemm_fc1_dgrad")),
                            ("gemm_wgrad", ("gemm_wgrad_w1", "gemm_wgrad_w2"))):
        assert algo[chain] == tuple(x + y for x, y in zip(algo[m1], algo[m2]))
    # the weight gradients: 1208 MB of bf16 dW1 and dW2 written, 420 MB read
    rd, wr, fl = algo["gemm_wgrad"]
    E, H, F, N = 128, 2048, 768, 4096 * 8
    assert wr == E * 3 * F * H * 2
    assert rd == N * (2 * F + H + H + F) * 2
    assert fl == 2.0 * N * 3 * F * H


def test_floor_is_the_copy_rate_when_writes_stream_faster():
    b = _bench()
    algo = b.algorithmic(SHAPE)
    agg = {"gemm_wgrad": [1, 0.3], "combine": [1, 0.026]}
    ks = b.kernel_stats(agg, algo, PEAKS, 7400.0)
    for name, (n, ms) in agg.items():
        by = algo[name][0] + algo[name][1]
        copy_floor_us = by / (PEAKS["hbm_gbs"] * 1e9) * 1e6
        assert abs(ks[name]["hbm_floor_us"] - copy_floor_us) < 0.11
        assert abs(ks[name]["roofline_frac"] - copy_floor_us / (ms * 1e3)) < 2e-3
        assert ks[name]["bound"] == "hbm"
    # a write-only rate below the copy rate would make the written bytes the floor
    slow = b.kernel_stats(agg, algo, PEAKS, 3000.0)
    assert slow["gemm_wgrad"]["hbm_floor_us"] > ks["gemm_wgrad"]["hbm_floor_us"]


def test_compute_bound_gemm_is_rated_against_the_sustained_tensor_peak():
    b = _bench()
    shape = {"T": 65536, "H": 2048, "E": 128, "k": 8, "F": 768}  # 4096 rows per expert
    algo = b.algorithmic(shape)
    ks = b.kernel_stats({"gemm_ffn_fwd": [1, 3.0]}, algo, PEAKS, 7400.0)
    fl = algo["gemm_ffn_fwd"][2]
    assert ks["gemm_ffn_fwd"]["bound"] == "tensor"
    assert abs(ks["gemm_ffn_fwd"]["roofline_frac"]
               - fl / (PEAKS["bf16_tflops_sustained"] * 1e12) / 3.0e-3) < 2e-3


def test_rows_histogram_buckets():
    b = _bench()
    cnt = torch.tensor([0, 5, 63, 64, 127, 128, 255, 256, 4095, 4096, 9000], dtype=torch.int32)
    h = b.rows_histogram(cnt)
    assert list(h) == [str(m) for m in b.BUCKET_ROWS]
    assert h["64"] == {"experts": 5, "rows": 0 + 5 + 63 + 64 + 127}  # the first takes fewer rows
    assert h["128"] == {"experts": 2, "rows": 128 + 255}
    assert h["256"] == {"experts": 1, "rows": 256}
    assert h["2048"] == {"experts": 1, "rows": 4095}
    assert h["4096"] == {"experts": 2, "rows": 4096 + 9000}  # the last takes more
    assert sum(v["experts"] for v in h.values()) == cnt.numel()
    assert sum(v["rows"] for v in h.values()) == int(cnt.sum())

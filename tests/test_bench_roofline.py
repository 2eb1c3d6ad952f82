"""The benchmark's roofline arithmetic (CPU): the algorithmic work of each
launch phase, the choice of peak by the length of the timed region, and the
fractions of the phase table."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

PEAKS = {"hbm_gbs": 6790.7, "bf16_tflops": 1917.9, "bf16_tflops_sustained": 1726.7}


def test_algorithmic_work_of_the_prefill_step():
    T, H, I, E, K = 4096, 2048, 1408, 64, 6
    a = bench.algo_work(T, H, I, E, K, fwd_only=False)
    F = 2.0 * T * K * H * I
    # each GEMM launch does 3F: 6 TK H I forward, 12 TK H I backward in two launches
    for k in ("gemm_fwd", "gemm_bwd_data", "gemm_bwd_weight"):
        assert a[k] == ("tensor", 3 * F)
    assert a["gemm_fwd"][1] + a["gemm_bwd_data"][1] + a["gemm_bwd_weight"][1] == 18 * T * K * H * I
    # dispatch: x once + K bf16 rows + their fp8 copies (training); combine: K rows + y + w
    assert a["dispatch_x"] == ("hbm", (T * H + T * K * H) * 2.0 + T * K * H)
    assert a["combine_y"] == ("hbm", (T * K * H + T * H) * 2.0 + T * K * 2.0)
    inf = bench.algo_work(T, H, I, E, K, fwd_only=True)
    assert inf["dispatch_x"] == ("hbm", (T * H + T * K * H) * 2.0)


def test_decode_gemm_is_weight_streaming():
    T, H, I, E, K = 128, 7168, 2048, 256, 8
    a = bench.algo_work(T, H, I, E, K, fwd_only=True, touched=250)
    bound, work = a["gemm_fwd"]
    assert bound == "hbm"
    assert work == 250 * (H * 2 * I + I * H) * 2.0 + T * K * (H + I) * 4.0


@pytest.mark.parametrize("region_ms,key", [(27.0, "bf16_tflops"), (1999.0, "bf16_tflops"),
                                           (2000.0, "bf16_tflops_sustained"),
                                           (550.0, "bf16_tflops")])
def test_peak_follows_the_timed_region(region_ms, key):
    assert bench.peak_for("tensor", region_ms, PEAKS) == (PEAKS[key], key)
    assert bench.peak_for("hbm", region_ms, PEAKS) == (PEAKS["hbm_gbs"], "hbm_gbs")


def test_phase_table_fractions():
    T, H, I, E, K = 4096, 2048, 1408, 64, 6
    algo = bench.algo_work(T, H, I, E, K, fwd_only=False)
    # 100 profiled steps: gemm_bwd_weight 46 ms in all, combine_y 2.3 ms
    prof = {"gemm_bwd_weight": (46.0, 100), "combine_y": (2.3, 100), "route": (0.0, 0)}
    ph = bench.phase_table(prof, 100, 1.33, algo, PEAKS, region_ms=26.6)
    assert "route" not in ph  # no launches: left out
    w = ph["gemm_bwd_weight"]
    tf = 3 * 2.0 * T * K * H * I / 0.46e-3 / 1e12
    assert w["achieved"] == pytest.approx(tf)
    assert w["frac"] == pytest.approx(tf / PEAKS["bf16_tflops"])   # short region: burst
    assert w["frac_sustained"] == pytest.approx(tf / PEAKS["bf16_tflops_sustained"])
    c = ph["combine_y"]
    assert c["unit"] == "GB/s"
    assert c["frac"] == pytest.approx(c["achieved"] / PEAKS["hbm_gbs"])
    assert c["share"] == pytest.approx(0.023 / 1.33)

"""bench.py's roofline model on CPU: the tensor peak follows the run's clock
and the recipe (bf16 burst or sustained figure; FP8 twice it, FP4 six times,
the nominal dense ratios), and the algorithmic bytes of a GEMM stage count
each operand once at its storage size."""
import pytest

import bench
import moe_inputs as mi

PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
         "clocks_under_load": {"sm_mhz_median": 1455.0}}


@pytest.mark.parametrize("mhz,fp8,fp4,want", [(2070.0, False, False, 1900.0), (1460.0, False, False, 1700.0),
                                             (2070.0, True, False, 3800.0), (2070.0, False, True, 11400.0),
                                             (1460.0, False, True, 10200.0)])
def test_peak_follows_clock_and_recipe(mhz, fp8, fp4, want):
    peak, desc = bench.choose_peak(PEAKS, "measured", {"sm_mhz": mhz}, fp8, fp4)
    assert peak == pytest.approx(want)
    assert ("6 x" in desc) == fp4 and ("2 x" in desc) == (fp8 and not fp4)


def test_stage_bytes_count_operands_at_their_storage_size():
    w = mi.WORKLOADS["qwen3_235b"]
    R, H, F, E = w.R, w.H, w.F, w.E
    RH, RF, EHF = R * H, R * F, E * H * F
    per = {mi.BF16: 2.0, mi.FP8_BLOCK: 1 + 4 / 128, mi.MXFP8: 1 + 1 / 32, mi.NVFP4: 0.5 + 1 / 16}
    for dt, a in per.items():
        wd = mi.scaled(w, dtype=dt)
        # fc2: reads h (R F) and Wd (E F H) as operands, writes Yp (R H) in bf16
        assert bench.stage_bytes("fc2", wd) == pytest.approx(a * (RF + EHF) + 2 * RH)
        # fc1 wgrad: reads Xp^T (R H) and [dA | dU] (2 R F), writes dWg, dWu in bf16
        assert bench.stage_bytes("fc1_wgrad", wd) == pytest.approx(a * (RH + 2 * RF) + 2 * 2 * EHF)
    # FLOPs do not depend on the recipe
    assert bench.stage_flops("fc1_swiglu", mi.scaled(w, dtype=mi.NVFP4)) == bench.stage_flops("fc1_swiglu", w)

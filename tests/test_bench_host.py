"""Host-side arithmetic of bench.py's JSON line (CPU): per-step sums over the phases, mean and
median step, the L2-warm key, and the dominant kernel's roofline from given per-phase times."""
import pytest

import bench


def test_config_numbers_from_given_phase_times():
    w = bench.WORKLOADS["C5"]
    per_phase = {"pi_attn_fwd": [0.1, 0.3, 0.2], "pi_attn_bwd": [0.5, 0.4, 0.6]}  # ms per step
    assert bench.step_times(per_phase, 3) == pytest.approx([0.6, 0.7, 0.8])
    out = bench.config_numbers(w, per_phase, 3, l2_warm_ms=0.5)
    assert out["ms_per_step"] == pytest.approx(0.7)
    assert out["median_ms_per_step"] == pytest.approx(0.7)
    assert out["l2_warm_ms_per_step"] == 0.5
    assert out["tokens_per_s"] == pytest.approx(w.B * w.N * 3 / 2.1e-3)
    assert out["per_phase_ms"] == pytest.approx({"pi_attn_fwd": 0.2, "pi_attn_bwd": 0.5})
    # the dominant kernel is the backward (1.5 of 2.1 ms); its algorithmic bytes over its mean time
    wk = bench.work(w, True)
    r = out["roofline"]
    assert r["kernel"] == "pi_attn_bwd"
    assert r["kernel_us"] == pytest.approx(500.0)
    peaks, _ = bench.load_peaks()
    t_hbm = wk["bwd_bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tensor = wk["bwd_flops"] / (peaks["bf16_tflops"] * 1e12)
    if r["bound"] == "hbm":
        assert r["achieved"] == pytest.approx(wk["bwd_bytes"] / 0.5e-3 / 1e9)
        assert r["unit"] == "GB/s"
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    full = bench.roofline_of(w, wk, per_phase)
    assert full["t_roof_us"] == pytest.approx(max(full["t_hbm_us"], full["t_tensor_us"]))
    assert full["t_hbm_us"] == pytest.approx(1e6 * t_hbm)
    assert full["t_tensor_us"] == pytest.approx(1e6 * t_tensor)
    assert full["algorithmic_bytes"] == wk["bwd_bytes"] and full["useful_flops"] == wk["bwd_flops"]


def test_l2_warm_key_only_when_given():
    w = bench.WORKLOADS["C2"]
    per_phase = {"pi_attn_fwd": [0.05, 0.07, 0.06, 0.30]}
    out = bench.config_numbers(w, per_phase, 4)
    assert "l2_warm_ms_per_step" not in out
    assert out["median_ms_per_step"] == pytest.approx(0.065)  # the median ignores the outlier
    assert out["ms_per_step"] == pytest.approx(0.12)

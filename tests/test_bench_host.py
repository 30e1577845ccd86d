"""Host-side pieces of bench.py that the JSON line depends on, checked on the CPU: the clock
sampler's parsing of nvidia-smi rows (the throttle reasons decide whether a run is kept), and
the roofline's operation count and derived FP32 peak."""
import pytest

import bench
from lapl_workloads import WORKLOADS


def _summary_of(tmp_path, text):
    path = tmp_path / "clocks.csv"
    path.write_text(text)
    cs = bench.ClockSampler(0)
    cs.path = str(path)
    return cs.summary()


def test_clock_summary_median_max_and_reasons(tmp_path):
    rows = ("0, 2070, 2070, 900.10, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active\n"
            "0, 2060, 2070, 1300.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n"
            "0, 2040, 2070, 1390.5, 0x0000000000000004, Not Active, Not Active, Not Active, Active\n")
    s = _summary_of(tmp_path, rows)
    assert s["sm_mhz"] == 2060.0 and s["sm_max_mhz"] == 2070.0 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]


def test_clock_summary_reports_every_slowdown_reason(tmp_path):
    rows = ("0, 1500, 2070, 1400.0, 0x48, Active, Active, Active, Not Active\n"
            "0, 1600, 2070, 1400.0, 0x48, Not Active, Not Active, Not Active, Not Active\n")
    s = _summary_of(tmp_path, rows)
    assert s["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert s["sm_mhz"] == 1550.0


def test_clock_summary_without_samples(tmp_path):
    s = _summary_of(tmp_path, "")
    assert s == {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}


def test_roofline_operation_count_and_peak():
    w = WORKLOADS["stage1_f32"]
    # 3 ops x (query block + key block) x B x H x N x m x d
    assert bench.cdist_ops_per_launch(w) == 3 * 2 * 8 * 2 * 3136 * 49 * 32 == 472055808
    assert bench.fp32_peak_tflops(152, 2070.0) == pytest.approx(80.54784)


def test_gemm_chain_roofline_bytes_and_fraction():
    """Algorithmic bytes of the two chain stages at the hires shape (bf16 inputs): B V stage
    reads B^T, V and (statistics) A^T; the output stage reads A^T and writes fp32 O."""
    import bench
    from lapl_workloads import WORKLOADS
    w = WORKLOADS["hires_bf16"]
    bh, n, m, d = 32, 16384, 64, 64
    e = bench.gemm_chain_roofline(w, {"bv": 0.1, "output": 0.05}, {"hbm_gbs": 5000.0},
                                  {"bv_tensor_core": 1})
    assert e[0]["bytes"] == bh * m * n * 4 * 2 + bh * n * d * 2
    assert e[1]["bytes"] == bh * m * n * 4 + bh * n * d * 4
    assert abs(e[0]["achieved"] - e[0]["bytes"] / 1e-4 / 1e9) < 1e-6
    assert abs(e[1]["frac"] - e[1]["bytes"] / 5e-5 / 1e9 / 5000.0) < 1e-12
    assert "tcgen05" in e[0]["kernel"] and e[0]["flops"] == 2.0 * bh * n * m * d
    assert e[1]["kernel"].startswith("output_kernel")
    e = bench.gemm_chain_roofline(w, {"bv": 0.1, "output": 0.05}, {"hbm_gbs": 5000.0},
                                  {"bv_tensor_core": 0, "out_tensor_core": 1})
    assert e[0]["kernel"].startswith("bv_kernel") and e[1]["kernel"].startswith("out_tc_kernel")


def test_dominant_kernel_entry():
    """The solve's tensor-core work: 2 x BH x 2T products x ceil(m'/8) MMAs of 128 x 128 x 8
    (m' = m rounded up to 4), against half the measured bf16 peak; absent without the
    tensor-core solve."""
    import bench
    from lapl_workloads import WORKLOADS
    w = WORKLOADS["stage1_f32"]
    e = bench.dominant_kernel_entry(w, {"newton_schulz": 0.05}, {"bf16_tflops": 2000.0},
                                    {"ns_tensor_core": 1}, 0.1)
    flops = 2.0 * 16 * 2 * 20 * 7 * 128 * 128 * 8
    assert abs(e["achieved"] - flops / 5e-5 / 1e12) < 1e-9
    assert e["peak"] == 1000.0 and e["bound"] == "latency" and e["share_of_forward"] == 0.5
    assert bench.dominant_kernel_entry(w, {"newton_schulz": 0.05}, {}, {"ns_tensor_core": 0},
                                       0.1) is None


def test_distance_traffic_taken_on_the_committed_sources():
    """Every distance-kernel source the traffic hash covers exists, and each recorded DRAM
    traffic figure was captured on exactly the sources in the tree (otherwise the bench reports
    traffic as null and the figure must be re-taken with ncu)."""
    import os
    import bench
    csrc = os.path.join(bench.ROOT, "laplacian_nystr_attention_gb300", "csrc")
    for f in bench.CDIST_SOURCES:
        assert os.path.isfile(os.path.join(csrc, f)), f
    sha = bench.cdist_sources_sha()
    assert sha == bench.cdist_sources_sha()                 # deterministic
    for key, (nbytes, taken_on) in bench.CDIST_TRAFFIC.items():
        assert nbytes > 0, key
        assert taken_on == sha, key

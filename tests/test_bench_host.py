"""Host-side logic of bench.py (no GPU): the layer-copy rotation that keeps
weights cold, and the config dict both arms print."""
import bench

L2 = 132 << 20  # an L2 of 132 MiB (GB300 reports about this)


def test_cold_copies_exceed_three_l2_between_reuses():
    for name in ("ling_m1", "ling_m6", "mxfp4_m1", "fp8_m1", "sweep_m1", "sweep_m16"):
        w = bench.WORKLOADS[name]
        c = bench.cold_copies(name, L2)
        assert c & (c - 1) == 0 and bench.PERIOD % c == 0
        assert (c - 1) * bench.min_step_bytes(bench.layer_shape(name), w["wfmt"], w["M"]) > 3 * L2
        assert c // 2 < w["copies"] or (c // 2 - 1) * bench.min_step_bytes(
            bench.layer_shape(name), w["wfmt"], w["M"]) <= 3 * L2  # the smallest such power of two
    assert bench.cold_copies("ling_m1", L2) == 8          # 108.8 MB per step
    assert bench.cold_copies("mxfp4_m1", L2) == 16        # 39.5 MB per step
    assert bench.cold_copies("ling_e128_m1", L2) == 2     # profiling case: fixed


def test_both_arms_print_the_same_config():
    a = bench.workload_config("ling_m1", 8, 1)
    b = bench.workload_config("ling_m1", 8, 1, res={"weights_gb": 48.4, "launch": "cuda-graph",
                                                   "distinct_experts_mean": 8.0, "reuse_bytes_min": 7e8},
                              l2_bytes=L2)
    assert all(b[k] == v for k, v in a.items())
    assert "8 layer copies" in a["workload"]


def test_sweep_covers_m_1_to_16():
    ms = sorted(bench.WORKLOADS[n]["M"] for n in bench.SWEEP.split(","))
    assert ms == list(range(1, 17))

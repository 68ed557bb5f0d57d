"""Host-side helpers of bench.py (CPU only): the clock-sample summary that
decides whether a timed region saw throttling, the whole-job rate and the
workload description in the JSON line."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
import hs_workloads as W  # noqa: E402


def _sample(sm, max_sm=2070, power=150.0, active="0x0", hw="Not Active", hw_th="Not Active",
            sw_th="Not Active", sw_pc="Not Active"):
    return ["0", str(sm), str(max_sm), str(power), active, hw, hw_th, sw_th, sw_pc]


def _sampler(samples):
    s = bench.ClockSampler.__new__(bench.ClockSampler)  # no nvidia-smi process
    s.samples = samples
    s.proc = None
    s.thread = None
    return s


def test_clock_summary_uses_the_samples_inside_the_region():
    s = _sampler([(0.5, _sample(1000)), (1.1, _sample(2070)), (1.2, _sample(2050, power=300)),
                  (1.3, _sample(2070)), (5.0, _sample(900))])
    out = s.summary(1.0, 2.0)
    assert out["samples_in_region"] == 3 and out["samples_used"] == 3
    assert out["sm_mhz"] == 2070.0 and out["sm_max_mhz"] == 2070.0
    assert out["power_w_max"] == 300.0
    assert out["reasons"] == []


def test_clock_summary_names_every_active_throttle_reason():
    s = _sampler([(1.1, _sample(1500, hw="Active", sw_pc="Active")),
                  (1.2, _sample(1600, sw_th="Active"))])
    out = s.summary(1.0, 2.0)
    assert out["reasons"] == ["hw_slowdown", "sw_power_cap", "sw_thermal_slowdown"]
    assert out["sm_mhz"] == 1550.0


def test_clock_summary_of_a_region_shorter_than_the_interval_takes_the_nearest_sample():
    s = _sampler([(0.0, _sample(1200)), (1.04, _sample(2070)), (2.0, _sample(1300))])
    out = s.summary(1.00, 1.01)  # no sample inside
    assert out["samples_in_region"] == 0 and out["samples_used"] == 1
    assert out["sm_mhz"] == 2070.0


def test_clock_summary_without_samples_reports_none():
    out = _sampler([]).summary(0.0, 1.0)
    assert out == {"samples_in_region": 0, "samples_used": 0}


def test_whole_job_rate_counts_every_replica():
    assert bench.whole_job_rate(131072, 1, 0.0774) == 131072 / 0.0774e-3
    assert bench.whole_job_rate(131072, 4, 0.0774) == 4 * bench.whole_job_rate(131072, 1, 0.0774)


def test_config_names_the_workload_and_the_flush():
    w = W.WORKLOADS["C2"]
    c = bench.config_dict(w, 1)
    assert c["workload"] == "dsa_decode_b64_k2048 (C2)"
    assert (c["batch"], c["steps"], c["top_k"], c["seq_len"]) == (64, 1, 2048, 32768)
    assert "flushed" in c["l2"] and c["parallelism"] == "single GPU"
    assert bench.config_dict(w, 8)["parallelism"] == "replicas x8"
    assert not any(k in c for k in ("model", "global_batch"))  # a workload, not a model


def test_cpu_baseline_times_the_oracle_on_a_bounded_sample():
    import numpy as np
    w = W.scaled(W.WORKLOADS["C2"], batch=2, seq_len=4096, top_k=256, hot_buffer=512)
    calls = W.TopkStream(w).calls(bench.PREROLL_CALLS + 4)
    pool = np.empty((w.batch, w.seq_len, w.row_bytes), dtype=np.uint8)
    W.fill_host_pool(pool, 0)
    out = bench.cpu_baseline_oracle(w, calls, W.req_pool_indices(w), W.seq_lens(w), 0.0, pool)
    assert out["kind"] == "oracle" and out["unit"] == bench.UNIT
    assert out["cores"] == min(w.batch, os.cpu_count() or 1)
    assert out["value"] > 0 and "steady-state calls" in out["sample"]
    assert out["sample"].startswith("2 ")  # at least two timed calls, even with no time budget


def test_phase_times_reads_the_kernel_timeline():
    """Two launches of a 3-row call in clusters of 2 (ns stamps): spans from
    the first CTA's start, the leaders' commits and the copy window."""
    import numpy as np
    t = np.zeros((2, 3, 8, 16), np.int64)
    for launch in range(2):
        for b in range(3):
            for r in range(2):
                t[launch, b, r, :11] = [1000 + 10 * b, 1500, 2000, 2500, 3000, 3500, 4000,
                                        4500, 5000 + 100 * b, 0, 9000 + 10 * r]
                t[launch, b, r, 15] = 2
            t[launch, b, 0, 9] = 7000 + 500 * b
    out = bench.phase_times(t)
    # lookup: last word 8 (5200) minus the first start (1000)
    assert out["gather_span_us"] == [4.2, 4.2]
    # commit span: last leader word 9 (8000) minus the first leader word 8 (5000)
    assert out["commit_span_us"] == [3.0, 3.0]
    assert sorted(out["commit_us"]) == [2.0, 2.0, 2.4, 2.4, 2.8, 2.8]
    # copy window: last word 10 (9010) minus the first word 8 (5000)
    assert out["copy_span_us"] == [4.01, 4.01]
    s = out["summary"]
    assert s["cluster_size"] == 2
    assert s["probed"]["median_cta"] == 0.5  # word 1 (1500) from t0 = 1000
    assert s["lists_written"]["last_cta"] == 4.2
    assert s["commit_done"]["last_cta"] == 7.0
    # a rank the call does not use (word 15 tells the cluster size) is ignored
    t[:, :, 2:, :] = 123456789
    assert bench.phase_times(t)["gather_span_us"] == [4.2, 4.2]

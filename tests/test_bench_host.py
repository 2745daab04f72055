"""Host-side logic of bench.py, on CPU: the clock record's window over the timed region, the
plan-balance report, and the kernel-source hash that keys the recorded traffic."""
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
import mla_paged_kv_decode_gb300 as mla  # noqa: E402
from mla_paged_kv_decode_gb300 import build as lib_build  # noqa: E402


def _row(mhz, reasons=("Not Active",) * 4):
    return ", ".join(["0", str(mhz), "2070", "500.0", "0x0", *reasons])


def test_clock_summary_takes_the_samples_inside_the_timed_region():
    s = bench.ClockSampler(0)
    s.samples = [(0.9, _row(1000)), (1.1, _row(2070)), (1.2, _row(2040)), (1.3, _row(2070)),
                 (1.6, _row(900, ("Active", "Not Active", "Not Active", "Not Active")))]
    c = s.summary(1.0, 1.5)
    assert c["samples"] == 3 and c["window"] == "timed region"
    assert c["sm_mhz"] == 2070.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == []                     # the slowdown at 1.6 s is outside the region


def test_clock_summary_reports_throttle_reasons_and_falls_back_to_the_nearest_samples():
    s = bench.ClockSampler(0)
    s.samples = [(1.0, _row(1500, ("Not Active", "Not Active", "Not Active", "Active"))), (2.0, _row(2070))]
    c = s.summary(1.01, 1.02)                     # shorter than the sampling period
    assert c["window"] == "nearest to the timed region" and c["samples"] == 2
    assert c["reasons"] == ["sw_power_cap"]
    assert bench.ClockSampler(0).summary(0, 1)["reasons"] == ["unsampled"]


def test_plan_balance_of_the_membound_plan():
    if lib_build.needs_build():
        lib_build.build()
    mla.load()
    B, P, L = 64, 64, 4096
    indptr = torch.arange(0, B + 1, dtype=torch.int32) * (L // P)
    last = torch.full((B,), P, dtype=torch.int32)
    plan = mla.mla_decode_plan(indptr, last, B, 16, P, 152)
    bal = bench.plan_balance(plan, 16, mla.MLA_KV_BF16)
    assert bal["units"] <= 152 and bal["tile"] == 32 and bal["segment_cost_tiles"] == 4
    assert 1.0 <= bal["tiles_max_over_mean"] <= 1.1
    assert bal["partials"] == mla.mla_plan_num_partials(plan)
    assert bal["segments"] == mla.mla_plan_num_segments(plan)


def test_source_hash_covers_the_attention_sources_only():
    h = bench.kernel_source_hash()
    assert len(h) == 16 and int(h, 16) >= 0
    csrc = os.path.join(ROOT, "mla_paged_kv_decode_gb300", "csrc")
    assert "prologue.cu" in os.listdir(csrc)      # present, and left out of the hash
    assert h == bench.kernel_source_hash()        # deterministic


def test_source_hash_ignores_comments_only():
    a = "int f(int x) {  // scale\n    return 2 * x;\n}\n"
    b = "// doubles x\nint f(int x) {\n    return 2 * x;  /* twice */\n}\n\n"
    c = "int f(int x) {\n    return 3 * x;\n}\n"
    assert bench.strip_comments(a) == bench.strip_comments(b) == "int f(int x) {\n    return 2 * x;\n}"
    assert bench.strip_comments(c) != bench.strip_comments(a)


def test_cpu_baseline_line():
    from workloads import WORKLOADS, make_inputs
    inp = make_inputs(WORKLOADS["tiny"])
    c = bench.cpu_baseline(inp, "tiny", 4)
    assert c["kind"] == "oracle" and c["unit"] == "GB/s" and c["cores"] >= 1 and c["value"] > 0
    assert c["single_thread"]["cores"] == 1 and c["single_thread"]["value"] > 0
    assert c["sample"].startswith("4 of 4 requests of tiny")


def test_reference_arm_line(capsys):
    """`bench.py --impl reference`: one JSON line with the oracle's own metric, unit, e2e and
    cpu_baseline keys, no host-device bytes."""
    import json
    import types
    args = types.SimpleNamespace(workload="tiny", sample_requests=4, steps=2, warmup=1, gpus=1)
    bench.run_reference(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "GB/s" and line["value"] > 0
    assert line["metric"] == bench.METRIC and line["higher_is_better"] is True
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["steps"] == 2 and line["warmup"] == 1 and line["config"]["workload"] == "tiny"

"""Host logic of the benchmark that decides what its JSON line reports (CPU).

The byte accounting is pinned to hand-computed totals, the nvidia-smi clock
parser to made-up sample lines, and the DRAM-traffic lookup to the rule that
a capture stops counting once the kernel source it was taken on changes.
"""
from __future__ import annotations

import json
import os
import time

import pytest

import bench
import ep_synth


def test_prefill_bytes_by_hand():
    """T=4096, H=7168, E=256, R=32, k=8, worked out term by term:
    route    T E 4 + T k 8                 =   4,194,304 +     262,144
    layout   T k 8 + (2E + 2R + 2) 4       =     262,144 +       2,312
    dispatch T H 2 + T k H 2 + T k 8       =  58,720,256 + 469,762,048 + 262,144
    combine  T k H 2 + T k 8 + T H 2       = 469,762,048 +     262,144 + 58,720,256"""
    w = ep_synth.CONFIGS["prefill"]
    kb = w.algorithmic_bytes()
    assert kb["route"] == 4_456_448
    assert kb["layout"] == 264_456
    assert kb["dispatch"] == 528_744_448
    assert kb["combine"] == 528_744_448
    assert w.total_bytes() == 1_062_209_800
    assert bench.call_bytes(w, "dispatch_fused") == 4_456_448 + 264_456 + 528_744_448
    assert bench.call_bytes(w, "combine") == 528_744_448


@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "mid", "sweep-zipf-T1", "sweep-uniform-T32768"])
def test_step_bytes_are_the_sum_of_the_calls(name):
    w = ep_synth.get_workload(name) if name.startswith("sweep") else ep_synth.CONFIGS[name]
    fused = sum(bench.call_bytes(w, n) for n in ("dispatch_fused", "combine"))
    separate = sum(bench.call_bytes(w, n) for n in ("route", "layout", "dispatch", "combine"))
    assert fused == separate == w.total_bytes()
    # collected by term: rows 4 T H (k + 1) (x read, k send rows written, k y rows read, out written),
    # logits 4 T E, the eight T k int32/fp32 arrays 32 T k, counts and offsets 8 (E + R + 1)
    T, H, E, R, k = w.T, w.H, w.E, w.R, w.k
    assert w.total_bytes() == 4 * T * H * (k + 1) + 4 * T * E + 32 * T * k + 8 * (E + R + 1)


def _line(sm, smax, *active):
    names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    flags = ", ".join("Active" if n in active else "Not Active" for n in names)
    return f"2026/12/02 10:00:00.000, 0, {sm}, {smax}, 812.40, 0x0000000000000000, {flags}"


def test_clock_parser_median_and_reasons():
    out = "\n".join([_line(2070, 2070), _line(1980, 2070, "sw_power_cap"), _line(2055, 2070)])
    c = bench.parse_clock_samples(out)
    assert c == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_clock_parser_reports_every_throttle_reason_seen():
    out = "\n".join([_line(1500, 2070, "hw_slowdown"), _line(1400, 2070, "hw_thermal_slowdown", "sw_thermal_slowdown")])
    c = bench.parse_clock_samples(out)
    assert c["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert c["sm_mhz"] == 1450.0


def test_clock_parser_skips_lines_it_cannot_read():
    out = "\n".join(["", "garbage", "a, b, [N/A], [N/A], x, y, z, w, v, u", _line(2070, 2070)])
    assert bench.parse_clock_samples(out) == {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 1}
    assert bench.parse_clock_samples("")["sm_mhz"] is None


def test_code_only_ignores_comments_and_blank_space():
    a = "int f(int x) {\n    return x + 1;  // one more\n}\n"
    b = "/* header\n   text */\nint f(int x) {\n\n        return x + 1;\n}\n"
    c = "int f(int x) {\n    return x + 2;\n}\n"
    assert bench._code_only(a) == bench._code_only(b)
    assert bench._code_only(a) != bench._code_only(c)


def test_traffic_summary_entries_are_complete():
    data = json.loads((bench.ROOT / "profiles" / "dram_traffic.txt").read_text())
    assert "ncu" in data["command"] and "--clock-control none" in data["command"]
    for workload in ("prefill", "sweep-zipf-T32768"):
        for kernel, ent in data[workload].items():
            assert kernel in bench.KERNEL_SOURCES
            assert isinstance(ent["dram_bytes_per_launch"], int) and ent["dram_bytes_per_launch"] > 0
            if "components" in ent:  # summed from other captures: valid while each of them is
                assert all(c in data[workload] and "components" not in data[workload][c] for c in ent["components"])
            else:
                assert len(ent["source_sha256_16"]) == 16
        p = data[workload]
        assert p["dispatch_fused"]["components"] == ["route", "layout", "dispatch"]
        assert p["dispatch_fused"]["dram_bytes_per_launch"] == sum(
            p[k]["dram_bytes_per_launch"] for k in ("route", "layout", "dispatch"))


def test_traffic_is_dropped_once_the_kernel_source_changes(monkeypatch):
    data = json.loads((bench.ROOT / "profiles" / "dram_traffic.txt").read_text())
    kernel = "combine"
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: data["prefill"][k]["source_sha256_16"])
    assert bench.ncu_traffic(kernel, "prefill") == data["prefill"][kernel]["dram_bytes_per_launch"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: "0" * 16)
    assert bench.ncu_traffic(kernel, "prefill") is None
    assert bench.ncu_traffic(kernel, "no-such-workload") is None


def test_summed_traffic_follows_its_components(monkeypatch):
    data = json.loads((bench.ROOT / "profiles" / "dram_traffic.txt").read_text())
    p = data["prefill"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: p[k].get("source_sha256_16", "?"))
    assert bench.ncu_traffic("dispatch_fused", "prefill") == p["dispatch_fused"]["dram_bytes_per_launch"]
    # one component changed: the sum is dropped too
    monkeypatch.setattr(bench, "kernel_source_hash",
                        lambda k: "0" * 16 if k == "layout" else p[k].get("source_sha256_16", "?"))
    assert bench.ncu_traffic("dispatch_fused", "prefill") is None


def test_clock_sampler_with_a_fake_nvidia_smi(tmp_path, monkeypatch):
    """The sampler starts nvidia-smi, stops it and parses what it printed; a
    stand-in script on PATH prints two samples, then waits to be stopped."""
    fake = tmp_path / "nvidia-smi"
    printed = tmp_path / "printed"
    fake.write_text("#!/bin/sh\n"
                    f"echo '{_line(2070, 2070)}'\n"
                    f"echo '{_line(2040, 2070, 'sw_power_cap')}'\n"
                    f"touch '{printed}'\n"
                    "exec sleep 30\n")
    fake.chmod(0o755)
    monkeypatch.setenv("PATH", f"{tmp_path}{os.pathsep}{os.environ['PATH']}")
    s = bench.ClockSampler(0)
    deadline = time.monotonic() + 20
    while not printed.exists() and time.monotonic() < deadline:
        time.sleep(0.05)
    c = s.stop()
    assert c == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 2}
    assert bench.ClockSampler(0, enabled=False).stop() is None


@pytest.mark.parametrize("R,W", [(32, 152), (64, 7), (5, 5), (1, 3)])
def test_rank_static_table_tiles_the_rows_once(R, W):
    """The ablation's rank-static table: worker r mod W takes rank r's whole
    segment; every send row is in exactly one chunk, each chunk inside one
    rank, and worker_begin indexes each worker's chunks (the form
    ep_dispatch_scheduled reads)."""
    import numpy as np

    g = np.random.default_rng(R * 1000 + W)
    counts = g.integers(0, 50, size=R)
    counts[g.integers(0, R)] = 0  # an empty rank
    rank_offset = np.concatenate([[0], np.cumsum(counts)])
    rows, wb = bench.rank_static_table(rank_offset, W)
    assert len(wb) == W + 1 and wb[0] == 0 and wb[-1] == len(rows)
    assert all(wb[i] <= wb[i + 1] for i in range(W))
    covered = np.zeros(int(rank_offset[-1]), np.int32)
    for w in range(W):
        for worker, hop, r, begin, n in rows[wb[w]:wb[w + 1]]:
            assert worker == w == r % W and hop == 0 and n > 0
            assert begin == rank_offset[r] and n == rank_offset[r + 1] - rank_offset[r]
            covered[begin:begin + n] += 1
    assert (covered == 1).all()


def test_whole_job_and_step_stats():
    # 3 ranks, 1.5 GB per step each, 10 steps, slowest rank 4 ms in total -> 0.4 ms per step
    v, ms = bench.whole_job(1_500_000_000, 3, 10, 4.0)
    assert ms == pytest.approx(0.4)
    assert v == pytest.approx(3 * 1.5 / 0.4e-3)
    st = bench.step_stats_us([0.003, 0.001, 0.002, 0.004, 0.005, 0.006, 0.007, 0.008, 0.009, 0.010])
    assert st == {"median": 6.0, "p10": 2.0, "p90": 10.0, "min": 1.0, "max": 10.0}
    assert bench.reduce_max_many({"a": 1, "b": 2.5}, 1) == {"a": 1.0, "b": 2.5}


def test_default_workload_is_the_largest_single_gpu_one():
    names = [w.name for w in ep_synth.sweep_workloads()] + list(ep_synth.CONFIGS)
    biggest = max(names, key=lambda n: ep_synth.get_workload(n).total_bytes())
    assert ep_synth.get_workload(bench.DEFAULT_WORKLOAD).total_bytes() == ep_synth.get_workload(biggest).total_bytes()
    assert bench.parse_args([]).config == bench.DEFAULT_WORKLOAD
    for n in bench.BLOCK_WORKLOADS + bench.LATENCY_WORKLOADS:
        ep_synth.get_workload(n)

"""Host-side bookkeeping of bench.py: the algorithmic work each workload's
number is divided by (per valid key 1152 B for bf16 rows or 656 B for FP8
rows + scales + RoPE; 2*576 + 2*512 flops per query row and valid key; a key
read once serves every head and every query token of its sequence), and the
clock summary taken from nvidia-smi samples."""
import time

import workloads as W
import bench

FLOP = 2 * 576 + 2 * 512


def test_work_of_named_workloads():
    assert bench.work_of(W.config(1)) == (2 * 256 * 1152, 2 * 256 * 64 * FLOP)
    assert bench.work_of(W.config(3)) == (1_289_370_240, 1_119_245 * 128 * FLOP)
    valid = 2048 - 102                                   # distinct top-k rows per sequence
    assert bench.work_of(W.config(4)) == (32 * valid * 656, 32 * valid * 64 * FLOP)
    causal_keys = sum(16384 - 4 + t + 1 for t in range(4))  # token t sees s_k - T + t + 1 keys
    assert bench.work_of(W.config(5)) == (32 * 16384 * 1152, 32 * causal_keys * 64 * FLOP)


def _row(ts, sm, active_mask, hw="Not Active", sw_power="Not Active"):
    return f"{ts}, 0, {sm}, 2070, 1390.5, {active_mask}, {hw}, Not Active, Not Active, {sw_power}"


def test_clock_summary_takes_samples_inside_the_timed_region():
    base = time.mktime(time.strptime("2026/12/03 01:00:00", "%Y/%m/%d %H:%M:%S"))
    text = "\n".join([
        _row("2026/12/03 01:00:00.100", 2070, "0x0"),                          # before
        _row("2026/12/03 01:00:01.000", 1700, "0x4", sw_power="Active"),
        _row("2026/12/03 01:00:01.500", 1650, "0x4", sw_power="Active"),
        "garbage line",
        _row("2026/12/03 01:00:02.000", 1750, "0x0"),
        _row("2026/12/03 01:00:05.000", 2070, "0x8", hw="Active"),             # after
    ])
    c = bench.summarise_clocks(text, base + 0.9, base + 2.0)
    assert c == {"sm_mhz": 1700.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3,
                 "in_timed_region": True}


def test_clock_summary_without_samples_inside():
    base = time.mktime(time.strptime("2026/12/03 01:00:00", "%Y/%m/%d %H:%M:%S"))
    text = "\n".join([_row("2026/12/03 01:00:00.000", 1980, "0x0"),
                      _row("2026/12/03 01:00:09.000", 2070, "0x8", hw="Active")])
    c = bench.summarise_clocks(text, base + 0.5, base + 0.6)               # nearest sample to the start
    assert c["samples"] == 1 and c["sm_mhz"] == 1980.0 and c["reasons"] == [] and not c["in_timed_region"]
    assert bench.summarise_clocks("", base, base + 1) == {"samples": 0}


def test_l2_flush_decision_of_named_workloads():
    """Workloads whose step touches less than twice the L2 (the tiny, paged
    and sparse ones) are timed with the L2 flushed before every step, and
    their `config.l2` label says so; the long ones are larger than L2."""
    l2 = 129 * 1024 * 1024
    flushed = {}
    for i in range(1, 6):
        w = W.config(i)
        kv, _ = bench.work_of(w)
        touched = bench.step_bytes(w, kv)
        flushed[i] = touched < 2 * l2
        label = bench.l2_label(touched, l2, flushed[i])
        assert ("flushed before every timed step" in label) == flushed[i]
        assert f"{touched / 1e6:.1f} MB touched" in label
    assert flushed == {1: True, 2: True, 3: False, 4: True, 5: False}
    w2 = W.config(2)
    rows = 16 * 128
    assert bench.step_bytes(w2, 75_497_472) == 75_497_472 + rows * (1152 + 1024 + 4)


def test_reference_arm_reports_the_same_config(capsys, monkeypatch):
    """`--impl reference` (the float64 oracle on the host) prints the same
    `config` object as the library's arm builds for the workload, so the two
    lines describe one benchmark."""
    import json
    import sys
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"])
    bench.main()
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    w = W.config(3)
    want, flush = bench.decode_config(w, 1, 1, bench.device_parts(0), bench.device_l2_bytes(0))
    assert line["config"] == want and not flush
    assert line["steps"] == 1 and line["warmup"] == 3 and line["dtype"] == "f64"

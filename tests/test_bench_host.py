"""Host logic of bench.py that needs no GPU: the clock record around the
timed region, the per-workload DRAM traffic lookup, and the workload
description both arms print."""
import argparse
import json
import os

import bench
from tree_speculative_decoding_jt_gb300 import workloads as wk


def _line(sm, mx=2070, reasons=("Not Active",) * 4):
    return f"0, {sm}, {mx}, 500.0, 0x0, " + ", ".join(reasons)


def test_clock_summary_keeps_the_region_and_its_neighbours():
    c = bench.ClockSampler(0)
    c.t_start, c.t_end = 10.0, 10.02   # a region much shorter than a sample period
    c.lines = [(9.5, _line(900)), (9.95, _line(2070)), (10.05, _line(2055)), (10.5, _line(800)),
               (10.07, "garbage")]
    s = c.summary()
    assert s["samples"] == 2 and s["samples_total"] == 4
    assert s["sm_mhz"] == (2070 + 2055) / 2 and s["sm_max_mhz"] == 2070
    assert s["reasons"] == []


def test_clock_summary_reports_throttle_reasons_and_empty_windows():
    c = bench.ClockSampler(0)
    c.t_start, c.t_end = 1.0, 2.0
    c.lines = [(1.5, _line(1800, reasons=("Not Active", "Not Active", "Not Active", "Active")))]
    assert c.summary()["reasons"] == ["sw_power_cap"]
    c.lines = [(5.0, _line(2070))]
    s = c.summary()
    assert s["samples"] == 0 and s["sm_mhz"] is None and "note" in s


def test_traffic_is_looked_up_per_workload_and_source(tmp_path, monkeypatch):
    kern = tmp_path / "k.cu"
    kern.write_text("kernel v1")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.source_hash(["k.cu"])
    entries = [{"workload": "a", "kernel": "k1", "source_hash": h, "dram_bytes_per_launch": 111},
               {"workload": "a", "kernel": "k2", "source_hash": h, "dram_bytes_per_launch": 333},
               {"workload": "b", "kernel": "k1", "source_hash": "0" * 16, "dram_bytes_per_launch": 222}]
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({"entries": entries}))
    assert bench.profiled_traffic("k.cu", "a", "k1") == 111
    assert bench.profiled_traffic("k.cu", "a", "k2") == 333   # per kernel
    assert bench.profiled_traffic("k.cu", "a", "k3") is None
    assert bench.profiled_traffic("k.cu", "b") is None        # taken on another source
    assert bench.profiled_traffic("k.cu", "c") is None        # no capture of this workload
    kern.write_text("kernel v2")
    assert bench.profiled_traffic("k.cu", "a", "k1") is None  # the kernel changed since


def test_committed_traffic_entries_are_keyed():
    p = os.path.join(bench.ROOT, "profiles", "traffic.json")
    d = json.load(open(p))
    names = {c["name"] for c in wk.CONFIGS.values()}
    for e in d["entries"]:
        assert e["workload"] in names and len(e["source_hash"]) == 16 and e["dram_bytes_per_launch"] > 0
        assert e["kernel"] in ("tree_attn_tc_kernel<128>", "tree_attn_pair_kernel")


def test_both_arms_describe_the_same_workload():
    args = argparse.Namespace(alpha=0.0, adaptive=False, stochastic=False, flush_mb=512)
    wl = wk.make(3, with_kv=False, with_draft=False)
    a = bench.config_dict(args, wl, 1)
    b = bench.config_dict(args, wk.make(3, with_kv=False, with_draft=False), 1)
    assert a == b and a["workload"] == wk.CONFIGS[3]["name"] and a["nseq"] == 16


def test_split_mode_rule_matches_the_workloads():
    """bench.py's launch count follows the library's plan: split mode only
    when the units are at most half the SMs (batch 1)."""
    sms = 152
    assert bench.attn_split_mode(1, 32, 8, 256, 273, sms)          # config 2: 32 units
    assert not bench.attn_split_mode(32, 32, 8, 64, 2053, sms)     # config 4: 256 units
    assert not bench.attn_split_mode(16, 32, 8, 256, 514, sms)     # config 3: 512 units at max_tree
    assert not bench.attn_split_mode(1, 32, 8, 256, 2, sms)        # too few key tiles to split
    # the CTA-pair kernel has one work slot per two SMs
    assert bench.attn_split_mode(1, 32, 8, 256, 273, sms // 2)     # config 2: 32 units, 2 splits
    assert bench.attn_split_mode(2, 32, 8, 256, 273, sms)           # 64 units: split on 152 slots,
    assert not bench.attn_split_mode(2, 32, 8, 256, 273, sms // 2)  # not on 76


def test_kernel_choice_rule(monkeypatch):
    """bench.py mirrors the library's choice of attention kernel."""
    monkeypatch.delenv("JT_ATTN_KERNEL", raising=False)
    assert bench.attn_kernel(128, 32, 8, 64) == "pair"      # config 4: one query-tile pair per head
    assert bench.attn_kernel(128, 32, 8, 256) == "single"   # configs 2, 3, 5: four pairs per head
    assert bench.attn_kernel(64, 32, 8, 64) == "single"     # head dim 64: single-SM kernel only
    monkeypatch.setenv("JT_ATTN_KERNEL", "single")
    assert bench.attn_kernel(128, 32, 8, 64) == "single"
    monkeypatch.setenv("JT_ATTN_KERNEL", "pair")
    assert bench.attn_kernel(128, 32, 8, 256) == "pair"

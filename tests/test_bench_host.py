"""Host logic of bench.py that needs no GPU: the profiled-traffic lookup.

`roofline.traffic` in the bench line comes from profiles/traffic.json only while the
kernel's sources hash to the digest recorded with the counters; a stale or missing entry
must give null, never an old number.
"""
from __future__ import annotations

import hashlib
import importlib.util
import json
import os
import sys
import types

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture()
def bench(monkeypatch, tmp_path):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    csrc = tmp_path / "quantized_routed_expert_sigmoid_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "k.cu").write_bytes(b"kernel source v1\n")
    digest = hashlib.sha1(b"kernel source v1\n").hexdigest()
    entries = {
        "k_kernel decode": {"dram_bytes_per_launch": 123, "sources": ["k.cu"], "sources_sha1": digest},
        "k_kernel stack T=64": {"dram_bytes_per_launch": 456, "sources": ["k.cu"], "sources_sha1": digest},
    }
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps(entries))
    monkeypatch.setattr(mod, "ROOT", str(tmp_path))
    return mod, csrc


def test_current_digest_gives_the_profiled_bytes(bench):
    mod, _ = bench
    assert mod.profiled_traffic("k_kernel", types.SimpleNamespace(workload="decode", tokens=0)) == 123
    assert mod.profiled_traffic("k_kernel", types.SimpleNamespace(workload="stack", tokens=64)) == 456


def test_missing_entry_or_other_T_gives_none(bench):
    mod, _ = bench
    assert mod.profiled_traffic("k_kernel", types.SimpleNamespace(workload="prefill", tokens=0)) is None
    assert mod.profiled_traffic("k_kernel", types.SimpleNamespace(workload="stack", tokens=8)) is None
    assert mod.profiled_traffic("other_kernel", types.SimpleNamespace(workload="decode", tokens=0)) is None


def test_changed_source_gives_none(bench):
    mod, csrc = bench
    (csrc / "k.cu").write_bytes(b"kernel source v2\n")
    assert mod.profiled_traffic("k_kernel", types.SimpleNamespace(workload="decode", tokens=0)) is None


def test_clock_samples_inside_the_timed_region(bench):
    # only the samples taken while the timed steps ran count; with none inside, all of them
    mod, _ = bench
    lines = [
        "2026/12/02 10:00:00.000, 0, 1200, 2070, 150.0, Active, Not Active, Not Active, Not Active, Not Active",
        "2026/12/02 10:00:00.200, 0, 2070, 2070, 900.0, Active, Not Active, Not Active, Not Active, Active",
        "2026/12/02 10:00:00.400, 0, 2055, 2070, 950.0, Active, Not Active, Not Active, Not Active, Active",
        "2026/12/02 10:00:00.600, 0, 1500, 2070, 200.0, Active, Active, Not Active, Not Active, Not Active",
        "garbage line",
    ]
    rows = mod.parse_clock_samples(lines)
    assert len(rows) == 4
    t0 = rows[1][0] - 0.05
    t1 = rows[2][0] + 0.05
    s = mod.summarize_clocks(rows, t0, t1)
    assert s["samples"] == 2 and s["sm_mhz"] == (2070 + 2055) / 2 and s["reasons"] == ["sw_power_cap"]
    assert s["window"] == "timed region"
    s_all = mod.summarize_clocks(rows, t1 + 10.0, t1 + 11.0)
    assert s_all["samples"] == 4 and "hw_slowdown" in s_all["reasons"] and s_all["window"].startswith("whole run")
    assert mod.summarize_clocks([], None, None) is None


def test_launch_count_per_layer(bench):
    mod, _ = bench
    import synth
    # the three chained decode kernels
    assert mod.launches_per_layer(synth.DECODE, 1, path="decode_chain") == 3
    # prefill T=4096, as listed by ncu: router split, router logits, top-k, permute (two
    # launches above 1024 pairs), fp16 copy of x, token-block list, gate/up, down, combine
    assert mod.launches_per_layer(synth.DECODE, 4096, path="tensor") == 10
    # stack at T=64 on the GEMV path: RMSNorm, logits, top-k, permute, gate/up, down, combine
    assert mod.launches_per_layer(synth.DECODE, 64, stack=True, path="gemv") == 7
    # DeepSeek-shaped T=2 on the GEMV path: + the shared expert's gate/up and down
    assert mod.launches_per_layer(synth.DEEPSEEK, 2, path="gemv") == 8
    # DeepSeek-shaped T=512 on the tensor cores: 4096 pairs, router on tcgen05, shared expert
    assert mod.launches_per_layer(synth.DEEPSEEK, 512, path="tensor") == 12


def test_algorithmic_bytes_of_the_decode_layer(bench):
    mod, _ = bench
    import numpy as np
    import synth
    # T = 1 with 8 distinct experts: 8 x 2,654,208 B of Q4_K rows, the fp32 router (1 MiB),
    # the bf16 token in and the fp32 row out
    offs = np.array([0] * 5 + list(range(1, 9)) + [8] * 116)
    assert len(offs) == 129
    total, gu, u = mod.algorithmic_bytes(synth.DECODE, 1, offs)
    assert u == 8
    assert synth.bytes_per_expert(synth.DECODE) == 2654208
    assert total == 8 * 2654208 + 128 * 2048 * 4 + 2048 * 2 + 2048 * 4
    # gate/up: 2 x 768 rows of 8 Q4_K blocks per chosen expert, the token, and h (fp32, k x I)
    assert gu == 8 * 2 * 768 * 8 * 144 + 2048 * 2 + 8 * 768 * 4
    # the DeepSeek-shaped layer: a routed expert of 24,772,608 B, a Q8_0 shared expert of 46.8 MB
    assert synth.bytes_per_expert(synth.DEEPSEEK) == 24772608
    assert synth.shared_bytes(synth.DEEPSEEK) == 46792704

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

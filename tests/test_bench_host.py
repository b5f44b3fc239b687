"""Host-side parts of bench.py on CPU: the reference arm's JSON line (the
oracle timed on the host, here on a small slice of the same workload), the
gating of the committed DRAM-traffic figure by the kernel source digest, and
the build and host metadata the result line carries."""
import argparse
import io
import json
import os
from contextlib import redirect_stdout

import pytest

import bench
import synth


def test_reference_arm_prints_one_valid_line(monkeypatch):
    small = synth.merge_u64(seed=2, m=1 << 16, n=1 << 16)
    monkeypatch.setattr(bench.synth, "merge_u64", lambda: small)
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    out = io.StringIO()
    with redirect_stdout(out):
        bench.run_reference(argparse.Namespace(gpus=1, steps=2, warmup=1, impl="reference"))
    lines = [ln for ln in out.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["steps"] == 2 and d["warmup"] == 1
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["config"] == bench.headline_config(1 << 16, 1 << 16)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1 and cb["value"] == d["value"]
    assert cb["host_cores"] == os.cpu_count() and "sample" in cb
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_do_nothing(monkeypatch):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    out = io.StringIO()
    with redirect_stdout(out):
        bench.run_reference(argparse.Namespace(gpus=2, steps=2, warmup=1, impl="reference"))
    assert out.getvalue() == ""


def test_traffic_is_reported_only_for_the_source_it_was_taken_on(monkeypatch):
    key = "merge_tile_kernel<u64,payload,11,2,1>"
    with open(os.path.join(bench.ROOT, "profiles", "ncu_traffic.json")) as f:
        ent = json.load(f)[key]
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: ent["source_digest"])
    assert bench.ncu_traffic(key) == pytest.approx(float(ent["dram_bytes_per_launch"]))
    monkeypatch.setattr(bench, "kernel_source_digest", lambda: "0" * 16)
    assert bench.ncu_traffic(key) is None
    assert bench.ncu_traffic("no such kernel") is None


def test_headline_config_names_the_workload_only():
    c = bench.headline_config(1 << 26, 1 << 26)
    assert c["m"] == c["n"] == 1 << 26 and c["key"] == "u64" and c["payload"] == "u32"
    assert "2^26" in c["workload"]
    assert not {"model", "global_batch", "seq_len", "items_per_thread", "tile"} & set(c)


def test_build_and_host_metadata():
    b = bench.build_info()
    assert "-gencode arch=compute_103a,code=sm_103a" in b["nvcc_flags"]
    assert bench.ROOT not in b["nvcc_flags"]      # paths relative to the tree
    assert len(b["source_digest"]) == 16
    h = bench.host_info()
    assert h["cpu_count"] == os.cpu_count() and h["machine"]


def test_peak_comes_from_the_measured_file_when_present(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.hbm_peak() == (bench.FALLBACK_HBM_GBS, "fallback")
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 6692.5}))
    assert bench.hbm_peak() == (6692.5, "measured")

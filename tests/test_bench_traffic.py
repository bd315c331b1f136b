"""The bench's DRAM-traffic record on CPU.

The bench line's `roofline.traffic` comes from committed ncu counters. It may be
reported only while the kernel's sources are the ones the counters were taken on,
so a kernel changed after its capture reads null instead of a stale figure.
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402

SRC = "two_stage_kv_snapkv_gb300/csrc/rkv_decode.cu"


def _record(tmp_path, sha):
    p = tmp_path / "traffic.json"
    p.write_text(json.dumps({"wl": {"hsa_step": {"bytes_per_launch": 1234, "source_file": SRC, "source_sha": sha}}}))
    return str(p)


def test_an_entry_matching_the_sources_is_reported(tmp_path):
    path = _record(tmp_path, bench._source_sha(SRC))
    assert bench.recorded_traffic("wl", "hsa_step", path) == 1234


def test_a_stale_or_missing_entry_reads_none(tmp_path):
    path = _record(tmp_path, "0" * 16)
    assert bench.recorded_traffic("wl", "hsa_step", path) is None
    assert bench.recorded_traffic("wl", "snap_compact", path) is None
    assert bench.recorded_traffic("other", "hsa_step", path) is None
    assert bench.recorded_traffic("wl", "hsa_step", str(tmp_path / "absent.json")) is None


def test_the_source_sha_covers_the_shared_headers(tmp_path, monkeypatch):
    # a change in a header every kernel includes changes every kernel's code
    base = bench._source_sha(SRC)
    hdr = tmp_path / "h.cuh"
    hdr.write_text("// a header\n")
    monkeypatch.setattr(bench, "KERNEL_HEADERS", (*bench.KERNEL_HEADERS, str(hdr)))
    assert bench._source_sha(SRC) != base


def test_the_committed_record_names_real_sources_and_kernels():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        rec = json.load(f)
    entries = [(w, k, e) for w, ks in rec.items() if isinstance(ks, dict) for k, e in ks.items()]
    assert entries
    for w, k, e in entries:
        assert os.path.exists(os.path.join(ROOT, e["source_file"])), (w, k)
        assert isinstance(e["bytes_per_launch"], int) and e["bytes_per_launch"] > 0, (w, k)
        assert len(e["source_sha"]) == 16, (w, k)

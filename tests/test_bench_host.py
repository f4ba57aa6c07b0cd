"""bench.py host logic that needs no GPU: the kernel-source hash that gates the
recorded ncu traffic, and the lookup that uses it."""
import json
import os
import shutil

import bench

SRCS = ("pa_decode.cu", "pa_device.cuh", "pa_fp8.cuh")


def _tree(tmp_path):
    csrc = tmp_path / "paged_kv_cache_294_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for f in SRCS:
        shutil.copy(os.path.join(bench.ROOT, "paged_kv_cache_294_gb300", "csrc", f), csrc / f)
    (tmp_path / "profiles").mkdir()
    return csrc


def test_hash_ignores_comments_and_blank_lines_but_not_code(tmp_path, monkeypatch):
    csrc = _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h0 = bench.kernel_source_hash()
    p = csrc / "pa_decode.cu"
    src = p.read_text()
    p.write_text("// a new comment\n\n/* and a\n   block comment */\n" + src.replace("\n", "  // trailing\n", 3))
    assert bench.kernel_source_hash() == h0
    p.write_text(src.replace("atom.acq_rel.gpu", "atom.relaxed.gpu", 1))
    assert bench.kernel_source_hash() != h0


def test_traffic_reported_only_for_the_recorded_kernel_and_split_count(tmp_path, monkeypatch):
    _tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    h = bench.kernel_source_hash()
    rec = {"8b": {"kernel_hash": h, "splits": 8, "dram_bytes_per_launch": 5.0e8}}
    (tmp_path / "profiles" / "decode_traffic.json").write_text(json.dumps(rec))
    assert bench.ncu_traffic("8b", 8) == 5.0e8
    assert bench.ncu_traffic("8b", 6) is None          # another split count
    assert bench.ncu_traffic("70b", 8) is None         # no record
    rec["8b"]["kernel_hash"] = "0" * 16                  # taken on other code
    (tmp_path / "profiles" / "decode_traffic.json").write_text(json.dumps(rec))
    assert bench.ncu_traffic("8b", 8) is None


def test_committed_traffic_is_one_capture_with_sane_ratios():
    """All workloads' records come from one kernel source, and each launch moved
    at least its algorithmic bytes and not much more (no re-reads)."""
    with open(os.path.join(bench.ROOT, "profiles", "decode_traffic.json")) as f:
        rec = json.load(f)
    assert len({e["kernel_hash"] for e in rec.values()}) == 1
    for w, e in rec.items():
        assert 1.0 <= e["dram_bytes_per_launch"] / e["algorithmic_bytes"] < 1.05, w

"""The bench reports the dominant kernel's DRAM traffic from a committed ncu
summary only while that summary was taken on the current kernel sources
(CPU only: the summaries are rewritten into a temporary tree)."""
import hashlib
import os

import bench


def _source_hash(files):
    h = hashlib.sha256()
    for f in files:
        h.update(open(f, "rb").read())
    return h.hexdigest()


def _with_profiles(monkeypatch, tmp_path, text, name):
    prof = tmp_path / "profiles"
    prof.mkdir(exist_ok=True)
    (prof / name).write_text(text)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))


def test_traffic_only_for_the_current_sources(monkeypatch, tmp_path):
    cur = _source_hash(bench.GEMM_SRC)
    text = f"kernel_source_sha256: {cur}\ndram_bytes_per_launch: 12.5e9\n"
    _with_profiles(monkeypatch, tmp_path, text, "expert_gate_up_mai-base-1.txt")
    assert bench.profiled_traffic("mai-base-1") == 12.5e9
    stale = text.replace(cur, "0" * 64)
    _with_profiles(monkeypatch, tmp_path, stale, "expert_gate_up_mai-base-1.txt")
    assert bench.profiled_traffic("mai-base-1") is None


def test_missing_summary_gives_no_traffic(monkeypatch, tmp_path):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("mai-base-1") is None
    assert bench.profiled_traffic("tiny") is None
    assert os.path.isdir(tmp_path)

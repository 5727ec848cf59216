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


def test_gate_up_algorithmic_bytes_are_the_touched_weights():
    """The dominant kernel's algorithmic bytes count the gate and up weights of
    the experts that got tokens only; z and h traffic is reported as built."""
    from mixture_experts_layer_router_gb300 import synth
    c = synth.CONFIGS["mai-base-1"]
    flops, algo, built = bench.gate_up_work(c, 512)
    assert algo == 512 * 2 * 10240 * 3072 * 2  # 64.42 GB
    assert built == algo + c.T * c.k * (3072 + 10240) * 2
    assert flops == 2 * c.T * c.k * 3072 * 2 * 10240
    _, algo8, _ = bench.gate_up_work(c, 300, eb=1)
    assert algo8 == 300 * 2 * 10240 * 3072


def test_layer_roofline_peak_follows_the_power_cap():
    from mixture_experts_layer_router_gb300 import synth
    c = synth.CONFIGS["mid"]
    peaks = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
    a = bench.layer_roofline(c, 64, 1.0, peaks, "measured", False, False, capped=False)
    b = bench.layer_roofline(c, 64, 1.0, peaks, "measured", False, False, capped=True)
    assert a["flops"] == c.T * bench.layer_flops_per_token(c)
    assert abs(a["tc_ms"] * 1900.0 - b["tc_ms"] * 1700.0) < 1e-9 * a["tc_ms"] * 1900.0
    assert a["frac"] == max(a["tc_ms"], a["hbm_ms"]) and "burst" in a["tensor_peak"]

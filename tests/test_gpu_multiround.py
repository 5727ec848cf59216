"""The multi-round fixed-capacity expert schedule on the GPU: the schedule
bit for bit against the oracle's, the layer output against the oracle's
layer routed from the GPU logits, and bitwise equal to the one-pass forward
(no slot is dropped; every slot's expert rows are computed by the same
kernels with the same arithmetic)."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_router_gb300 import capi, synth
import gpu_helpers as gh
from oracle import latentmoe_ref as ref
from oracle import multiround as mr

pytestmark = pytest.mark.gpu


def _layer(name, seed=0, fp8=False):
    cfg = synth.CONFIGS[name]
    w = synth.make_weights(cfg, seed, "cuda")
    x = synth.make_x(cfg, seed, "cuda")
    return cfg, w, x, gh.make_layer(cfg, w, fp8=fp8)


_ORACLE_Y = {}


def _oracle_y(name, seed, w, x, logits):
    """The oracle's layer output routed from the GPU logits, once per workload."""
    key = (name, seed)
    if key not in _ORACLE_Y:
        cfg = synth.CONFIGS[name]
        _ORACLE_Y[key] = (logits.clone(), ref.forward(gh.f64(x), gh.oracle_weights(w), cfg.k,
                                                      logits=gh.f64(logits))["y"])
    L0, y = _ORACLE_Y[key]
    assert torch.equal(L0, logits)  # the same routing as the cached oracle run
    return y


def _forward(layer, x, fp8):
    if fp8:
        layer.set_fp8_scales([0.02, 0.01])
    y = layer.forward(x).clone()
    torch.cuda.synchronize()
    return y


@pytest.mark.parametrize("name,C,G", [("imbalanced", 48, 8), ("imbalanced", 16, 4),
                                      ("imbalanced", 300, 64), ("mid", 200, 1),
                                      ("mid", 10, 64), ("tiny", 3, 4)])
def test_schedule_matches_oracle_and_output_matches_one_pass(name, C, G):
    cfg, w, x, layer = _layer(name, seed=1)
    y0 = _forward(layer, x, False)
    counts = layer.get_routing(cfg.T, "cuda")["counts"].cpu().numpy().astype(np.int64)
    layer.set_capacity(C, G)
    y1 = _forward(layer, x, False)
    assert layer.status() == 0
    got = layer.rounds()
    want = mr.schedule(counts, cfg.E, C, G)
    assert got["left_over"] == 0
    assert got["needed"] == want["R"]
    take = got["take"].cpu().numpy()
    assert np.array_equal(take[:want["R"]], want["take"])
    assert not take[want["R"]:].any()
    assert torch.equal(y0, y1)
    L1 = layer.get_routing(cfg.T, "cuda")["logits"]
    gh.assert_y_close(y1, _oracle_y(name, 1, w, x, L1), what=f"{name} C={C} G={G}")


@pytest.mark.parametrize("pairs", [True, False])
def test_e4m3_rounds_equal_one_pass(pairs):
    cfg, w, x, layer = _layer("imbalanced", seed=2, fp8=True)
    layer.set_sm_pairs(pairs)
    y0 = _forward(layer, x, True)
    s0 = layer.fp8_state()
    layer.set_capacity(32, 8)
    y1 = _forward(layer, x, True)
    s1 = layer.fp8_state()
    assert layer.status() == 0 and layer.rounds()["needed"] > 1
    assert torch.equal(y0, y1)
    assert s0["last_amax"] == s1["last_amax"]  # same h values, same maxima


def test_too_few_rounds_sets_the_status():
    cfg, w, x, layer = _layer("imbalanced", seed=3)
    counts = None
    layer.forward(x)
    counts = layer.get_routing(cfg.T, "cuda")["counts"].cpu().numpy()
    want = mr.schedule(counts, cfg.E, 16, 4)
    assert want["R"] > 2
    layer.set_capacity(16, 4, 2)
    layer.forward(x)
    got = layer.rounds()
    assert got["launched"] == 2 and got["left_over"] == int(want["take"][2:].sum())
    assert layer.status() == capi.STATUS_ROUNDS
    assert layer.status() == 0  # read and cleared


def test_worst_case_rounds_launch_count_and_errors():
    cfg, w, x, layer = _layer("tiny", seed=4)
    C, G = 5, 4
    layer.set_capacity(C, G)
    per = cfg.T * min(cfg.k, G)
    launched_want = -(-per // (G * C))
    n0 = layer.launch_count()
    layer.forward(x)
    got = layer.rounds()
    assert got["launched"] == launched_want
    assert layer.launch_count() - n0 == 7 + 1 + 2 * launched_want - 2
    for bad in [(-1, 1, 0), (4, 0, 0), (4, cfg.E + 1, 0), (4, 2, -1)]:
        with pytest.raises(capi.LatentMoEError):
            layer.set_capacity(*bad)
    layer.set_capacity(0)
    with pytest.raises(capi.LatentMoEError):
        layer.rounds()


def test_all_e4m3_rounds_and_replay_equal_one_pass():
    """All-E4M3 GEMMs with the capacity schedule, and router replay of the
    same choices and gates: every variant reproduces the one-pass forward
    bit for bit (same codes, same scales, same fp32 expert outputs)."""
    cfg = synth.LayerConfig("tiny-shared", T=300, d=256, l=512, E=8, k=3, F=512, Fs=256)
    w = synth.make_weights(cfg, 11, "cuda")
    x = synth.make_x(cfg, 11, "cuda")
    layer = gh.make_layer(cfg, w, fp8=True, fp8_dense=True)
    scales = [0.02, 0.01, 0.01, 0.005, 0.01]
    layer.set_fp8_scales(scales)
    y0 = layer.forward(x).clone()
    r = layer.get_routing(cfg.T, "cuda")
    idx, gates = r["idx"].clone(), r["gates"].clone()
    layer.set_capacity(40, 4)
    layer.set_fp8_scales(scales)
    y1 = layer.forward(x).clone()
    assert layer.rounds()["needed"] > 1
    layer.set_fp8_scales(scales)
    y2 = layer.forward_routed(x, idx, gates).clone()
    layer.set_capacity(0)
    layer.set_fp8_scales(scales)
    y3 = layer.forward_routed(x, idx).clone()
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(y0, y1) and torch.equal(y0, y2) and torch.equal(y0, y3)

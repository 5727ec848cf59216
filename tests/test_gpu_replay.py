"""Router replay on the GPU (latentmoe_forward_routed) against the oracle."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_router_gb300 import capi, synth
import gpu_helpers as gh
from oracle import latentmoe_ref as ref

pytestmark = pytest.mark.gpu


def _setup(name="tiny", seed=0, renorm=False):
    cfg = synth.CONFIGS[name]
    w = synth.make_weights(cfg, seed, "cuda")
    x = synth.make_x(cfg, seed, "cuda")
    return cfg, w, x, gh.make_layer(cfg, w, renorm=renorm)


@pytest.mark.parametrize("renorm", [False, True])
def test_replaying_own_choices_reproduces_forward(renorm):
    cfg, w, x, layer = _setup("mid", 3, renorm)
    y = layer.forward(x).clone()
    r = layer.get_routing(cfg.T, "cuda")
    y_gates = layer.forward_routed(x, r["idx"], r["gates"]).clone()
    y_nogates = layer.forward_routed(x, r["idx"]).clone()
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(y_gates, y)
    assert torch.equal(y_nogates, y)


def test_replay_foreign_choices_matches_oracle():
    cfg, w, x, layer = _setup("tiny", 5)
    rng = np.random.default_rng(9)
    idx = np.stack([rng.permutation(cfg.E)[:cfg.k] for _ in range(cfg.T)]).astype(np.int32)
    gates = rng.uniform(0.05, 0.6, (cfg.T, cfg.k)).astype(np.float32)
    W = gh.oracle_weights(w)
    xs = gh.f64(x)
    for g in (gates, None):
        yt = layer.forward_routed(x, torch.from_numpy(idx).cuda(),
                                  None if g is None else torch.from_numpy(g).cuda())
        r = layer.get_routing(cfg.T, "cuda")
        torch.cuda.synchronize()
        assert layer.status() == 0
        ora = ref.forward_routed(xs, W, idx, None if g is None else g.astype(np.float64),
                                 logits=None if g is not None else gh.f64(r["logits"]))
        gh.assert_routing_equal(r, {**ora, "idx": idx}, cfg.T, cfg.k)
        gh.assert_y_close(yt, ora["y"])


def test_replay_with_out_of_range_ids_drops_those_slots():
    cfg, w, x, layer = _setup("tiny", 6)
    rng = np.random.default_rng(2)
    idx = np.stack([rng.permutation(cfg.E)[:cfg.k] for _ in range(cfg.T)]).astype(np.int32)
    gates = rng.uniform(0.05, 0.6, (cfg.T, cfg.k)).astype(np.float32)
    bad = [(3, 0, cfg.E), (10, 1, -1), (77, 1, cfg.E + 100)]
    idx_bad = idx.copy()
    for t, j, e in bad:
        idx_bad[t, j] = e
    y = layer.forward_routed(x, torch.from_numpy(idx_bad).cuda(), torch.from_numpy(gates).cuda())
    torch.cuda.synchronize()
    assert layer.status() & capi.STATUS_BAD_EXPERT
    # oracle: the same choices with those slots' gates set to zero
    g0 = gates.astype(np.float64).copy()
    for t, j, _ in bad:
        g0[t, j] = 0.0
    ora = ref.forward_routed(gh.f64(x), gh.oracle_weights(w), idx, g0)
    gh.assert_y_close(y, ora["y"])
    # the handle recovers: a normal forward afterwards is clean
    layer.forward(x)
    torch.cuda.synchronize()
    assert layer.status() == 0


def test_replay_argument_errors():
    cfg, w, x, layer = _setup("tiny", 7)
    lib = capi.load()
    y = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    idx = torch.zeros((cfg.T, cfg.k), dtype=torch.int32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert lib.latentmoe_forward_routed(layer.handle, x.data_ptr(), None, None, y.data_ptr(),
                                        cfg.T, s) == capi.ERR_INVALID_ARG
    assert lib.latentmoe_forward_routed(layer.handle, x.data_ptr(), idx.data_ptr() + 2, None,
                                        y.data_ptr(), cfg.T, s) == capi.ERR_INVALID_ARG

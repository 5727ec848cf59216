"""The seeded workloads have the structure the configs promise (CPU, oracle routing)."""
import numpy as np
import torch

from mixture_experts_layer_router_gb300 import synth
from oracle import latentmoe_ref as ref


def _route(cfg):
    x = synth.make_x(cfg, 0, "cpu").float().numpy().astype(np.float64)
    w = synth.make_weights(cfg, 0, "cpu", experts=False)
    b = None if w["b_r"] is None else w["b_r"].numpy().astype(np.float64)
    L = ref.router_logits(x, w["w_r"].float().numpy().astype(np.float64), b)
    return ref.route(L, cfg.E, cfg.k)


def test_imbalanced_loads():
    cfg = synth.CONFIGS["imbalanced"]
    r = _route(cfg)
    counts = r["counts"]
    assert counts.sum() == cfg.slots
    assert counts.max() > 0.10 * cfg.slots      # one expert takes more than 10% of slots
    assert (counts == 0).sum() >= 3             # several experts get no token


def test_mid_loads_near_uniform():
    cfg = synth.CONFIGS["mid"]
    r = _route(cfg)
    counts = r["counts"]
    assert (counts > 0).all()
    assert counts.max() < 3 * cfg.slots / cfg.E


def test_generator_is_seeded_and_bf16():
    cfg = synth.CONFIGS["tiny"]
    a = synth.make_weights(cfg, 0, "cpu")
    b = synth.make_weights(cfg, 0, "cpu")
    c = synth.make_weights(cfg, 1, "cpu")
    for key in ("w_r", "w_dn", "w_g", "w_d", "w_up"):
        assert a[key].dtype == torch.bfloat16
        assert torch.equal(a[key], b[key])
        assert not torch.equal(a[key], c[key])
    # one expert regenerates on its own
    wg, wu, wd = synth.make_expert(cfg, 5, 0, "cpu")
    assert torch.equal(wg, a["w_g"][5]) and torch.equal(wd, a["w_d"][5])


def test_zipf_bias_formula_inputs():
    b = synth.zipf_router_bias(64, 123)
    ranks = np.exp(-b.numpy().astype(np.float64) / 1.8)  # b = -1.8 ln(rank)
    assert np.allclose(np.sort(ranks), np.arange(1, 65), rtol=1e-5)

"""Load-balancing statistics and the selection-only bias on the GPU, against
the oracle. Expert choices under a selection bias are compared with the
ranking key L + b formed in fp32, the precision the kernels decide in."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_router_gb300 import capi, synth
import gpu_helpers as gh
from oracle import latentmoe_ref as ref

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny", "mid", "imbalanced"])
def test_lbl_stats_match_oracle(name):
    cfg = synth.CONFIGS[name]
    w = synth.make_weights(cfg, 2, "cuda")
    x = synth.make_x(cfg, 2, "cuda")
    layer = gh.make_layer(cfg, w)
    layer.forward(x)
    r = layer.get_routing(cfg.T, "cuda")
    ps, cn = layer.lbl_stats("cuda")
    ps2, cn2 = layer.lbl_stats("cuda")
    torch.cuda.synchronize()
    counts, psum = ref.lbl_stats(gh.f64(r["logits"]), r["idx"].cpu().numpy(), cfg.E)
    assert np.array_equal(cn.cpu().numpy(), counts)
    np.testing.assert_allclose(gh.f64(ps), psum, rtol=2e-5, atol=1e-6)
    assert abs(float(ps.double().sum()) - cfg.T) <= 1e-3 * cfg.T
    assert torch.equal(ps, ps2) and torch.equal(cn, cn2)


@pytest.mark.parametrize("name,renorm", [("tiny", False), ("mid", True), ("imbalanced", False)])
def test_selection_bias_matches_oracle(name, renorm):
    cfg = synth.CONFIGS[name]
    w = synth.make_weights(cfg, 3, "cuda")
    x = synth.make_x(cfg, 3, "cuda")
    b = synth.zipf_router_bias(cfg.E, 77) * 0.5
    w["b_r"] = b.cuda()
    layer = capi.LatentMoE(cfg.d, cfg.l, cfg.E, cfg.k, cfg.F, cfg.Fs, max_tokens=cfg.T,
                           renorm=renorm, select_bias=True)
    layer.load_weights(w)
    y = layer.forward(x)
    r = layer.get_routing(cfg.T, "cuda")
    torch.cuda.synchronize()
    assert layer.status() == 0
    W = gh.oracle_weights({**w, "b_r": None})
    xs = gh.f64(x)
    L32 = r["logits"].cpu().numpy()
    # exported logits are unbiased
    assert np.abs(L32.astype(np.float64) - ref.router_logits(xs, W.w_r)).max() <= gh.LOGIT_MAX_ABS
    key32 = (L32 + b.numpy()[None, :]).astype(np.float32)
    ora = ref.forward(xs, W, cfg.k, renorm=renorm, logits=L32.astype(np.float64),
                      select_logits=key32)
    gh.assert_routing_equal(r, ora, cfg.T, cfg.k)
    gh.assert_y_close(y, ora["y"])
    # the bias did move choices (the test would be vacuous otherwise)
    plain = ref.route(L32.astype(np.float64), cfg.E, cfg.k)
    assert not np.array_equal(plain["idx"], ora["idx"])
    # the standalone routing kernel decides the same, bitwise, from the same logits
    alone = layer.route_from_logits(r["logits"].clone())
    torch.cuda.synchronize()
    for key in ("idx", "gates", "counts", "offsets", "perm", "pos"):
        assert torch.equal(r[key], alone[key]), key


def test_bias_flags_are_exclusive():
    gh.lib()
    with pytest.raises(capi.LatentMoEError):
        capi.LatentMoE(256, 128, 16, 2, 256, 0, max_tokens=8, router_bias=True, select_bias=True)

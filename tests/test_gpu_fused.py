"""Both expert GEMMs in one launch (latentmoe_set_expert_fusion) against the
two launches and the oracle (GPU).

The fused kernel runs the same tiles with the same MMAs in another order and
hands h from the gate+up tiles to the down tiles through completion counts,
so the layer output must be bitwise the one of the two launches; and it must
stay so over consecutive forwards (the counts are reset by the kernel
itself), with and without programmatic launch, in bf16 and E4M3."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_router_gb300 import capi, synth
import gpu_helpers as gh
from oracle import latentmoe_ref as ref

pytestmark = pytest.mark.gpu

# F % 256 == 0 and l % 512 == 0: the fused kernel's shapes. "small" has 8
# experts of ~256 slots (one or two token chunks), "skewed" a router bias that
# puts more than 512 slots on some experts (wide down tiles, several gate+up
# chunks) and none on others.
SMALL = synth.LayerConfig("fused-small", T=1024, d=512, l=512, E=8, k=2, F=512,
                          router_std=0.02)
SKEWED = synth.LayerConfig("fused-skewed", T=2048, d=512, l=1024, E=16, k=4, F=768,
                           router_std=0.02, zipf_bias=True)
SHARED = synth.LayerConfig("fused-shared", T=512, d=1024, l=512, E=8, k=3, F=256, Fs=512)


def _forwards(layer, x, fused, n=3, scales=None):
    layer.set_expert_fusion(1 if fused else 0)
    outs = []
    for _ in range(n):
        if scales is not None:
            layer.set_fp8_scales(scales)
        outs.append(layer.forward(x).clone())
    torch.cuda.synchronize()
    assert layer.status() == 0
    return outs


@pytest.mark.parametrize("cfg", [SMALL, SKEWED, SHARED, synth.CONFIGS["mid"],
                                 synth.CONFIGS["imbalanced"]], ids=lambda c: c.name)
def test_fused_equals_two_launches_and_oracle(cfg):
    w = synth.make_weights(cfg, 5, "cuda")
    x = synth.make_x(cfg, 5, "cuda")
    layer = gh.make_layer(cfg, w)
    two = _forwards(layer, x, False, n=1)[0]
    fused = _forwards(layer, x, True, n=3)
    for y in fused:
        assert torch.equal(y, two)
    r = layer.get_routing(cfg.T, "cuda")
    ora = ref.forward(gh.f64(x), gh.oracle_weights(w), cfg.k, logits=gh.f64(r["logits"]))
    gh.assert_y_close(fused[-1], ora["y"], what=cfg.name)
    layer.close()


@pytest.mark.parametrize("cfg", [SKEWED, synth.CONFIGS["imbalanced"]], ids=lambda c: c.name)
def test_fused_without_programmatic_launch(cfg):
    w = synth.make_weights(cfg, 6, "cuda")
    x = synth.make_x(cfg, 6, "cuda")
    layer = gh.make_layer(cfg, w)
    layer.set_pdl(False)
    y0 = _forwards(layer, x, False, n=1)[0]
    y1 = _forwards(layer, x, True, n=2)
    layer.set_pdl(True)
    y2 = _forwards(layer, x, True, n=2)
    for y in y1 + y2:
        assert torch.equal(y, y0)
    layer.close()


@pytest.mark.parametrize("dense", [False, True])
@pytest.mark.parametrize("cfg", [SKEWED, synth.CONFIGS["mid"]], ids=lambda c: c.name)
def test_fused_e4m3_equals_two_launches(cfg, dense):
    w = synth.make_weights(cfg, 7, "cuda")
    x = synth.make_x(cfg, 7, "cuda")
    layer = gh.make_layer(cfg, w, fp8=True, fp8_dense=dense)
    scales = [0.02, 0.01, 0.02, 0.01, 0.02][:capi.FP8_TENSORS if dense else 2]
    two = _forwards(layer, x, False, n=1, scales=scales)[0]
    s_two = layer.fp8_state()
    fused = _forwards(layer, x, True, n=2, scales=scales)
    s_fused = layer.fp8_state()
    for y in fused:
        assert torch.equal(y, two)
    # the amax the fused kernel records for h is the two launches' one
    np.testing.assert_array_equal(np.asarray(s_fused["last_amax"]),
                                  np.asarray(s_two["last_amax"]))
    layer.close()


def test_fused_routed_replay():
    """The replay entry (router bypassed, expert ids given) on the fused path."""
    cfg = SMALL
    w = synth.make_weights(cfg, 8, "cuda")
    x = synth.make_x(cfg, 8, "cuda")
    layer = gh.make_layer(cfg, w)
    g = torch.Generator(device="cpu")
    g.manual_seed(3)
    # distinct experts per token, skewed towards expert 0 (more than 256 slots)
    idx = torch.stack([torch.randperm(cfg.E, generator=g)[:cfg.k] for _ in range(cfg.T)])
    idx[: cfg.T // 2, 0] = 0
    idx[: cfg.T // 2, 1] = torch.where(idx[: cfg.T // 2, 1] == 0, 1, idx[: cfg.T // 2, 1])
    idx = idx.to(torch.int32).cuda()
    outs = []
    for fused in (0, 1):
        layer.set_expert_fusion(fused)
        outs.append(layer.forward_routed(x, idx).clone())
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(outs[0], outs[1])
    layer.close()


def test_automatic_mode_matches_both():
    """Mode 2 (the default) picks one of the two forms: the output is the same
    bitwise as both of them."""
    cfg = SKEWED
    w = synth.make_weights(cfg, 9, "cuda")
    x = synth.make_x(cfg, 9, "cuda")
    layer = gh.make_layer(cfg, w)
    y_auto = layer.forward(x).clone()
    y_two = _forwards(layer, x, False, n=1)[0]
    y_one = _forwards(layer, x, True, n=1)[0]
    assert torch.equal(y_auto, y_two) and torch.equal(y_auto, y_one)
    layer.close()


def test_set_expert_fusion_rejects_bad_values():
    cfg = SMALL
    w = synth.make_weights(cfg, 0, "cuda")
    layer = gh.make_layer(cfg, w)
    lib = capi.load()
    assert lib.latentmoe_set_expert_fusion(layer.handle, 3) == capi.ERR_INVALID_ARG
    assert lib.latentmoe_set_expert_fusion(layer.handle, -1) == capi.ERR_INVALID_ARG
    assert lib.latentmoe_set_expert_fusion(None, 1) == capi.ERR_INVALID_ARG
    for mode in (0, 1, 2):
        assert lib.latentmoe_set_expert_fusion(layer.handle, mode) == capi.OK
    layer.close()

"""E4M3 for the latent projections and the shared expert (LATENTMOE_FP8_DENSE)
on the GPU against the oracle's E4M3 layer.

Stage by stage on the GPU's own codes: x's codes (an input in bf16, decided
in fp32 on both sides) bit for bit; z, h and the shared hidden within one
E4M3 step and rarely off; c (an fp32 sum of fp32 expert outputs) within the
propagated fp32 rounding of its terms; the output on all of
the GPU's codes within the bf16 path's bounds; and, end to end, far inside
the FP8 method's own distance from the exact layer."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_router_gb300 import capi, synth
import gpu_helpers as gh
from oracle import fp8 as ofp8
from oracle import latentmoe_ref as ref
from test_gpu_fp8 import _codes_close, _decode

pytestmark = pytest.mark.gpu


def _c_codes_close(got, ora, s_c):
    """The GPU forms o by fp32 accumulation and sums it in fp32, so its c may
    differ from the oracle's by B[t] = sum_j |g_tj| |o_tj| 2^-14 (fp32
    accumulation over K <= 10240 terms, with room); where terms cancel that
    can exceed an E4M3 step of c. Each GPU code must be a rounding of some
    value within B of the oracle's c: |got - c| <= B + half a step at the
    larger of |c|, |got|."""
    c, g, pos, o = ora["c"], ora["gates"], ora["pos"], ora["o"]
    T, k = pos.shape
    B = np.zeros_like(c)
    for j in range(k):
        B += np.abs(g[:, j:j + 1]) * np.abs(o[pos[:, j]])
    B *= 2.0 ** -14
    mag = np.maximum(np.abs(c), np.abs(got))
    half_step = np.maximum(mag * 2.0 ** -4, 2.0 ** -10 * s_c)
    err = np.abs(got - c)
    bad = err > B + half_step * (1 + 1e-9)
    assert not bad.any(), (int(bad.sum()), float(err[bad].max()))
    assert (got != ora["c_q"] * s_c).mean() < 1e-2


def _dense_case(cfg, seed, renorm=False, T=None):
    w = synth.make_weights(cfg, seed, "cuda")
    x = synth.make_x(cfg, seed, "cuda")
    layer = gh.make_layer(cfg, w, renorm=renorm, fp8=True, fp8_dense=True)
    return w, x[: (T or cfg.T)], layer


def _check_dense(cfg, w, x, layer, renorm=False):
    T = x.shape[0]
    layer.forward(x)
    s_z, s_h, s_x, s_c, s_sh = layer.fp8_state()["scales"]
    y = layer.forward(x)
    r = layer.get_routing(T, "cuda")
    zc, hc = layer.fp8_codes(T, "cuda")
    xc, cc, shc = layer.fp8_dense_codes(T, "cuda")
    torch.cuda.synchronize()
    assert layer.status() == 0
    W = gh.oracle_weights(w)
    xs = gh.f64(x)
    L = gh.f64(r["logits"])
    dense = {"s_x": s_x, "s_c": s_c, "s_sh": s_sh}
    kw = dict(s_z=s_z, s_h=s_h, renorm=renorm, logits=L)
    # x: bit for bit
    xq = _decode(xc)
    assert np.array_equal(xq, ofp8.quantize_input(xs, s_x))
    # z from the GPU's x codes
    on_x = ofp8.forward_fp8(xs, W, cfg.k, dense={**dense, "x_codes": xq}, **kw)
    gh.assert_routing_equal(r, on_x, T, cfg.k)
    zq, hq = _decode(zc), _decode(hc)
    _codes_close(zq * s_z, on_x["z_q"] * s_z, s_z, "z codes")
    # h from the GPU's z codes
    on_z = ofp8.forward_fp8(xs, W, cfg.k, z_codes=zq, dense={**dense, "x_codes": xq}, **kw)
    _codes_close(hq * s_h, on_z["h_q"] * s_h, s_h, "h codes")
    # c from the GPU's h codes; the shared hidden from the GPU's x codes
    on_h = ofp8.forward_fp8(xs, W, cfg.k, z_codes=zq, h_codes=hq,
                            dense={**dense, "x_codes": xq}, **kw)
    cq = _decode(cc)
    _c_codes_close(cq * s_c, on_h, s_c)
    codes = {**dense, "x_codes": xq, "c_codes": cq}
    if cfg.Fs:
        shq = _decode(shc)
        _codes_close(shq * s_sh, on_h["sh_q"] * s_sh, s_sh, "shared hidden codes")
        codes["sh_codes"] = shq
    # the output on all of the GPU's codes
    on_all = ofp8.forward_fp8(xs, W, cfg.k, z_codes=zq, h_codes=hq, dense=codes, **kw)
    gh.assert_y_close(y, on_all["y"], "y on the GPU's codes")
    # end to end: far inside the E4M3 layer's own distance from the exact layer
    own = ofp8.forward_fp8(xs, W, cfg.k, dense=dense, **kw)
    exact = ref.forward(xs, W, cfg.k, renorm=renorm, logits=L)["y"]
    yg = gh.f64(y)
    rel = np.linalg.norm(yg - own["y"]) / np.linalg.norm(own["y"])
    rel_fp8 = np.linalg.norm(own["y"] - exact) / np.linalg.norm(exact)
    assert rel < 0.5 * rel_fp8, (rel, rel_fp8)
    # recorded maxima of the forward
    last = layer.fp8_state()["last_amax"]
    assert last[2] == np.abs(xs).max()
    assert abs(last[3] - on_h["c_amax"]) <= 1e-2 * on_h["c_amax"]
    if cfg.Fs:
        assert abs(last[4] - on_h["sh_amax"]) <= 1e-2 * on_h["sh_amax"]


@pytest.mark.parametrize("name", ["tiny", "mid", "imbalanced"])
def test_dense_e4m3_layer(name):
    cfg = synth.CONFIGS[name]
    w, x, layer = _dense_case(cfg, 5)
    _check_dense(cfg, w, x, layer)


def test_dense_e4m3_shared_expert_ragged_renorm_out_fp32():
    cfg = synth.LayerConfig("tiny-shared", T=200, d=256, l=128, E=8, k=3, F=256, Fs=384)
    w, x, _ = _dense_case(cfg, 6)
    layer = gh.make_layer(cfg, w, renorm=True, fp8=True, fp8_dense=True)
    for T in (1, 77, 200):
        layer.set_fp8_scales([1.0] * capi.FP8_TENSORS)
        _check_dense(cfg, w, x[:T], layer, renorm=True)
    layer32 = gh.make_layer(cfg, w, out_fp32=True, fp8=True, fp8_dense=True)
    _check_dense(cfg, w, x, layer32)


def test_dense_weight_scales_and_launches():
    cfg = synth.LayerConfig("tiny-shared", T=64, d=256, l=128, E=8, k=2, F=256, Fs=256)
    w, x, layer = _dense_case(cfg, 7)
    experts, dense = layer.fp8_all_weight_scales()
    for key in ("w_dn", "w_up", "w_gs", "w_us", "w_ds"):
        assert dense[key] == np.float32(ofp8.weight_scale(gh.f64(w[key]))), key
    n0 = layer.launch_count()
    layer.forward(x)
    # router, sort x3, quantize x, down, gate+up, down, combine, shared gate+up,
    # up (fp32 partial), shared down (+ partial), scale update
    assert layer.launch_count() - n0 == 11
    plain = gh.make_layer(cfg, w, fp8=True)
    _, d2 = plain.fp8_all_weight_scales()
    assert all(v == 1.0 for v in d2.values())
    with pytest.raises(capi.LatentMoEError):
        plain.fp8_dense_codes(cfg.T, "cuda")
    with pytest.raises(capi.LatentMoEError):  # dense needs the expert flag
        capi.LatentMoE(cfg.d, cfg.l, cfg.E, cfg.k, cfg.F, cfg.Fs, max_tokens=cfg.T,
                       fp8_dense=True)

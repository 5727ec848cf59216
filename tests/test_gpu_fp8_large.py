"""The E4M3 expert path at the two large shapes at full size, in the launch
configuration the benchmark times (after a calibrating forward, as the
benchmark's warm-up does): routing in full, bit-exact from the GPU logits;
on seeded token samples, the GPU's z and h codes against the oracle's and
the output against the oracle's E4M3 layer evaluated on the GPU's codes."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_router_gb300 import synth
import gpu_helpers as gh
from oracle import fp8 as ofp8
from oracle import latentmoe_ref as ref
from test_gpu_fp8 import _codes_close, _decode

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,n_y", [("mai-base-1", 4), ("mai-base-2", 4)])
def test_large_shape_e4m3_sampled(name, n_y):
    cfg = synth.CONFIGS[name]
    free, _ = torch.cuda.mem_get_info()
    need = 3 * (3 * cfg.E * cfg.F * cfg.l) + 4 * (3 * cfg.d * cfg.Fs + 2 * cfg.d * cfg.l) + \
        cfg.slots * (2 * cfg.l + cfg.F) * 2 + (8 << 30)
    if free < need:
        pytest.skip(f"needs {need / 2**30:.0f} GiB free, {free / 2**30:.0f} GiB available")
    w = synth.make_weights(cfg, 0, "cuda")
    x = synth.make_x(cfg, 0, "cuda")
    layer = gh.make_layer(cfg, w, fp8=True)
    layer.forward(x)
    s_z, s_h = layer.fp8_state()["scales"][:2]
    y = layer.forward(x)
    r = layer.get_routing(cfg.T, "cuda")
    zc, hc = layer.fp8_codes(cfg.T, "cuda")
    torch.cuda.synchronize()
    assert layer.status() == 0
    W = gh.oracle_weights(w, stacked=False)
    L_gpu = gh.f64(r["logits"])
    gh.assert_routing_equal(r, ref.route(L_gpu, cfg.E, cfg.k), cfg.T, cfg.k)

    # weight scales of a few experts, bit for bit
    got_ws = layer.fp8_weight_scales()
    for e in (0, cfg.E // 2, cfg.E - 1):
        for m, key in enumerate(("w_g", "w_u", "w_d")):
            assert got_ws[m][e] == np.float32(ofp8.weight_scale(gh.f64(w[key][e])))

    s = synth.sample_tokens(cfg.T, n_y, seed=1).numpy()
    st = torch.from_numpy(s).cuda()
    xs = gh.f64(x[st])
    Ls = L_gpu[s]
    pos_gpu = r["pos"].cpu().numpy().reshape(cfg.T, cfg.k)[s]
    cache = {}
    own = ofp8.forward_fp8(xs, W, cfg.k, s_z=s_z, s_h=s_h, logits=Ls, wq_cache=cache)
    # the GPU's codes of the sampled tokens, in the oracle's slot order
    zq_all, hq_all = _decode(zc), _decode(hc)
    zq = np.zeros_like(own["z_q"])
    hq = np.zeros_like(own["h_q"])
    for i in range(n_y):
        for j in range(cfg.k):
            zq[own["pos"][i, j]] = zq_all[pos_gpu[i, j]]
            hq[own["pos"][i, j]] = hq_all[pos_gpu[i, j]]
    _codes_close(zq * s_z, own["z_q"] * s_z, s_z, "z codes", max_frac=2e-3)
    on_z = ofp8.forward_fp8(xs, W, cfg.k, s_z=s_z, s_h=s_h, logits=Ls, z_codes=zq,
                            wq_cache=cache)
    _codes_close(hq * s_h, on_z["h_q"] * s_h, s_h, "h codes", max_frac=2e-3)
    on_codes = ofp8.forward_fp8(xs, W, cfg.k, s_z=s_z, s_h=s_h, logits=Ls, z_codes=zq,
                                h_codes=hq, wq_cache=cache)
    gh.assert_y_close(y[st], on_codes["y"], what=f"{name} E4M3 on the GPU's codes")
    rel = np.linalg.norm(gh.f64(y[st]) - own["y"]) / np.linalg.norm(own["y"])
    assert rel <= gh.Y_REL_FRO, rel
    del layer, w, x, y
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,n_y", [("mai-base-1", 3), ("mai-base-2", 3)])
def test_large_shape_all_e4m3_sampled(name, n_y):
    """All GEMMs but the router in E4M3 at full size: x codes of sampled
    tokens bit for bit, then z, h, c and the shared hidden stage by stage on
    the GPU's own codes, and y on all of them within the bf16 bounds."""
    from test_gpu_fp8_dense import _c_codes_close
    cfg = synth.CONFIGS[name]
    free, _ = torch.cuda.mem_get_info()
    need = 3 * (3 * cfg.E * cfg.F * cfg.l) + 4 * (3 * cfg.d * cfg.Fs + 2 * cfg.d * cfg.l) + \
        cfg.slots * (2 * cfg.l + cfg.F) * 4 + (8 << 30)
    if free < need:
        pytest.skip(f"needs {need / 2**30:.0f} GiB free, {free / 2**30:.0f} GiB available")
    w = synth.make_weights(cfg, 0, "cuda")
    x = synth.make_x(cfg, 0, "cuda")
    layer = gh.make_layer(cfg, w, fp8=True, fp8_dense=True)
    layer.forward(x)
    s_z, s_h, s_x, s_c, s_sh = layer.fp8_state()["scales"]
    y = layer.forward(x)
    r = layer.get_routing(cfg.T, "cuda")
    zc, hc = layer.fp8_codes(cfg.T, "cuda")
    xc, cc, shc = layer.fp8_dense_codes(cfg.T, "cuda")
    torch.cuda.synchronize()
    assert layer.status() == 0
    W = gh.oracle_weights(w, stacked=False)
    L_gpu = gh.f64(r["logits"])
    s = synth.sample_tokens(cfg.T, n_y, seed=2).numpy()
    st = torch.from_numpy(s).cuda()
    xs = gh.f64(x[st])
    Ls = L_gpu[s]
    pos_gpu = r["pos"].cpu().numpy().reshape(cfg.T, cfg.k)[s]
    xq = _decode(xc[st])
    assert np.array_equal(xq, ofp8.quantize_input(xs, s_x))
    dense = {"s_x": s_x, "s_c": s_c, "s_sh": s_sh, "x_codes": xq}
    cache = {}
    kw = dict(s_z=s_z, s_h=s_h, logits=Ls, wq_cache=cache)
    on_x = ofp8.forward_fp8(xs, W, cfg.k, dense=dense, **kw)
    zq_all, hq_all = _decode(zc), _decode(hc)
    zq = np.zeros_like(on_x["z_q"])
    hq = np.zeros_like(on_x["h_q"])
    for i in range(n_y):
        for j in range(cfg.k):
            zq[on_x["pos"][i, j]] = zq_all[pos_gpu[i, j]]
            hq[on_x["pos"][i, j]] = hq_all[pos_gpu[i, j]]
    _codes_close(zq * s_z, on_x["z_q"] * s_z, s_z, "z codes", max_frac=2e-3)
    on_z = ofp8.forward_fp8(xs, W, cfg.k, z_codes=zq, dense=dense, **kw)
    _codes_close(hq * s_h, on_z["h_q"] * s_h, s_h, "h codes", max_frac=2e-3)
    on_h = ofp8.forward_fp8(xs, W, cfg.k, z_codes=zq, h_codes=hq, dense=dense, **kw)
    cq = _decode(cc[st])
    _c_codes_close(cq * s_c, on_h, s_c)
    codes = {**dense, "c_codes": cq}
    if cfg.Fs:
        shq = _decode(shc[st])
        _codes_close(shq * s_sh, on_h["sh_q"] * s_sh, s_sh, "shared hidden codes",
                     max_frac=2e-3)
        codes["sh_codes"] = shq
    on_all = ofp8.forward_fp8(xs, W, cfg.k, z_codes=zq, h_codes=hq, dense=codes, **kw)
    gh.assert_y_close(y[st], on_all["y"], what=f"{name} all-E4M3 on the GPU's codes")
    del layer, w, x, y
    torch.cuda.empty_cache()

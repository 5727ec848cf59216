"""The E4M3 paths at the two large shapes at full size, in the launch
configuration the benchmark times (after a calibrating forward, as the
benchmark's warm-up does): routing in full, bit-exact from the GPU logits;
on 32 tokens chosen to reach as many expert GEMM tiles as 32 tokens can
(each slot a different expert where possible, the last chunk of split
experts included), the GPU's codes against the oracle's stage by stage and
the output against the oracle evaluated on the GPU's codes.

Both variants, E4M3 expert GEMMs and E4M3 for every GEMM but the router,
run in one test per shape: their routers are the same bf16 GEMM, so they
route identically, touch the same experts, and share one set of the
oracle's weight codes (quantized once)."""
import time

import numpy as np
import pytest
import torch

from mixture_experts_layer_router_gb300 import synth
import gpu_helpers as gh
from oracle import fp8 as ofp8
from oracle import latentmoe_ref as ref
from test_gpu_fp8 import _codes_close, _decode
from test_gpu_fp8_dense import _c_codes_close

pytestmark = pytest.mark.gpu

N_TOKENS = 32


def _slot_codes(all_codes, pos_gpu, pos_ora, shape):
    """The GPU's codes of the sampled tokens' slots, in the oracle's slot order."""
    out = np.zeros(shape)
    n, k = pos_ora.shape
    for i in range(n):
        for j in range(k):
            out[pos_ora[i, j]] = all_codes[pos_gpu[i, j]]
    return out


def _run(cfg, w, x, dense):
    layer = gh.make_layer(cfg, w, fp8=True, fp8_dense=dense)
    layer.forward(x)  # calibrates the delayed scales
    scales = layer.fp8_state()["scales"][:5 if dense else 2]
    y = layer.forward(x)
    r = layer.get_routing(cfg.T, "cuda")
    codes = {"z": layer.fp8_codes(cfg.T, "cuda")}
    if dense:
        codes["dense"] = layer.fp8_dense_codes(cfg.T, "cuda")
    torch.cuda.synchronize()
    assert layer.status() == 0
    weight_scales = layer.fp8_weight_scales()
    layer.close()
    return y, r, codes, scales, weight_scales


@pytest.mark.parametrize("name", ["mai-base-1", "mai-base-2"])
def test_large_shape_e4m3_sampled(name):
    cfg = synth.CONFIGS[name]
    free, _ = torch.cuda.mem_get_info()
    need = 3 * (3 * cfg.E * cfg.F * cfg.l) + 4 * (3 * cfg.d * cfg.Fs + 2 * cfg.d * cfg.l) + \
        cfg.slots * (2 * cfg.l + cfg.F) * 4 + (8 << 30)
    if free < need:
        pytest.skip(f"needs {need / 2**30:.0f} GiB free, {free / 2**30:.0f} GiB available")
    w = synth.make_weights(cfg, 0, "cuda")
    x = synth.make_x(cfg, 0, "cuda")

    # ---- E4M3 expert GEMMs
    y, r, codes, (s_z, s_h), got_ws = _run(cfg, w, x, dense=False)
    L_gpu = gh.f64(r["logits"])
    gh.assert_routing_equal(r, ref.route(L_gpu, cfg.E, cfg.k), cfg.T, cfg.k)
    for e in (0, cfg.E // 2, cfg.E - 1):  # weight scales, bit for bit
        for m, key in enumerate(("w_g", "w_u", "w_d")):
            assert got_ws[m][e] == np.float32(ofp8.weight_scale(gh.f64(w[key][e])))

    s = gh.covering_tokens(r, cfg.T, cfg.k, n_min=N_TOKENS, last_slots=False, n_max=N_TOKENS)
    assert len(s) == N_TOKENS
    st = torch.from_numpy(s).cuda()
    xs = gh.f64(x[st])
    Ls = L_gpu[s]
    pos_gpu = r["pos"].cpu().numpy().reshape(cfg.T, cfg.k)[s]
    touched = np.unique(r["idx"].cpu().numpy().reshape(cfg.T, cfg.k)[s])
    t0 = time.perf_counter()
    cache = gh.E4M3WeightCodes(w, touched)
    W = gh.oracle_weights(w, stacked=False)
    kw = dict(logits=Ls, wq_cache=cache)

    own = ofp8.forward_fp8(xs, W, cfg.k, s_z=s_z, s_h=s_h, **kw)
    zc, hc = codes["z"]
    zq = _slot_codes(_decode(zc), pos_gpu, own["pos"], own["z_q"].shape)
    hq = _slot_codes(_decode(hc), pos_gpu, own["pos"], own["h_q"].shape)
    _codes_close(zq * s_z, own["z_q"] * s_z, s_z, "z codes", max_frac=2e-3)
    # on the GPU's codes: h from the GPU's z codes, y from both
    on = ofp8.forward_fp8(xs, W, cfg.k, s_z=s_z, s_h=s_h, z_codes=zq, h_codes=hq, **kw)
    _codes_close(hq * s_h, ofp8.quantize_act(on["h"], s_h) * s_h, s_h, "h codes", max_frac=2e-3)
    gh.assert_y_close(y[st], on["y"], what=f"{name} E4M3 on the GPU's codes")
    rel = np.linalg.norm(gh.f64(y[st]) - own["y"]) / np.linalg.norm(own["y"])
    assert rel <= gh.Y_REL_FRO, rel
    del y

    # ---- every GEMM but the router in E4M3, same weights, same routing
    y, r2, codes, (s_z, s_h, s_x, s_c, s_sh), _ = _run(cfg, w, x, dense=True)
    for key in ("idx", "counts", "offsets", "perm", "pos"):
        assert torch.equal(r2[key], r[key]), key
    xc, cc, shc = codes["dense"]
    xq = _decode(xc[st])
    assert np.array_equal(xq, ofp8.quantize_input(xs, s_x))
    dense = {"s_x": s_x, "s_c": s_c, "s_sh": s_sh, "x_codes": xq}
    on_x = ofp8.forward_fp8(xs, W, cfg.k, s_z=s_z, s_h=s_h, dense=dense, **kw)
    zc, hc = codes["z"]
    zq = _slot_codes(_decode(zc), pos_gpu, on_x["pos"], on_x["z_q"].shape)
    hq = _slot_codes(_decode(hc), pos_gpu, on_x["pos"], on_x["h_q"].shape)
    _codes_close(zq * s_z, on_x["z_q"] * s_z, s_z, "z codes", max_frac=2e-3)
    cq = _decode(cc[st])
    all_codes = {**dense, "c_codes": cq}
    if cfg.Fs:
        all_codes["sh_codes"] = _decode(shc[st])
    # on every one of the GPU's codes: h from its z codes, c from its h
    # codes, the shared hidden from its x codes, and y from all of them
    on = ofp8.forward_fp8(xs, W, cfg.k, s_z=s_z, s_h=s_h, z_codes=zq, h_codes=hq,
                          dense=all_codes, **kw)
    _codes_close(hq * s_h, ofp8.quantize_act(on["h"], s_h) * s_h, s_h, "h codes", max_frac=2e-3)
    _c_codes_close(cq * s_c, {**on, "c_q": ofp8.quantize_act(on["c"], s_c)}, s_c)
    if cfg.Fs:
        _codes_close(all_codes["sh_codes"] * s_sh, ofp8.quantize_act(on["sh"], s_sh) * s_sh,
                     s_sh, "shared hidden codes", max_frac=2e-3)
    gh.assert_y_close(y[st], on["y"], what=f"{name} all-E4M3 on the GPU's codes")
    print(f"{name}: E4M3 checked on {len(s)} tokens reaching {len(touched)} experts "
          f"({time.perf_counter() - t0:.1f} s of oracle)")
    del y, cache, w, x
    torch.cuda.empty_cache()

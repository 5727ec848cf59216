"""FP8 E4M3 expert GEMMs on the GPU against the oracle's E4M3 layer.

Weight codes and scales are decided in fp32 on both sides and must match
bit for bit. The grouped E4M3 GEMM is exact on small-integer codes. The
layer output is compared with the oracle's FP8 layer run at the scales the
GPU used (the scales come from the GPU's own recorded maxima, which the
oracle's delayed-scaling recurrence reproduces exactly). Activation codes
are decided from values that differ in the last fp32 bits between the two
sides, so a code may differ by one step where a value sits within that
difference of a rounding midpoint; such moves are checked to be rare and
one step at most, and the output is then checked against the oracle run on
the GPU's own codes with the bounds of the bf16 path.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_router_gb300 import capi, synth
import gpu_helpers as gh
from oracle import fp8 as ofp8
from oracle import latentmoe_ref as ref

pytestmark = pytest.mark.gpu


def _decode(codes: torch.Tensor) -> np.ndarray:
    return codes.view(torch.float8_e4m3fn).float().cpu().numpy().astype(np.float64)


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * scale).to(torch.bfloat16)


# ---------------------------------------------------------------- quantizer

def test_quantize_matches_oracle_bit_for_bit():
    gh.lib()
    G, R, C = 4, 96, 272
    src = torch.stack([_bf16((R, C), 1, 0.02), _bf16((R, C), 2, 3.0),
                       torch.zeros((R, C), dtype=torch.bfloat16, device="cuda"),
                       _bf16((R, C), 3, 1e-3)])
    codes = torch.empty((G, R, C), dtype=torch.uint8, device="cuda")
    scales = torch.empty((G,), dtype=torch.float32, device="cuda")
    assert capi.quantize_e4m3(src, codes, scales) == capi.OK
    torch.cuda.synchronize()
    got = _decode(codes)
    sc = scales.cpu().numpy()
    for g in range(G):
        want, s = ofp8.quantize_weight(gh.f64(src[g]))
        assert sc[g] == np.float32(s), g
        assert np.array_equal(got[g], want), g


def test_quantize_ties_round_to_even():
    """A grid with max 56 (scale 1/8 exactly, reciprocal 8): the scaled values
    land exactly on E4M3 midpoints, where the rounding direction is fixed."""
    gh.lib()
    v = ofp8.e4m3_values()
    v = v[v <= 448]
    mids = (v[:-1] + v[1:]) / 2
    vals = np.concatenate([mids, -mids, [448.0]]) / 8.0
    n = (len(vals) + 15) // 16 * 16
    row = np.zeros(n)
    row[:len(vals)] = vals
    src = torch.tensor(row, dtype=torch.float64).to(torch.bfloat16).reshape(1, 1, n).cuda()
    assert np.array_equal(gh.f64(src).ravel(), row)  # midpoints are exact in bf16
    codes = torch.empty((1, 1, n), dtype=torch.uint8, device="cuda")
    scales = torch.empty((1,), dtype=torch.float32, device="cuda")
    assert capi.quantize_e4m3(src, codes, scales) == capi.OK
    torch.cuda.synchronize()
    assert scales.item() == 0.125
    want, _ = ofp8.quantize_weight(row.reshape(1, n))
    assert np.array_equal(_decode(codes).ravel(), want.ravel())


# ---------------------------------------------------------------- grouped GEMM

def _int_codes(shape, seed, lo=-4, hi=4):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    vals = torch.randint(lo, hi + 1, shape, generator=g, device="cuda").float()
    return vals.to(torch.float8_e4m3fn).view(torch.uint8), vals.double().cpu()


@pytest.mark.parametrize("counts", [[0, 37, 256, 300, 5, 0, 130], [1], [513, 0, 0, 16]])
def test_grouped_e4m3_plain_exact(counts):
    """Integer codes: products and sums are exact in fp32, so C is the
    bf16 rounding of the exact result times the power-of-two scales."""
    gh.lib()
    G, N, K = len(counts), 384, 256
    M = sum(counts)
    A, Af = _int_codes((M, K), 11)
    B, Bf = _int_codes((G * N, K), 12)
    s_a = 0.5
    s_b = [2.0 ** -(g % 5) for g in range(G)]
    scales = torch.tensor([s_a, 1.0] + s_b, dtype=torch.float32, device="cuda")
    offs = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32,
                        device="cuda")
    C = torch.full((M, N), 7.0, dtype=torch.bfloat16, device="cuda")
    assert capi.debug_grouped_gemm_e4m3(A, B, scales, C, None, offs, G, M, N, K, 1) == capi.OK
    assert capi.debug_status() == 0
    want = torch.empty((M, N), dtype=torch.float64)
    o = 0
    for g, n in enumerate(counts):
        want[o:o + n] = (Af[o:o + n] @ Bf[g * N:(g + 1) * N].T) * (s_a * s_b[g])
        o += n
    assert torch.equal(C.cpu(), want.to(torch.bfloat16))


def test_grouped_e4m3_swiglu_codes_and_amax():
    gh.lib()
    counts = [40, 0, 260, 17]
    G, N, K = len(counts), 256, 384
    M = sum(counts)
    A, Af = _int_codes((M, K), 21, -2, 2)
    B, Bf = _int_codes((2 * G * N, K), 22, -2, 2)
    s_a, s_out = 2.0 ** -4, 2.0 ** -3
    s_g = [2.0 ** -(3 + g) for g in range(G)]
    s_u = [2.0 ** -(2 + g) for g in range(G)]
    scales = torch.tensor([s_a, s_out] + s_g + s_u, dtype=torch.float32, device="cuda")
    offs = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32,
                        device="cuda")
    C = torch.zeros((M, N), dtype=torch.uint8, device="cuda")
    amax = torch.zeros((1,), dtype=torch.int32, device="cuda")
    assert capi.debug_grouped_gemm_e4m3(A, B, scales, C, amax, offs, G, M, N, K, 2) == capi.OK
    assert capi.debug_status() == 0
    h = np.zeros((M, N))
    o = 0
    for g, n in enumerate(counts):
        a = Af[o:o + n].numpy()
        gate = (a @ Bf[g * N:(g + 1) * N].numpy().T) * (s_a * s_g[g])
        up = (a @ Bf[(G + g) * N:(G + g + 1) * N].numpy().T) * (s_a * s_u[g])
        h[o:o + n] = ref.silu(gate) * up
        o += n
    want = ofp8.quantize_act(h, s_out) * s_out
    got = _decode(C) * s_out
    # SiLU differs from the float64 one in the last fp32 bits: a code may
    # move by one step where h sits on a midpoint, nowhere else
    diff = got != want
    step = np.maximum(np.abs(want), 2.0 ** -6 * s_out) * 2.0 ** -3
    assert np.all(np.abs(got - want)[diff] <= step[diff] * (1 + 1e-9))
    assert diff.mean() < 1e-3
    amax_gpu = amax.view(torch.float32).item()
    assert abs(amax_gpu - np.abs(h).max()) <= 1e-5 * np.abs(h).max()


# ---------------------------------------------------------------- the layer

def _layer_case(name, seed=0, T=None, renorm=False):
    cfg = synth.CONFIGS[name] if isinstance(name, str) else name
    w = synth.make_weights(cfg, seed, "cuda")
    x = synth.make_x(cfg, seed, "cuda")
    layer = gh.make_layer(cfg, w, renorm=renorm, fp8=True)
    return cfg, w, x[: (T or cfg.T)], layer


def _weight_scales_exact(layer, w, E):
    got = layer.fp8_weight_scales()
    for m, key in enumerate(("w_g", "w_u", "w_d")):
        for e in range(E):
            assert got[m][e] == np.float32(ofp8.weight_scale(gh.f64(w[key][e]))), (key, e)


def _codes_close(got, want, scale, what, max_frac=1e-3):
    """E4M3 code values (times scale) equal except for rare one-step moves."""
    diff = got != want
    step = np.maximum(np.abs(want), 2.0 ** -6 * scale) * 2.0 ** -3
    assert np.all(np.abs(got - want)[diff] <= step[diff] * (1 + 1e-9)), what
    assert diff.mean() <= max_frac, (what, diff.mean())


def _check_fp8_layer(cfg, w, x, layer, renorm=False):
    """Calibrate with one forward, then compare the next against the oracle.

    Three checks: (1) the GPU's z and h codes against the oracle's, (2) the
    output against the oracle evaluated on the GPU's own codes, with the
    bounds of the bf16 path, (3) the output against the oracle's own FP8
    layer in Frobenius norm, far inside the FP8 method's own error."""
    T = x.shape[0]
    layer.forward(x)
    st = layer.fp8_state()
    s_z, s_h = st["scales"][:2]
    y = layer.forward(x)
    r = layer.get_routing(T, "cuda")
    zc, hc = layer.fp8_codes(T, "cuda")
    torch.cuda.synchronize()
    assert layer.status() == 0
    W = gh.oracle_weights(w)
    xs = gh.f64(x)
    L = gh.f64(r["logits"])
    ora = ofp8.forward_fp8(xs, W, cfg.k, s_z=s_z, s_h=s_h, renorm=renorm, logits=L)
    gh.assert_routing_equal(r, ora, T, cfg.k)
    zq, hq = _decode(zc), _decode(hc)
    _codes_close(zq * s_z, ora["z_q"] * s_z, s_z, "z codes")
    # h codes against the oracle's h computed from the GPU's z codes
    on_z = ofp8.forward_fp8(xs, W, cfg.k, s_z=s_z, s_h=s_h, renorm=renorm, logits=L,
                            z_codes=zq)
    _codes_close(hq * s_h, on_z["h_q"] * s_h, s_h, "h codes")
    on_codes = ofp8.forward_fp8(xs, W, cfg.k, s_z=s_z, s_h=s_h, renorm=renorm, logits=L,
                                z_codes=zq, h_codes=hq)
    gh.assert_y_close(y, on_codes["y"], "y on the GPU's codes")
    # the GPU really ran E4M3: it sits far closer to the FP8 oracle than the
    # FP8 oracle sits to the exact layer
    yg = gh.f64(y)
    rel = np.linalg.norm(yg - ora["y"]) / np.linalg.norm(ora["y"])
    exact = ref.forward(xs, W, cfg.k, renorm=renorm, logits=L)["y"]
    rel_fp8 = np.linalg.norm(ora["y"] - exact) / np.linalg.norm(exact)
    assert rel <= gh.Y_REL_FRO and rel < 0.3 * rel_fp8, (rel, rel_fp8)
    st2 = layer.fp8_state()
    assert st2["steps"] == 2
    az, ah = st2["last_amax"][:2]
    assert abs(az - ora["z_amax"]) <= 1e-3 * ora["z_amax"]
    assert abs(ah - ora["h_amax"]) <= 1e-2 * ora["h_amax"]
    return st, st2


@pytest.mark.parametrize("name", ["tiny", "mid", "imbalanced"])
def test_fp8_layer_matches_oracle(name):
    cfg, w, x, layer = _layer_case(name)
    _weight_scales_exact(layer, w, cfg.E)
    _check_fp8_layer(cfg, w, x, layer)


def test_fp8_shared_expert_ragged_renorm():
    cfg = synth.LayerConfig("tiny-shared", T=200, d=256, l=128, E=8, k=3, F=256, Fs=384)
    w = synth.make_weights(cfg, 7, "cuda")
    x = synth.make_x(cfg, 7, "cuda")
    layer = gh.make_layer(cfg, w, renorm=True, fp8=True)
    for T in (1, 77, 200):
        layer.set_fp8_scales([1.0, 1.0])
        _check_fp8_layer(cfg, w, x[:T], layer, renorm=True)


def test_delayed_scaling_recurrence_over_the_history():
    """1026 forwards, the first on 8x larger input: the GPU's scales follow
    the oracle recurrence fed with the GPU's maxima, bit for bit, and the
    spike leaves the window after 1024 forwards."""
    cfg, w, x, layer = _layer_case("tiny", seed=9)
    ds = ofp8.DelayedScaling(capi.FP8_TENSORS)
    big = (x.float() * 8).to(torch.bfloat16)
    amax0 = None
    for n in range(1026):
        layer.forward(big if n == 0 else x)
        st = layer.fp8_state()
        want = ds.record(st["last_amax"])
        assert st["steps"] == n + 1
        assert [np.float32(s) for s in st["scales"]] == list(want), n
        if n == 0:
            amax0 = st["last_amax"]
        elif n < 1024:
            assert st["scales"][0] == np.float32(np.float32(amax0[0]) / np.float32(448))
    assert st["scales"][0] < np.float32(np.float32(amax0[0]) / np.float32(448))
    assert layer.status() == 0


def test_set_scales_errors_and_launch_count():
    cfg, w, x, layer = _layer_case("tiny", seed=2)
    layer.set_fp8_scales([0.01, 0.02])
    st = layer.fp8_state()
    assert st["scales"][:2] == [np.float32(0.01), np.float32(0.02)] and st["steps"] == 0
    for bad in ([0.0, 1.0], [-1.0, 1.0], [float("inf"), 1.0], [1.0, float("nan")]):
        with pytest.raises(capi.LatentMoEError):
            layer.set_fp8_scales(bad)
    n0 = layer.launch_count()
    layer.forward(x)
    assert layer.launch_count() - n0 == 8
    plain = gh.make_layer(cfg, w)
    with pytest.raises(capi.LatentMoEError):
        plain.fp8_state()
    with pytest.raises(capi.LatentMoEError):
        plain.fp8_weight_scales()


def test_fp8_forward_is_deterministic_and_zero_input_is_zero():
    cfg, w, x, layer = _layer_case("imbalanced", seed=4)
    layer.set_fp8_scales([0.05, 0.01])
    a = layer.forward(x).clone()
    layer.set_fp8_scales([0.05, 0.01])
    b = layer.forward(x).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    z = layer.forward(torch.zeros_like(x))
    torch.cuda.synchronize()
    assert torch.all(z == 0)

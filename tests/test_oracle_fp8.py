"""The oracle's E4M3 rounding and FP8 expert path against the format's
definition, torch's float8 conversion, and the bf16 oracle (CPU)."""
import numpy as np
import pytest
import torch

from oracle import fp8, latentmoe_ref as ref
import oracle_pins


def test_every_code_is_a_fixed_point():
    v = fp8.e4m3_values()
    assert len(v) == 127 and v[-1] == 448.0 and v[1] == 2.0 ** -9
    assert np.array_equal(fp8.round_e4m3(v), v)
    assert np.array_equal(fp8.round_e4m3(-v), -v)


def test_midpoints_round_to_even_mantissa():
    v = fp8.e4m3_values()
    mids = (v[:-1] + v[1:]) / 2
    r = fp8.round_e4m3(mids)
    for lo, hi, got in zip(v[:-1], v[1:], r):
        # the neighbour whose mantissa (position in the value list) is even
        want = lo if int(np.where(v == lo)[0][0]) % 2 == 0 else hi
        assert got == want, (lo, hi, got)


def test_saturation_and_underflow():
    assert fp8.round_e4m3([460.0, 470.0, 1e9, -1e9]).tolist() == [448.0, 448.0, 448.0, -448.0]
    assert fp8.round_e4m3([2.0 ** -10, 3 * 2.0 ** -11, 2.0 ** -12]).tolist() == [0.0, 2.0 ** -9, 0.0]


def test_matches_torch_float8_in_range():
    g = torch.Generator().manual_seed(0)
    x = torch.randn(20000, generator=g) * torch.exp2(torch.randint(-12, 9, (20000,), generator=g).float())
    x = x.clamp(-440, 440)
    want = x.to(torch.float8_e4m3fn).double().numpy()
    got = fp8.round_e4m3(x.double().numpy())
    assert np.array_equal(got, want)


def test_weight_codes_use_fp32_scale():
    w = np.array([[0.5, -1.75], [3.0, 0.0078125]])
    q, s = fp8.quantize_weight(w)
    assert s == float(np.float32(3.0) / np.float32(448.0))
    assert np.all(np.abs(q) <= 448) and q[1, 0] == 448.0


def test_fp8_path_reduces_to_bf16_oracle_within_fp8_error():
    """With scales that keep values in range, the FP8 layer stays within a few
    percent of the exact layer (3 mantissa bits: <= 2^-4 relative per value)."""
    w = oracle_pins.tiny_layer(81, T=40, d=16, l=32, E=4, k=2, F=64)
    W = oracle_pins.oracle_weights(ref, w)
    exact = ref.forward(w["x"], W, 2)
    first = fp8.forward_fp8(w["x"], W, 2, s_z=1.0, s_h=1.0)
    got = fp8.forward_fp8(w["x"], W, 2, s_z=first["z_amax"] / 448, s_h=first["h_amax"] / 448)
    rel = np.linalg.norm(got["y"] - exact["y"]) / np.linalg.norm(exact["y"])
    assert rel < 0.1
    assert np.array_equal(got["idx"], exact["idx"])


def _grid_layer(seed, T=30, d=16, E=4, k=2, F=24):
    """A layer whose expert weights and latent are E4M3 codes times distinct
    powers of two, so the weights and z quantize exactly and the only FP8
    rounding left is that of h."""
    rng = np.random.default_rng(seed)
    v = fp8.e4m3_values()
    codes = lambda shape: rng.choice(np.concatenate([v, -v]), size=shape)
    def with_max(shape):
        c = codes(shape)
        c.flat[rng.integers(c.size)] = 448.0  # amax 448 makes the scale the power of two
        return c
    sz = 2.0 ** -7
    w = {
        "x": codes((T, d)) * sz,
        "w_r": rng.standard_normal((E, d)),
        "w_dn": np.eye(d),
        "w_up": rng.standard_normal((d, d)),
        "w_g": np.stack([with_max((F, d)) * 2.0 ** -(8 + e) for e in range(E)]),
        "w_u": np.stack([with_max((F, d)) * 2.0 ** -(10 + e) for e in range(E)]),
        "w_d": np.stack([with_max((d, F)) * 2.0 ** -(9 + 2 * e) for e in range(E)]),
    }
    return w, sz


def test_fp8_error_is_only_the_rounding_of_h():
    """Exact weights and z: |y_fp8 - y| is bounded elementwise by the
    propagated half-ulp of h (2^-4 relative, 2^-10 s_h absolute below the
    normal range). A wrong scale, a swapped operand or a missing factor breaks
    the bound by orders of magnitude."""
    w, sz = _grid_layer(5)
    W = ref.OracleWeights.from_stacked(w["w_r"], w["w_dn"], w["w_up"], w["w_g"], w["w_u"],
                                       w["w_d"])
    k = 2
    exact = ref.forward(w["x"], W, k)
    probe = fp8.forward_fp8(w["x"], W, k, s_z=sz, s_h=1.0)
    s_h = probe["h_amax"] / 448
    got = fp8.forward_fp8(w["x"], W, k, s_z=sz, s_h=s_h)
    assert np.array_equal(got["idx"], exact["idx"])
    # elementwise bound from the exact h of every slot
    z = w["x"]
    bound = np.zeros_like(exact["y"])
    for t in range(z.shape[0]):
        for j in range(k):
            e = exact["idx"][t, j]
            g = z[t] @ w["w_g"][e].T
            u = z[t] @ w["w_u"][e].T
            h = ref.silu(g) * u
            dh = np.maximum(np.abs(h) * 2.0 ** -4, 2.0 ** -10 * s_h)
            bound[t] += exact["gates"][t, j] * (np.abs(w["w_up"]) @ (np.abs(w["w_d"][e]) @ dh))
    err = np.abs(got["y"] - exact["y"])
    assert np.all(err <= bound * (1 + 1e-9) + 1e-300)
    assert err.max() > 0  # h really was rounded


def test_weight_scale_of_a_power_of_two_grid_is_exact():
    w, _ = _grid_layer(6)
    for e in range(4):
        q, s = fp8.quantize_weight(w["w_g"][e])
        assert s == 2.0 ** -(8 + e) and np.array_equal(q * s, w["w_g"][e])


def test_tiny_activation_scale_flushes_h_to_zero_and_huge_saturates():
    w, sz = _grid_layer(7)
    W = ref.OracleWeights.from_stacked(w["w_r"], w["w_dn"], w["w_up"], w["w_g"], w["w_u"],
                                       w["w_d"])
    flushed = fp8.forward_fp8(w["x"], W, 2, s_z=sz, s_h=1e30)
    assert np.all(flushed["y"] == 0)
    sat = fp8.forward_fp8(w["x"], W, 2, s_z=sz * 2.0 ** -20, s_h=1.0)
    # z saturates at 448 * s_z: the latent the experts see is at most 448 s_z in magnitude
    assert np.isfinite(sat["y"]).all()


# ---------------------------------------------------------------- planted mistakes

FP8_CHECKS = [test_every_code_is_a_fixed_point, test_midpoints_round_to_even_mantissa,
              test_saturation_and_underflow, test_matches_torch_float8_in_range,
              test_weight_codes_use_fp32_scale, test_fp8_error_is_only_the_rounding_of_h,
              test_weight_scale_of_a_power_of_two_grid_is_exact,
              test_tiny_activation_scale_flushes_h_to_zero_and_huge_saturates]


def _round_ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    e = np.maximum(np.floor(np.log2(np.maximum(a, 2.0 ** -9))), -6.0)
    q = np.exp2(e - 3.0)
    r = np.minimum(np.floor(a / q + 0.5) * q, 448.0)
    return np.where(x < 0, -r, r)


def _round_no_subnormals(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -30)))
    q = np.exp2(e - 3.0)
    r = np.round(a / q) * q
    r = np.where(a < 2.0 ** -6, 0.0, np.minimum(r, 448.0))
    return np.where(x < 0, -r, r)


def _round_two_mantissa_bits(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    e = np.maximum(np.floor(np.log2(np.maximum(a, 2.0 ** -9))), -6.0)
    q = np.exp2(e - 2.0)
    r = np.minimum(np.round(a / q) * q, 448.0)
    return np.where(x < 0, -r, r)


_orig_quantize_weight = fp8.quantize_weight


def _weight_scale_unused(w):
    q, s = _orig_quantize_weight(w)
    return q, 1.0


def _act_scale_multiplied(t, s):
    return fp8.round_e4m3(np.asarray(t, dtype=np.float64) * s)


FP8_MUTATIONS = {
    "ties_away": ("round_e4m3", _round_ties_away),
    "no_subnormals": ("round_e4m3", _round_no_subnormals),
    "two_mantissa_bits": ("round_e4m3", _round_two_mantissa_bits),
    "weight_scale_unused": ("quantize_weight", _weight_scale_unused),
    "act_scale_multiplied": ("quantize_act", _act_scale_multiplied),
}


@pytest.mark.parametrize("name", sorted(FP8_MUTATIONS))
def test_planted_fp8_mistake_is_caught(name, monkeypatch):
    attr, fn = FP8_MUTATIONS[name]
    monkeypatch.setattr(fp8, attr, fn)
    caught = []
    for check in FP8_CHECKS:
        try:
            check()
        except Exception as exc:
            caught.append(check.__name__)
    assert caught, f"mutation {name} passed every FP8 pin"


def test_delayed_scaling_window():
    """The scale follows the largest maximum of the last 1024 forwards: a
    spike at forward 0 sets it for exactly 1024 steps, then it falls back."""
    ds = fp8.DelayedScaling(2)
    assert ds.scales.tolist() == [1.0, 1.0]
    s = ds.record([896.0, 0.0])
    assert s[0] == 2.0 and s[1] == 1.0  # zero maxima keep the initial scale
    for n in range(1, 1024):
        s = ds.record([44.8, 4.48])
        assert s[0] == 2.0 and s[1] == np.float32(np.float32(4.48) / np.float32(448))
    s = ds.record([44.8, 4.48])  # forward 1024 overwrites the spike
    assert s[0] == np.float32(np.float32(44.8) / np.float32(448))
    assert ds.steps == 1025


def test_given_codes_reproduce_own_codes():
    """Passing back the codes the oracle formed itself changes nothing."""
    w = oracle_pins.tiny_layer(83, T=33, d=16, l=32, E=5, k=2, F=48)
    W = oracle_pins.oracle_weights(ref, w)
    a = fp8.forward_fp8(w["x"], W, 2, s_z=0.01, s_h=0.003)
    b = fp8.forward_fp8(w["x"], W, 2, s_z=0.01, s_h=0.003, z_codes=a["z_q"], h_codes=a["h_q"])
    assert np.array_equal(a["y"], b["y"])
    # slot i holds token perm[i]'s latent codes
    z = ref.latent_down(w["x"], W.w_dn)
    assert np.array_equal(a["z_q"], fp8.quantize_act(z, 0.01)[a["perm"]])


def test_weight_cache_changes_nothing():
    w = oracle_pins.tiny_layer(84, T=20, d=16, l=32, E=4, k=2, F=32)
    W = oracle_pins.oracle_weights(ref, w)
    cache = {}
    a = fp8.forward_fp8(w["x"], W, 2, s_z=0.01, s_h=0.003)
    b = fp8.forward_fp8(w["x"], W, 2, s_z=0.01, s_h=0.003, wq_cache=cache)
    c = fp8.forward_fp8(w["x"], W, 2, s_z=0.01, s_h=0.003, wq_cache=cache)
    assert np.array_equal(a["y"], b["y"]) and np.array_equal(a["y"], c["y"]) and cache


def _grid_layer_dense(seed, T=24, d=32, l=16, E=4, k=2, F=24, Fs=40):
    """Like _grid_layer, with the dense weights on E4M3 grids too (power-of-
    two scales): x, W_dn, W_up and the shared weights quantize exactly."""
    rng = np.random.default_rng(seed)
    v = fp8.e4m3_values()
    codes = lambda shape: rng.choice(np.concatenate([v, -v]), size=shape)

    def with_max(shape, e2):
        c = codes(shape)
        c.flat[rng.integers(c.size)] = 448.0
        return c * 2.0 ** e2
    sx = 2.0 ** -8
    w = {
        "x": codes((T, d)) * sx,
        "w_r": rng.standard_normal((E, d)),
        "w_dn": with_max((l, d), -12), "w_up": with_max((d, l), -11),
        "w_g": np.stack([with_max((F, l), -(9 + e)) for e in range(E)]),
        "w_u": np.stack([with_max((F, l), -(10 + e)) for e in range(E)]),
        "w_d": np.stack([with_max((l, F), -(10 + e)) for e in range(E)]),
        "w_gs": with_max((Fs, d), -12), "w_us": with_max((Fs, d), -11),
        "w_ds": with_max((d, Fs), -12),
    }
    W = ref.OracleWeights.from_stacked(w["w_r"], w["w_dn"], w["w_up"], w["w_g"], w["w_u"],
                                       w["w_d"], w_gs=w["w_gs"], w_us=w["w_us"], w_ds=w["w_ds"])
    return w, W, sx


def test_dense_e4m3_error_is_the_rounding_of_c_and_sh():
    """Exact x and dense weights: the dense E4M3 layer differs from the
    expert-only E4M3 layer (same z and h codes) only by the rounding of c
    and of the shared hidden, each bounded elementwise by its half-step."""
    w, W, sx = _grid_layer_dense(11)
    k = 2
    base = fp8.forward_fp8(w["x"], W, k, s_z=1.0, s_h=1.0)
    s_z, s_h = base["z_amax"] / 448, base["h_amax"] / 448
    experts = fp8.forward_fp8(w["x"], W, k, s_z=s_z, s_h=s_h)
    probe = fp8.forward_fp8(w["x"], W, k, s_z=s_z, s_h=s_h,
                            dense={"s_x": sx, "s_c": 1.0, "s_sh": 1.0})
    s_c, s_sh = probe["c_amax"] / 448, probe["sh_amax"] / 448
    got = fp8.forward_fp8(w["x"], W, k, s_z=s_z, s_h=s_h,
                          dense={"s_x": sx, "s_c": s_c, "s_sh": s_sh})
    assert np.array_equal(got["x_q"] * sx, w["x"])             # x exact on its grid
    assert np.array_equal(got["z_q"], experts["z_q"])          # so z and h codes agree
    assert np.array_equal(got["h_q"], experts["h_q"])
    shared = ref.shared_expert(w["x"], w["w_gs"], w["w_us"], w["w_ds"])
    y_exp_noshared = experts["y"] - shared
    c, sh = got["c"], got["sh"]
    hc = np.maximum(np.abs(c) * 2.0 ** -4, 2.0 ** -10 * s_c)
    hs = np.maximum(np.abs(sh) * 2.0 ** -4, 2.0 ** -10 * s_sh)
    bound = hc @ np.abs(w["w_up"]).T + hs @ np.abs(w["w_ds"]).T
    err = np.abs(got["y"] - (y_exp_noshared + shared))
    assert np.all(err <= bound * (1 + 1e-9) + 1e-300) and err.max() > 0
    # the maxima the dense path records
    assert got["x_amax"] == np.abs(w["x"]).max()
    assert got["c_amax"] == np.abs(c).max() and got["sh_amax"] == np.abs(sh).max()


def test_dense_given_codes_reproduce_own_codes():
    w, W, sx = _grid_layer_dense(12)
    d = {"s_x": sx * 3, "s_c": 0.01, "s_sh": 0.02}
    a = fp8.forward_fp8(w["x"], W, 2, s_z=0.01, s_h=0.003, dense=d)
    b = fp8.forward_fp8(w["x"], W, 2, s_z=0.01, s_h=0.003, z_codes=a["z_q"], h_codes=a["h_q"],
                        dense={**d, "x_codes": a["x_q"], "c_codes": a["c_q"],
                               "sh_codes": a["sh_q"]})
    assert np.array_equal(a["y"], b["y"])


FP8_CHECKS += [test_dense_e4m3_error_is_the_rounding_of_c_and_sh]


def test_quantize_input_matches_act_when_the_product_is_exact():
    """bf16 values times a power-of-two reciprocal: the fp32 product is exact,
    so the fp32 and float64 decisions agree everywhere; with a general scale
    they differ only where the fp32 product lands on the other side of a
    midpoint."""
    rng = np.random.default_rng(3)
    t = np.asarray(torch.from_numpy(rng.standard_normal(5000)).to(torch.bfloat16).double())
    assert np.array_equal(fp8.quantize_input(t, 2.0 ** -5), fp8.quantize_act(t, 2.0 ** -5))
    a, b = fp8.quantize_input(t, 0.0137), fp8.quantize_act(t, 0.0137)
    assert (a != b).mean() < 1e-2

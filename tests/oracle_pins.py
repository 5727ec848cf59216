"""Pins for the float64 oracle: checks against facts that do not come from it.

Each ``check_*`` takes the oracle module and raises on a mismatch. They are
collected by ``test_oracle_pins.py`` against the real oracle and by
``test_oracle_mutations.py`` against copies with planted mistakes, which shows
that every planted mistake trips at least one of them.

What pins what:
- brute force (scalar loops, dense over all experts, no sort) on tiny
  non-square shapes: every step, including transposed operands;
- closed forms on a 2-wide hand-built layer: logits, softmax gates, SiLU,
  the combine, non-symmetric down/up projections, the shared expert;
- E=1, k=1 reduces to a dense SwiGLU between the down- and up-projection
  (written here with einsum index strings);
- k=E without renorm is the dense softmax mixture (scipy's softmax);
- the counting sort equals numpy's stable argsort of the flattened choices;
- slot invariants, zero-input ties, token and expert permutation symmetry.
"""
from __future__ import annotations

import math

import numpy as np

try:
    from scipy.special import softmax as scipy_softmax
except ImportError:  # pragma: no cover - scipy is present on both machines
    scipy_softmax = None


def _softmax(L):
    if scipy_softmax is not None:
        return scipy_softmax(L, axis=1)
    m = L.max(axis=1, keepdims=True)
    e = np.exp(L - m)
    return e / e.sum(axis=1, keepdims=True)


def _sigmoid(a):
    return 1.0 / (1.0 + math.exp(-a))


def _bf16_grid(rng, shape, scale):
    """Random values on a coarse dyadic grid (exact in bf16 and float64)."""
    return np.round(rng.standard_normal(shape) * scale * 64.0) / 64.0


def tiny_layer(seed, T=7, d=6, l=4, E=5, k=2, F=3, Fs=0, bias=False):
    rng = np.random.default_rng(seed)
    w = {
        "x": _bf16_grid(rng, (T, d), 1.0),
        "w_r": _bf16_grid(rng, (E, d), 0.5),
        "b_r": _bf16_grid(rng, (E,), 0.5) if bias else None,
        "w_dn": _bf16_grid(rng, (l, d), 0.4),
        "w_up": _bf16_grid(rng, (d, l), 0.5),
        "w_g": _bf16_grid(rng, (E, F, l), 0.5),
        "w_u": _bf16_grid(rng, (E, F, l), 0.5),
        "w_d": _bf16_grid(rng, (E, l, F), 0.6),
        "w_gs": _bf16_grid(rng, (Fs, d), 0.4) if Fs else None,
        "w_us": _bf16_grid(rng, (Fs, d), 0.4) if Fs else None,
        "w_ds": _bf16_grid(rng, (d, Fs), 0.5) if Fs else None,
        "k": k,
    }
    return w


def oracle_weights(ref, w):
    return ref.OracleWeights.from_stacked(
        w["w_r"], w["w_dn"], w["w_up"], w["w_g"], w["w_u"], w["w_d"],
        b_r=w["b_r"], w_gs=w["w_gs"], w_us=w["w_us"], w_ds=w["w_ds"])


# ---------------------------------------------------------------- brute force

def check_brute_force(ref):
    from oracle import latentmoe_brute as brute
    cases = [
        dict(seed=1),
        dict(seed=2, bias=True),
        dict(seed=3, Fs=3),
        dict(seed=4, k=3, E=4, bias=True, Fs=2),
        dict(seed=5, k=1, E=3, T=5),
    ]
    for c in cases:
        renorm_modes = (False, True)
        w = tiny_layer(**c)
        for renorm in renorm_modes:
            out = ref.forward(w["x"], oracle_weights(ref, w), w["k"], renorm=renorm)
            bf = brute.forward(w["x"].tolist(), w["w_r"].tolist(), w["w_dn"].tolist(),
                               w["w_up"].tolist(), w["w_g"].tolist(), w["w_u"].tolist(),
                               w["w_d"].tolist(), w["k"],
                               b_r=None if w["b_r"] is None else w["b_r"].tolist(),
                               renorm=renorm,
                               w_gs=None if w["w_gs"] is None else w["w_gs"].tolist(),
                               w_us=None if w["w_us"] is None else w["w_us"].tolist(),
                               w_ds=None if w["w_ds"] is None else w["w_ds"].tolist())
            assert np.array_equal(out["idx"], np.array(bf["idx"])), ("idx", c)
            np.testing.assert_allclose(out["gates"], np.array(bf["gates"]), rtol=0, atol=1e-12)
            np.testing.assert_allclose(out["y"], np.array(bf["y"]), rtol=0, atol=1e-12)
            assert np.array_equal(out["counts"], np.array(bf["counts"]))
            assert np.array_equal(out["offsets"], np.array(bf["offsets"]))
            assert np.array_equal(out["pos"], np.array(bf["pos"]))
            assert np.array_equal(out["perm"], np.array(bf["perm"]))


# ---------------------------------------------------------------- closed forms

def _hand_layer(w_up=None, w_dn=None):
    """A 2-wide layer whose output can be written down by hand.

    x = [1, 0]; router rows are the unit vectors, so L = [1, 0] and
    p = [s, 1-s] with s = sigmoid(1). Expert 0 has gate row [1, 0], up row
    [2, 0], down column [1, 0]; expert 1 has gate row [-1, 0], up row [1, 0],
    down column [0, 3].
    """
    w = {
        "x": np.array([[1.0, 0.0]]),
        "w_r": np.eye(2),
        "b_r": None,
        "w_dn": np.eye(2) if w_dn is None else w_dn,
        "w_up": np.eye(2) if w_up is None else w_up,
        "w_g": np.array([[[1.0, 0.0]], [[-1.0, 0.0]]]),
        "w_u": np.array([[[2.0, 0.0]], [[1.0, 0.0]]]),
        "w_d": np.array([[[1.0], [0.0]], [[0.0], [3.0]]]),
        "w_gs": None, "w_us": None, "w_ds": None,
    }
    return w


def check_closed_forms(ref):
    s = _sigmoid(1.0)
    # k = 1: only expert 0; silu(1) = s, h = 2s, o = [2s, 0], gate s.
    w = _hand_layer()
    out = ref.forward(w["x"], oracle_weights(ref, w), 1)
    np.testing.assert_allclose(out["logits"], [[1.0, 0.0]], atol=1e-15)
    assert out["idx"].tolist() == [[0]]
    np.testing.assert_allclose(out["gates"], [[s]], rtol=1e-14)
    np.testing.assert_allclose(out["y"], [[2 * s * s, 0.0]], rtol=1e-14, atol=1e-15)
    # k = 2: expert 1 adds gate (1-s) times [0, 3 * silu(-1)], silu(-1) = -(1-s).
    out = ref.forward(w["x"], oracle_weights(ref, w), 2)
    assert out["idx"].tolist() == [[0, 1]]
    np.testing.assert_allclose(out["y"], [[2 * s * s, -3 * (1 - s) ** 2]], rtol=1e-14)
    # renorm with k = E leaves the gates unchanged (they already sum to 1)
    out_r = ref.forward(w["x"], oracle_weights(ref, w), 2, renorm=True)
    np.testing.assert_allclose(out_r["y"], out["y"], rtol=1e-14)
    # non-symmetric projections: y = W_up c with c = [2s^2, -3(1-s)^2]
    wu = np.array([[1.0, 2.0], [0.0, 1.0]])
    w2 = _hand_layer(w_up=wu)
    out = ref.forward(w2["x"], oracle_weights(ref, w2), 2)
    c0, c1 = 2 * s * s, -3 * (1 - s) ** 2
    np.testing.assert_allclose(out["y"], [[c0 + 2 * c1, c1]], rtol=1e-14)
    # W_dn = [[1,0],[1,1]] with x = [0,1]: L = [0,1] picks expert 1 first,
    # z = W_dn x = [0,1], and both experts read only z[0] = 0, so y = 0
    # exactly; a transposed W_dn would give z = [1,1] and a non-zero y.
    wdn = np.array([[1.0, 0.0], [1.0, 1.0]])
    w3 = _hand_layer(w_dn=wdn)
    w3["x"] = np.array([[0.0, 1.0]])
    out = ref.forward(w3["x"], oracle_weights(ref, w3), 2)
    assert out["idx"].tolist() == [[1, 0]]
    np.testing.assert_allclose(out["y"], [[0.0, 0.0]], atol=1e-15)
    # shared expert on the full width, weight 1: with x = [1, 0],
    # gate row [1, 0] -> s, up row [0.5, 0] -> 0.5, down column [4, -2]
    w4 = _hand_layer()
    w4["w_gs"] = np.array([[1.0, 0.0]])
    w4["w_us"] = np.array([[0.5, 0.0]])
    w4["w_ds"] = np.array([[4.0], [-2.0]])
    out = ref.forward(w4["x"], oracle_weights(ref, w4), 1)
    np.testing.assert_allclose(out["y"], [[2 * s * s + 2 * s, -s]], rtol=1e-14)


def check_tie_break(ref):
    L = np.array([[0.5, 0.5, 0.2, 0.5], [0.1, 0.3, 0.3, 0.3], [2.0, 1.0, 2.0, 2.0]])
    idx = ref.top_k_stable(L, 3)
    assert idx.tolist() == [[0, 1, 3], [1, 2, 3], [0, 2, 3]], idx.tolist()
    r = ref.route(L, 4, 2)
    assert r["idx"].tolist() == [[0, 1], [1, 2], [0, 2]]


# ---------------------------------------------------------------- reductions

def check_dense_sandwich(ref):
    """E = 1, k = 1: gate 1, y = W_up (SiLU(W_g z) * (W_u z)) W_d with z = W_dn x."""
    rng = np.random.default_rng(11)
    T, d, l, F = 9, 6, 4, 5
    x = _bf16_grid(rng, (T, d), 1.0)
    w_dn = _bf16_grid(rng, (l, d), 0.4)
    w_up = _bf16_grid(rng, (d, l), 0.5)
    wg = _bf16_grid(rng, (1, F, l), 0.5)
    wu = _bf16_grid(rng, (1, F, l), 0.5)
    wd = _bf16_grid(rng, (1, l, F), 0.5)
    w_r = _bf16_grid(rng, (1, d), 0.5)
    W = ref.OracleWeights.from_stacked(w_r, w_dn, w_up, wg, wu, wd)
    out = ref.forward(x, W, 1)
    z = np.einsum("ld,td->tl", w_dn, x)
    a = np.einsum("fl,tl->tf", wg[0], z)
    b = np.einsum("fl,tl->tf", wu[0], z)
    h = a * (1.0 / (1.0 + np.exp(-a))) * b
    o = np.einsum("lf,tf->tl", wd[0], h)
    y = np.einsum("dl,tl->td", w_up, o)
    np.testing.assert_allclose(out["gates"], np.ones((T, 1)), rtol=0, atol=0)
    np.testing.assert_allclose(out["y"], y, rtol=1e-12, atol=1e-12)


def check_full_mixture(ref):
    """k = E, no renorm: y = W_up sum_e p_e FFN_e(z), p = scipy softmax."""
    w = tiny_layer(21, T=6, d=5, l=4, E=4, k=4, F=3, bias=True)
    out = ref.forward(w["x"], oracle_weights(ref, w), 4)
    L = np.einsum("ed,td->te", w["w_r"], w["x"]) + w["b_r"][None, :]
    p = _softmax(L)
    z = np.einsum("ld,td->tl", w["w_dn"], w["x"])
    c = np.zeros_like(z)
    for e in range(4):
        a = np.einsum("fl,tl->tf", w["w_g"][e], z)
        b = np.einsum("fl,tl->tf", w["w_u"][e], z)
        h = a / (1.0 + np.exp(-a)) * b
        c += p[:, e:e + 1] * np.einsum("lf,tf->tl", w["w_d"][e], h)
    y = np.einsum("dl,tl->td", w["w_up"], c)
    np.testing.assert_allclose(out["y"], y, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out["gates"].sum(axis=1), np.ones(6), rtol=1e-14)


def check_gates(ref):
    rng = np.random.default_rng(5)
    L = rng.standard_normal((40, 9)) * 2.0
    for k in (1, 3, 9):
        r = ref.route(L, 9, k)
        p = _softmax(L)
        np.testing.assert_allclose(r["gates"], np.take_along_axis(p, r["idx"], 1), rtol=1e-13)
        g = r["gates"]
        assert np.all(g > 0) and np.all(g <= 1)
        assert np.all(np.diff(g, axis=1) <= 0)
        assert np.all(g.sum(axis=1) <= 1 + 1e-12)
        rn = ref.route(L, 9, k, renorm=True)
        np.testing.assert_allclose(rn["gates"].sum(axis=1), 1.0, rtol=1e-13)
        np.testing.assert_allclose(rn["gates"], g / g.sum(axis=1, keepdims=True), rtol=1e-13)


# ---------------------------------------------------------------- counting sort

def _random_choices(rng, T, E, k):
    return np.stack([rng.permutation(E)[:k] for _ in range(T)])


def check_counting_sort(ref):
    rng = np.random.default_rng(7)
    for T, E, k in ((50, 7, 3), (1, 4, 4), (33, 16, 1), (64, 5, 2)):
        idx = _random_choices(rng, T, E, k)
        counts, offsets, perm, pos = ref.counting_sort(idx, E)
        S = T * k
        # a library stable sort of the flattened choices gives the same layout
        order = np.argsort(idx.ravel(), kind="stable")
        assert np.array_equal(perm, order // k)
        inv = np.empty(S, dtype=np.int64)
        inv[order] = np.arange(S)
        assert np.array_equal(pos.ravel(), inv)
        assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
        assert offsets[0] == 0 and offsets[E] == S
        assert np.array_equal(np.diff(offsets), counts)
        assert np.array_equal(np.bincount(perm, minlength=T), np.full(T, k))
        for e in range(E):
            seg = perm[offsets[e]:offsets[e + 1]]
            assert np.all(np.diff(seg) > 0)
            assert np.all([e in idx[t] for t in seg])
        for t in range(T):
            for j in range(k):
                s = pos[t, j]
                assert perm[s] == t
                assert offsets[idx[t, j]] <= s < offsets[idx[t, j] + 1]


# ---------------------------------------------------------------- symmetries

def check_zero_input(ref):
    w = tiny_layer(31, T=5, d=6, l=4, E=6, k=3, F=3, Fs=2)
    x = np.zeros_like(w["x"])
    out = ref.forward(x, oracle_weights(ref, w), 3)
    assert out["idx"].tolist() == [[0, 1, 2]] * 5
    np.testing.assert_allclose(out["gates"], np.full((5, 3), 1 / 6), rtol=1e-14)
    assert out["counts"].tolist() == [5, 5, 5, 0, 0, 0]
    assert out["perm"].tolist() == list(range(5)) * 3
    assert np.all(out["y"] == 0.0)


def check_token_permutation(ref):
    w = tiny_layer(41, T=8, Fs=2, bias=True)
    W = oracle_weights(ref, w)
    out = ref.forward(w["x"], W, w["k"])
    P = np.random.default_rng(3).permutation(8)
    outp = ref.forward(w["x"][P], W, w["k"])
    np.testing.assert_allclose(outp["y"], out["y"][P], rtol=1e-13, atol=1e-13)
    assert np.array_equal(outp["idx"], out["idx"][P])


def check_expert_permutation(ref):
    w = tiny_layer(43, T=8, E=6, bias=True)
    out = ref.forward(w["x"], oracle_weights(ref, w), w["k"])
    Q = np.random.default_rng(4).permutation(6)
    wq = dict(w)
    for key in ("w_r", "b_r", "w_g", "w_u", "w_d"):
        wq[key] = w[key][Q]
    outq = ref.forward(w["x"], oracle_weights(ref, wq), w["k"])
    np.testing.assert_allclose(outq["y"], out["y"], rtol=1e-13, atol=1e-13)
    assert np.array_equal(Q[outq["idx"]], out["idx"])


def check_shared_only(ref):
    w = tiny_layer(51, T=6, Fs=3)
    w["w_d"] = np.zeros_like(w["w_d"])
    out = ref.forward(w["x"], oracle_weights(ref, w), w["k"])
    a = w["x"] @ w["w_gs"].T
    b = w["x"] @ w["w_us"].T
    s = (a / (1.0 + np.exp(-a)) * b) @ w["w_ds"].T
    np.testing.assert_allclose(out["y"], s, rtol=1e-13, atol=1e-13)


def check_replay(ref):
    """Router replay: the layer's own choices reproduce forward(); foreign
    choices and gates match brute force with the same replayed routing."""
    from oracle import latentmoe_brute as brute
    for c in (dict(seed=61, bias=True), dict(seed=62, Fs=2, k=3, E=4)):
        w = tiny_layer(**c)
        W = oracle_weights(ref, w)
        out = ref.forward(w["x"], W, w["k"])
        rep = ref.forward_routed(w["x"], W, out["idx"])
        np.testing.assert_allclose(rep["y"], out["y"], rtol=0, atol=1e-14)
        rng = np.random.default_rng(c["seed"])
        T, E, k = w["x"].shape[0], w["w_r"].shape[0], w["k"]
        idx = np.stack([rng.permutation(E)[:k] for _ in range(T)])
        for gates in (None, rng.uniform(0.1, 1.0, (T, k))):
            got = ref.forward_routed(w["x"], W, idx, gates)
            bf = brute.forward(w["x"].tolist(), w["w_r"].tolist(), w["w_dn"].tolist(),
                               w["w_up"].tolist(), w["w_g"].tolist(), w["w_u"].tolist(),
                               w["w_d"].tolist(), k,
                               b_r=None if w["b_r"] is None else w["b_r"].tolist(),
                               w_gs=None if w["w_gs"] is None else w["w_gs"].tolist(),
                               w_us=None if w["w_us"] is None else w["w_us"].tolist(),
                               w_ds=None if w["w_ds"] is None else w["w_ds"].tolist(),
                               replay_idx=idx.tolist(),
                               replay_gates=None if gates is None else gates.tolist())
            np.testing.assert_allclose(got["y"], np.array(bf["y"]), rtol=0, atol=1e-12)
            np.testing.assert_allclose(got["gates"], np.array(bf["gates"]), rtol=0, atol=1e-12)
            assert np.array_equal(got["pos"], np.array(bf["pos"]))


def check_select_bias(ref):
    """Selection-only bias: zero bias changes nothing; a bias moves only the
    choice (gates stay unbiased softmax probabilities); a dominant bias forces
    its expert into every token's top-k."""
    w = tiny_layer(71, T=9, E=6, k=2)
    W = oracle_weights(ref, w)
    base = ref.forward(w["x"], W, 2)
    zero = ref.forward(w["x"], W, 2, select_bias=np.zeros(6))
    np.testing.assert_allclose(zero["y"], base["y"], rtol=0, atol=0)
    b = np.zeros(6)
    b[4] = 1e6
    forced = ref.forward(w["x"], W, 2, select_bias=b)
    assert np.all(forced["idx"][:, 0] == 4)
    np.testing.assert_allclose(forced["gates"][:, 0], base["p"][:, 4], rtol=1e-14)
    # the second choice is the unbiased top-1 unless that was expert 4
    top1 = np.argsort(-base["logits"], axis=1, kind="stable")
    want2 = np.where(top1[:, 0] == 4, top1[:, 1], top1[:, 0])
    assert np.array_equal(forced["idx"][:, 1], want2)


def check_lbl_stats(ref):
    """Counts sum to T*k and match a direct tally; probability sums add up to
    T (each token's softmax sums to 1) and equal a per-token scipy softmax."""
    rng = np.random.default_rng(12)
    T, E, k = 40, 7, 3
    L = rng.standard_normal((T, E)) * 2
    idx = ref.top_k_stable(L, k)
    counts, psum = ref.lbl_stats(L, idx, E)
    assert counts.sum() == T * k
    tally = [sum(1 for t in range(T) for j in range(k) if idx[t, j] == e) for e in range(E)]
    assert counts.tolist() == tally
    np.testing.assert_allclose(psum.sum(), T, rtol=1e-13)
    np.testing.assert_allclose(psum, _softmax(L).sum(axis=0), rtol=1e-13)


ALL_CHECKS = [
    check_brute_force, check_closed_forms, check_tie_break, check_dense_sandwich,
    check_full_mixture, check_gates, check_counting_sort, check_zero_input,
    check_token_permutation, check_expert_permutation, check_shared_only, check_replay,
    check_select_bias, check_lbl_stats,
]

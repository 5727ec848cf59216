"""Planted mistakes in the oracle must each trip at least one pin (CPU only).

Every mutation below replaces one function of the float64 oracle with a
plausible wrong version (a dropped term, a wrong sign, a transposed operand,
a wrong index or order). The pins in ``oracle_pins`` are then run against the
mutated oracle; the test fails if all of them still pass, since that would
mean the pins cannot tell the mistake from the real thing.
"""
import numpy as np
import pytest

import oracle_pins
from oracle import latentmoe_ref as ref


def _silu_wrong_sign(a):
    return a / (1.0 + np.exp(a))


def _silu_is_sigmoid(a):
    return 1.0 / (1.0 + np.exp(-a))


def _gates_all_one(p, idx, renorm=False):
    return np.ones(idx.shape)


def _gates_always_renorm(p, idx, renorm=False):
    g = np.take_along_axis(p, idx, axis=1)
    return g / g.sum(axis=1, keepdims=True)


def _topk_ties_high_first(L, k):
    order = np.argsort(L, axis=1, kind="stable")[:, ::-1]
    return order[:, :k].astype(np.int64)


def _topk_ascending(L, k):
    return np.argsort(L, axis=1, kind="stable")[:, :k].astype(np.int64)


def _logits_no_bias(x, w_r, b_r=None):
    return x @ w_r.T


def _down_transposed(x, w_dn):
    return x @ w_dn


def _up_transposed(c, w_up):
    return c @ w_up


def _combine_drop_last(H, gates, pos):
    T, k = pos.shape
    c = np.zeros((T, H.shape[1]))
    for j in range(k - 1):
        c += gates[:, j:j + 1] * H[pos[:, j]]
    return c


def _combine_unweighted(H, gates, pos):
    T, k = pos.shape
    c = np.zeros((T, H.shape[1]))
    for j in range(k):
        c += H[pos[:, j]]
    return c


def _sort_tokens_reversed(idx, E):
    T, k = idx.shape
    counts = np.bincount(idx.ravel(), minlength=E)
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    fill = np.zeros(E, dtype=np.int64)
    perm = np.full(T * k, -1, dtype=np.int64)
    pos = np.full((T, k), -1, dtype=np.int64)
    for t in reversed(range(T)):
        for j in range(k):
            e = idx[t, j]
            s = offsets[e] + fill[e]
            fill[e] += 1
            perm[s] = t
            pos[t, j] = s
    return counts, offsets, perm, pos


def _swiglu_silu_on_up(a, w_g, w_u, w_d):
    return ((a @ w_g.T) * ref_silu(a @ w_u.T)) @ w_d.T


def _swiglu_no_gate(a, w_g, w_u, w_d):
    return (a @ w_u.T) @ w_d.T


def _shared_dropped(x, w_gs, w_us, w_ds):
    return np.zeros((x.shape[0], w_ds.shape[0]))


def _softmax_no_exp(L):
    return L / L.sum(axis=1, keepdims=True)


def _softmax_over_k_only(L):
    # softmax restricted to the largest two entries (top-k before softmax)
    out = np.zeros_like(L)
    order = np.argsort(-L, axis=1, kind="stable")[:, :2]
    v = np.take_along_axis(L, order, 1)
    e = np.exp(v - v.max(axis=1, keepdims=True))
    np.put_along_axis(out, order, e / e.sum(axis=1, keepdims=True), 1)
    return out


def ref_silu(a):
    return a / (1.0 + np.exp(-a))


def _experts_shifted(z, perm, offsets, weights):
    S = perm.shape[0]
    H = np.zeros((S, z.shape[1]))
    E = weights.num_experts
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        w_g, w_u, w_d = weights.expert((e + 1) % E)
        H[lo:hi] = ref.swiglu_ffn(z[perm[lo:hi]], w_g, w_u, w_d)
    return H


MUTATIONS = {
    "silu_wrong_sign": ("silu", _silu_wrong_sign),
    "silu_is_sigmoid": ("silu", _silu_is_sigmoid),
    "gates_all_one": ("select_gates", _gates_all_one),
    "gates_always_renorm": ("select_gates", _gates_always_renorm),
    "topk_ties_high_first": ("top_k_stable", _topk_ties_high_first),
    "topk_ascending": ("top_k_stable", _topk_ascending),
    "logits_no_bias": ("router_logits", _logits_no_bias),
    "down_transposed": ("latent_down", _down_transposed),
    "up_transposed": ("latent_up", _up_transposed),
    "combine_drop_last": ("combine", _combine_drop_last),
    "combine_unweighted": ("combine", _combine_unweighted),
    "sort_tokens_reversed": ("counting_sort", _sort_tokens_reversed),
    "swiglu_silu_on_up": ("swiglu_ffn", _swiglu_silu_on_up),
    "swiglu_no_gate": ("swiglu_ffn", _swiglu_no_gate),
    "shared_dropped": ("shared_expert", _shared_dropped),
    "softmax_no_exp": ("softmax_rows", _softmax_no_exp),
    "softmax_over_k_only": ("softmax_rows", _softmax_over_k_only),
    "experts_shifted": ("run_experts", _experts_shifted),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTATIONS[name]
    monkeypatch.setattr(ref, attr, fn)
    caught = []
    for check in oracle_pins.ALL_CHECKS:
        try:
            check(ref)
        except Exception as exc:  # an assertion, or a shape error from a transposed operand
            caught.append((check.__name__, type(exc).__name__))
    assert caught, f"mutation {name} passed every pin"

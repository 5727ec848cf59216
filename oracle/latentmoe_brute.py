"""Brute-force second form of the LatentMoE oracle (test infrastructure).

Only ``tests/`` may import this module. It restates the same layer as
``latentmoe_ref`` with scalar Python loops and no library routine beyond
``math.exp``: every expert is evaluated on every token and multiplied by a
0/1 selection mask, top-k is picked by repeated scans, and slots come from
counting earlier tokens directly. It exists to pin the vectorised oracle on
tiny shapes; it is far too slow for anything else.

Passages followed are those of ``latentmoe_ref``: "The Training and RL
Infrastructure Behind MAI-Thinking-1" (sections "The model the systems run",
"2. Numerics", "Bitwise determinism") and "MAI-Base-2: Microsoft's 2.8T base
model, and whether its compute numbers add up" (section "The model").
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional


def _matvec(w, v) -> List[float]:
    """w [out][in] times v [in] with a plain double loop."""
    out = []
    for r in range(len(w)):
        s = 0.0
        row = w[r]
        for i in range(len(v)):
            s += row[i] * v[i]
        out.append(s)
    return out


def _silu(a: float) -> float:
    return a / (1.0 + math.exp(-a))


def _ffn(v, wg, wu, wd) -> List[float]:
    g = _matvec(wg, v)
    u = _matvec(wu, v)
    h = [_silu(g[i]) * u[i] for i in range(len(g))]
    return _matvec(wd, h)


def _pick_top_k(L: List[float], k: int) -> List[int]:
    """Repeated scan: the largest remaining logit, lowest index on equal values."""
    chosen: List[int] = []
    for _ in range(k):
        best = -1
        for e in range(len(L)):
            if e in chosen:
                continue
            if best < 0 or L[e] > L[best]:
                best = e
        chosen.append(best)
    return chosen


def forward(x, w_r, w_dn, w_up, w_g, w_u, w_d, k: int, b_r=None,
            renorm: bool = False, w_gs=None, w_us=None, w_ds=None,
            logits=None, replay_idx=None, replay_gates=None) -> Dict[str, object]:
    """All arguments are nested lists (or arrays indexable as lists).

    ``replay_idx`` [T][k] replaces the top-k choice (router replay); with
    ``replay_gates`` the gates are taken as given as well."""
    T = len(x)
    E = len(w_r)
    idx_all, gates_all, y_all, L_all = [], [], [], []
    for t in range(T):
        xt = [float(v) for v in x[t]]
        if logits is None:
            L = _matvec(w_r, xt)
            if b_r is not None:
                L = [L[e] + float(b_r[e]) for e in range(E)]
        else:
            L = [float(v) for v in logits[t]]
        m = max(L)
        ex = [math.exp(L[e] - m) for e in range(E)]
        tot = 0.0
        for v in ex:
            tot += v
        p = [v / tot for v in ex]
        idx = _pick_top_k(L, k) if replay_idx is None else [int(e) for e in replay_idx[t]]
        gates = [p[e] for e in idx]
        if replay_gates is not None:
            gates = [float(g) for g in replay_gates[t]]
        elif renorm:
            gs = sum(gates)
            gates = [g / gs for g in gates]
        # dense over all experts: weight 0 unless selected
        z = _matvec(w_dn, xt)
        c = [0.0] * len(z)
        for j in range(k):
            for e in range(E):
                mask = 1.0 if idx[j] == e else 0.0
                if mask == 0.0:
                    continue
                o = _ffn(z, w_g[e], w_u[e], w_d[e])
                for i in range(len(c)):
                    c[i] += mask * gates[j] * o[i]
        y = _matvec(w_up, c)
        if w_gs is not None:
            s = _ffn(xt, w_gs, w_us, w_ds)
            y = [y[i] + s[i] for i in range(len(y))]
        idx_all.append(idx)
        gates_all.append(gates)
        y_all.append(y)
        L_all.append(L)
    # slots by definition: segment start of e plus earlier tokens choosing e
    counts = [0] * E
    for t in range(T):
        for e in idx_all[t]:
            counts[e] += 1
    pos = []
    for t in range(T):
        row = []
        for e in idx_all[t]:
            start = sum(counts[:e])
            earlier = sum(1 for t2 in range(t) if e in idx_all[t2])
            row.append(start + earlier)
        pos.append(row)
    perm = [-1] * (T * k)
    for t in range(T):
        for j in range(k):
            perm[pos[t][j]] = t
    offsets = [0]
    for e in range(E):
        offsets.append(offsets[-1] + counts[e])
    return {"logits": L_all, "idx": idx_all, "gates": gates_all, "y": y_all,
            "counts": counts, "offsets": offsets, "perm": perm, "pos": pos}

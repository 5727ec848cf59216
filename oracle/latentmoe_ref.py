"""Float64 CPU oracle of the LatentMoE layer forward (test infrastructure).

This module is test infrastructure. Only ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference legs of ``bench.py`` may import it. The
product path (the CUDA library and its Python binding) never calls it, and it
shares no code with that path.

What it computes, step by step, with the passage each step follows:

1. Router logits on the full hidden state, ``L = x W_r^T (+ b)``.
   "The Training and RL Infrastructure Behind MAI-Thinking-1", section "The
   model the systems run": the router reads the whole hidden vector, and only
   the experts see the compressed latent. Section "2. Numerics" ("Pre-training
   and mid-training precision") keeps router logits in FP32; here they are
   float64, and the parity modes can feed the GPU's fp32 logits instead.
   The per-expert bias ``b`` is an input of the skewed-load workload only.
2. Softmax gating over all experts, ``p = softmax(L)`` per row (the MoE row of
   that section's shape table: top-8 of 512 experts, gated by a softmax).
3. Top-k selection by a stable sort on ``-L``: larger logit first, lower
   expert index first among equals (section "Bitwise determinism": the MoE
   top-k uses a stable sort so that equal values always resolve alike).
4. Gates are the chosen probabilities ``g[t,j] = p[t, idx[t,j]]``; dividing by
   their sum is an explicit option (``renorm``), off by default.
5. Shared latent down-projection ``z = x W_dn^T`` before dispatch (MoE row of
   the shape table: one down-projection to width 3072, shared by all experts,
   applied before the tokens are dispatched).
6. Counting sort of the T*k (token, choice) slots by expert, stable in token
   order: ``n_e`` = slots of expert e, ``o_e`` = exclusive prefix sum, the slot
   of (t, j) is ``o_e + #{t' < t : e in idx[t']}``; ``perm[slot] = t`` and
   ``pos[t, j] = slot``. This is the dropless "expert encode" layout
   (section "3. Training", "Custom kernels"; "Memory and dropless MoE").
7. Per-expert SwiGLU FFN on the latent rows of its segment,
   ``H_e = (SiLU(Z_e W_g^T) * (Z_e W_u^T)) W_d^T`` with ``SiLU(a) = a/(1+e^-a)``
   (shape table: the feed-forward blocks are SwiGLU; expert FFN width 10240).
8. Gate-weighted combine ``c[t] = sum_j g[t,j] H[pos[t,j]]`` in j order
   (section "2. Numerics" lists the MoE combine among the FP32 steps).
9. Up-projection back to hidden width, ``y = c W_up^T``; with a shared expert,
   ``y += (SiLU(x W_gs^T) * (x W_us^T)) W_ds^T`` on the full width, unweighted
   ("MAI-Base-2: Microsoft's 2.8T base model, and whether its compute numbers
   add up", section "The model": each token also goes through one shared
   expert, which works on the full width without the down/up projection).

Readings where the pages leave a step open: softmax over all E experts before
selection; no renorm by default; selection compares logits; projections carry
no bias; the shared expert has weight 1 and is added after the up-projection.

Inputs are the bf16-rounded tensors upcast exactly to float64. No
intermediate is rounded.
"""
from __future__ import annotations

from typing import Callable, Dict, Optional, Tuple

import numpy as np

ExpertFn = Callable[[int], Tuple[np.ndarray, np.ndarray, np.ndarray]]


class OracleWeights:
    """Float64 weights in nn.Linear layout [out, in].

    ``expert(e)`` returns ``(w_g [F,l], w_u [F,l], w_d [l,F])``; for the large
    shapes it can fetch one expert at a time so that all experts never sit in
    host memory together.
    """

    def __init__(self, w_r, w_dn, w_up, expert: ExpertFn, b_r=None,
                 w_gs=None, w_us=None, w_ds=None):
        self.w_r = np.asarray(w_r, dtype=np.float64)
        self.b_r = None if b_r is None else np.asarray(b_r, dtype=np.float64)
        self.w_dn = np.asarray(w_dn, dtype=np.float64)
        self.w_up = np.asarray(w_up, dtype=np.float64)
        self.expert = expert
        self.w_gs = None if w_gs is None else np.asarray(w_gs, dtype=np.float64)
        self.w_us = None if w_us is None else np.asarray(w_us, dtype=np.float64)
        self.w_ds = None if w_ds is None else np.asarray(w_ds, dtype=np.float64)

    @property
    def num_experts(self) -> int:
        return self.w_r.shape[0]

    @staticmethod
    def from_stacked(w_r, w_dn, w_up, w_g, w_u, w_d, b_r=None,
                     w_gs=None, w_us=None, w_ds=None) -> "OracleWeights":
        """From stacked expert arrays w_g/w_u [E,F,l] and w_d [E,l,F]."""
        w_g = np.asarray(w_g, dtype=np.float64)
        w_u = np.asarray(w_u, dtype=np.float64)
        w_d = np.asarray(w_d, dtype=np.float64)
        return OracleWeights(w_r, w_dn, w_up, lambda e: (w_g[e], w_u[e], w_d[e]),
                             b_r=b_r, w_gs=w_gs, w_us=w_us, w_ds=w_ds)


def silu(a: np.ndarray) -> np.ndarray:
    """SiLU(a) = a * sigmoid(a) = a / (1 + exp(-a))."""
    return a / (1.0 + np.exp(-a))


def router_logits(x: np.ndarray, w_r: np.ndarray, b_r: Optional[np.ndarray] = None) -> np.ndarray:
    """Step 1: L = x W_r^T (+ b), shape [T, E]."""
    L = x @ w_r.T
    if b_r is not None:
        L = L + b_r[None, :]
    return L


def softmax_rows(L: np.ndarray) -> np.ndarray:
    """Step 2: row softmax over all experts (max subtracted for range only)."""
    m = L.max(axis=1, keepdims=True)
    e = np.exp(L - m)
    return e / e.sum(axis=1, keepdims=True)


def top_k_stable(L: np.ndarray, k: int) -> np.ndarray:
    """Step 3: first k experts of a stable sort on -L (ties: lower index first)."""
    order = np.argsort(-L, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def select_gates(p: np.ndarray, idx: np.ndarray, renorm: bool = False) -> np.ndarray:
    """Step 4: g[t,j] = p[t, idx[t,j]], divided by sum_j g[t,j] if renorm."""
    g = np.take_along_axis(p, idx, axis=1)
    if renorm:
        g = g / g.sum(axis=1, keepdims=True)
    return g


def latent_down(x: np.ndarray, w_dn: np.ndarray) -> np.ndarray:
    """Step 5: z = x W_dn^T, shape [T, l]."""
    return x @ w_dn.T


def counting_sort(idx: np.ndarray, E: int):
    """Step 6: counts [E], offsets [E+1], perm [T*k], pos [T,k].

    Slots are handed out by walking tokens in order and, inside a token, its
    choices in slot order j; each expert's next free slot is o_e plus the
    number of earlier tokens that chose it.
    """
    T, k = idx.shape
    counts = np.zeros(E, dtype=np.int64)
    for e in idx.ravel():
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts)
    fill = np.zeros(E, dtype=np.int64)
    perm = np.full(T * k, -1, dtype=np.int64)
    pos = np.full((T, k), -1, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            slot = offsets[e] + fill[e]
            fill[e] += 1
            perm[slot] = t
            pos[t, j] = slot
    return counts, offsets, perm, pos


def swiglu_ffn(a: np.ndarray, w_g: np.ndarray, w_u: np.ndarray, w_d: np.ndarray) -> np.ndarray:
    """(SiLU(a W_g^T) * (a W_u^T)) W_d^T."""
    return (silu(a @ w_g.T) * (a @ w_u.T)) @ w_d.T


def run_experts(z: np.ndarray, perm: np.ndarray, offsets: np.ndarray,
                weights: OracleWeights) -> np.ndarray:
    """Step 7: H [T*k, l]; segment e holds expert e's outputs in slot order."""
    S = perm.shape[0]
    H = np.zeros((S, z.shape[1]), dtype=np.float64)
    for e in range(weights.num_experts):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        w_g, w_u, w_d = weights.expert(e)
        H[lo:hi] = swiglu_ffn(z[perm[lo:hi]], w_g, w_u, w_d)
    return H


def combine(H: np.ndarray, gates: np.ndarray, pos: np.ndarray) -> np.ndarray:
    """Step 8: c[t] = sum_j g[t,j] H[pos[t,j]], summed in j order."""
    T, k = pos.shape
    c = np.zeros((T, H.shape[1]), dtype=np.float64)
    for j in range(k):
        c += gates[:, j:j + 1] * H[pos[:, j]]
    return c


def latent_up(c: np.ndarray, w_up: np.ndarray) -> np.ndarray:
    """Step 9a: y = c W_up^T, shape [T, d]."""
    return c @ w_up.T


def shared_expert(x: np.ndarray, w_gs, w_us, w_ds) -> np.ndarray:
    """Step 9b: full-width SwiGLU shared expert, weight 1."""
    return swiglu_ffn(x, w_gs, w_us, w_ds)


def forward(x: np.ndarray, weights: OracleWeights, k: int, renorm: bool = False,
            logits: Optional[np.ndarray] = None,
            select_bias: Optional[np.ndarray] = None,
            select_logits: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """The whole layer on x [T, d]; returns every intermediate.

    ``logits`` (e.g. the GPU's fp32 router logits) replaces step 1 when given;
    selection and gates then follow from those values exactly.

    ``select_bias`` [E] is the selection-only reading of the loss-free
    balancer that "The Training and RL Infrastructure Behind MAI-Thinking-1"
    names without a mechanism (section "Sharding and parallelism"): the bias
    moves the top-k choice (step 3 ranks L + b) while the gates stay the
    softmax probabilities of the unbiased logits (steps 2 and 4).
    ``select_logits`` [T, E] gives that ranking key directly (L + b as another
    implementation rounded it), so that a comparison can take the choice in
    the other side's precision.
    """
    x = np.asarray(x, dtype=np.float64)
    E = weights.num_experts
    if logits is None:
        L = router_logits(x, weights.w_r, weights.b_r)
    else:
        L = np.asarray(logits, dtype=np.float64)
    p = softmax_rows(L)
    if select_logits is not None:
        idx = top_k_stable(np.asarray(select_logits, dtype=np.float64), k)
    elif select_bias is None:
        idx = top_k_stable(L, k)
    else:
        idx = top_k_stable(L + np.asarray(select_bias, dtype=np.float64)[None, :], k)
    g = select_gates(p, idx, renorm)
    z = latent_down(x, weights.w_dn)
    counts, offsets, perm, pos = counting_sort(idx, E)
    H = run_experts(z, perm, offsets, weights)
    c = combine(H, g, pos)
    y = latent_up(c, weights.w_up)
    if weights.w_gs is not None:
        y = y + shared_expert(x, weights.w_gs, weights.w_us, weights.w_ds)
    return {"logits": L, "p": p, "idx": idx, "gates": g, "z": z,
            "counts": counts, "offsets": offsets, "perm": perm, "pos": pos,
            "H": H, "c": c, "y": y}


def forward_routed(x: np.ndarray, weights: OracleWeights, idx: np.ndarray,
                   gates: Optional[np.ndarray] = None, renorm: bool = False,
                   logits: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """The layer with the expert choices given (router replay).

    "The Training and RL Infrastructure Behind MAI-Thinking-1": the MoE layer
    supports router replay (section "Sharding and parallelism"), and the
    expert choices made during inference are recorded and replayed in the
    learner's pass (section "4. RL infrastructure"). ``idx`` [T, k] replaces
    steps 1-3. Gates are taken as given; when ``gates`` is None they are the
    softmax probabilities of the replayed experts under this layer's router
    (step 4 on the replayed choices).
    """
    x = np.asarray(x, dtype=np.float64)
    idx = np.asarray(idx, dtype=np.int64)
    E = weights.num_experts
    if gates is None:
        L = router_logits(x, weights.w_r, weights.b_r) if logits is None else \
            np.asarray(logits, dtype=np.float64)
        g = select_gates(softmax_rows(L), idx, renorm)
    else:
        g = np.asarray(gates, dtype=np.float64)
    z = latent_down(x, weights.w_dn)
    counts, offsets, perm, pos = counting_sort(idx, E)
    H = run_experts(z, perm, offsets, weights)
    c = combine(H, g, pos)
    y = latent_up(c, weights.w_up)
    if weights.w_gs is not None:
        y = y + shared_expert(x, weights.w_gs, weights.w_us, weights.w_ds)
    return {"idx": idx, "gates": g, "counts": counts, "offsets": offsets, "perm": perm,
            "pos": pos, "c": c, "y": y}


def route(logits: np.ndarray, E: int, k: int, renorm: bool = False,
          select_bias: Optional[np.ndarray] = None,
          select_logits: Optional[np.ndarray] = None) -> Dict[str, np.ndarray]:
    """Steps 2-4 and 6 from given logits: the routing half of the layer."""
    L = np.asarray(logits, dtype=np.float64)
    p = softmax_rows(L)
    if select_logits is not None:
        idx = top_k_stable(np.asarray(select_logits, dtype=np.float64), k)
    elif select_bias is None:
        idx = top_k_stable(L, k)
    else:
        idx = top_k_stable(L + np.asarray(select_bias, dtype=np.float64)[None, :], k)
    g = select_gates(p, idx, renorm)
    counts, offsets, perm, pos = counting_sort(idx, E)
    return {"idx": idx, "gates": g, "counts": counts, "offsets": offsets,
            "perm": perm, "pos": pos}



def lbl_stats(logits: np.ndarray, idx: np.ndarray, E: int):
    """Load-balancing statistics of one batch: slots per expert and the sum
    over tokens of each expert's router probability.

    "The Training and RL Infrastructure Behind MAI-Thinking-1" (section
    "Sharding and parallelism") uses a global-batch load-balancing loss,
    aggregated across data-parallel workers and micro-batches; "Frontier
    Pre-training at Microsoft AI" (section "Reducing per-expert overhead")
    batches it across layers. The loss formula and its coefficient are not on
    the pages, so these are the per-batch statistics such a loss is built
    from: counts n_e (sum them over batches, divide by the total slots for
    f_e) and prob_sum_e = sum_t softmax(L_t)_e (sum over batches, divide by
    the total tokens for the mean probability P_e).
    """
    p = softmax_rows(np.asarray(logits, dtype=np.float64))
    counts = np.zeros(E, dtype=np.int64)
    for e in np.asarray(idx).ravel():
        counts[e] += 1
    return counts, p.sum(axis=0)

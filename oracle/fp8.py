"""FP8 E4M3 forward of the expert FFNs in the oracle (test infrastructure).

Only ``tests/`` and ``bench.py``'s CPU legs may import this module; it shares
no code with the CUDA library.

"The Training and RL Infrastructure Behind MAI-Thinking-1", section
"2. Numerics": forward GEMMs run in FP8 E4M3, and every FP8 operation uses
delayed scaling with a 1,024-step history of the absolute maximum. This
module restates that for the two expert GEMMs of the layer:

- E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinities, the
  largest finite value 448, subnormals down to 2^-9. Rounding is to nearest,
  ties to even; magnitudes above 448 saturate to 448.
- A tensor t with scale s is stored as q = E4M3(t / s) and stands for q * s.
- Weights (static): s = amax(W_e) / 448 per expert matrix.
- Activations: z (input of gate/up) and h (input of down) use per-tensor
  scales from delayed scaling; the scales are inputs here (the GPU reports
  the ones it used).
- g = (q_z q_g^T) s_z s_g, u = (q_z q_u^T) s_z s_u, h = SiLU(g) u,
  o = (q_h q_d^T) s_h s_d.
- With the dense GEMMs in E4M3 too (forward_fp8's ``dense``): x, the
  combined latent c and the shared expert's hidden are quantized with their
  own per-tensor scales, and the latent projections and the shared expert's
  weights with one scale per matrix; the router keeps fp32 logits (the
  pages keep routing in FP32).

Readings where the pages are silent: scales are per tensor, and per expert
for the expert weights; the history starts empty and a scale of 1 is used
until it holds a non-zero maximum.

Delayed scaling (DelayedScaling below): forward n quantizes with the scale
made from the maxima of forwards n-1024 .. n-1 (s = max / 448, formed in
fp32); the maximum forward n records enters the history afterwards. A window
whose maxima are all zero leaves the scale as it was.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np

from oracle import latentmoe_ref as ref

E4M3_MAX = 448.0


def round_e4m3(x) -> np.ndarray:
    """Nearest E4M3 value (ties to even), saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    # spacing of representable values: 2^(e-3) in binade e >= -6, 2^-9 below
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -9)))
    e = np.maximum(e, -6.0)
    q = np.exp2(e - 3.0)
    r = np.round(a / q) * q  # np.round rounds half to even
    r = np.minimum(r, E4M3_MAX)
    return np.where(x < 0, -r, r)


def e4m3_values() -> np.ndarray:
    """All non-negative finite E4M3 values, from the bit layout."""
    vals = []
    for exp in range(16):
        for man in range(8):
            if exp == 15 and man == 7:
                continue  # the NaN code
            if exp == 0:
                vals.append(man * 2.0 ** -9)
            else:
                vals.append((1.0 + man / 8.0) * 2.0 ** (exp - 7))
    return np.array(sorted(set(vals)))


HISTORY = 1024


class DelayedScaling:
    """Scales of a few activation tensors from a ring of recorded maxima."""

    def __init__(self, n: int, length: int = HISTORY):
        self.length = length
        self.hist = np.zeros((n, length), dtype=np.float32)
        self.scales = np.ones(n, dtype=np.float32)
        self.steps = 0

    def record(self, amax) -> np.ndarray:
        """Enter one forward's maxima (fp32) and return the next scales."""
        amax = np.asarray(amax, dtype=np.float32)
        self.hist[:, self.steps % self.length] = amax
        self.steps += 1
        m = self.hist.max(axis=1)
        for i in range(m.shape[0]):
            if m[i] > 0:
                self.scales[i] = np.float32(m[i]) / np.float32(E4M3_MAX)
        return self.scales.copy()


def weight_scale(w: np.ndarray) -> float:
    """amax / 448 in fp32, the way the kernel forms it (1 for an all-zero matrix)."""
    amax = np.float32(np.max(np.abs(w))) if w.size else np.float32(0)
    if amax == 0:
        return 1.0
    return float(np.float32(amax) / np.float32(E4M3_MAX))


def quantize_weight(w: np.ndarray):
    """(codes as float64 values, scale): the codes are E4M3(fp32(w) * fp32(1/s)),
    the fp32 operations the kernel uses, so the codes match it exactly."""
    s = weight_scale(w)
    inv = np.float32(1.0) / np.float32(s)
    prod = (np.asarray(w, dtype=np.float32) * inv).astype(np.float64)
    return round_e4m3(prod), s


def quantize_input(t: np.ndarray, s: float) -> np.ndarray:
    """Codes of a tensor given in bf16 (exact in fp32) with scale s, the
    product taken in fp32 as the kernel does: E4M3(fp32(t) * fp32(1/s))."""
    inv = np.float32(1.0) / np.float32(s)
    return round_e4m3((np.asarray(t, dtype=np.float32) * inv).astype(np.float64))


def quantize_act(t: np.ndarray, s: float) -> np.ndarray:
    """Activation codes E4M3(t * (1/s)); t is the float64 oracle value."""
    inv = float(np.float32(1.0) / np.float32(s))
    return round_e4m3(np.asarray(t, dtype=np.float64) * inv)


def forward_fp8(x: np.ndarray, weights: ref.OracleWeights, k: int, s_z: float, s_h: float,
                renorm: bool = False, logits: Optional[np.ndarray] = None,
                z_codes: Optional[np.ndarray] = None,
                h_codes: Optional[np.ndarray] = None,
                wq_cache: Optional[dict] = None,
                dense: Optional[dict] = None) -> Dict[str, np.ndarray]:
    """The layer with FP8 E4M3 expert GEMMs; everything else as ref.forward.

    z_codes [T*k, l] / h_codes [T*k, F] (E4M3 code values, slot order), when
    given, replace the codes this function would form for z and h: the
    expert GEMMs are then evaluated on exactly those codes. The returned
    "z_q" and "h_q" are the codes used, and "h" the unquantized h.
    wq_cache, a dict kept by the caller, holds each expert's quantized
    weights across calls on the same weights.

    dense, when given, runs the other forward GEMMs in E4M3 as well (the
    router keeps its fp32 logits): {"s_x", "s_c", "s_sh"} are the scales of
    x, of the combined latent c and of the shared expert's hidden SiLU(g)*u;
    optional "x_codes" [T, d], "c_codes" [T, l], "sh_codes" [T, F_s] replace
    the codes formed here. Then z = s_x s_dn (x_q W_dn_q^T), y = s_c s_up
    (c_q W_up_q^T) + s_sh s_ds (sh_q W_ds_q^T) with sh from s_x-scaled
    products of x_q and the shared weights' codes."""
    x = np.asarray(x, dtype=np.float64)
    E = weights.num_experts
    L = ref.router_logits(x, weights.w_r, weights.b_r) if logits is None else \
        np.asarray(logits, dtype=np.float64)
    p = ref.softmax_rows(L)
    idx = ref.top_k_stable(L, k)
    g = ref.select_gates(p, idx, renorm)
    out = {}
    if dense is None:
        z = ref.latent_down(x, weights.w_dn)
    else:
        s_x = dense["s_x"]
        # x is given in bf16: its codes are decided from the fp32 product, as
        # in the kernel, so both sides start from the same codes
        xq = quantize_input(x, s_x) if dense.get("x_codes") is None else \
            np.asarray(dense["x_codes"], dtype=np.float64)
        qdn, sdn = quantize_weight(weights.w_dn)
        z = (xq @ qdn.T) * (s_x * sdn)
        out.update({"x_q": xq, "x_amax": float(np.abs(x).max()) if x.size else 0.0, "z": z})
    counts, offsets, perm, pos = ref.counting_sort(idx, E)
    zq_slots = quantize_act(z, s_z)[perm] if z_codes is None else \
        np.asarray(z_codes, dtype=np.float64)
    H = np.zeros((perm.shape[0], z.shape[1]), dtype=np.float64)
    h_all = hq_all = None  # [T*k, F], allocated once F is known
    h_amax = 0.0
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue
        if wq_cache is not None and e in wq_cache:
            (qg, sg), (qu, su), (qd, sd) = wq_cache[e]
        else:
            w_g, w_u, w_d = weights.expert(e)
            qg, sg = quantize_weight(w_g)
            qu, su = quantize_weight(w_u)
            qd, sd = quantize_weight(w_d)
            if wq_cache is not None:
                wq_cache[e] = ((qg, sg), (qu, su), (qd, sd))
        zq = zq_slots[lo:hi]
        gate = (zq @ qg.T) * (s_z * sg)
        up = (zq @ qu.T) * (s_z * su)
        h = ref.silu(gate) * up
        h_amax = max(h_amax, float(np.abs(h).max()))
        qh = quantize_act(h, s_h) if h_codes is None else \
            np.asarray(h_codes[lo:hi], dtype=np.float64)
        if h_all is None:
            h_all = np.zeros((perm.shape[0], qg.shape[0]), dtype=np.float64)
            hq_all = np.zeros_like(h_all)
        h_all[lo:hi] = h
        hq_all[lo:hi] = qh
        H[lo:hi] = (qh @ qd.T) * (s_h * sd)
    c = ref.combine(H, g, pos)
    if dense is None:
        y = ref.latent_up(c, weights.w_up)
        if weights.w_gs is not None:
            y = y + ref.shared_expert(x, weights.w_gs, weights.w_us, weights.w_ds)
    else:
        s_c, s_sh = dense["s_c"], dense["s_sh"]
        cq = quantize_act(c, s_c) if dense.get("c_codes") is None else \
            np.asarray(dense["c_codes"], dtype=np.float64)
        qup, sup = quantize_weight(weights.w_up)
        y = (cq @ qup.T) * (s_c * sup)
        out.update({"c": c, "c_q": cq, "c_amax": float(np.abs(c).max()) if c.size else 0.0})
        if weights.w_gs is not None:
            qgs, sgs = quantize_weight(weights.w_gs)
            qus, sus = quantize_weight(weights.w_us)
            qds, sds = quantize_weight(weights.w_ds)
            sh = ref.silu((xq @ qgs.T) * (s_x * sgs)) * ((xq @ qus.T) * (s_x * sus))
            shq = quantize_act(sh, s_sh) if dense.get("sh_codes") is None else \
                np.asarray(dense["sh_codes"], dtype=np.float64)
            y = y + (shq @ qds.T) * (s_sh * sds)
            out.update({"sh": sh, "sh_q": shq, "sh_amax": float(np.abs(sh).max())})
    # the maxima delayed scaling records for the next step's scales
    z_amax = float(np.abs(z).max()) if z.size else 0.0
    out.update({"idx": idx, "gates": g, "counts": counts, "offsets": offsets, "pos": pos,
                "perm": perm, "y": y, "z_amax": z_amax, "h_amax": h_amax, "z_q": zq_slots,
                "h": h_all, "h_q": hq_all, "o": H})
    return out

"""Shared helpers for the GPU parity tests (GPU path vs the float64 oracle)."""
from __future__ import annotations

import numpy as np
import torch

from mixture_experts_layer_router_gb300 import build, capi, synth
from oracle import latentmoe_ref as ref

# Parity bounds for the layer output (bf16 data, fp32 accumulation) and the
# router logits; the integer routing outputs are compared exactly.
Y_REL_FRO = 1e-2
Y_MAX_ABS = 3e-2
LOGIT_MAX_ABS = 1e-2

_built = False


def lib():
    global _built
    if not _built:
        build.build()
        _built = True
    return capi.load()


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def oracle_weights(w, stacked: bool = True) -> ref.OracleWeights:
    """Float64 oracle weights from the device tensors the GPU path uses."""
    if stacked:
        return ref.OracleWeights.from_stacked(
            f64(w["w_r"]), f64(w["w_dn"]), f64(w["w_up"]), f64(w["w_g"]), f64(w["w_u"]),
            f64(w["w_d"]), b_r=None if w["b_r"] is None else f64(w["b_r"]),
            w_gs=None if w["w_gs"] is None else f64(w["w_gs"]),
            w_us=None if w["w_us"] is None else f64(w["w_us"]),
            w_ds=None if w["w_ds"] is None else f64(w["w_ds"]))

    def expert(e):  # one expert at a time: the large shapes do not fit in host fp64
        return f64(w["w_g"][e]), f64(w["w_u"][e]), f64(w["w_d"][e])

    return ref.OracleWeights(
        f64(w["w_r"]), f64(w["w_dn"]), f64(w["w_up"]), expert,
        b_r=None if w["b_r"] is None else f64(w["b_r"]),
        w_gs=None if w["w_gs"] is None else f64(w["w_gs"]),
        w_us=None if w["w_us"] is None else f64(w["w_us"]),
        w_ds=None if w["w_ds"] is None else f64(w["w_ds"]))


def make_layer(cfg: synth.LayerConfig, w, max_tokens=None, renorm=False, out_fp32=False,
               fp8=False, fp8_dense=False):
    lib()
    layer = capi.LatentMoE(cfg.d, cfg.l, cfg.E, cfg.k, cfg.F, cfg.Fs,
                           max_tokens=max_tokens or cfg.T, renorm=renorm,
                           router_bias=w["b_r"] is not None, out_fp32=out_fp32, fp8=fp8,
                           fp8_dense=fp8_dense)
    layer.load_weights(w)
    return layer


def assert_y_close(y_gpu: torch.Tensor, y_ref: np.ndarray, what: str = "y"):
    y = f64(y_gpu)
    diff = y - y_ref
    rel = np.linalg.norm(diff) / max(np.linalg.norm(y_ref), 1e-30)
    mx = np.abs(diff).max()
    assert rel <= Y_REL_FRO and mx <= Y_MAX_ABS, f"{what}: rel fro {rel:.3e}, max abs {mx:.3e}"
    return rel, mx


def assert_routing_equal(gpu: dict, ora: dict, T: int, k: int):
    """idx, counts, offsets, perm, pos bit-exact; gates to fp32 rounding."""
    assert np.array_equal(gpu["idx"].cpu().numpy().reshape(T, k), ora["idx"])
    assert np.array_equal(gpu["counts"].cpu().numpy(), ora["counts"])
    assert np.array_equal(gpu["offsets"].cpu().numpy(), ora["offsets"])
    assert np.array_equal(gpu["perm"].cpu().numpy(), ora["perm"])
    assert np.array_equal(gpu["pos"].cpu().numpy().reshape(T, k), ora["pos"])
    np.testing.assert_allclose(f64(gpu["gates"]).reshape(T, k), ora["gates"], rtol=2e-6,
                               atol=1e-9)


# ---------------------------------------------------------------- token samples at full size

def slot_chunks(n: int):
    """[(first, end)) slot ranges, relative to an expert's first slot, of every
    token chunk the expert GEMMs cut an expert of n slots into: the one-SM
    kernels' and the SM-pair gate+up kernel's chunks (at most 256 slots,
    split evenly, each a multiple of 16 slots except the last) and, for
    n > 256, the SM-pair down GEMM's wide chunks (at most 512 slots, split
    the same way) with the two token ranges of a wide chunk of more than 256
    slots (its first 256 slots, which one MMA covers, and the rest, which a
    second MMA covers)."""
    if n <= 0:
        return []

    def even(limit):
        nch = -(-n // limit)
        cs = (-(-n // nch) + 15) & ~15
        return [(c * cs, min((c + 1) * cs, n)) for c in range(nch)]

    out = even(256)
    if n > 256:
        for lo, hi in even(512):
            out.append((lo, hi))
            if hi - lo > 256:
                out += [(lo, lo + 256), (lo + 256, hi)]
    return sorted(set(out))


def covering_tokens(routing: dict, T: int, k: int, n_min: int, seed: int = 1,
                    last_slots: bool = True, n_max: int = None) -> np.ndarray:
    """Sorted token ids whose slots reach every expert GEMM tile of the forward.

    From the GPU's routing (counts, offsets, perm): (1) with ``last_slots``,
    the token holding the last slot of every non-empty expert (the ragged
    tail of its last tile); (2) greedily, tokens until every chunk of every
    expert has a sampled slot; (3) the seeded sample ``synth.sample_tokens``
    until there are ``n_min`` tokens. With ``n_max``, step (2) stops there
    (it picks the token covering the most uncovered chunks first)."""
    counts = routing["counts"].cpu().numpy().astype(np.int64)
    offsets = routing["offsets"].cpu().numpy().astype(np.int64)
    perm = routing["perm"].cpu().numpy().astype(np.int64)
    chosen = set()
    if last_slots:
        for e in np.nonzero(counts)[0]:
            chosen.add(int(perm[offsets[e + 1] - 1]))
    # every (expert, chunk) as a requirement; a token meets those its slots fall in
    need = {}
    for e in np.nonzero(counts)[0]:
        for c, (lo, hi) in enumerate(slot_chunks(int(counts[e]))):
            toks = perm[offsets[e] + lo:offsets[e] + hi]
            if not any(int(t) in chosen for t in toks):
                need[(int(e), c)] = set(int(t) for t in toks)
    by_token = {}
    for req, toks in need.items():
        for t in toks:
            by_token.setdefault(t, set()).add(req)
    while need and (n_max is None or len(chosen) < n_max):
        t = max(by_token, key=lambda u: (len(by_token[u]), -u))
        for req in list(by_token[t]):
            for u in need.pop(req):
                if u != t:
                    by_token[u].discard(req)
        del by_token[t]
        by_token = {u: r for u, r in by_token.items() if r}
        chosen.add(t)
    for t in synth.sample_tokens(T, T, seed=seed).numpy():
        if len(chosen) >= n_min:
            break
        chosen.add(int(t))
    return np.array(sorted(chosen), dtype=np.int64)


class ExpertPrefetch:
    """Float64 expert weights for ``ref.OracleWeights``, copied from the
    device a few experts ahead of the oracle's expert loop (which asks in
    ascending order) on worker threads; nothing is kept once handed out."""

    def __init__(self, w, experts, window: int = 6):
        from concurrent.futures import ThreadPoolExecutor
        self.w = w
        self.order = sorted(int(e) for e in experts)
        self.window = window
        self.pool = ThreadPoolExecutor(window)
        self.futs = {}
        self.next = 0
        self._fill()

    def _load(self, e):
        return f64(self.w["w_g"][e]), f64(self.w["w_u"][e]), f64(self.w["w_d"][e])

    def _fill(self):
        while self.next < len(self.order) and len(self.futs) < self.window:
            e = self.order[self.next]
            self.next += 1
            self.futs[e] = self.pool.submit(self._load, e)

    def __call__(self, e):
        fut = self.futs.pop(int(e), None)
        self._fill()
        return self._load(e) if fut is None else fut.result()

    def close(self):
        self.pool.shutdown(wait=True, cancel_futures=True)


class E4M3WeightCodes:
    """``wq_cache`` for ``oracle.fp8.forward_fp8``: the oracle's own
    ``quantize_weight`` of each listed expert's three matrices, computed once
    on worker threads and kept as float16 (every E4M3 value is exact in
    float16, so the copy loses nothing), handed out as float64."""

    def __init__(self, w, experts, threads: int = 8):
        from concurrent.futures import ThreadPoolExecutor
        from oracle import fp8 as ofp8
        self.store = {}

        def quantize(e):
            out = []
            for key in ("w_g", "w_u", "w_d"):
                q, s = ofp8.quantize_weight(f64(w[key][e]))
                q16 = q.astype(np.float16)
                out.append((q16, s))
            return e, out

        with ThreadPoolExecutor(threads) as ex:
            for e, out in ex.map(quantize, sorted(int(e) for e in experts)):
                self.store[e] = out
        first = next(iter(self.store.values()), None)
        if first is not None:  # the float16 copy is exact
            q, _ = ofp8.quantize_weight(f64(w["w_g"][next(iter(self.store))]))
            assert np.array_equal(first[0][0].astype(np.float64), q)

    def __contains__(self, e):
        return int(e) in self.store

    def __getitem__(self, e):
        return tuple((q.astype(np.float64), s) for q, s in self.store[int(e)])

    def __setitem__(self, e, v):
        self.store[int(e)] = [(q.astype(np.float16), s) for q, s in v]

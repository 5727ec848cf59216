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

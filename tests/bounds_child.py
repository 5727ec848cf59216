"""Run by tests/test_gpu_bounds.py in a child process whose LATENTMOE_LIB
names the bounds-checked debug build of the library (-DLMOE_BOUNDS: every
epilogue store, scatter write and combine read checks its row and reports an
access outside its buffer through LATENTMOE_STATUS_BOUNDS instead of making
it). Each case runs a forward path, requires the device status to carry no
bounds bit, and checks the output against the oracle. Prints one line per
case and "bounds build: all cases clean" at the end; exits non-zero on the
first failure."""
import os
import sys

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, HERE)
sys.path.insert(0, os.path.dirname(HERE))

from mixture_experts_layer_router_gb300 import capi, synth  # noqa: E402
import gpu_helpers as gh  # noqa: E402
from oracle import latentmoe_ref as ref  # noqa: E402


def _layer(cfg, seed, **kw):
    w = synth.make_weights(cfg, seed, "cuda")
    x = synth.make_x(cfg, seed, "cuda")
    return w, x, gh.make_layer(cfg, w, **kw)


def _status(layer):
    torch.cuda.synchronize()
    return layer.status()


def _check_forward(name, cfg, seed, T=None, **kw):
    w, x, layer = _layer(cfg, seed, **kw)
    x = x[: (T or cfg.T)]
    y = layer.forward(x)
    r = layer.get_routing(x.shape[0], "cuda")
    st = _status(layer)
    assert st == 0, (name, st)
    ora = ref.forward(gh.f64(x), gh.oracle_weights(w), cfg.k, logits=gh.f64(r["logits"]),
                      renorm=kw.get("renorm", False))
    gh.assert_y_close(y, ora["y"], what=name)
    print(f"{name}: status 0, y within the parity bounds", flush=True)
    return w, x, layer, y


def main():
    assert capi.LIB_PATH == os.environ.get("LATENTMOE_LIB"), capi.LIB_PATH
    gh.lib()
    tiny = synth.CONFIGS["tiny"]
    _check_forward("tiny", tiny, 0)
    _check_forward("tiny, ragged T = 77, renorm", tiny, 1, T=77, renorm=True)
    mid_ragged = synth.LayerConfig("mid-ragged", T=1000, d=512, l=512, E=24, k=3, F=512)
    _check_forward("ragged T = 1000 across tiles", mid_ragged, 2)
    shared = synth.LayerConfig("shared", T=300, d=256, l=512, E=8, k=3, F=512, Fs=256)
    _check_forward("shared expert, fp32 out", shared, 3, out_fp32=True)
    imb = synth.CONFIGS["imbalanced"]
    w, x, layer, y0 = _check_forward("imbalanced", imb, 4)

    # multi-round fixed capacity on the same layer: every round's stores
    layer.set_capacity(32, 8)
    y1 = layer.forward(x)
    st = _status(layer)
    assert st == 0, ("rounds", st)
    assert layer.rounds()["needed"] > 1
    assert torch.equal(y0, y1)
    print("imbalanced, capacity 32 in groups of 8: status 0, bitwise the one-pass output",
          flush=True)

    # router replay with expert ids outside [0, E): those slots are dropped
    # (BAD_EXPERT), and nothing is stored or read out of bounds
    w, x, layer = _layer(tiny, 6)
    rng = np.random.default_rng(2)
    idx = np.stack([rng.permutation(tiny.E)[:tiny.k] for _ in range(tiny.T)]).astype(np.int32)
    gates = rng.uniform(0.05, 0.6, (tiny.T, tiny.k)).astype(np.float32)
    bad = [(3, 0, tiny.E), (10, 1, -1), (77, 1, tiny.E + 100)]
    idx_bad = idx.copy()
    for t, j, e in bad:
        idx_bad[t, j] = e
    y = layer.forward_routed(x, torch.from_numpy(idx_bad).cuda(), torch.from_numpy(gates).cuda())
    st = _status(layer)
    assert st == capi.STATUS_BAD_EXPERT, ("replay", st)
    g0 = gates.astype(np.float64).copy()
    for t, j, _ in bad:
        g0[t, j] = 0.0
    gh.assert_y_close(y, ref.forward_routed(gh.f64(x), gh.oracle_weights(w), idx, g0)["y"])
    print("replay with out-of-range ids: status BAD_EXPERT only, y within the parity bounds",
          flush=True)

    # the E4M3 expert path (its codes and fp32 outputs go through the same checks)
    w, x, layer = _layer(tiny, 8, fp8=True)
    layer.set_fp8_scales([0.02, 0.01])
    layer.forward(x)
    st = _status(layer)
    assert st == 0, ("e4m3", st)
    print("tiny, E4M3 experts: status 0", flush=True)
    print("bounds build: all cases clean", flush=True)


if __name__ == "__main__":
    main()

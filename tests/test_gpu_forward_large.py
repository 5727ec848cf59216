"""The two large shapes at full size, in the launch configuration the
benchmark times: routing checked in full (bit-exact from the GPU logits);
logits on a seeded token sample; the layer output on a token sample that
reaches every expert GEMM tile of the forward (the last slot of every
expert, a slot in every token chunk of every expert, topped up with seeded
tokens to at least 256), computed by the oracle one expert at a time."""
import time

import numpy as np
import pytest
import torch

from mixture_experts_layer_router_gb300 import synth
import gpu_helpers as gh
from oracle import latentmoe_ref as ref

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,n_logit,n_y", [("mai-base-1", 256, 256), ("mai-base-2", 256, 256)])
def test_large_shape_sampled(name, n_logit, n_y):
    cfg = synth.CONFIGS[name]
    free, _ = torch.cuda.mem_get_info()
    need = 2 * (3 * cfg.E * cfg.F * cfg.l + 3 * cfg.d * cfg.Fs + 2 * cfg.d * cfg.l) + \
        cfg.slots * (2 * cfg.l + cfg.F) * 2 + (8 << 30)
    if free < need:
        pytest.skip(f"needs {need / 2**30:.0f} GiB free, {free / 2**30:.0f} GiB available")
    w = synth.make_weights(cfg, 0, "cuda")
    x = synth.make_x(cfg, 0, "cuda")
    layer = gh.make_layer(cfg, w)
    y = layer.forward(x)
    r = layer.get_routing(cfg.T, "cuda")
    torch.cuda.synchronize()
    assert layer.status() == 0
    L_gpu = gh.f64(r["logits"])

    # full routing, bit-exact from the same logits
    ora_r = ref.route(L_gpu, cfg.E, cfg.k)
    gh.assert_routing_equal(r, ora_r, cfg.T, cfg.k)

    # logits on a token sample
    W0 = gh.oracle_weights(w, stacked=False)
    s = synth.sample_tokens(cfg.T, n_logit, seed=1).numpy()
    xs = gh.f64(x[torch.from_numpy(s).cuda()])
    L_ref = ref.router_logits(xs, W0.w_r, W0.b_r)
    assert np.abs(L_gpu[s] - L_ref).max() <= gh.LOGIT_MAX_ABS

    # layer outputs on tokens that reach every tile: each expert's last slot
    # and a slot in each of its token chunks
    s2 = gh.covering_tokens(r, cfg.T, cfg.k, n_min=n_y, seed=1)
    idx = ora_r["idx"][s2]
    touched = np.unique(idx)
    assert len(touched) == int((ora_r["counts"] > 0).sum())
    t0 = time.perf_counter()
    fetch = gh.ExpertPrefetch(w, touched)
    W = ref.OracleWeights(W0.w_r, W0.w_dn, W0.w_up, fetch, b_r=W0.b_r, w_gs=W0.w_gs,
                          w_us=W0.w_us, w_ds=W0.w_ds)
    ora = ref.forward(gh.f64(x[torch.from_numpy(s2).cuda()]), W, cfg.k, logits=L_gpu[s2])
    fetch.close()
    gh.assert_y_close(y[torch.from_numpy(s2).cuda()], ora["y"], what=name)
    print(f"{name}: y checked on {len(s2)} tokens reaching {len(touched)} experts "
          f"({time.perf_counter() - t0:.1f} s of oracle)")
    del layer, w, x, y
    torch.cuda.empty_cache()

"""The two large shapes at full size, in the launch configuration the
benchmark times: routing checked in full (bit-exact from the GPU logits),
logits and layer outputs on seeded token samples that the oracle computes
one expert at a time."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_router_gb300 import synth
import gpu_helpers as gh
from oracle import latentmoe_ref as ref

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name,n_logit,n_y", [("mai-base-1", 256, 12), ("mai-base-2", 256, 8)])
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
    W = gh.oracle_weights(w, stacked=False)
    L_gpu = gh.f64(r["logits"])

    # full routing, bit-exact from the same logits
    ora_r = ref.route(L_gpu, cfg.E, cfg.k)
    gh.assert_routing_equal(r, ora_r, cfg.T, cfg.k)

    # logits on a token sample
    s = synth.sample_tokens(cfg.T, n_logit, seed=1).numpy()
    xs = gh.f64(x[torch.from_numpy(s).cuda()])
    L_ref = ref.router_logits(xs, W.w_r, W.b_r)
    assert np.abs(L_gpu[s] - L_ref).max() <= gh.LOGIT_MAX_ABS

    # layer outputs on a smaller sample (each token pulls its k experts)
    s2 = s[:n_y]
    ora = ref.forward(gh.f64(x[torch.from_numpy(s2).cuda()]), W, cfg.k, logits=L_gpu[s2])
    gh.assert_y_close(y[torch.from_numpy(s2).cuda()], ora["y"], what=name)
    del layer, w, x, y
    torch.cuda.empty_cache()

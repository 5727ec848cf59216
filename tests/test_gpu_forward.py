"""The whole layer on the GPU against the float64 oracle, on the small
configs in full (tiny, mid, imbalanced) and on flag variants.

Output parity routes the oracle from the GPU's own fp32 logits (exported by
latentmoe_get_routing), because near-equal logits can legitimately pick a
different expert in float64; the logits themselves are checked separately.
"""
import numpy as np
import pytest
import torch

from mixture_experts_layer_router_gb300 import capi, synth
import gpu_helpers as gh
from oracle import latentmoe_ref as ref

pytestmark = pytest.mark.gpu


def _setup(name, seed=0, bias_override=None):
    cfg = synth.CONFIGS[name]
    w = synth.make_weights(cfg, seed, "cuda")
    if bias_override is not None:
        w["b_r"] = bias_override
    x = synth.make_x(cfg, seed, "cuda")
    return cfg, w, x


def _check_layer(cfg, w, x, layer, T=None):
    T = cfg.T if T is None else T
    y = layer.forward(x[:T])
    r = layer.get_routing(T, "cuda")
    torch.cuda.synchronize()
    assert layer.status() == 0
    W = gh.oracle_weights(w)
    xs = gh.f64(x[:T])
    # logits: GPU fp32 vs float64
    L_ref = ref.router_logits(xs, W.w_r, W.b_r)
    L_gpu = gh.f64(r["logits"])
    assert np.abs(L_gpu - L_ref).max() <= gh.LOGIT_MAX_ABS
    # routing from the GPU logits: bit-exact integers
    renorm = bool(layer.flags & capi.RENORM)
    ora = ref.forward(xs, W, cfg.k, renorm=renorm, logits=L_gpu)
    gh.assert_routing_equal(r, ora, T, cfg.k)
    rel, mx = gh.assert_y_close(y, ora["y"])
    return y, ora


@pytest.mark.parametrize("name", ["tiny", "mid", "imbalanced"])
def test_forward_matches_oracle(name):
    cfg, w, x = _setup(name)
    layer = gh.make_layer(cfg, w)
    _check_layer(cfg, w, x, layer)


def test_tiny_flag_variants():
    cfg, w, x = _setup("tiny", seed=3)
    g = torch.Generator(device="cpu")
    g.manual_seed(4)
    w["b_r"] = (torch.randn(cfg.E, generator=g) * 0.5).cuda()
    for renorm in (False, True):
        for out_fp32 in (False, True):
            layer = gh.make_layer(cfg, w, renorm=renorm, out_fp32=out_fp32)
            y, _ = _check_layer(cfg, w, x, layer)
            assert y.dtype == (torch.float32 if out_fp32 else torch.bfloat16)


def test_ragged_token_counts():
    """T not a multiple of the 128-row tile, and T = 1."""
    cfg, w, x = _setup("tiny", seed=5)
    layer = gh.make_layer(cfg, w)
    for T in (1, 77, 128):
        _check_layer(cfg, w, x, layer, T=T)


def test_shared_expert_small():
    """A small layer with a shared expert (the MAI-Base-2 structure)."""
    cfg = synth.LayerConfig("tiny-shared", T=200, d=256, l=128, E=8, k=3, F=256, Fs=384)
    w = synth.make_weights(cfg, 7, "cuda")
    x = synth.make_x(cfg, 7, "cuda")
    layer = gh.make_layer(cfg, w)
    _check_layer(cfg, w, x, layer)


def test_zero_input_routes_to_first_experts():
    cfg, w, x = _setup("tiny", seed=8)
    x = torch.zeros_like(x)
    layer = gh.make_layer(cfg, w)
    y = layer.forward(x)
    r = layer.get_routing(cfg.T, "cuda")
    torch.cuda.synchronize()
    assert torch.all(r["idx"].cpu() == torch.arange(cfg.k, dtype=torch.int32)[None, :])
    counts = r["counts"].cpu()
    assert counts[:cfg.k].tolist() == [cfg.T] * cfg.k and counts[cfg.k:].sum() == 0
    assert torch.all(y == 0)


def test_forward_is_bitwise_deterministic():
    cfg, w, x = _setup("imbalanced", seed=1)
    layer = gh.make_layer(cfg, w)
    a = layer.forward(x).clone()
    b = layer.forward(x).clone()
    torch.cuda.synchronize()
    assert torch.equal(a, b)


def test_forward_host_matches_device_forward():
    cfg, w, x = _setup("mid", seed=2)
    layer = gh.make_layer(cfg, w)
    y_dev = layer.forward(x)
    torch.cuda.synchronize()
    xh = x.cpu().pin_memory()
    yh = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16).pin_memory()
    layer.forward_host(xh, yh)
    assert torch.equal(yh, y_dev.cpu())


@pytest.mark.parametrize("out_fp32", [False, True])
def test_forward_host_async_pipeline_matches_device_forwards(out_fp32):
    """Five pipelined host-buffer forwards of different inputs into different
    outputs (the copies of one step overlapping the neighbours' forwards),
    then one wait: each output equals the device forward of its input bit for
    bit. Then the bench's pattern, one input and one output buffer reused for
    three steps, and the synchronous entry afterwards."""
    cfg = synth.LayerConfig("host-async", T=1500, d=512, l=256, E=8, k=2, F=512, Fs=256)
    w = synth.make_weights(cfg, 17, "cuda")
    layer = gh.make_layer(cfg, w, out_fp32=out_fp32)
    dt = torch.float32 if out_fp32 else torch.bfloat16
    xs = [synth.make_x(cfg, 100 + i, "cuda") for i in range(5)]
    ys_dev = [layer.forward(x).clone() for x in xs]
    torch.cuda.synchronize()
    xh = [x.cpu().pin_memory() for x in xs]
    yh = [torch.full((cfg.T, cfg.d), -1.0, dtype=dt).pin_memory() for _ in xs]
    for a, b in zip(xh, yh):
        layer.forward_host_async(a, b)
    layer.host_wait()
    for b, y in zip(yh, ys_dev):
        assert torch.equal(b, y.cpu())
    y1 = torch.full((cfg.T, cfg.d), -1.0, dtype=dt).pin_memory()
    for _ in range(3):
        layer.forward_host_async(xh[1], y1)
    layer.host_wait()
    assert torch.equal(y1, ys_dev[1].cpu())
    y2 = torch.full((cfg.T, cfg.d), -1.0, dtype=dt).pin_memory()
    layer.forward_host(xh[2], y2)
    assert torch.equal(y2, ys_dev[2].cpu())
    assert layer.status() == 0
    layer.close()


def test_launch_count_and_stage_times():
    cfg, w, x = _setup("tiny")
    layer = gh.make_layer(cfg, w)
    layer.set_profiling(2)
    n0 = layer.launch_count()
    layer.forward(x)
    assert layer.launch_count() - n0 == 7  # the sort is one cooperative launch
    t = layer.stage_times(0)
    assert set(t) == {"router", "replay_gates", "sort", "down_proj", "expert_gate_up",
                      "expert_down", "combine", "shared_gate_up", "up_proj",
                      "fp8_scales"}
    assert all(v >= 0 for v in t.values())


def test_error_paths_on_device():
    cfg, w, x = _setup("tiny")
    gh.lib()
    layer = capi.LatentMoE(cfg.d, cfg.l, cfg.E, cfg.k, cfg.F, 0, max_tokens=cfg.T)
    y = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    lib = capi.load()
    s = torch.cuda.current_stream().cuda_stream
    assert lib.latentmoe_forward(layer.handle, x.data_ptr(), y.data_ptr(), cfg.T, s) == \
        capi.ERR_NOT_LOADED
    layer.load_weights(w)
    assert lib.latentmoe_forward(layer.handle, x.data_ptr(), y.data_ptr(), cfg.T + 1, s) == \
        capi.ERR_INVALID_ARG
    assert lib.latentmoe_forward(layer.handle, x.data_ptr(), y.data_ptr(), 0, s) == \
        capi.ERR_INVALID_ARG
    assert lib.latentmoe_forward(layer.handle, x.data_ptr() + 2, y.data_ptr(), cfg.T, s) == \
        capi.ERR_UNSUPPORTED
    w2 = dict(w)
    w2["w_g"] = None
    with pytest.raises(capi.LatentMoEError):
        layer.load_weights(w2)
    assert layer.status() == 0


@pytest.mark.parametrize("name,renorm", [("tiny", False), ("mid", True), ("imbalanced", False)])
def test_fused_router_matches_standalone_routing(name, renorm):
    """The router kernel's in-epilogue softmax/top-k gives the same idx and
    bitwise the same gates as the warp-per-token routing of its own logits."""
    cfg, w, x = _setup(name, seed=4)
    layer = gh.make_layer(cfg, w, renorm=renorm)
    layer.forward(x)
    r = layer.get_routing(cfg.T, "cuda")
    alone = layer.route_from_logits(r["logits"].clone())
    torch.cuda.synchronize()
    for key in ("idx", "gates", "counts", "offsets", "perm", "pos"):
        assert torch.equal(r[key], alone[key]), key


@pytest.mark.parametrize("fp8,dense", [(False, False), (True, False), (True, True)])
def test_single_sm_expert_shapes(fp8, dense):
    """F = l = 384 (F % 256 and l % 512 nonzero): both expert GEMMs run the
    single-SM kernels inside the layer; bf16 against the oracle, and the
    E4M3 variants against their bf16 counterpart within the E4M3 error."""
    cfg = synth.LayerConfig("odd", T=333, d=256, l=384, E=12, k=3, F=384, Fs=384)
    w = synth.make_weights(cfg, 21, "cuda")
    x = synth.make_x(cfg, 21, "cuda")
    layer = gh.make_layer(cfg, w, fp8=fp8, fp8_dense=dense)
    if not fp8:
        _check_layer(cfg, w, x, layer)
        return
    layer.forward(x)
    y = layer.forward(x)
    r = layer.get_routing(cfg.T, "cuda")
    torch.cuda.synchronize()
    assert layer.status() == 0
    W = gh.oracle_weights(w)
    exact = ref.forward(gh.f64(x), W, cfg.k, logits=gh.f64(r["logits"]))["y"]
    rel = np.linalg.norm(gh.f64(y) - exact) / np.linalg.norm(exact)
    assert rel < 0.15, rel


@pytest.mark.parametrize("out_fp32", [False, True])
def test_forward_host_chunks_all_e4m3_shared(out_fp32):
    """The host-buffer forward with all-E4M3 GEMMs and a shared expert (the
    up-projection's fp32 partial) equals the device forward bit for bit."""
    cfg = synth.LayerConfig("host", T=2600, d=512, l=256, E=8, k=2, F=512, Fs=256)
    w = synth.make_weights(cfg, 13, "cuda")
    x = synth.make_x(cfg, 13, "cuda")
    layer = gh.make_layer(cfg, w, out_fp32=out_fp32, fp8=True, fp8_dense=True)
    scales = [0.02, 0.01, 0.01, 0.005, 0.01]
    layer.set_fp8_scales(scales)
    y_dev = layer.forward(x)
    torch.cuda.synchronize()
    layer.set_fp8_scales(scales)
    xh = x.cpu().pin_memory()
    yh = torch.empty((cfg.T, cfg.d), dtype=y_dev.dtype).pin_memory()
    layer.forward_host(xh, yh)
    assert torch.equal(yh, y_dev.cpu())
    assert layer.status() == 0


@pytest.mark.parametrize("shape", [
    dict(T=200, d=256, l=128, E=1, k=1, F=256),     # one expert: the dense SwiGLU sandwich
    dict(T=150, d=256, l=128, E=16, k=16, F=128),   # every expert chosen: the full mixture
    dict(T=100, d=384, l=256, E=5, k=3, F=256),     # odd expert count
    dict(T=256, d=256, l=128, E=512, k=16, F=128),  # widest top-k at the largest E
])
def test_degenerate_and_extreme_routing(shape):
    """The fused router and the rest of the layer at the edges of the routing
    space: E = 1, k = E, odd E, and k = 16 with E = 512."""
    cfg = synth.LayerConfig("edge", Fs=0, **shape)
    w = synth.make_weights(cfg, 17, "cuda")
    x = synth.make_x(cfg, 17, "cuda")
    layer = gh.make_layer(cfg, w)
    y, ora = _check_layer(cfg, w, x, layer)
    if cfg.E == 1:
        # every token in the one expert with gate 1: y = W_up SwiGLU(W_dn x)
        W = gh.oracle_weights(w)
        z = ref.latent_down(gh.f64(x), W.w_dn)
        wg, wu, wd = W.expert(0)
        dense = ref.latent_up(ref.swiglu_ffn(z, wg, wu, wd), W.w_up)
        assert np.allclose(ora["y"], dense, rtol=0, atol=1e-12)
    # the E4M3 path on the same edges: routing identical, output near bf16
    layer8 = gh.make_layer(cfg, w, fp8=True, fp8_dense=True)
    layer8.forward(x)
    y8 = layer8.forward(x)
    r8 = layer8.get_routing(cfg.T, "cuda")
    torch.cuda.synchronize()
    assert layer8.status() == 0
    assert torch.equal(r8["idx"], layer.get_routing(cfg.T, "cuda")["idx"])
    rel = (y8.float() - y.float()).norm() / y.float().norm()
    assert rel < 0.15, rel.item()


@pytest.mark.parametrize("fp8", [False, True])
def test_forward_captures_into_a_cuda_graph(fp8):
    """The forward enqueues no host synchronisation, so it can be captured
    into a CUDA graph (after one call outside the capture sets the kernel
    attributes) and replayed; replays match eager forwards bit for bit,
    E4M3 scale updates included."""
    cfg = synth.CONFIGS["tiny"]
    w = synth.make_weights(cfg, 23, "cuda")
    x = synth.make_x(cfg, 23, "cuda")
    layer = gh.make_layer(cfg, w, fp8=fp8, fp8_dense=fp8)
    y = torch.empty((cfg.T, cfg.d), dtype=torch.bfloat16, device="cuda")
    layer.forward(x, y)  # outside the capture: per-device kernel setup
    torch.cuda.synchronize()
    if fp8:
        layer.set_fp8_scales([0.02, 0.01, 0.01, 0.005, 0.01])
    eager = []
    for _ in range(3):
        eager.append(layer.forward(x, y).clone())
    torch.cuda.synchronize()
    if fp8:
        layer.set_fp8_scales([0.02, 0.01, 0.01, 0.005, 0.01])
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            layer.forward(x, y, stream=s)
    torch.cuda.synchronize()
    # the capture enqueued nothing; replay the same three forwards
    for i in range(3):
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(y, eager[i]), i
    assert layer.status() == 0


@pytest.mark.parametrize("fp8", [False, True])
def test_reloading_weights_matches_a_fresh_handle(fp8):
    """load_weights twice on one handle (the owned copy, packed tiles and
    E4M3 scales rebuilt) gives the same output as a new handle."""
    cfg = synth.CONFIGS["tiny"]
    wa = synth.make_weights(cfg, 31, "cuda")
    wb = synth.make_weights(cfg, 32, "cuda")
    x = synth.make_x(cfg, 31, "cuda")
    scales = [0.02, 0.01, 0.01, 0.005, 0.01]
    layer = gh.make_layer(cfg, wa, fp8=fp8, fp8_dense=fp8)
    layer.forward(x)
    layer.load_weights(wb)
    if fp8:
        layer.set_fp8_scales(scales)
    y1 = layer.forward(x).clone()
    fresh = gh.make_layer(cfg, wb, fp8=fp8, fp8_dense=fp8)
    if fp8:
        fresh.set_fp8_scales(scales)
        assert fresh.fp8_all_weight_scales() == layer.fp8_all_weight_scales()
    y2 = fresh.forward(x)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


@pytest.mark.parametrize("name", ["tiny", "mid", "imbalanced"])
def test_programmatic_launch_on_and_off_bitwise_equal(name):
    """The forward's kernels with programmatic dependent launch (the default)
    and in plain stream order give the same bits, forward after forward."""
    cfg = synth.CONFIGS[name]
    w = synth.make_weights(cfg, 5, "cuda")
    x = synth.make_x(cfg, 5, "cuda")
    layer = gh.make_layer(cfg, w)
    ys = [layer.forward(x).clone() for _ in range(3)]
    layer.set_pdl(False)
    ys += [layer.forward(x).clone() for _ in range(2)]
    layer.set_pdl(True)
    ys.append(layer.forward(x).clone())
    torch.cuda.synchronize()
    assert layer.status() == 0
    for y in ys[1:]:
        assert torch.equal(ys[0], y)


@pytest.mark.parametrize("name,variant", [("tiny", "bf16"), ("mid", "bf16"),
                                          ("imbalanced", "bf16"), ("mid", "one_sm"),
                                          ("mid", "e4m3"), ("mid", "e4m3_dense")])
def test_back_to_back_forwards_on_new_inputs(name, variant):
    """Forwards enqueued back to back, each on new inputs (so each routes its
    tokens differently), give the bits of the same forwards run one at a time
    in plain stream order with a synchronisation between them. Under
    programmatic launch each kernel's set-up overlaps the kernel before it,
    across forwards too; every kernel must still read this forward's routing
    and slots, never the previous forward's."""
    cfg = synth.CONFIGS[name]
    fp8 = variant.startswith("e4m3")
    w = synth.make_weights(cfg, 11, "cuda")
    xs = [synth.make_x(cfg, 20 + i, "cuda") for i in range(4)]
    layer = gh.make_layer(cfg, w, fp8=fp8, fp8_dense=variant == "e4m3_dense")
    if variant == "one_sm":
        layer.set_sm_pairs(False)
    scales = [0.02, 0.01, 0.02, 0.01, 0.02][:capi.FP8_TENSORS if variant == "e4m3_dense" else 2]

    def run(pdl, sync):
        layer.set_pdl(pdl)
        if fp8:
            layer.set_fp8_scales(scales)
        ys = []
        for x in xs:
            ys.append(layer.forward(x).clone())
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        assert layer.status() == 0
        return ys

    ys_fast = run(True, False)
    ys_ref = run(False, True)
    routes = set()
    for i, (a, b) in enumerate(zip(ys_fast, ys_ref)):
        assert torch.equal(a, b), f"forward {i}"
    # the inputs do route differently (otherwise stale slots would go unseen)
    for x in xs[:2]:
        layer.forward(x)
        routes.add(layer.get_routing(cfg.T, "cuda")["idx"].cpu().numpy().tobytes())
    assert len(routes) == 2
    layer.close()


@pytest.mark.parametrize("E,k", [(64, 4), (512, 8)])
def test_router_several_tiles_per_cta(E, k):
    """More 128-token tiles than SMs: each router CTA runs several tiles in
    turn (its stage ring and TMEM hand-off carry over from tile to tile), at
    both k-block widths (128 columns for E <= 128, 32 columns and two MMAs
    for E = 512)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    T = 128 * (2 * sms + 3) + 17  # every CTA two tiles or more, a ragged last tile
    cfg = synth.LayerConfig("many-tiles", T=T, d=256, l=128, E=E, k=k, F=256)
    w = synth.make_weights(cfg, 23, "cuda")
    x = synth.make_x(cfg, 23, "cuda")
    layer = gh.make_layer(cfg, w)
    _check_layer(cfg, w, x, layer)
    layer.close()


def test_two_handles_on_two_streams():
    """Two layers of different shapes, each on its own stream, forwards
    interleaved with nothing ordering the streams: each output is bitwise the
    one of the same forward run alone. The handles share no device state (each
    has its own workspace, counters and scratch), so concurrency changes
    nothing."""
    cfg_a = synth.CONFIGS["mid"]
    cfg_b = synth.LayerConfig("shared-b", T=1000, d=512, l=256, E=16, k=3, F=512, Fs=512)
    wa = synth.make_weights(cfg_a, 31, "cuda")
    wb = synth.make_weights(cfg_b, 32, "cuda")
    xa = [synth.make_x(cfg_a, 40 + i, "cuda") for i in range(3)]
    xb = [synth.make_x(cfg_b, 50 + i, "cuda") for i in range(3)]
    la = gh.make_layer(cfg_a, wa)
    lb = gh.make_layer(cfg_b, wb)
    ref_a = [la.forward(x).clone() for x in xa]
    ref_b = [lb.forward(x).clone() for x in xb]
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    ya = [torch.empty_like(y) for y in ref_a]
    yb = [torch.empty_like(y) for y in ref_b]
    for _ in range(2):
        for i in range(3):
            la.forward(xa[i], ya[i], stream=sa)
            lb.forward(xb[i], yb[i], stream=sb)
    torch.cuda.synchronize()
    assert la.status() == 0 and lb.status() == 0
    for a, b in zip(ya, ref_a):
        assert torch.equal(a, b)
    for a, b in zip(yb, ref_b):
        assert torch.equal(a, b)
    la.close()
    lb.close()

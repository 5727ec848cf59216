"""The SM-pair grouped kernels (tcgen05 cta_group::2) against the one-SM
kernels and the float64 products: the debug GEMM entries on ragged groups,
then the whole layer with pairs on and off against the oracle."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_router_gb300 import capi, synth
import gpu_helpers as gh
from oracle import latentmoe_ref as ref
from test_gpu_fp8 import _int_codes

pytestmark = pytest.mark.gpu
PAIR = 4


def _rand(shape, seed, scale=1.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * scale).to(torch.bfloat16)


def _offs(counts):
    return torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int32,
                        device="cuda")


# 300, 513, 257, 512, 511, 1000 and 1537 slots: more than one token chunk in the
# SwiGLU GEMM (even chunks of at most 256) and wide tiles in the down GEMM (one
# accumulator over chunks of up to 512 tokens, the tokens past 256 in a second MMA)
@pytest.mark.parametrize("counts", [[16], [1, 0, 300, 37], [256, 513, 0, 8, 130],
                                    [257, 512, 1000], [1537, 3, 511]])
@pytest.mark.parametrize("mode,N", [(2, 256), (2, 512), (0, 512), (0, 1024)])
def test_pair_grouped_bf16_equals_single_sm(counts, mode, N):
    gh.lib()
    G, K = len(counts), 256
    M = sum(counts)
    A = _rand((M, K), 1)
    B = _rand(((2 if mode == 2 else 1) * G * N, K), 2, 0.05)
    offs = _offs(counts)
    C1 = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    C2 = torch.full((M, N), -3.0, dtype=torch.bfloat16, device="cuda")
    assert capi.debug_grouped_gemm(A, B, C1, offs, G, M, N, K, mode) == capi.OK
    assert capi.debug_status() == 0
    assert capi.debug_grouped_gemm(A, B, C2, offs, G, M, N, K, mode | PAIR) == capi.OK
    assert capi.debug_status() == 0
    torch.cuda.synchronize()
    # same products, same k order: the pair kernel must agree bit for bit
    assert torch.equal(C1, C2)
    # and with float64
    Ad, Bd = A.double().cpu(), B.double().cpu()
    o = 0
    for g, n in enumerate(counts):
        if n == 0:
            continue
        a = Ad[o:o + n]
        if mode == 2:
            gate = a @ Bd[g * N:(g + 1) * N].T
            up = a @ Bd[(G + g) * N:(G + g + 1) * N].T
            want = gate / (1 + torch.exp(-gate)) * up
        else:
            want = a @ Bd[g * N:(g + 1) * N].T
        err = (C2[o:o + n].double().cpu() - want).abs()
        assert (err <= want.abs() * 2 ** -7 + 1e-3 * want.abs().max()).all()
        o += n


@pytest.mark.parametrize("counts", [[0, 37, 256, 300, 5, 130], [513, 257, 1000, 512]])
@pytest.mark.parametrize("mode,N", [(1, 512), (2, 256)])
def test_pair_grouped_e4m3_equals_single_sm(mode, N, counts):
    gh.lib()
    G, K = len(counts), 384
    M = sum(counts)
    A, _ = _int_codes((M, K), 31)
    B, _ = _int_codes(((2 if mode == 2 else 1) * G * N, K), 32)
    nsc = 2 + (2 if mode == 2 else 1) * G
    scales = torch.tensor([0.5, 4.0] + [2.0 ** -(i % 4) for i in range(nsc - 2)],
                          dtype=torch.float32, device="cuda")
    offs = _offs(counts)
    out_dt = torch.uint8 if mode == 2 else torch.bfloat16
    C1 = torch.zeros((M, N), dtype=out_dt, device="cuda")
    C2 = torch.ones((M, N), dtype=out_dt, device="cuda")
    am1 = torch.zeros((1,), dtype=torch.int32, device="cuda")
    am2 = torch.zeros((1,), dtype=torch.int32, device="cuda")
    assert capi.debug_grouped_gemm_e4m3(A, B, scales, C1, am1, offs, G, M, N, K, mode) == capi.OK
    assert capi.debug_grouped_gemm_e4m3(A, B, scales, C2, am2, offs, G, M, N, K,
                                        mode | PAIR) == capi.OK
    assert capi.debug_status() == 0
    assert torch.equal(C1, C2)
    assert torch.equal(am1, am2)


@pytest.mark.parametrize("name", ["mid", "imbalanced"])
@pytest.mark.parametrize("fp8", [False, True])
def test_layer_with_and_without_pairs(name, fp8):
    """mid/imbalanced (F = 2048, l = 1024) run both expert GEMMs on pairs."""
    cfg = synth.CONFIGS[name]
    w = synth.make_weights(cfg, 3, "cuda")
    x = synth.make_x(cfg, 3, "cuda")
    layer = gh.make_layer(cfg, w, fp8=fp8)
    scales = [0.02, 0.01]
    outs = []
    for pairs in (False, True):
        layer.set_sm_pairs(pairs)
        if fp8:
            layer.set_fp8_scales(scales)
        outs.append(layer.forward(x).clone())
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(outs[0], outs[1])
    if not fp8:
        r = layer.get_routing(cfg.T, "cuda")
        W = gh.oracle_weights(w)
        ora = ref.forward(gh.f64(x), W, cfg.k, logits=gh.f64(r["logits"]))
        gh.assert_y_close(outs[1], ora["y"])


def test_set_sm_pairs_rejects_bad_values():
    cfg = synth.CONFIGS["tiny"]
    w = synth.make_weights(cfg, 0, "cuda")
    layer = gh.make_layer(cfg, w)
    lib = capi.load()
    assert lib.latentmoe_set_sm_pairs(layer.handle, 2) == capi.ERR_INVALID_ARG
    assert lib.latentmoe_set_sm_pairs(None, 1) == capi.ERR_INVALID_ARG
    layer.set_sm_pairs(False)
    layer.set_sm_pairs(True)


# ---------------------------------------------------------------- dense GEMMs

@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("M,N,K", [(1, 256, 128), (300, 384, 256), (1000, 1024, 512),
                                   (4096, 256, 1024), (513, 128, 384)])
def test_pair_dense_equals_single_sm(mode, M, N, K):
    """The dense SM-pair kernel (M = 256 pair tiles; ragged last tile, whose
    second CTA may hold no rows) agrees bit for bit with the one-SM kernel."""
    gh.lib()
    A = _rand((M, K), 11)
    B = _rand(((2 if mode == 2 else 1) * N, K), 12, 0.05)
    dt = torch.float32 if mode == 1 else torch.bfloat16
    C1 = torch.full((M, N), 3.0, dtype=dt, device="cuda")
    C2 = torch.full((M, N), -3.0, dtype=dt, device="cuda")
    assert capi.debug_gemm(A, B, C1, M, N, K, mode) == capi.OK
    assert capi.debug_gemm(A, B, C2, M, N, K, mode | PAIR) == capi.OK
    torch.cuda.synchronize()
    assert capi.debug_status() == 0
    assert torch.equal(C1, C2)
    Ad, Bd = A.double().cpu(), B.double().cpu()
    if mode == 2:
        gate, up = Ad @ Bd[:N].T, Ad @ Bd[N:].T
        want = gate / (1 + torch.exp(-gate)) * up
    else:
        want = Ad @ Bd.T
    err = (C2.double().cpu() - want).abs()
    assert (err <= want.abs() * 2 ** -7 + 1e-3 * want.abs().max()).all()


SHARED = synth.LayerConfig("shared-ragged", T=300, d=512, l=256, E=16, k=2, F=256, Fs=512)


@pytest.mark.parametrize("fp8_dense", [False, True])
@pytest.mark.parametrize("out_fp32", [False, True])
def test_layer_dense_pairs_on_and_off(fp8_dense, out_fp32):
    """Every dense GEMM of the forward (the scatter down-projection, the
    shared expert's SwiGLU, the up-projection with the shared down-projection,
    fp32 output, E4M3 operands) gives the same output on SM pairs."""
    cfg = SHARED
    w = synth.make_weights(cfg, 5, "cuda")
    x = synth.make_x(cfg, 5, "cuda")
    layer = gh.make_layer(cfg, w, out_fp32=out_fp32, fp8=fp8_dense, fp8_dense=fp8_dense)
    outs = []
    for pairs in (False, True):
        layer.set_sm_pairs(pairs)
        if fp8_dense:
            layer.set_fp8_scales([0.02, 0.01, 0.03, 0.02, 0.01])
        outs.append(layer.forward(x).clone())
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(outs[0], outs[1])
    if not fp8_dense:
        r = layer.get_routing(cfg.T, "cuda")
        ora = ref.forward(gh.f64(x), gh.oracle_weights(w), cfg.k, logits=gh.f64(r["logits"]))
        gh.assert_y_close(outs[1], ora["y"])


@pytest.mark.parametrize("T", [129, 256, 257, 383, 511, 600])
def test_layer_ragged_tokens_across_pair_tiles(T):
    """Token counts around the 256-row pair tile of the dense kernels (the
    second CTA of the last pair tile holds part of a tile, or no rows): the
    forward matches the oracle and is bitwise the same with pairs off."""
    cfg = synth.LayerConfig("pair-ragged", T=600, d=384, l=256, E=12, k=3, F=256, Fs=256)
    w = synth.make_weights(cfg, 9, "cuda")
    x = synth.make_x(cfg, 9, "cuda")[:T].contiguous()
    layer = gh.make_layer(cfg, w)
    outs = []
    for pairs in (True, False):
        layer.set_sm_pairs(pairs)
        outs.append(layer.forward(x).clone())
    torch.cuda.synchronize()
    assert layer.status() == 0
    assert torch.equal(outs[0], outs[1])
    r = layer.get_routing(T, "cuda")
    ora = ref.forward(gh.f64(x), gh.oracle_weights(w), cfg.k, logits=gh.f64(r["logits"]))
    gh.assert_y_close(outs[0], ora["y"])

"""Routing on the GPU (softmax, stable top-k, counting sort) against the
oracle fed the same fp32 logits: integers bit-exact."""
import numpy as np
import pytest
import torch

from mixture_experts_layer_router_gb300 import capi
import gpu_helpers as gh
from oracle import latentmoe_ref as ref

pytestmark = pytest.mark.gpu


def _layer(E, k, T, renorm=False):
    gh.lib()
    return capi.LatentMoE(128, 128, E, k, 128, 0, max_tokens=T, renorm=renorm)


def _logits(T, E, seed, kind="normal"):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    if kind == "normal":
        L = torch.randn((T, E), generator=g)
    elif kind == "ties":  # few distinct values: many exact ties
        L = torch.randint(0, 4, (T, E), generator=g).float() * 0.25
    elif kind == "zeros":
        L = torch.zeros((T, E))
    elif kind == "skewed":  # a Zipf-like bias: one expert takes most tokens
        L = torch.randn((T, E), generator=g) * 0.1 - 1.8 * torch.log(
            1.0 + torch.randperm(E, generator=g).float())
    return L.float()


@pytest.mark.parametrize("T,E,k,kind", [
    (128, 16, 2, "normal"), (1000, 64, 4, "normal"), (4096, 64, 4, "skewed"),
    (777, 100, 5, "ties"), (64, 512, 8, "ties"), (33, 16, 16, "normal"),
    (256, 8, 3, "zeros"), (16384, 512, 8, "normal"), (8192, 256, 7, "normal"), (1, 4, 1, "normal"),
    # around the one-CTA sort's limit (4096 slots): one CTA, then the cooperative launch
    (1024, 512, 4, "skewed"), (4097, 64, 1, "ties"),
    # 2M slots: more 1024-slot chunks than the cooperative sort keeps resident
    # on the SMs at once, so the three-launch sort runs
    (262144, 32, 8, "normal"),
])
def test_route_matches_oracle(T, E, k, kind):
    layer = _layer(E, k, T)
    L = _logits(T, E, T * 31 + E, kind).cuda()
    n0 = layer.launch_count()
    out = layer.route_from_logits(L)
    torch.cuda.synchronize()
    if T * k > 1024 * 8 * torch.cuda.get_device_properties(0).multi_processor_count:
        # top-k, then the sort's histogram, scan and scatter launches
        assert layer.launch_count() - n0 == 4
    ora = ref.route(L.cpu().double().numpy(), E, k)
    gh.assert_routing_equal(out, ora, T, k)
    assert layer.status() == 0


def test_route_renorm():
    T, E, k = 500, 32, 4
    layer = _layer(E, k, T, renorm=True)
    L = _logits(T, E, 5)
    out = layer.route_from_logits(L.cuda())
    ora = ref.route(L.double().numpy(), E, k, renorm=True)
    gh.assert_routing_equal(out, ora, T, k)


def test_route_is_deterministic():
    T, E, k = 4096, 512, 8
    layer = _layer(E, k, T)
    L = _logits(T, E, 9, "ties").cuda()
    a = layer.route_from_logits(L)
    b = layer.route_from_logits(L)
    for key in a:
        assert torch.equal(a[key], b[key]), key

"""The allocation-free routing entry point against the oracle and the
regular entry point (GPU).

latentmoe_route_from_logits_static serves callers that cannot allocate
device memory (an application whose own pool owns the whole device, or a
latency-critical loop that cannot pay for cudaFree's synchronisation). It
keeps the sort's scratch in a fixed array inside the library instead of a
handle's workspace. This file is collected last on purpose, and it must pass
both alone in a fresh process and after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_layer_router_gb300 import capi
import gpu_helpers as gh
from oracle import latentmoe_ref as ref

pytestmark = pytest.mark.gpu


def _logits(T, E, seed, ties=False):
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    if ties:
        return (torch.randint(0, 4, (T, E), generator=g).float() * 0.25).cuda()
    return torch.randn((T, E), generator=g).cuda()


def _static_route(L, k, renorm):
    lib = gh.lib()
    T, E = L.shape
    out = {
        "idx": torch.full((T, k), -7, dtype=torch.int32, device="cuda"),
        "gates": torch.full((T, k), -7.0, dtype=torch.float32, device="cuda"),
        "counts": torch.full((E,), -7, dtype=torch.int32, device="cuda"),
        "offsets": torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
        "perm": torch.full((T * k,), -7, dtype=torch.int32, device="cuda"),
        "pos": torch.full((T, k), -7, dtype=torch.int32, device="cuda"),
    }
    rc = lib.latentmoe_route_from_logits_static(
        L.data_ptr(), T, E, k, capi.RENORM if renorm else 0,
        *(out[n].data_ptr() for n in ("idx", "gates", "counts", "offsets", "perm", "pos")),
        torch.cuda.current_stream().cuda_stream)
    assert rc == capi.OK, rc
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("T,E,k,renorm", [(4096, 64, 4, False), (16384, 512, 8, False),
                                          (777, 100, 5, True)])
def test_static_entry_matches_oracle_and_regular_entry_twice(T, E, k, renorm):
    gh.lib()
    layer = capi.LatentMoE(128, 128, E, k, 128, 0, max_tokens=T, renorm=renorm)
    for call, seed in enumerate((11, 12)):  # two calls in a row, different inputs
        L = _logits(T, E, seed + 100 * E, ties=(call == 1))
        want = layer.route_from_logits(L)
        torch.cuda.synchronize()
        got = _static_route(L, k, renorm)
        for key in ("idx", "counts", "offsets", "perm", "pos"):
            assert torch.equal(got[key], want[key]), (call, key)
        np.testing.assert_allclose(got["gates"].cpu().numpy(), want["gates"].cpu().numpy(),
                                   rtol=2e-6, atol=1e-9)
        # and against the oracle's routing of the same logits
        gh.assert_routing_equal(got, ref.route(gh.f64(L), E, k, renorm=renorm), T, k)
    layer.close()


def test_static_entry_allocates_nothing():
    """After the first call on the device (which loads the library's module
    and looks up the array's address), further calls leave the device's free
    memory exactly as it was."""
    T, E, k = 16384, 512, 8
    L = _logits(T, E, 7)
    _static_route(L, k, False)  # first call on this device: set-up
    outs = _static_route(L, k, False)  # outputs allocated before the measurement
    lib = gh.lib()
    s = torch.cuda.current_stream().cuda_stream
    ptrs = [outs[n].data_ptr() for n in ("idx", "gates", "counts", "offsets", "perm", "pos")]
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert lib.latentmoe_route_from_logits_static(L.data_ptr(), T, E, k, 0, *ptrs, s) == \
            capi.OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    gh.assert_routing_equal(outs, ref.route(gh.f64(L), E, k), T, k)


def test_static_entry_rejects_sizes_beyond_its_scratch():
    lib = gh.lib()
    L = torch.zeros((1, 1), device="cuda")
    buf = torch.zeros(16, dtype=torch.int32, device="cuda")
    p = buf.data_ptr()
    s = torch.cuda.current_stream().cuda_stream
    # ceil(T*k/1024) * E = 258 * 512 > 131072
    rc = lib.latentmoe_route_from_logits_static(L.data_ptr(), 32897, 512, 8, 0,
                                                p, p, p, p, p, p, s)
    assert rc == capi.ERR_UNSUPPORTED
    rc = lib.latentmoe_route_from_logits_static(L.data_ptr(), 4, 8, 2, capi.OUT_FP32,
                                                p, p, p, p, p, p, s)
    assert rc == capi.ERR_INVALID_ARG
    rc = lib.latentmoe_route_from_logits_static(L.data_ptr(), 4, 8, 2, 0,
                                                None, p, p, p, p, p, s)
    assert rc == capi.ERR_INVALID_ARG

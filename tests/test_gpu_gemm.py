"""The tcgen05 GEMM core on its own, against a float64 matmul of the same
bf16 operands (debug entry points of the C ABI)."""
import pytest
import torch

from mixture_experts_layer_router_gb300 import capi
import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _rand(shape, seed, scale=1.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * scale).to(torch.bfloat16)


def _ref(A, B):
    return A.double().cpu() @ B.double().cpu().T


def _check(C, ref, out_bf16=True):
    C = C.double().cpu()
    scale = ref.abs().max().item() + 1e-30
    err = (C - ref).abs()
    tol = (ref.abs() * (2.0 ** -8) if out_bf16 else 0) + 1e-5 * scale
    bad = (err > tol).sum().item()
    assert bad == 0, f"{bad} of {ref.numel()} wrong; max err {err.max().item():.3e} (scale {scale:.3e})"


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (256, 512, 256), (300, 384, 640),
                                   (1, 128, 128), (1000, 1024, 1024), (4096, 2048, 1024)])
def test_dense_bf16(M, N, K):
    gh.lib()
    A, B = _rand((M, K), 1), _rand((N, K), 2, 0.1)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert capi.debug_gemm(A, B, C, M, N, K, 0) == capi.OK
    assert capi.debug_status() == 0
    _check(C, _ref(A, B))


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (200, 100, 256), (128, 16, 256), (513, 512, 384)])
def test_dense_f32(M, N, K):
    gh.lib()
    A, B = _rand((M, K), 3), _rand((N, K), 4, 0.1)
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    assert capi.debug_gemm(A, B, C, M, N, K, 1) == capi.OK
    assert capi.debug_status() == 0
    _check(C, _ref(A, B), out_bf16=False)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (130, 384, 512)])
def test_dense_swiglu(M, N, K):
    gh.lib()
    A, B = _rand((M, K), 5, 0.5), _rand((2 * N, K), 6, 0.1)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert capi.debug_gemm(A, B, C, M, N, K, 2) == capi.OK
    assert capi.debug_status() == 0
    r = _ref(A, B)
    g, u = r[:, :N], r[:, N:]
    _check(C, g / (1 + torch.exp(-g)) * u)


@pytest.mark.parametrize("mode,N,offsets", [
    (0, 256, [0, 0, 130, 130, 400, 700, 701]),
    (2, 256, [0, 0, 130, 130, 400, 700, 701]),
    (0, 128, [0, 1, 18, 618, 874, 875]),          # second accumulator unused
    (0, 384, [0, 255, 256, 513, 1200]),           # chunked groups, half-used block
    (2, 128, [0, 17, 17, 300, 1100, 1101, 1357]),
    (2, 384, [0, 64, 64, 64, 320]),
])
def test_grouped(mode, N, offsets):
    gh.lib()
    G, M, K = len(offsets) - 1, offsets[-1], 256
    A = _rand((M, K), 7)
    Bn = N * G * (2 if mode == 2 else 1)
    B = _rand((Bn, K), 8, 0.1)
    C = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    off = torch.tensor(offsets, dtype=torch.int32, device="cuda")
    assert capi.debug_grouped_gemm(A, B, C, off, G, M, N, K, mode) == capi.OK
    assert capi.debug_status() == 0
    ref = torch.zeros((M, N), dtype=torch.float64)
    for g in range(G):
        lo, hi = offsets[g], offsets[g + 1]
        if hi == lo:
            continue
        if mode == 0:
            ref[lo:hi] = _ref(A[lo:hi], B[g * N:(g + 1) * N])
        else:
            gg = _ref(A[lo:hi], B[g * N:(g + 1) * N])
            uu = _ref(A[lo:hi], B[G * N + g * N:G * N + (g + 1) * N])
            ref[lo:hi] = gg / (1 + torch.exp(-gg)) * uu
    _check(C, ref)


def test_bounded_wait_gives_up():
    """A wait nobody completes ends by itself and reports a timeout."""
    import ctypes
    lib = gh.lib()
    v = ctypes.c_uint32(0)
    assert lib.latentmoe_debug_wait_timeout(1_000_000, ctypes.byref(v)) == capi.ERR_TIMEOUT
    assert v.value == capi.STATUS_TIMEOUT
    # the context stays usable
    assert capi.debug_status() == 0
    A, B = _rand((128, 128), 9), _rand((256, 128), 10)
    C = torch.empty((128, 256), dtype=torch.bfloat16, device="cuda")
    assert capi.debug_gemm(A, B, C, 128, 256, 128, 0) == capi.OK
    _check(C, _ref(A, B))

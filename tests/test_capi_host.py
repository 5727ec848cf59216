"""The C-ABI library loads, exports every declared symbol, and validates
arguments on the host before touching the GPU (CPU only)."""
import ctypes
import os
import re

import pytest

from mixture_experts_layer_router_gb300 import build, capi

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "latentmoe.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return capi.load()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(latentmoe_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), n
        assert n in capi.SIGNATURES, f"{n} has no binding"


def test_binding_declares_nothing_extra():
    assert set(capi.SIGNATURES) == set(_declared())


def _dims(**kw):
    base = dict(hidden=256, latent=128, num_experts=16, ffn=256, shared_ffn=0, max_tokens=128)
    base.update(kw)
    return capi.latentmoe_dims(**base)


@pytest.mark.parametrize("kw,k,flags,code", [
    (dict(), 0, 0, capi.ERR_INVALID_ARG),                 # k < 1
    (dict(), 17, 0, capi.ERR_INVALID_ARG),                # k > 16
    (dict(num_experts=4), 5, 0, capi.ERR_INVALID_ARG),    # k > E
    (dict(max_tokens=0), 2, 0, capi.ERR_INVALID_ARG),
    (dict(num_experts=0), 1, 0, capi.ERR_INVALID_ARG),
    (dict(shared_ffn=-128), 2, 0, capi.ERR_INVALID_ARG),
    (dict(), 2, 64, capi.ERR_INVALID_ARG),                # unknown flag bit
    (dict(), 2, 2 | 8, capi.ERR_INVALID_ARG),             # both bias modes
    (dict(hidden=200), 2, 0, capi.ERR_UNSUPPORTED),       # not a multiple of 128
    (dict(latent=64), 2, 0, capi.ERR_UNSUPPORTED),
    (dict(ffn=100), 2, 0, capi.ERR_UNSUPPORTED),
    (dict(shared_ffn=64), 2, 0, capi.ERR_UNSUPPORTED),
    (dict(num_experts=513), 2, 0, capi.ERR_UNSUPPORTED),  # E > 512
    (dict(max_tokens=1 << 28), 16, 0, capi.ERR_UNSUPPORTED),  # slots exceed int32 range
])
def test_create_rejects_bad_arguments(lib, kw, k, flags, code):
    h = ctypes.c_void_p(123)
    d = _dims(**kw)
    assert lib.latentmoe_create(ctypes.byref(d), k, flags, ctypes.byref(h)) == code
    assert h.value is None


def test_null_arguments(lib):
    h = ctypes.c_void_p()
    assert lib.latentmoe_create(None, 2, 0, ctypes.byref(h)) == capi.ERR_INVALID_ARG
    d = _dims()
    assert lib.latentmoe_create(ctypes.byref(d), 2, 0, None) == capi.ERR_INVALID_ARG
    assert lib.latentmoe_destroy(None) == capi.OK
    assert lib.latentmoe_forward(None, None, None, 1, None) == capi.ERR_INVALID_ARG
    assert lib.latentmoe_forward_host(None, None, None, 1, None) == capi.ERR_INVALID_ARG
    assert lib.latentmoe_forward_host_async(None, None, None, 1, None) == capi.ERR_INVALID_ARG
    assert lib.latentmoe_host_wait(None) == capi.ERR_INVALID_ARG
    assert lib.latentmoe_load_weights(None, None, None) == capi.ERR_INVALID_ARG
    assert lib.latentmoe_get_status(None, None) == capi.ERR_INVALID_ARG
    assert lib.latentmoe_debug_gemm(None, None, None, 1, 128, 128, 0, None) == capi.ERR_INVALID_ARG
    # E4M3 entries
    f = (ctypes.c_float * 2)()
    n = ctypes.c_int64()
    assert lib.latentmoe_get_fp8_state(None, f, f, ctypes.byref(n)) == capi.ERR_INVALID_ARG
    assert lib.latentmoe_set_fp8_scales(None, f) == capi.ERR_INVALID_ARG
    assert lib.latentmoe_get_fp8_weight_scales(None, f) == capi.ERR_INVALID_ARG
    assert lib.latentmoe_get_fp8_codes(None, None, None, None) == capi.ERR_INVALID_ARG
    assert lib.latentmoe_quantize_e4m3(None, 1, 1, 16, None, None, None) == capi.ERR_INVALID_ARG
    assert lib.latentmoe_debug_grouped_gemm_e4m3(None, None, None, None, None, None, 1, 1, 128,
                                                 128, 1, None) == capi.ERR_INVALID_ARG


def test_strings_and_stages(lib):
    assert lib.latentmoe_strerror(capi.ERR_TIMEOUT) == b"a bounded device wait timed out"
    n = lib.latentmoe_num_stages()
    names = [lib.latentmoe_stage_name(i).decode() for i in range(n)]
    assert names == ["router", "replay_gates", "sort", "down_proj", "expert_gate_up",
                     "expert_down", "combine", "shared_gate_up", "up_proj",
                     "fp8_scales"]
    assert lib.latentmoe_stage_name(n) is None


def test_missing_library_fails_loudly():
    """No CPU fallback: with the library absent, loading it and creating a
    layer raise instead of computing anything."""
    import subprocess
    import sys
    code = (
        "import mixture_experts_layer_router_gb300.capi as c\n"
        "c._lib = None\n"
        "c.load.__defaults__ = ('/nonexistent/liblatentmoe.so',)\n"
        "try:\n"
        "    c.LatentMoE(256, 128, 16, 2, 256)\n"
        "except RuntimeError as e:\n"
        "    print('raised:', e)\n"
        "    raise SystemExit(3)\n"
        "raise SystemExit(0)\n")
    root = os.path.dirname(os.path.dirname(__file__))
    r = subprocess.run([sys.executable, "-c", code], cwd=root, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 3, r.stdout + r.stderr
    assert "is missing" in r.stdout

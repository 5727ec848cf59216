"""ctypes binding of liblatentmoe.so (include/latentmoe.h), same names.

Argument marshalling only: every step of the layer runs in the library's
CUDA kernels. PyTorch provides device memory (``tensor.data_ptr()``) and
streams (``torch.cuda.current_stream().cuda_stream``). There is no fallback:
``load()`` raises if the library is missing or cannot be loaded.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, Optional  # noqa: F401

_PKG = os.path.dirname(os.path.abspath(__file__))
# LATENTMOE_LIB names another build of the same library (the bounds-checked
# debug build, _build/bounds/liblatentmoe.so); there is no other fallback
LIB_PATH = os.environ.get("LATENTMOE_LIB") or os.path.join(_PKG, "_build", "liblatentmoe.so")

OK = 0
ERR_INVALID_ARG = -1
ERR_UNSUPPORTED = -2
ERR_NOT_LOADED = -3
ERR_CUDA = -4
ERR_TIMEOUT = -5
ERR_DEVICE_STATUS = -6
ERR_OUT_OF_MEMORY = -7

RENORM = 1
ROUTER_BIAS = 2
OUT_FP32 = 4
SELECT_BIAS = 8
FP8_EXPERTS = 16
FP8_DENSE = 32
FP8_TENSORS = 5  # scaled activations: z, h, x, c, shared hidden

STATUS_TIMEOUT = 1
STATUS_BAD_EXPERT = 2
STATUS_ROUNDS = 4
STATUS_BOUNDS = 8

_c_void_p = ctypes.c_void_p
_i64 = ctypes.c_int64


class latentmoe_dims(ctypes.Structure):
    _fields_ = [("hidden", _i64), ("latent", _i64), ("num_experts", _i64),
                ("ffn", _i64), ("shared_ffn", _i64), ("max_tokens", _i64)]


class latentmoe_weights(ctypes.Structure):
    _fields_ = [(n, _c_void_p) for n in
                ("w_r", "b_r", "w_dn", "w_g", "w_u", "w_d", "w_up", "w_gs", "w_us", "w_ds")]


# name -> (restype, argtypes)
SIGNATURES = {
    "latentmoe_create": (ctypes.c_int, [ctypes.POINTER(latentmoe_dims), ctypes.c_int,
                                        ctypes.c_uint32, ctypes.POINTER(_c_void_p)]),
    "latentmoe_load_weights": (ctypes.c_int, [_c_void_p, ctypes.POINTER(latentmoe_weights),
                                                _c_void_p]),
    "latentmoe_forward": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _i64, _c_void_p]),
    "latentmoe_forward_routed": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                                _c_void_p, _i64, _c_void_p]),
    "latentmoe_forward_host": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _i64, _c_void_p]),
    "latentmoe_forward_host_async": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _i64,
                                                    _c_void_p]),
    "latentmoe_host_wait": (ctypes.c_int, [_c_void_p]),
    "latentmoe_destroy": (ctypes.c_int, [_c_void_p]),
    "latentmoe_route_from_logits": (ctypes.c_int, [_c_void_p, _c_void_p, _i64] + [_c_void_p] * 7),
    "latentmoe_route_from_logits_static": (ctypes.c_int, [_c_void_p, _i64, _i64, ctypes.c_int,
                                                          ctypes.c_uint32] + [_c_void_p] * 7),
    "latentmoe_lbl_stats": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "latentmoe_get_routing": (ctypes.c_int, [_c_void_p] + [_c_void_p] * 7 + [_c_void_p]),
    "latentmoe_get_status": (ctypes.c_int, [_c_void_p, ctypes.POINTER(ctypes.c_uint32)]),
    "latentmoe_set_profiling": (ctypes.c_int, [_c_void_p, ctypes.c_int]),
    "latentmoe_get_stage_times": (ctypes.c_int, [_c_void_p, ctypes.c_int,
                                                 ctypes.POINTER(ctypes.c_float), ctypes.c_int]),
    "latentmoe_num_stages": (ctypes.c_int, []),
    "latentmoe_stage_name": (ctypes.c_char_p, [ctypes.c_int]),
    "latentmoe_get_launch_count": (ctypes.c_int, [_c_void_p, ctypes.POINTER(_i64)]),
    "latentmoe_set_pdl": (ctypes.c_int, [_c_void_p, ctypes.c_int]),
    "latentmoe_set_sm_pairs": (ctypes.c_int, [_c_void_p, ctypes.c_int]),
    "latentmoe_set_expert_fusion": (ctypes.c_int, [_c_void_p, ctypes.c_int]),
    "latentmoe_set_capacity": (ctypes.c_int, [_c_void_p, _i64, _i64, _i64]),
    "latentmoe_get_rounds": (ctypes.c_int, [_c_void_p, _c_void_p, ctypes.POINTER(ctypes.c_int32)]),
    "latentmoe_last_cuda_error": (ctypes.c_int, [_c_void_p]),
    "latentmoe_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "latentmoe_debug_gemm": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _i64, _i64, _i64,
                                            ctypes.c_int, _c_void_p]),
    "latentmoe_debug_grouped_gemm": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p,
                                                    _i64, _i64, _i64, _i64, ctypes.c_int,
                                                    _c_void_p]),
    "latentmoe_get_fp8_state": (ctypes.c_int, [_c_void_p, ctypes.POINTER(ctypes.c_float),
                                               ctypes.POINTER(ctypes.c_float),
                                               ctypes.POINTER(_i64)]),
    "latentmoe_get_fp8_codes": (ctypes.c_int, [_c_void_p, _c_void_p, _c_void_p, _c_void_p]),
    "latentmoe_set_fp8_scales": (ctypes.c_int, [_c_void_p, ctypes.POINTER(ctypes.c_float)]),
    "latentmoe_get_fp8_dense_codes": (ctypes.c_int, [_c_void_p] * 5),
    "latentmoe_get_fp8_weight_scales": (ctypes.c_int, [_c_void_p,
                                                       ctypes.POINTER(ctypes.c_float)]),
    "latentmoe_quantize_e4m3": (ctypes.c_int, [_c_void_p, _i64, _i64, _i64, _c_void_p,
                                               _c_void_p, _c_void_p]),
    "latentmoe_debug_grouped_gemm_e4m3": (ctypes.c_int, [_c_void_p] * 6 + [_i64] * 4 +
                                          [ctypes.c_int, _c_void_p]),
    "latentmoe_debug_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint32)]),
    "latentmoe_debug_wait_timeout": (ctypes.c_int, [ctypes.c_uint64,
                                                    ctypes.POINTER(ctypes.c_uint32)]),
}

_lib: Optional[ctypes.CDLL] = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the library (once) and declare every entry point."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it first "
                           "(python -m mixture_experts_layer_router_gb300.build)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


class LatentMoEError(RuntimeError):
    def __init__(self, code: int, what: str, cuda_error: int = 0):
        self.code = code
        self.cuda_error = cuda_error
        msg = load().latentmoe_strerror(code).decode()
        extra = f", cudaError {cuda_error}" if cuda_error else ""
        super().__init__(f"{what}: {msg} ({code}{extra})")


def check(code: int, what: str, handle=None) -> None:
    if code != OK:
        cuda = load().latentmoe_last_cuda_error(handle) if handle is not None else 0
        raise LatentMoEError(code, what, cuda)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


class LatentMoE:
    """A handle on one layer. ``load_weights`` takes a dict as made by
    ``synth.make_weights`` (device bf16 tensors, ``b_r`` fp32 or None); the
    library copies them, so the caller may drop its tensors afterwards."""

    def __init__(self, d: int, l: int, E: int, k: int, F: int, Fs: int = 0,
                 max_tokens: int = 1, renorm: bool = False, router_bias: bool = False,
                 out_fp32: bool = False, select_bias: bool = False, fp8: bool = False,
                 fp8_dense: bool = False):
        lib = load()
        self.dims = latentmoe_dims(d, l, E, F, Fs, max_tokens)
        self.k = k
        self.flags = (RENORM if renorm else 0) | (ROUTER_BIAS if router_bias else 0) | \
            (OUT_FP32 if out_fp32 else 0) | (SELECT_BIAS if select_bias else 0) | \
            (FP8_EXPERTS if fp8 else 0) | (FP8_DENSE if fp8_dense else 0)
        h = _c_void_p()
        check(lib.latentmoe_create(ctypes.byref(self.dims), k, self.flags, ctypes.byref(h)),
              "latentmoe_create")
        self.handle = h

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            load().latentmoe_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def load_weights(self, w: Dict[str, object], stream=None) -> None:
        lw = latentmoe_weights(*(_ptr(w.get(n)) for n in
                                 ("w_r", "b_r", "w_dn", "w_g", "w_u", "w_d", "w_up",
                                  "w_gs", "w_us", "w_ds")))
        check(load().latentmoe_load_weights(self.handle, ctypes.byref(lw), _stream(stream)),
              "latentmoe_load_weights", self.handle)

    def forward(self, x, out=None, stream=None):
        import torch
        T = x.shape[0]
        if out is None:
            dt = torch.float32 if self.flags & OUT_FP32 else torch.bfloat16
            out = torch.empty((T, self.dims.hidden), dtype=dt, device=x.device)
        check(load().latentmoe_forward(self.handle, x.data_ptr(), out.data_ptr(), T,
                                       _stream(stream)), "latentmoe_forward", self.handle)
        return out

    def forward_routed(self, x, idx, gates=None, out=None, stream=None):
        """Router replay: idx [T, k] int32 (and optionally gates [T, k] fp32) given."""
        import torch
        T = x.shape[0]
        if out is None:
            dt = torch.float32 if self.flags & OUT_FP32 else torch.bfloat16
            out = torch.empty((T, self.dims.hidden), dtype=dt, device=x.device)
        check(load().latentmoe_forward_routed(self.handle, x.data_ptr(), idx.data_ptr(),
                                              _ptr(gates), out.data_ptr(), T, _stream(stream)),
              "latentmoe_forward_routed", self.handle)
        return out

    def forward_host(self, x_host, out_host, stream=None):
        check(load().latentmoe_forward_host(self.handle, x_host.data_ptr(), out_host.data_ptr(),
                                            x_host.shape[0], _stream(stream)),
              "latentmoe_forward_host")
        return out_host

    def forward_host_async(self, x_host, out_host, stream=None):
        """Pipelined host-buffer forward: returns at once; x_host must stay
        unchanged and out_host unread until host_wait()."""
        check(load().latentmoe_forward_host_async(self.handle, x_host.data_ptr(),
                                                  out_host.data_ptr(), x_host.shape[0],
                                                  _stream(stream)),
              "latentmoe_forward_host_async")
        return out_host

    def host_wait(self) -> None:
        check(load().latentmoe_host_wait(self.handle), "latentmoe_host_wait")

    def route_from_logits(self, logits, stream=None):
        import torch
        T, E = logits.shape
        dev = logits.device
        k = self.k
        out = {
            "idx": torch.empty((T, k), dtype=torch.int32, device=dev),
            "gates": torch.empty((T, k), dtype=torch.float32, device=dev),
            "counts": torch.empty((E,), dtype=torch.int32, device=dev),
            "offsets": torch.empty((E + 1,), dtype=torch.int32, device=dev),
            "perm": torch.empty((T * k,), dtype=torch.int32, device=dev),
            "pos": torch.empty((T, k), dtype=torch.int32, device=dev),
        }
        check(load().latentmoe_route_from_logits(
            self.handle, logits.data_ptr(), T, out["idx"].data_ptr(), out["gates"].data_ptr(),
            out["counts"].data_ptr(), out["offsets"].data_ptr(), out["perm"].data_ptr(),
            out["pos"].data_ptr(), _stream(stream)), "latentmoe_route_from_logits")
        return out

    def get_routing(self, T: int, device, stream=None):
        import torch
        E, k = self.dims.num_experts, self.k
        out = {
            "logits": torch.empty((T, E), dtype=torch.float32, device=device),
            "idx": torch.empty((T, k), dtype=torch.int32, device=device),
            "gates": torch.empty((T, k), dtype=torch.float32, device=device),
            "counts": torch.empty((E,), dtype=torch.int32, device=device),
            "offsets": torch.empty((E + 1,), dtype=torch.int32, device=device),
            "perm": torch.empty((T * k,), dtype=torch.int32, device=device),
            "pos": torch.empty((T, k), dtype=torch.int32, device=device),
        }
        check(load().latentmoe_get_routing(
            self.handle, *(out[n].data_ptr() for n in
                           ("logits", "idx", "gates", "counts", "offsets", "perm", "pos")),
            _stream(stream)), "latentmoe_get_routing")
        return out

    def lbl_stats(self, device, stream=None):
        """(prob_sum [E] fp32, counts [E] int32) of the last forward."""
        import torch
        E = self.dims.num_experts
        ps = torch.empty((E,), dtype=torch.float32, device=device)
        cn = torch.empty((E,), dtype=torch.int32, device=device)
        check(load().latentmoe_lbl_stats(self.handle, ps.data_ptr(), cn.data_ptr(),
                                         _stream(stream)), "latentmoe_lbl_stats")
        return ps, cn

    def status(self) -> int:
        v = ctypes.c_uint32(0)
        load().latentmoe_get_status(self.handle, ctypes.byref(v))
        return v.value

    def set_profiling(self, slots: int) -> None:
        check(load().latentmoe_set_profiling(self.handle, slots), "latentmoe_set_profiling")

    def stage_times(self, slot: int):
        n = load().latentmoe_num_stages()
        buf = (ctypes.c_float * n)()
        check(load().latentmoe_get_stage_times(self.handle, slot, buf, n),
              "latentmoe_get_stage_times")
        return {stage_name(i): buf[i] for i in range(n)}

    def fp8_state(self):
        """{"scales": [s_z, s_h] for the next forward, "last_amax": the last
        forward's maxima, "steps": forwards entered into the history}."""
        sc = (ctypes.c_float * FP8_TENSORS)()
        am = (ctypes.c_float * FP8_TENSORS)()
        st = _i64(0)
        check(load().latentmoe_get_fp8_state(self.handle, sc, am, ctypes.byref(st)),
              "latentmoe_get_fp8_state")
        return {"scales": list(sc), "last_amax": list(am), "steps": st.value}

    def fp8_codes(self, T: int, device, stream=None):
        """(z codes [T*k, l], h codes [T*k, F]) uint8 of the last forward."""
        import torch
        S = T * self.k
        zc = torch.empty((S, self.dims.latent), dtype=torch.uint8, device=device)
        hc = torch.empty((S, self.dims.ffn), dtype=torch.uint8, device=device)
        check(load().latentmoe_get_fp8_codes(self.handle, zc.data_ptr(), hc.data_ptr(),
                                             _stream(stream)), "latentmoe_get_fp8_codes")
        return zc, hc

    def set_fp8_scales(self, scales) -> None:
        """Scales for z, h[, x, c, shared hidden]; the ones not given are 1."""
        vals = list(scales) + [1.0] * (FP8_TENSORS - len(scales))
        sc = (ctypes.c_float * FP8_TENSORS)(*vals)
        check(load().latentmoe_set_fp8_scales(self.handle, sc), "latentmoe_set_fp8_scales")

    def fp8_weight_scales(self):
        """[3, E] list of lists: scales of W_g, W_u, W_d per expert."""
        return self.fp8_all_weight_scales()[0]

    def fp8_all_weight_scales(self):
        """([3, E] expert scales, {w_dn, w_up, w_gs, w_us, w_ds} dense scales)."""
        E = self.dims.num_experts
        buf = (ctypes.c_float * (3 * E + 5))()
        check(load().latentmoe_get_fp8_weight_scales(self.handle, buf),
              "latentmoe_get_fp8_weight_scales")
        dense = dict(zip(("w_dn", "w_up", "w_gs", "w_us", "w_ds"), buf[3 * E:3 * E + 5]))
        return [list(buf[m * E:(m + 1) * E]) for m in range(3)], dense

    def fp8_dense_codes(self, T: int, device, stream=None):
        """(x codes [T, d], c codes [T, l], shared hidden codes [T, F_s] or None)."""
        import torch
        xc = torch.empty((T, self.dims.hidden), dtype=torch.uint8, device=device)
        cc = torch.empty((T, self.dims.latent), dtype=torch.uint8, device=device)
        sc = torch.empty((T, self.dims.shared_ffn), dtype=torch.uint8, device=device) \
            if self.dims.shared_ffn else None
        check(load().latentmoe_get_fp8_dense_codes(self.handle, xc.data_ptr(), cc.data_ptr(),
                                                   _ptr(sc), _stream(stream)),
              "latentmoe_get_fp8_dense_codes")
        return xc, cc, sc

    def set_capacity(self, capacity: int, group_size: int = 1, max_rounds: int = 0) -> None:
        """Multi-round fixed-capacity expert schedule (capacity 0: one pass)."""
        check(load().latentmoe_set_capacity(self.handle, capacity, group_size, max_rounds),
              "latentmoe_set_capacity", self.handle)

    def rounds(self, device="cuda"):
        """{"needed", "left_over", "launched", "take" [launched, E] int32} of the last forward."""
        import torch
        info = (ctypes.c_int32 * 3)()
        check(load().latentmoe_get_rounds(self.handle, None, info), "latentmoe_get_rounds")
        take = torch.empty((info[2], self.dims.num_experts), dtype=torch.int32, device=device)
        check(load().latentmoe_get_rounds(self.handle, take.data_ptr(), info),
              "latentmoe_get_rounds")
        return {"needed": info[0], "left_over": info[1], "launched": info[2], "take": take}

    def set_sm_pairs(self, enable: bool) -> None:
        check(load().latentmoe_set_sm_pairs(self.handle, int(enable)),
              "latentmoe_set_sm_pairs")

    def set_expert_fusion(self, mode) -> None:
        """0 (or False): two expert launches; 1 (or True): one fused launch where
        the shapes allow; 2: automatic (the default)."""
        check(load().latentmoe_set_expert_fusion(self.handle, int(mode)),
              "latentmoe_set_expert_fusion", self.handle)

    def set_pdl(self, enable: bool) -> None:
        check(load().latentmoe_set_pdl(self.handle, 1 if enable else 0), "latentmoe_set_pdl",
              self.handle)

    def launch_count(self) -> int:
        v = _i64(0)
        check(load().latentmoe_get_launch_count(self.handle, ctypes.byref(v)),
              "latentmoe_get_launch_count")
        return v.value


def stage_name(i: int) -> str:
    return load().latentmoe_stage_name(i).decode()


def debug_gemm(A, B, C, M: int, N: int, K: int, mode: int, stream=None) -> int:
    return load().latentmoe_debug_gemm(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K, mode,
                                       _stream(stream))


def debug_grouped_gemm(A, B, C, offsets, groups: int, M: int, N: int, K: int, mode: int,
                       stream=None) -> int:
    return load().latentmoe_debug_grouped_gemm(A.data_ptr(), B.data_ptr(), C.data_ptr(),
                                               offsets.data_ptr(), groups, M, N, K, mode,
                                               _stream(stream))


def quantize_e4m3(src, codes, scales, stream=None) -> int:
    """src bf16 [G, R, C] (device) -> codes uint8 [G, R, C], scales fp32 [G]."""
    G, R, C = src.shape
    return load().latentmoe_quantize_e4m3(src.data_ptr(), G, R, C, codes.data_ptr(),
                                          scales.data_ptr(), _stream(stream))


def debug_grouped_gemm_e4m3(A, B, scales, C, amax, offsets, groups: int, M: int, N: int, K: int,
                            mode: int, stream=None) -> int:
    return load().latentmoe_debug_grouped_gemm_e4m3(
        A.data_ptr(), B.data_ptr(), scales.data_ptr(), C.data_ptr(), _ptr(amax),
        offsets.data_ptr(), groups, M, N, K, mode, _stream(stream))


def debug_status() -> int:
    v = ctypes.c_uint32(0)
    load().latentmoe_debug_status(ctypes.byref(v))
    return v.value

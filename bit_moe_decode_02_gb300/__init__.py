"""Python binding of libmoe (the C ABI in include/moe.h), argument marshalling only.

Every step of the routed-expert block runs in the library's CUDA kernels; this
module turns torch tensors into pointers and streams and raises on a non-zero
status.  There is no CPU fallback: if libmoe.so is missing the import of the
library fails loudly (build it with ``python -m bit_moe_decode_02_gb300.build_ext``).

The function names are the C names: moe_create, moe_load_experts, moe_load_experts_ex,
moe_forward, moe_forward_host, moe_forward_stack, moe_forward_stack_steps, moe_forward_steps,
moe_load_router, moe_debug_router_logits, moe_set_batched_numerics, moe_set_swiglu, moe_get_status,
moe_debug_dequant, moe_debug_route, moe_debug_stack_trace, moe_debug_forward_f32,
moe_debug_set_wait, moe_last_bytes, moe_expert_bytes, moe_last_launches, moe_last_error,
moe_forward_noalloc, moe_debug_stream_weights, moe_destroy.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_OOM = -3
MOE_ERR_CUDA = -4
MOE_ERR_NOT_LOADED = -5
MOE_ERR_DEVICE_TIMEOUT = -6
MOE_ERR_DEVICE_FAULT = -7
MOE_FMT_MXFP4 = 1
MOE_FMT_INT4 = 2
MOE_LOAD_GATE_UP_INTERLEAVED = 1
MOE_LOAD_TRANSPOSED = 2
MOE_BATCHED_MXFP4 = 0
MOE_BATCHED_BF16 = 1

# every symbol include/moe.h declares
EXPORTS = ("moe_create", "moe_load_experts", "moe_load_experts_ex", "moe_forward", "moe_forward_host",
           "moe_forward_stack", "moe_forward_stack_steps", "moe_forward_steps", "moe_load_router",
           "moe_debug_router_logits", "moe_set_batched_numerics", "moe_set_swiglu", "moe_get_status", "moe_debug_dequant",
           "moe_debug_route",
           "moe_debug_stack_trace", "moe_debug_mx_quantize", "moe_debug_batched_h",
           "moe_debug_forward_f32", "moe_debug_set_wait",
           "moe_last_bytes", "moe_expert_bytes", "moe_last_launches", "moe_last_error",
           "moe_forward_noalloc", "moe_debug_stream_weights", "moe_destroy")


class MoeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"libmoe status {status}: {msg}")
        self.status = status


class moe_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int), ("intermediate", ctypes.c_int),
                ("num_experts", ctypes.c_int), ("num_layers", ctypes.c_int),
                ("max_tokens", ctypes.c_int), ("max_top_k", ctypes.c_int),
                ("format", ctypes.c_int), ("group", ctypes.c_int), ("has_bias", ctypes.c_int)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmoe.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run python -m bit_moe_decode_02_gb300.build_ext")
        L = ctypes.CDLL(LIB_PATH)
        p, i, ll = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong
        L.moe_create.argtypes = [ctypes.POINTER(moe_config), ctypes.POINTER(p)]
        L.moe_create.restype = i
        L.moe_load_experts.argtypes = [p, i, p, p, p, p, p, p, p]
        L.moe_load_experts.restype = i
        L.moe_load_experts_ex.argtypes = [p, i, p, p, p, p, p, p, i, p]
        L.moe_load_experts_ex.restype = i
        L.moe_debug_stream_weights.argtypes = [p, i, i, ll, p]
        L.moe_debug_stream_weights.restype = i
        L.moe_set_batched_numerics.argtypes = [p, i]
        L.moe_set_batched_numerics.restype = i
        L.moe_set_swiglu.argtypes = [p, ctypes.c_float, ctypes.c_float, ctypes.c_float]
        L.moe_set_swiglu.restype = i
        L.moe_forward.argtypes = [p, i, p, p, i, i, p, p]
        L.moe_forward.restype = i
        L.moe_forward_host.argtypes = [p, i, p, p, i, i, p, p]
        L.moe_forward_host.restype = i
        L.moe_forward_stack.argtypes = [p, p, p, i, i, p]
        L.moe_forward_stack.restype = i
        L.moe_forward_stack_steps.argtypes = [p, i, p, p, i, i, p]
        L.moe_forward_stack_steps.restype = i
        L.moe_load_router.argtypes = [p, i, p, p]
        L.moe_load_router.restype = i
        L.moe_debug_router_logits.argtypes = [p, p, i, p]
        L.moe_debug_router_logits.restype = i
        L.moe_forward_steps.argtypes = [p, i, i, p, p, i, i, p, p]
        L.moe_forward_steps.restype = i
        L.moe_get_status.argtypes = [p, p]
        L.moe_get_status.restype = i
        L.moe_debug_dequant.argtypes = [p, i, i, i, p, p]
        L.moe_debug_dequant.restype = i
        L.moe_debug_route.argtypes = [p, p, i, i, p, p, p]
        L.moe_debug_route.restype = i
        L.moe_debug_stack_trace.argtypes = [p, p, p, i, i, p, p]
        L.moe_debug_stack_trace.restype = i
        L.moe_debug_mx_quantize.argtypes = [p, ll, p, p, p]
        L.moe_debug_mx_quantize.restype = i
        L.moe_debug_batched_h.argtypes = [p, p, p, p]
        L.moe_debug_batched_h.restype = i
        L.moe_debug_forward_f32.argtypes = [p, i, p, p, i, i, p, p, p]
        L.moe_debug_forward_f32.restype = i
        L.moe_debug_set_wait.argtypes = [p, i, i]
        L.moe_debug_set_wait.restype = i
        L.moe_last_bytes.argtypes = [p, p, ctypes.POINTER(ll)]
        L.moe_last_bytes.restype = i
        L.moe_expert_bytes.argtypes = [p]
        L.moe_expert_bytes.restype = ll
        L.moe_last_launches.argtypes = [p]
        L.moe_last_launches.restype = i
        L.moe_last_error.argtypes = []
        L.moe_last_error.restype = ctypes.c_char_p
        L.moe_forward_noalloc.argtypes = [ctypes.POINTER(moe_config), p, p, p, p, p, p, p, p, i, i,
                                          p, p]
        L.moe_forward_noalloc.restype = i
        L.moe_destroy.argtypes = [p]
        L.moe_destroy.restype = None
        _lib = L
    return _lib


def moe_last_error() -> str:
    return lib().moe_last_error().decode()


def _check(rc: int) -> int:
    if rc != MOE_OK:
        raise MoeError(rc, moe_last_error())
    return rc


def _ptr(t):
    """device or host address of a torch tensor / numpy array / int / None"""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        return t.data_ptr()
    return t.ctypes.data


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def moe_create(hidden, intermediate, num_experts, num_layers=1, max_tokens=1, max_top_k=4,
               format=MOE_FMT_MXFP4, group=32, has_bias=1) -> int:
    cfg = moe_config(hidden, intermediate, num_experts, num_layers, max_tokens, max_top_k,
                     format, group, int(has_bias))
    h = ctypes.c_void_p()
    _check(lib().moe_create(ctypes.byref(cfg), ctypes.byref(h)))
    return h.value


def moe_load_experts(h, layer, gu_codes, gu_scales, gu_bias, dn_codes, dn_scales, dn_bias,
                     stream=None):
    return _check(lib().moe_load_experts(h, layer, _ptr(gu_codes), _ptr(gu_scales), _ptr(gu_bias),
                                         _ptr(dn_codes), _ptr(dn_scales), _ptr(dn_bias),
                                         _stream(stream)))


def moe_load_experts_ex(h, layer, gu_codes, gu_scales, gu_bias, dn_codes, dn_scales, dn_bias, flags,
                        stream=None):
    return _check(lib().moe_load_experts_ex(h, layer, _ptr(gu_codes), _ptr(gu_scales), _ptr(gu_bias),
                                            _ptr(dn_codes), _ptr(dn_scales), _ptr(dn_bias), flags,
                                            _stream(stream)))


def moe_forward(h, layer, x, logits, M, top_k, out, stream=None):
    return _check(lib().moe_forward(h, layer, _ptr(x), _ptr(logits), M, top_k, _ptr(out),
                                    _stream(stream)))


def moe_forward_host(h, layer, x, logits, M, top_k, out, stream=None):
    return _check(lib().moe_forward_host(h, layer, _ptr(x), _ptr(logits), M, top_k, _ptr(out),
                                         _stream(stream)))


def moe_forward_stack(h, resid, logits, M, top_k, stream=None):
    return _check(lib().moe_forward_stack(h, _ptr(resid), _ptr(logits), M, top_k, _stream(stream)))


def moe_forward_stack_steps(h, n, resid, logits, M, top_k, stream=None):
    return _check(lib().moe_forward_stack_steps(h, n, _ptr(resid), _ptr(logits), M, top_k, _stream(stream)))


def moe_load_router(h, layer, w, bias=None):
    """Router weights w bf16 bits [E][H] and bias [E] (numpy uint16 arrays or tensors)."""
    return _check(lib().moe_load_router(h, layer, _ptr(w), _ptr(bias)))


def moe_debug_stream_weights(h, layer0, n, nbytes, stream=None):
    return _check(lib().moe_debug_stream_weights(h, layer0, n, nbytes, _stream(stream)))


def moe_set_swiglu(h, alpha, limit, beta):
    return _check(lib().moe_set_swiglu(h, alpha, limit, beta))


def moe_set_batched_numerics(h, numerics):
    return _check(lib().moe_set_batched_numerics(h, numerics))


def moe_debug_router_logits(h, out, M, stream=None):
    return _check(lib().moe_debug_router_logits(h, _ptr(out), M, _stream(stream)))


def moe_forward_steps(h, n, layer0, x, logits, M, top_k, out, stream=None):
    return _check(lib().moe_forward_steps(h, n, layer0, _ptr(x), _ptr(logits), M, top_k, _ptr(out),
                                          _stream(stream)))


def moe_get_status(h, stream=None) -> int:
    return lib().moe_get_status(h, _stream(stream))


def moe_debug_dequant(h, layer, expert, proj, out, stream=None):
    return _check(lib().moe_debug_dequant(h, layer, expert, proj, _ptr(out), _stream(stream)))


def moe_debug_route(h, logits, M, top_k, idx, w, stream=None):
    return _check(lib().moe_debug_route(h, _ptr(logits), M, top_k, _ptr(idx), _ptr(w),
                                        _stream(stream)))


def moe_debug_stack_trace(h, resid, logits, M, top_k, trace, stream=None):
    return _check(lib().moe_debug_stack_trace(h, _ptr(resid), _ptr(logits), M, top_k, _ptr(trace),
                                              _stream(stream)))


def moe_debug_mx_quantize(x, n, codes, scales, stream=None):
    return _check(lib().moe_debug_mx_quantize(_ptr(x), n, _ptr(codes), _ptr(scales), _stream(stream)))


def moe_debug_batched_h(h, codes, scales, stream=None):
    return _check(lib().moe_debug_batched_h(h, _ptr(codes), _ptr(scales), _stream(stream)))


def moe_debug_forward_f32(h, layer, x, logits, M, top_k, out, out_f32, stream=None):
    return _check(lib().moe_debug_forward_f32(h, layer, _ptr(x), _ptr(logits), M, top_k, _ptr(out),
                                              _ptr(out_f32), _stream(stream)))


def moe_debug_set_wait(h, spin_limit, skip_cta=-1):
    return _check(lib().moe_debug_set_wait(h, spin_limit, skip_cta))


def moe_last_bytes(h, stream=None) -> int:
    b = ctypes.c_longlong()
    _check(lib().moe_last_bytes(h, _stream(stream), ctypes.byref(b)))
    return b.value


def moe_expert_bytes(h) -> int:
    return lib().moe_expert_bytes(h)


def moe_last_launches(h) -> int:
    return lib().moe_last_launches(h)


def moe_forward_noalloc(cfg: moe_config, gu_codes, gu_scales, gu_bias, dn_codes, dn_scales, dn_bias,
                        x, logits, M, top_k, out, stream=None):
    """The allocation-free layer forward (see include/moe.h): caller-layout
    weights, inputs and outputs are all caller memory; scratch is the
    library's fixed device array."""
    return _check(lib().moe_forward_noalloc(ctypes.byref(cfg), _ptr(gu_codes), _ptr(gu_scales),
                                            _ptr(gu_bias), _ptr(dn_codes), _ptr(dn_scales),
                                            _ptr(dn_bias), _ptr(x), _ptr(logits), M, top_k,
                                            _ptr(out), _stream(stream)))


def moe_destroy(h) -> None:
    lib().moe_destroy(h)

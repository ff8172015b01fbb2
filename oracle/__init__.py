"""Plain fp64 CPU oracle for the routed-expert block of a 4-bit MoE decode step.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers.  The product library never
imports, links or executes anything in this directory, and this directory never
imports the product package: the two paths share no code.  Seeded inputs come
from ``bit_moe_decode_02_gb300.synth``, which holds no arithmetic of the method.

The arithmetic lives in ``moe_oracle.c`` (fp64, textbook loops); this module
compiles it with gcc on first use and wraps it with ctypes.  Every function
cites the passage it follows in the C source.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

FMT_MXFP4 = 1
FMT_INT4 = 2


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into libmoe_oracle.so (gcc, -O2, no fast-math)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
            "-ffp-contract=off", _SRC, "-o", _LIB_PATH + ".tmp", "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(_LIB_PATH + ".tmp", _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            d, i, p, u16, i64 = (ctypes.c_double, ctypes.c_int, ctypes.c_void_p,
                                 ctypes.c_uint16, ctypes.c_int64)
            L.moe_oracle_e2m1.restype = d
            L.moe_oracle_e2m1.argtypes = [i]
            L.moe_oracle_e8m0.restype = d
            L.moe_oracle_e8m0.argtypes = [i]
            L.moe_oracle_fp16.restype = d
            L.moe_oracle_fp16.argtypes = [u16]
            L.moe_oracle_bf16.restype = d
            L.moe_oracle_bf16.argtypes = [u16]
            L.moe_oracle_to_bf16.restype = u16
            L.moe_oracle_to_bf16.argtypes = [d]
            L.moe_oracle_dequant.restype = None
            L.moe_oracle_dequant.argtypes = [i, p, p, i, i, i, p]
            L.moe_oracle_route.restype = None
            L.moe_oracle_route.argtypes = [p, i, i, i, p, p]
            L.moe_oracle_layer.restype = i
            L.moe_oracle_layer.argtypes = [i, i, i, i, i, i, i, p, p, p, p, p, p, p, p, p, p, p, p, i]
            L.moe_oracle_stack.restype = i
            L.moe_oracle_stack.argtypes = [i, i, i, i, i, i, i, i, p, p, p, p, p, p, p, p, p, p, i]
            L.moe_oracle_set_swiglu.restype = None
            L.moe_oracle_set_swiglu.argtypes = [d, d, d]
            L.moe_oracle_router.restype = None
            L.moe_oracle_router.argtypes = [i, i, i, p, p, p, p]
            L.moe_oracle_mx_quantize.restype = None
            L.moe_oracle_mx_quantize.argtypes = [p, i64, p, p]
            L.moe_oracle_layer_batched.restype = i
            L.moe_oracle_layer_batched.argtypes = [i, i, i, i, i] + [p] * 14 + [i]
            L.moe_oracle_max_threads.restype = i
            L.moe_oracle_max_threads.argtypes = []
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------
# Scalar formats (OCP MX v1.0 E2M1 / E8M0; IEEE binary16; bfloat16)
# --------------------------------------------------------------------------

def e2m1(code: int) -> float:
    return lib().moe_oracle_e2m1(int(code))


def e8m0(byte: int) -> float:
    return lib().moe_oracle_e8m0(int(byte))


def fp16(bits: int) -> float:
    return lib().moe_oracle_fp16(int(bits))


def bf16(bits: int) -> float:
    return lib().moe_oracle_bf16(int(bits))


def to_bf16(v: float) -> int:
    return int(lib().moe_oracle_to_bf16(float(v)))


def bf16_array(bits: np.ndarray) -> np.ndarray:
    f = np.vectorize(lambda b: lib().moe_oracle_bf16(int(b)), otypes=[np.float64])
    return f(np.asarray(bits, dtype=np.uint16))


def to_bf16_array(v: np.ndarray) -> np.ndarray:
    f = np.vectorize(lambda x: lib().moe_oracle_to_bf16(float(x)), otypes=[np.uint16])
    return f(np.asarray(v, dtype=np.float64))


def max_threads() -> int:
    return int(lib().moe_oracle_max_threads())


# --------------------------------------------------------------------------
# Weights, router, layer, stack
# --------------------------------------------------------------------------

def dequant(fmt: int, codes: np.ndarray, scales: np.ndarray, N: int, K: int,
            group: int = 32) -> np.ndarray:
    """W [N][K] fp64 of one packed projection (codes [N][K/2], scales per block)."""
    codes = _c(codes, np.uint8)
    scales = _c(scales, np.uint8 if fmt == FMT_MXFP4 else np.uint16)
    out = np.empty((N, K), dtype=np.float64)
    lib().moe_oracle_dequant(fmt, _ptr(codes), _ptr(scales), N, K, group, _ptr(out))
    return out


def route(logits: np.ndarray, k: int):
    """(idx [M][k] int32 in selection order, w [M][k] fp64)."""
    logits = _c(logits, np.float32)
    M, E = logits.shape
    idx = np.empty((M, k), dtype=np.int32)
    w = np.empty((M, k), dtype=np.float64)
    lib().moe_oracle_route(_ptr(logits), M, E, k, _ptr(idx), _ptr(w))
    return idx, w


def _scale_dtype(fmt):
    return np.uint8 if fmt == FMT_MXFP4 else np.uint16


def layer(fmt: int, H: int, I: int, E: int, k: int, t, x: np.ndarray, logits: np.ndarray,
          r: np.ndarray | None = None, group: int = 32, nthreads: int = 1):
    """One decode layer in fp64.  ``t`` holds gu_codes, gu_scales, gu_bias,
    dn_codes, dn_scales, dn_bias (numpy; biases may be None), laid out as
    [E][2I][H/2] / [E][2I][H/blk] / [E][2I] and [E][H][I/2] / [E][H][I/blk] / [E][H].
    x, r are bf16 bit patterns (uint16) [M][H]; logits fp32 [M][E].
    Returns (out fp64 [M][H], idx [M][k], w [M][k])."""
    x = _c(x, np.uint16)
    M = x.shape[0]
    logits = _c(logits, np.float32)
    r = _c(r, np.uint16)
    sd = _scale_dtype(fmt)
    arrs = [_c(t.gu_codes, np.uint8), _c(t.gu_scales, sd), _c(t.gu_bias, np.uint16),
            _c(t.dn_codes, np.uint8), _c(t.dn_scales, sd), _c(t.dn_bias, np.uint16)]
    out = np.empty((M, H), dtype=np.float64)
    idx = np.empty((M, k), dtype=np.int32)
    w = np.empty((M, k), dtype=np.float64)
    rc = lib().moe_oracle_layer(fmt, H, I, E, group, M, k, *[_ptr(a) for a in arrs],
                                _ptr(x), _ptr(logits), _ptr(r), _ptr(out), _ptr(idx), _ptr(w),
                                nthreads)
    if rc != 0:
        raise ValueError("oracle layer: bad arguments")
    return out, idx, w


class swiglu:
    """Context manager: the SwiGLU form h = gc sigmoid(alpha gc) (uc + beta),
    gc = min(g, limit), uc = clamp(u, -limit, limit), for the oracle calls
    inside it; (1, inf, 0) -- the plain silu(g) u -- outside."""

    def __init__(self, alpha: float = 1.0, limit: float = float("inf"), beta: float = 0.0):
        self.args = (float(alpha), float(limit), float(beta))

    def __enter__(self):
        lib().moe_oracle_set_swiglu(*self.args)
        return self

    def __exit__(self, *exc):
        lib().moe_oracle_set_swiglu(1.0, float("inf"), 0.0)
        return False


def router(x: np.ndarray, w: np.ndarray, b: np.ndarray | None = None) -> np.ndarray:
    """Router GEMV in fp64: logits [M][E] = b + x W^T for bf16 bit patterns
    x [M][H], w [E][H], b [E] (or None)."""
    x = _c(x, np.uint16)
    w = _c(w, np.uint16)
    b = _c(b, np.uint16)
    M, H = x.shape
    E = w.shape[0]
    out = np.empty((M, E), dtype=np.float64)
    lib().moe_oracle_router(H, E, M, _ptr(x), _ptr(w), _ptr(b), _ptr(out))
    return out


def stack(fmt: int, H: int, I: int, E: int, k: int, layers, logits: np.ndarray | None,
          resid: np.ndarray, group: int = 32, nthreads: int = 1, routers=None) -> np.ndarray:
    """Expert stack with the weightless RMSNorm coupling; returns r_L (bf16 bits).
    With ``routers`` (one (W bf16 [E][H], b bf16 [E] or None) per layer) each
    layer's logits are the router GEMV of its input, rounded to fp32, and
    ``logits`` is not read (it may be None)."""
    L = len(layers)
    M = np.asarray(resid).shape[0]
    logits = _c(np.zeros((L, M, E), np.float32) if logits is None else logits, np.float32)
    resid = np.array(resid, dtype=np.uint16, copy=True, order="C")
    sd = _scale_dtype(fmt)
    keep = []

    def parr(name, dt):
        vals = []
        for t in layers:
            a = getattr(t, name)
            a = _c(a, dt)
            keep.append(a)
            vals.append(0 if a is None else a.ctypes.data)
        if all(v == 0 for v in vals):
            return None
        return (ctypes.c_void_p * L)(*vals)

    ptrs = [parr("gu_codes", np.uint8), parr("gu_scales", sd), parr("gu_bias", np.uint16),
            parr("dn_codes", np.uint8), parr("dn_scales", sd), parr("dn_bias", np.uint16)]
    rw = rb = None
    if routers is not None:
        assert len(routers) == L
        ws = [_c(w_, np.uint16) for w_, _ in routers]
        bs = [_c(b_, np.uint16) for _, b_ in routers]
        keep.extend(ws + bs)
        rw = (ctypes.c_void_p * L)(*[a.ctypes.data for a in ws])
        if any(a is not None for a in bs):
            rb = (ctypes.c_void_p * L)(*[0 if a is None else a.ctypes.data for a in bs])
    rc = lib().moe_oracle_stack(fmt, H, I, E, group, L, M, k,
                                *[ctypes.cast(p, ctypes.c_void_p) if p is not None else None
                                  for p in ptrs],
                                _ptr(logits), _ptr(resid),
                                ctypes.cast(rw, ctypes.c_void_p) if rw is not None else None,
                                ctypes.cast(rb, ctypes.c_void_p) if rb is not None else None, nthreads)
    if rc != 0:
        raise ValueError("oracle stack: bad arguments")
    return resid


def mx_quantize(v: np.ndarray):
    """OCP MX conversion of a vector (length multiple of 32) to MXFP4:
    (codes [n/2] u8, scales [n/32] u8)."""
    v = _c(v, np.float64).ravel()
    n = v.size
    codes = np.empty(n // 2, dtype=np.uint8)
    scales = np.empty(n // 32, dtype=np.uint8)
    lib().moe_oracle_mx_quantize(_ptr(v), n, _ptr(codes), _ptr(scales))
    return codes, scales


def layer_batched(H: int, I: int, E: int, k: int, t, x: np.ndarray, logits: np.ndarray,
                  r: np.ndarray | None = None, h_codes_in=None, h_scales_in=None,
                  want_h: bool = False, nthreads: int = 1):
    """Batched MXFP4 layer with MX-quantised x and h (see moe_oracle.c).
    Returns out fp64 [M][H] and, if want_h, the oracle's (h_codes [M][k][I/2],
    h_scales [M][k][I/32])."""
    x = _c(x, np.uint16)
    M = x.shape[0]
    logits = _c(logits, np.float32)
    r = _c(r, np.uint16)
    arrs = [_c(t.gu_codes, np.uint8), _c(t.gu_scales, np.uint8), _c(t.gu_bias, np.uint16),
            _c(t.dn_codes, np.uint8), _c(t.dn_scales, np.uint8), _c(t.dn_bias, np.uint16)]
    hci = _c(h_codes_in, np.uint8)
    hsi = _c(h_scales_in, np.uint8)
    hco = np.empty((M, k, I // 2), dtype=np.uint8) if want_h else None
    hso = np.empty((M, k, I // 32), dtype=np.uint8) if want_h else None
    out = np.empty((M, H), dtype=np.float64)
    rc = lib().moe_oracle_layer_batched(H, I, E, M, k, *[_ptr(a) for a in arrs], _ptr(x),
                                        _ptr(logits), _ptr(r), _ptr(hci), _ptr(hsi),
                                        _ptr(hco), _ptr(hso), _ptr(out), nthreads)
    if rc != 0:
        raise ValueError("oracle batched layer: bad arguments")
    if want_h:
        return out, hco, hso
    return out

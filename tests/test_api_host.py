"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/moe.h declares, and rejects bad arguments before any
CUDA call."""
import ctypes
import os
import re

import pytest

import bit_moe_decode_02_gb300 as moe
from bit_moe_decode_02_gb300 import build_ext

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build_ext.build()
    return moe.lib()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_function(L):
    declared = _declared_functions()
    assert set(declared) == set(moe.EXPORTS)
    for name in declared:
        assert hasattr(L, name), name


def _cfg(**kw):
    base = dict(hidden=256, intermediate=256, num_experts=8, num_layers=1, max_tokens=1,
                max_top_k=2, format=moe.MOE_FMT_MXFP4, group=32, has_bias=1)
    base.update(kw)
    return moe.moe_config(*[base[f] for f, _ in moe.moe_config._fields_])


@pytest.mark.parametrize("bad,needle", [
    (dict(hidden=100), "hidden"), (dict(hidden=0), "hidden"), (dict(hidden=8192), "hidden"),
    (dict(hidden=96), "hidden"), (dict(intermediate=3136), "intermediate"),
    (dict(intermediate=48), "intermediate"), (dict(num_experts=0), "num_experts"),
    (dict(num_experts=300), "num_experts"), (dict(num_layers=0), "num_layers"),
    (dict(max_tokens=0), "max_tokens"), (dict(max_tokens=8193), "max_tokens"),
    (dict(max_top_k=0), "max_top_k"), (dict(max_top_k=9), "max_top_k"),
    (dict(max_top_k=17, num_experts=64), "max_top_k"), (dict(format=3), "format"),
    (dict(group=64), "group"), (dict(format=moe.MOE_FMT_INT4, group=48), "group"),
    (dict(format=moe.MOE_FMT_INT4, group=512), "group"), (dict(has_bias=2), "has_bias"),
])
def test_create_rejects_bad_config(L, bad, needle):
    h = ctypes.c_void_p(123)
    rc = L.moe_create(ctypes.byref(_cfg(**bad)), ctypes.byref(h))
    assert rc == moe.MOE_ERR_INVALID_ARG
    assert h.value is None
    assert needle in moe.moe_last_error()


def test_batched_path_needs_mxfp4(L):
    """max_tokens > 4 enables the tensor-core path, which runs MXFP4 only."""
    h = ctypes.c_void_p(123)
    rc = L.moe_create(ctypes.byref(_cfg(max_tokens=8, format=moe.MOE_FMT_INT4, group=64)), ctypes.byref(h))
    assert rc == moe.MOE_ERR_UNSUPPORTED
    assert h.value is None
    assert "MXFP4" in moe.moe_last_error()


def test_debug_entry_points_check_arguments(L):
    buf = ctypes.create_string_buffer(4096)
    addr = (ctypes.addressof(buf) + 15) & ~15
    assert L.moe_debug_mx_quantize(None, 32, addr, addr, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_debug_mx_quantize(addr, 33, addr, addr, None) == moe.MOE_ERR_INVALID_ARG
    assert "multiple of 32" in moe.moe_last_error()
    assert L.moe_debug_mx_quantize(addr + 4, 32, addr, addr, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_debug_batched_h(None, addr, addr, None) == moe.MOE_ERR_INVALID_ARG


def test_null_arguments_rejected(L):
    assert L.moe_create(None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_create(ctypes.byref(_cfg()), None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_load_experts(None, 0, None, None, None, None, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_forward(None, 0, None, None, 1, 1, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_forward_host(None, 0, None, None, 1, 1, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_forward_stack(None, None, None, 1, 1, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_get_status(None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_debug_dequant(None, 0, 0, 0, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_debug_route(None, None, 1, 1, None, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_debug_stack_trace(None, None, None, 1, 1, None, None) == moe.MOE_ERR_INVALID_ARG
    b = ctypes.c_longlong()
    assert L.moe_last_bytes(None, None, ctypes.byref(b)) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_expert_bytes(None) == 0
    assert L.moe_last_launches(None) == 0
    L.moe_destroy(None)


def test_create_without_gpu_fails_cleanly(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    h = ctypes.c_void_p(123)
    rc = L.moe_create(ctypes.byref(_cfg()), ctypes.byref(h))
    assert rc == moe.MOE_ERR_CUDA and h.value is None
    assert moe.moe_last_error()

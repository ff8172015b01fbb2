"""Helpers shared by the tests: tolerance, marshalling between the seeded
numpy inputs and device tensors, handle set-up.  No arithmetic of the method
lives here: the expected values come from the oracle."""
from __future__ import annotations

import numpy as np

import oracle
from bit_moe_decode_02_gb300 import synth

# Parity bar: max |gpu - oracle| <= REL * max|oracle| + ULPS * ulp_bf16(oracle)
# per element.  REL is the stated 2e-3 of the output's max-norm for
# fp32-accumulated outputs; the ULPS term is the bf16 output rounding itself
# (half an ulp for one rounding; one ulp where both sides round a residual
# at every layer and may land on either side of a rounding boundary).
REL = 2e-3


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    a = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    import torch
    b = np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)
    return torch.from_numpy(b).view(torch.bfloat16).to(torch.float64).numpy()


def assert_parity(gpu: np.ndarray, ref: np.ndarray, ulps: float = 0.5, rel: float = REL, what=""):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    assert gpu.shape == ref.shape
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite GPU output"
    err = np.abs(gpu - ref)
    bound = rel * np.abs(ref).max() + ulps * bf16_ulp(ref)
    bad = np.flatnonzero(err > bound)
    assert bad.size == 0, (f"{what}: {bad.size} elements out of tolerance; worst at "
                           f"{bad[np.argmax((err - bound).ravel()[bad])]}: "
                           f"max err {err.max():.4g} vs max|ref| {np.abs(ref).max():.4g}")
    return float(err.max() / max(np.abs(ref).max(), 1e-300))


def assert_parity_f32(got32: np.ndarray, ref: np.ndarray, what=""):
    """The stated bar on the fp32-accumulated output itself (before its bf16
    rounding): max |gpu - oracle| <= 2e-3 * max|oracle|, nothing added."""
    return assert_parity(got32, ref, ulps=0.0, what=what + " (fp32, before rounding)")


def forward_both(moe, h, layer, x, r, logits, k):
    """One forward through moe_debug_forward_f32: (bf16 output as f64, fp32
    output before rounding as f64)."""
    import torch
    xd = to_dev_bf16(x)
    out = to_dev_bf16(r)
    o32 = torch.empty(out.shape, dtype=torch.float32, device="cuda")
    ld = torch.from_numpy(np.ascontiguousarray(logits, np.float32)).cuda()
    moe.moe_debug_forward_f32(h, layer, xd, ld, x.shape[0], k, out, o32)
    torch.cuda.synchronize()
    assert moe.moe_get_status(h) == 0
    return bf16_bits_to_f64(dev_to_bits(out)), o32.cpu().numpy().astype(np.float64)


def to_dev_bf16(bits: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)).cuda()


def dev_to_bits(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def create_handle(shape: synth.Shape, layers: int = 1, max_tokens: int = 4, max_top_k=None):
    import bit_moe_decode_02_gb300 as moe
    return moe.moe_create(shape.hidden, shape.intermediate, shape.experts, layers, max_tokens,
                          max_top_k or shape.top_k,
                          moe.MOE_FMT_MXFP4 if shape.fmt == synth.FMT_MXFP4 else moe.MOE_FMT_INT4,
                          shape.group, 1 if shape.has_bias else 0)


def load_layer(h, layer: int, t: synth.LayerTensors):
    import bit_moe_decode_02_gb300 as moe
    moe.moe_load_experts(h, layer, t.gu_codes, t.gu_scales, t.gu_bias, t.dn_codes, t.dn_scales,
                         t.dn_bias)


def oracle_layer(shape: synth.Shape, t, x, logits, r, k=None, nthreads=None):
    nthreads = nthreads or oracle.max_threads()
    return oracle.layer(shape.fmt, shape.hidden, shape.intermediate, shape.experts,
                        k or shape.top_k, t, x, logits, r, group=shape.group, nthreads=nthreads)


def sparse_layer(shape: synth.Shape, layer: int, experts) -> synth.LayerTensors:
    """A layer's tensors with only `experts` generated (the rest zero): enough
    for the oracle, which reads only the experts the router selects."""
    return synth.layer_tensors(shape, layer, experts)

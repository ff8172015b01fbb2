"""The allocation-free layer forward (moe_forward_noalloc).

It is for callers whose runtime forbids cudaMalloc -- an engine that hands out
memory from its own pool, code running under CUDA graph capture, a plug-in that
may not touch the allocator -- and therefore cannot create a moe_handle.  The
GPU tests check, on two calls in a row, that it gives the same layer output as
the handle-based moe_forward on identical inputs, within the tolerance the
parity tests use, and that it matches the fp64 oracle directly, on shapes
only it accepts too (H or I an odd multiple of 32).  This file is named to be
collected last.
"""
import numpy as np
import pytest

import bit_moe_decode_02_gb300 as moe
from bit_moe_decode_02_gb300 import build_ext, synth


def _cfg(shape: synth.Shape):
    fmt = moe.MOE_FMT_MXFP4 if shape.fmt == synth.FMT_MXFP4 else moe.MOE_FMT_INT4
    return moe.moe_config(shape.hidden, shape.intermediate, shape.experts, 1, 4, shape.top_k, fmt,
                          shape.group, 1 if shape.has_bias else 0)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    """Argument checks run before any CUDA call, so this needs no GPU."""
    build_ext.build()
    L = moe.lib()
    shape = synth.TINY
    for kw, M, k in [(dict(hidden=4096), 1, 2), (dict(intermediate=3104), 1, 2), ({}, 5, 2),
                     ({}, 1, 17), ({}, 0, 2)]:
        cfg = _cfg(shape)
        for f, v in kw.items():
            setattr(cfg, f, v)
        dummy = 1 << 20   # never dereferenced: the call must fail on the sizes first
        rc = L.moe_forward_noalloc(cfg, dummy, dummy, dummy, dummy, dummy, dummy, dummy, dummy, M, k,
                                   dummy + (1 << 16), None)
        assert rc == moe.MOE_ERR_INVALID_ARG, (kw, M, k)
        assert "moe_forward_noalloc" in moe.moe_last_error()
    # misaligned scale arrays, logits or biases are rejected before any CUDA call
    a = 1 << 20
    cfg = _cfg(shape)
    for args in [(a, a + 8, a, a, a, a, a, a),        # gu_scales
                 (a, a, a, a, a + 4, a, a, a),        # dn_scales
                 (a, a, a + 1, a, a, a, a, a),        # gu_bias
                 (a, a, a, a, a, a + 1, a, a),        # dn_bias
                 (a, a, a, a, a, a, a, a + 2)]:       # router logits
        rc = L.moe_forward_noalloc(cfg, *args, 1, 2, a + (1 << 16), None)
        assert rc == moe.MOE_ERR_INVALID_ARG, args
        assert "aligned" in moe.moe_last_error()


NOALLOC_SHAPES = [
    synth.TINY,
    synth.Shape("ragged H=96 I=160 E=5 top-3 (odd multiples of 32)", 96, 160, 5, 3, bias_sigma=0.5, seed=71),
    synth.Shape("int4 biased group 32 H=192 I=96 E=6 top-2", 192, 96, 6, 2, fmt=synth.FMT_INT4, group=32,
                has_bias=True, bias_sigma=0.1, seed=72),
    synth.Shape("int4 group 64 H=128 I=64 E=6 top-2", 128, 64, 6, 2, fmt=synth.FMT_INT4, group=64,
                has_bias=False, seed=73),
    synth.Shape("top-16 of 32 H=I=128", 128, 128, 32, 16, bias_sigma=0.3, seed=74),
]


def _dev(torch, a):
    if a is None:
        return None
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16 if a.dtype == np.uint16 else a.dtype)).cuda()


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 2, 4])
@pytest.mark.parametrize("shape", NOALLOC_SHAPES, ids=lambda s: s.name)
def test_noalloc_matches_oracle(shape, M):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_testlib import assert_parity, bf16_bits_to_f64, oracle_layer

    build_ext.build()
    t = synth.layer_tensors(shape)
    w = [_dev(torch, a) for a in (t.gu_codes, t.gu_scales, t.gu_bias, t.dn_codes, t.dn_scales, t.dn_bias)]
    cfg = _cfg(shape)
    for step in range(2):
        x, r, logits = synth.step_inputs(shape, 60 + step, M=M, layers=1)
        lg = np.ascontiguousarray(logits[0])
        if step == 1 and M >= 2:   # ties and NaN logits
            lg[0, :] = 0.0
            lg[1, ::2] = np.nan
        out = _dev(torch, r)
        moe.moe_forward_noalloc(cfg, *w, _dev(torch, x), torch.from_numpy(lg).cuda(), M, shape.top_k, out)
        torch.cuda.synchronize()
        got = bf16_bits_to_f64(out.cpu().numpy().view(np.uint16))
        ref, _, _ = oracle_layer(shape, t, x, lg, r)
        assert_parity(got, ref, what=f"noalloc vs oracle, {shape.name}, M={M}, step {step}")


@pytest.mark.gpu
@pytest.mark.parametrize("shape,M", [
    (synth.GPTOSS_LAYER, 1),
    (synth.GPTOSS_LAYER, 3),
    (synth.Shape("int4 H=2048 I=768 E=128 top-8", 2048, 768, 128, 8, fmt=synth.FMT_INT4, group=64,
                 has_bias=False, seed=3), 4),
], ids=lambda v: getattr(v, "name", str(v)))
def test_noalloc_matches_moe_forward_on_two_calls(shape, M):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from moe_testlib import assert_parity, bf16_bits_to_f64, create_handle, load_layer

    build_ext.build()
    t = synth.layer_tensors(shape)
    dev = lambda a: None if a is None else torch.from_numpy(
        np.ascontiguousarray(a).view(np.int16 if a.dtype == np.uint16 else a.dtype)).cuda()
    w = [dev(a) for a in (t.gu_codes, t.gu_scales, t.gu_bias, t.dn_codes, t.dn_scales, t.dn_bias)]
    cfg = _cfg(shape)
    h = create_handle(shape)
    try:
        load_layer(h, 0, t)
        for step in range(2):   # two calls in a row share the scratch array
            x, r, logits = synth.step_inputs(shape, 40 + step, M=M, layers=1)
            xd = dev(x)
            ld = torch.from_numpy(np.ascontiguousarray(logits[0])).cuda()
            out_ref = dev(r)
            moe.moe_forward(h, 0, xd, ld, M, shape.top_k, out_ref)
            out_na = dev(r)
            moe.moe_forward_noalloc(cfg, *w, xd, ld, M, shape.top_k, out_na)
            torch.cuda.synchronize()
            got = bf16_bits_to_f64(out_na.cpu().numpy().view(np.uint16))
            ref = bf16_bits_to_f64(out_ref.cpu().numpy().view(np.uint16))
            assert_parity(got, ref, ulps=1.0, what=f"noalloc vs moe_forward, {shape.name}, step {step}")
    finally:
        moe.moe_destroy(h)

"""GPU parity of the batched path's bf16 numerics (moe_set_batched_numerics:
tcgen05.mma kind::f16 on weights dequantised to bf16, x as given, h as bf16
hi + lo).  Nothing on the activation side is quantised to FP4, so the layer is
compared with the plain fp64 oracle layer -- the same oracle as the decode
kernels -- at both bars (the fp32 result at 2e-3 of the max-norm; the bf16
output with half a bf16 ulp more).  Its error is also compared with the MXFP4
numerics' error on the same inputs, and the numeric edges of the weight
exponents run through it.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from bit_moe_decode_02_gb300 import synth
from moe_testlib import assert_parity, assert_parity_f32, forward_both, load_layer, sparse_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_moe_decode_02_gb300 import build_ext
    build_ext.build()
    import bit_moe_decode_02_gb300 as m
    return m


def _create(moe, shape, M, k=None, bf16=True):
    h = moe.moe_create(shape.hidden, shape.intermediate, shape.experts, 1, M, k or shape.top_k,
                       moe.MOE_FMT_MXFP4, 32, 1 if shape.has_bias else 0)
    if bf16:
        moe.moe_set_batched_numerics(h, moe.MOE_BATCHED_BF16)
    return h


SMALL = [
    # name, H, I, E, k, M, bias, hot experts
    ("square H=I=256 E=8 top-2 M=64", 256, 256, 8, 2, 64, True, ()),
    ("ragged H=320 I=192 E=4 top-2 M=300 (token tiles > 1 per expert)", 320, 192, 4, 2, 300, True, ()),
    ("smallest batch M=5 H=I=128 E=8 top-4", 128, 128, 8, 4, 5, True, ()),
    ("no bias H=384 I=640 E=16 top-4 M=96", 384, 640, 16, 4, 96, False, ()),
    ("skewed E=16 top-2 M=200, +2 on experts 0..3", 256, 320, 16, 2, 200, True, (0, 1, 2, 3)),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_bf16_batched_layer_small(moe, case):
    name, H, I, E, k, M, bias, hot = case
    shape = synth.Shape(name, H, I, E, k, has_bias=bias, e8m0_lo=117, e8m0_hi=124, seed=31,
                        tokens=M, hot_experts=hot, hot_bias=2.0 if hot else 0.0)
    t = synth.layer_tensors(shape)
    x, r, logits = synth.step_inputs(shape, 0, M=M, layers=1)
    h = _create(moe, shape, M)
    try:
        load_layer(h, 0, t)
        got, got32 = forward_both(moe, h, 0, x, r, logits[0], k)
        ref, _, _ = oracle.layer(oracle.FMT_MXFP4, H, I, E, k, t, x, logits[0], r, nthreads=oracle.max_threads())
        assert_parity(got, ref, what=f"bf16 batched {name}")
        assert_parity_f32(got32, ref, what=f"bf16 batched {name}")
        again, _ = forward_both(moe, h, 0, x, r, logits[0], k)
        assert np.array_equal(got, again)   # deterministic
        assert moe.moe_last_launches(h) == 6
    finally:
        moe.moe_destroy(h)


def test_bf16_more_accurate_than_mxfp4_activations(moe):
    """On the same inputs the bf16 numerics sit much closer to the exact layer
    than the MXFP4-activation numerics (measured on the fp32 results)."""
    shape = synth.Shape("accuracy H=I=512 E=8 top-2 M=128", 512, 512, 8, 2, e8m0_lo=117, e8m0_hi=124, seed=32,
                        tokens=128)
    t = synth.layer_tensors(shape)
    x, r, logits = synth.step_inputs(shape, 1, M=128, layers=1)
    ref, _, _ = oracle.layer(oracle.FMT_MXFP4, 512, 512, 8, 2, t, x, logits[0], r, nthreads=oracle.max_threads())
    errs = {}
    for bf16 in (False, True):
        h = _create(moe, shape, 128, bf16=bf16)
        try:
            load_layer(h, 0, t)
            _, got32 = forward_both(moe, h, 0, x, r, logits[0], 2)
            errs[bf16] = np.abs(got32 - ref).max() / np.abs(ref).max()
        finally:
            moe.moe_destroy(h)
    assert errs[True] < 1e-4, errs
    assert errs[True] * 20 < errs[False], errs


# (down E8M0 byte D, gate_up E8M0 byte G, x scale exponent X) per expert, as the
# decode kernels' edge test: products from the fp32 subnormal range to 2^34
EXP_TABLE = [(0, 240, -123), (1, 220, -103), (3, 200, -84), (8, 180, -67), (20, 160, -53),
             (40, 254, -92), (70, 250, -103), (100, 127, 5), (127, 110, 9), (150, 90, 17),
             (180, 70, 22), (200, 50, 32), (220, 30, 42), (240, 10, 62), (250, 2, 70), (254, 0, 72)]


def test_bf16_batched_weight_exponents_0_to_252(moe):
    """E8M0 bytes 0..252: every dequantised weight is a finite bf16 value (bytes
    253 with code 6 and 254 exceed the bf16 range, which is fp32's: this
    numerics does not take them; the MXFP4 decode and batched paths do)."""
    H = I = 256
    E = len(EXP_TABLE)
    shape = synth.Shape("bf16 E8M0 edges H=I=256 E=16 top-1", H, I, E, 1, has_bias=False, seed=61)
    t = synth.layer_tensors(shape)
    for e, (D, G, _) in enumerate(EXP_TABLE):
        t.gu_scales[e] = G
        t.dn_scales[e] = D
    rng = np.random.default_rng(7)
    experts = [e for e, (D, G, _) in enumerate(EXP_TABLE) if max(D, G) <= 252]
    x = synth.bf16_bits_from_f32(np.stack([np.ldexp(rng.standard_normal(H), EXP_TABLE[e][2])
                                           for e in experts]).astype(np.float32))
    M = len(experts)
    r = np.zeros((M, H), np.uint16)
    lg = np.zeros((M, E), np.float32)
    for m, e in enumerate(experts):
        lg[m, e] = 8.0
    h = _create(moe, shape, M, k=1)
    try:
        load_layer(h, 0, t)
        got, got32 = forward_both(moe, h, 0, x, r, lg, 1)
        ref, idx, _ = oracle.layer(oracle.FMT_MXFP4, H, I, E, 1, t, x, lg, r, nthreads=oracle.max_threads())
        assert list(idx[:, 0]) == experts
        for m, e in enumerate(experts):
            assert_parity(got[m], ref[m], what=f"bf16 edges token {m} (D, G, X) = {EXP_TABLE[e]}")
            assert_parity_f32(got32[m], ref[m], what=f"bf16 edges token {m}")
    finally:
        moe.moe_destroy(h)


@pytest.mark.parametrize("shape", [synth.BATCHED, synth.BATCHED_SKEWED], ids=["uniform", "skewed"])
def test_bf16_batched_full_size_sampled(moe, shape):
    """H=I=2880, 128 experts, top-4, M=512: every output of sampled tokens
    against the plain oracle (only the sampled tokens' experts generated)."""
    t = synth.layer_tensors(shape)
    x, r, logits = synth.step_inputs(shape, 0)
    lg = logits[0]
    M, k = x.shape[0], shape.top_k
    h = _create(moe, shape, M)
    try:
        load_layer(h, 0, t)
        got, got32 = forward_both(moe, h, 0, x, r, lg, k)
        top = np.argsort(-lg, axis=1, kind="stable")[:, :k]
        counts = np.bincount(top.ravel(), minlength=shape.experts)
        busiest = int(np.argmax(counts))
        rows = np.flatnonzero((top == busiest).any(axis=1))
        sample = sorted({0, M - 1, 137, int(rows[0]), int(rows[-1])})
        ts = sparse_layer(shape, 0, np.unique(top[sample]).tolist())
        ref, _, _ = oracle.layer(oracle.FMT_MXFP4, shape.hidden, shape.intermediate, shape.experts, k, ts,
                                 x[sample], lg[sample], r[sample], nthreads=oracle.max_threads())
        assert_parity(got[sample], ref, what=f"bf16 batched full size {shape.name}")
        assert_parity_f32(got32[sample], ref, what=f"bf16 batched full size {shape.name}")
    finally:
        moe.moe_destroy(h)


def test_set_batched_numerics_errors(moe):
    shape = synth.TINY
    h = moe.moe_create(shape.hidden, shape.intermediate, shape.experts, 1, 4, shape.top_k, moe.MOE_FMT_MXFP4, 32, 1)
    try:
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_set_batched_numerics(h, moe.MOE_BATCHED_BF16)
        assert ei.value.status == moe.MOE_ERR_UNSUPPORTED
    finally:
        moe.moe_destroy(h)
    h = moe.moe_create(shape.hidden, shape.intermediate, shape.experts, 1, 8, shape.top_k, moe.MOE_FMT_MXFP4, 32, 1)
    try:
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_set_batched_numerics(h, 7)
        assert ei.value.status == moe.MOE_ERR_INVALID_ARG
        moe.moe_set_batched_numerics(h, moe.MOE_BATCHED_BF16)
        moe.moe_set_batched_numerics(h, moe.MOE_BATCHED_MXFP4)
    finally:
        moe.moe_destroy(h)

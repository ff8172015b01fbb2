"""GPU parity of the SwiGLU form setting (moe_set_swiglu): the gpt-oss expert
activation h = min(g, 7) sigmoid(1.702 min(g, 7)) (clamp(u, -7, 7) + 1)
through every kernel that computes SwiGLU -- the MXFP4 decode layer (M = 1, 4),
the int4 layer, the batched path in both numerics -- against the oracle with
the same form; weight scales large enough that the clamps bite.  Back at the
default (1, +inf, 0) a handle gives the same bits as a fresh one.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from bit_moe_decode_02_gb300 import synth
from moe_testlib import assert_parity, assert_parity_f32, create_handle, forward_both, load_layer, oracle_layer

pytestmark = pytest.mark.gpu

GPTOSS = (1.702, 7.0, 1.0)


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_moe_decode_02_gb300 import build_ext
    build_ext.build()
    import bit_moe_decode_02_gb300 as m
    return m


def _clamped_share(shape, t, x, lg):
    """Share of the chosen experts' gate sums above the limit (the test's data
    must exercise the clamp)."""
    w = oracle.dequant(oracle.FMT_MXFP4 if shape.fmt == synth.FMT_MXFP4 else oracle.FMT_INT4, t.gu_codes[0],
                       t.gu_scales[0], 2 * shape.intermediate, shape.hidden, group=shape.group)
    g = oracle.bf16_array(x) @ w[:shape.intermediate].T
    return np.mean(np.abs(g) > GPTOSS[1])


SHAPES = [
    synth.Shape("swiglu MXFP4 H=I=256 E=8 top-2", 256, 256, 8, 2, e8m0_lo=124, e8m0_hi=127, bias_sigma=0.5, seed=91),
    synth.Shape("swiglu int4 H=256 I=128 E=8 top-2", 256, 128, 8, 2, fmt=synth.FMT_INT4, group=64, has_bias=False,
                int4_scale_sigma=0.2, seed=92),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("M", [1, 4])
def test_decode_gptoss_swiglu(moe, shape, M):
    t = synth.layer_tensors(shape, 0)
    x, r, lg = synth.step_inputs(shape, 50 + M, M=M, layers=1)
    assert _clamped_share(shape, t, x, lg[0]) > 0.05
    h = create_handle(shape)
    fresh = create_handle(shape)
    try:
        load_layer(h, 0, t)
        load_layer(fresh, 0, t)
        plain, _ = forward_both(moe, fresh, 0, x, r, lg[0], shape.top_k)
        moe.moe_set_swiglu(h, *GPTOSS)
        got, got32 = forward_both(moe, h, 0, x, r, lg[0], shape.top_k)
        with oracle.swiglu(*GPTOSS):
            ref, _, _ = oracle_layer(shape, t, x, lg[0], r)
        assert_parity(got, ref, what=f"{shape.name} M={M} gpt-oss SwiGLU")
        assert_parity_f32(got32, ref, what=f"{shape.name} M={M} gpt-oss SwiGLU")
        assert not np.array_equal(got, plain)
        moe.moe_set_swiglu(h, 1.0, float("inf"), 0.0)
        back, _ = forward_both(moe, h, 0, x, r, lg[0], shape.top_k)
        assert np.array_equal(back, plain)
    finally:
        moe.moe_destroy(h)
        moe.moe_destroy(fresh)


@pytest.mark.parametrize("bf16", [False, True], ids=["mxfp4 activations", "bf16 numerics"])
def test_batched_gptoss_swiglu(moe, bf16):
    shape = SHAPES[0]
    M = 48
    t = synth.layer_tensors(shape, 0)
    x, r, lg = synth.step_inputs(shape, 60, M=M, layers=1)
    h = create_handle(shape, max_tokens=M)
    try:
        if bf16:
            moe.moe_set_batched_numerics(h, moe.MOE_BATCHED_BF16)
        load_layer(h, 0, t)
        moe.moe_set_swiglu(h, *GPTOSS)
        got, got32 = forward_both(moe, h, 0, x, r, lg[0], shape.top_k)
        H, I, E, k = shape.hidden, shape.intermediate, shape.experts, shape.top_k
        with oracle.swiglu(*GPTOSS):
            if bf16:
                ref, _, _ = oracle_layer(shape, t, x, lg[0], r)
            else:
                # the MXFP4-activation numerics: h (the SwiGLU output, quantised) code by
                # code against the oracle's, then the oracle fed the GPU's own h codes
                codes = torch.zeros(M * k * I // 2, dtype=torch.uint8, device="cuda")
                scales = torch.zeros(M * k * I // 32, dtype=torch.uint8, device="cuda")
                moe.moe_debug_batched_h(h, codes, scales)
                torch.cuda.synchronize()
                gh = codes.cpu().numpy().reshape(M * k, I // 2)
                gs = scales.cpu().numpy().reshape(M * k, I // 32)
                _, oh, os_ = oracle.layer_batched(H, I, E, k, t, x, lg[0], r, want_h=True,
                                                  nthreads=oracle.max_threads())
                oh = oh.reshape(M * k, I // 2)
                nib = lambda c: np.stack([c & 15, c >> 4], axis=-1)
                assert np.count_nonzero(nib(gh) != nib(oh)) / (M * k * I) < 1e-3
                assert np.count_nonzero(gs != os_.reshape(M * k, -1)) / gs.size < 1e-3
                ref = oracle.layer_batched(H, I, E, k, t, x, lg[0], r, h_codes_in=gh, h_scales_in=gs,
                                           nthreads=oracle.max_threads())
        assert_parity(got, ref, what=f"batched gpt-oss SwiGLU bf16={bf16}")
        assert_parity_f32(got32, ref, what=f"batched gpt-oss SwiGLU bf16={bf16}")
    finally:
        moe.moe_destroy(h)


def test_set_swiglu_argument_errors(moe):
    shape = SHAPES[0]
    h = create_handle(shape)
    try:
        for args in [(float("nan"), 7.0, 1.0), (1.0, 0.0, 1.0), (1.0, -1.0, 0.0), (1.0, float("nan"), 0.0),
                     (1.0, 7.0, float("inf"))]:
            with pytest.raises(moe.MoeError) as ei:
                moe.moe_set_swiglu(h, *args)
            assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    finally:
        moe.moe_destroy(h)

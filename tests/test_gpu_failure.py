"""Failure detection on the GPU without a fault: a device-side wait that runs
out reports MOE_ERR_DEVICE_TIMEOUT, and the handle works again afterwards.

moe_debug_set_wait lowers the polling limit of the decode layer's cross-CTA
waits and makes one CTA skip its arrival at the layer's grid barrier, so the
other CTAs' waits give up (nothing traps, nothing reads outside the handle's
buffers, the launch ends).  moe_get_status must then report the timeout and
reset the counters, and the next normal call must match the oracle.
"""
import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from bit_moe_decode_02_gb300 import synth
from moe_testlib import assert_parity, bf16_bits_to_f64, create_handle, dev_to_bits, load_layer, \
    oracle_layer, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_moe_decode_02_gb300 import build_ext
    build_ext.build()
    import bit_moe_decode_02_gb300 as m
    return m


def _forward(moe, h, x, r, logits, k):
    out = to_dev_bf16(r)
    moe.moe_forward(h, 0, to_dev_bf16(x), torch.from_numpy(np.ascontiguousarray(logits)).cuda(),
                    x.shape[0], k, out)
    return out


@pytest.mark.parametrize("skip_cta", [0, 77])
def test_grid_barrier_timeout_is_reported_and_recovered(moe, skip_cta):
    shape = synth.TINY
    t = synth.layer_tensors(shape)
    h = create_handle(shape)
    try:
        load_layer(h, 0, t)
        x, r, logits = synth.step_inputs(shape, 3, M=2, layers=1)
        assert moe.moe_get_status(h) == moe.MOE_OK
        moe.moe_debug_set_wait(h, 20000, skip_cta)
        t0 = time.perf_counter()
        _forward(moe, h, x, r, logits[0], shape.top_k)
        status = moe.moe_get_status(h)          # synchronises; resets the counters
        elapsed = time.perf_counter() - t0
        assert status == moe.MOE_ERR_DEVICE_TIMEOUT
        assert elapsed < 10.0, elapsed
        assert moe.moe_get_status(h) == moe.MOE_OK   # read and cleared
        moe.moe_debug_set_wait(h, 0, -1)
        for step in range(2):                   # the same handle, normal calls again
            x, r, logits = synth.step_inputs(shape, 10 + step, M=2, layers=1)
            out = _forward(moe, h, x, r, logits[0], shape.top_k)
            assert moe.moe_get_status(h) == moe.MOE_OK
            ref, _, _ = oracle_layer(shape, t, x, logits[0], r)
            assert_parity(bf16_bits_to_f64(dev_to_bits(out)), ref, what=f"after the timeout, step {step}")
    finally:
        moe.moe_destroy(h)


def test_set_wait_rejects_bad_arguments(moe):
    h = create_handle(synth.TINY)
    try:
        for args in [(-1, -1), (10, -2)]:
            with pytest.raises(moe.MoeError) as ei:
                moe.moe_debug_set_wait(h, *args)
            assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    finally:
        moe.moe_destroy(h)


def test_timeout_inside_a_multi_step_launch(moe):
    """The same inside one persistent launch of several steps: every call's
    barrier gives up in bounded time, the launch ends, the status reports it,
    and afterwards the steps match single calls again."""
    shape = synth.Shape("tiny steps L=2", 256, 256, 8, 2, layers=2, bias_sigma=0.02, seed=35)
    layers = [synth.layer_tensors(shape, l) for l in range(2)]
    h = create_handle(shape, layers=2, max_tokens=1)
    try:
        for l, t in enumerate(layers):
            load_layer(h, l, t)
        ins = [synth.step_inputs(shape, 20 + s, M=1, layers=1) for s in range(3)]
        x = np.stack([a for a, _, _ in ins])
        r = np.stack([b for _, b, _ in ins])
        lg = np.ascontiguousarray(np.stack([c[0] for _, _, c in ins]))
        moe.moe_debug_set_wait(h, 20000, 3)
        t0 = time.perf_counter()
        moe.moe_forward_steps(h, 3, 0, to_dev_bf16(x), torch.from_numpy(lg).cuda(), 1, 2, to_dev_bf16(r))
        assert moe.moe_get_status(h) == moe.MOE_ERR_DEVICE_TIMEOUT
        assert time.perf_counter() - t0 < 10.0
        moe.moe_debug_set_wait(h, 0, -1)
        od = to_dev_bf16(r)
        moe.moe_forward_steps(h, 3, 0, to_dev_bf16(x), torch.from_numpy(lg).cuda(), 1, 2, od)
        assert moe.moe_get_status(h) == moe.MOE_OK
        got = dev_to_bits(od)
        for s in range(3):
            ref, _, _ = oracle_layer(shape, layers[s % 2], x[s], lg[s], r[s])
            assert_parity(bf16_bits_to_f64(got[s]), ref, what=f"after the timeout, step {s}")
    finally:
        moe.moe_destroy(h)

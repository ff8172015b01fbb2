"""GPU parity of the in-library router GEMV (logits = b + x W^T in fp32) and of
the layers, stacks and steps that route on it inside the launch.

The logits are checked against the oracle's fp64 GEMV within the fp32
summation bound.  The top-k decision then rests on fp32 values on both
sides: a layer that routed on its own logits must give the same bits as the
same layer given those logits, and that layer is compared with the oracle fed
the GPU's logits (the decision taken in the kernel's precision).  All kernels
sum in one order, so the decode, int4 and batched paths give the same logits
for the same input, bit for bit.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from bit_moe_decode_02_gb300 import synth
from moe_testlib import (assert_parity, bf16_bits_to_f64, create_handle, dev_to_bits, load_layer, oracle_layer,
                         sparse_layer, to_dev_bf16)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_moe_decode_02_gb300 import build_ext
    build_ext.build()
    import bit_moe_decode_02_gb300 as m
    return m


SHAPES = [
    synth.Shape("router tiny H=256 I=256 E=8 top-2", 256, 256, 8, 2, bias_sigma=0.02, seed=81),
    synth.Shape("router E=200 > SMs H=128 I=64 top-4", 128, 64, 200, 4, bias_sigma=0.02, seed=82),
    synth.Shape("router int4 H=256 I=128 E=40 top-3", 256, 128, 40, 3, fmt=synth.FMT_INT4, group=64,
                has_bias=False, seed=83),
]


def _logits_bound(x, w, b):
    """fp32 summation bound for each logit: a few hundred roundings of
    2^-24 relative to the sum of |x_h W_eh| (plus the bias add)."""
    xv, wv, bv = oracle.bf16_array(x), oracle.bf16_array(w), oracle.bf16_array(b)
    return 2.0 ** -15 * (np.abs(xv) @ np.abs(wv).T + np.abs(bv)) + 1e-30


def _gpu_logits(moe, h, M, E):
    out = torch.empty((M, E), dtype=torch.float32, device="cuda")
    moe.moe_debug_router_logits(h, out, M)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _forward(moe, h, layer, x, r, logits, M, k):
    xd, od = to_dev_bf16(x), to_dev_bf16(r)
    ld = None if logits is None else torch.from_numpy(np.ascontiguousarray(logits, np.float32)).cuda()
    moe.moe_forward(h, layer, xd, ld, M, k, od)
    torch.cuda.synchronize()
    assert moe.moe_get_status(h) == 0
    return dev_to_bits(od)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("M", [1, 3, 4])
def test_layer_routes_on_its_own_logits(moe, shape, M):
    t = synth.layer_tensors(shape, 0)
    w, b = synth.router_tensors(shape, 0)
    h = create_handle(shape)
    try:
        load_layer(h, 0, t)
        moe.moe_load_router(h, 0, w, b)
        x, r, _ = synth.step_inputs(shape, 40 + M, M=M, layers=1)
        got = _forward(moe, h, 0, x, r, None, M, shape.top_k)
        lg = _gpu_logits(moe, h, M, shape.experts)
        ref_lg = oracle.router(x, w, b)
        err = np.abs(lg - ref_lg)
        assert np.all(err <= _logits_bound(x, w, b)), f"max logit err {err.max():.3g}"
        # the same bits as the layer given those logits, and the oracle on them
        given = _forward(moe, h, 0, x, r, lg, M, shape.top_k)
        assert np.array_equal(got, given)
        ref, _, _ = oracle_layer(shape, t, x, lg, r)
        assert_parity(bf16_bits_to_f64(got), ref, what=f"{shape.name} M={M} routed in-kernel")
    finally:
        moe.moe_destroy(h)


def test_full_size_gptoss_layer_with_router(moe):
    shape = synth.Shape("gpt-oss router", 2880, 2880, 32, 4, layers=1, e8m0_lo=117, e8m0_hi=124, seed=84)
    w, b = synth.router_tensors(shape, 0)
    h = create_handle(shape, max_tokens=4)
    try:
        load_layer(h, 0, synth.layer_tensors(shape, 0))
        moe.moe_load_router(h, 0, w, b)
        for M in (1, 4):
            x, r, _ = synth.step_inputs(shape, 90 + M, M=M, layers=1)
            got = _forward(moe, h, 0, x, r, None, M, 4)
            lg = _gpu_logits(moe, h, M, 32)
            assert np.all(np.abs(lg - oracle.router(x, w, b)) <= _logits_bound(x, w, b))
            assert np.array_equal(got, _forward(moe, h, 0, x, r, lg, M, 4))
            idx, _ = oracle.route(lg, 4)
            t = sparse_layer(shape, 0, idx.ravel())
            ref, _, _ = oracle_layer(shape, t, x, lg, r)
            assert_parity(bf16_bits_to_f64(got), ref, what=f"gpt-oss router M={M}")
    finally:
        moe.moe_destroy(h)


def test_batched_router_matches_decode_bits(moe):
    """M = 16 (batched path: a router kernel, then the grouped GEMMs) routes on
    logits bit-identical to the decode kernel's for the same rows."""
    shape = SHAPES[0]
    t = synth.layer_tensors(shape, 0)
    w, b = synth.router_tensors(shape, 0)
    h = create_handle(shape, max_tokens=16)
    try:
        load_layer(h, 0, t)
        moe.moe_load_router(h, 0, w, b)
        x, r, _ = synth.step_inputs(shape, 77, M=16, layers=1)
        got = _forward(moe, h, 0, x, r, None, 16, shape.top_k)
        lg16 = _gpu_logits(moe, h, 16, shape.experts)
        assert np.all(np.abs(lg16 - oracle.router(x, w, b)) <= _logits_bound(x, w, b))
        assert np.array_equal(got, _forward(moe, h, 0, x, r, lg16, 16, shape.top_k))
        _forward(moe, h, 0, x[:4], r[:4], None, 4, shape.top_k)
        assert np.array_equal(_gpu_logits(moe, h, 4, shape.experts), lg16[:4])
    finally:
        moe.moe_destroy(h)


@pytest.mark.parametrize("shape", [SHAPES[0], SHAPES[2]], ids=lambda s: s.name)
def test_steps_with_router_equal_single_calls(moe, shape):
    L, n, M = 3, 5, 2
    layers = [synth.layer_tensors(shape, l) for l in range(L)]
    h = create_handle(shape, layers=L)
    try:
        for l in range(L):
            load_layer(h, l, layers[l])
            moe.moe_load_router(h, l, *synth.router_tensors(shape, l))
        ins = [synth.step_inputs(shape, 300 + s, M=M, layers=1) for s in range(n)]
        x = np.stack([a for a, _, _ in ins])
        r = np.stack([c for _, c, _ in ins])
        xd, od = to_dev_bf16(x), to_dev_bf16(r)
        moe.moe_forward_steps(h, n, 1, xd, None, M, shape.top_k, od)
        torch.cuda.synchronize()
        assert moe.moe_get_status(h) == 0
        got = dev_to_bits(od)
        for s in range(n):
            single = _forward(moe, h, (1 + s) % L, x[s], r[s], None, M, shape.top_k)
            assert np.array_equal(got[s], single), f"step {s}"
    finally:
        moe.moe_destroy(h)


@pytest.mark.parametrize("shape", [SHAPES[0], SHAPES[2]], ids=lambda s: s.name)
def test_stack_with_router(moe, shape):
    """The stack routing every layer on its own input inside one launch: n
    steps equal n single stacks, the layer-by-layer trace ends on the same
    bits, and every transition matches the oracle stack's layer (router GEMV of
    x_l in fp64, rounded to fp32, then top-k) applied to the GPU's r_l."""
    L, n, M = 3, 2, 2
    layers = [synth.layer_tensors(shape, l) for l in range(L)]
    routers = [synth.router_tensors(shape, l) for l in range(L)]
    h = create_handle(shape, layers=L)
    try:
        for l in range(L):
            load_layer(h, l, layers[l])
            moe.moe_load_router(h, l, *routers[l])
        rs = np.stack([synth.step_inputs(shape, 500 + s, M=M)[1] for s in range(n)])
        rd = to_dev_bf16(rs)
        moe.moe_forward_stack_steps(h, n, rd, None, M, shape.top_k)
        torch.cuda.synchronize()
        assert moe.moe_get_status(h) == 0
        got = dev_to_bits(rd)
        for s in range(n):
            one = to_dev_bf16(rs[s])
            moe.moe_forward_stack(h, one, None, M, shape.top_k)
            torch.cuda.synchronize()
            assert np.array_equal(got[s], dev_to_bits(one)), f"step {s}"
            trace = torch.empty((L + 1, M, shape.hidden), dtype=torch.int16, device="cuda")
            moe.moe_debug_stack_trace(h, to_dev_bf16(rs[s]), None, M, shape.top_k, trace)
            torch.cuda.synchronize()
            tr = trace.cpu().numpy().view(np.uint16)
            assert np.array_equal(tr[L], got[s])
            for l in range(L):
                ref = oracle.stack(shape.fmt, shape.hidden, shape.intermediate, shape.experts, shape.top_k,
                                   [layers[l]], None, tr[l], group=shape.group, nthreads=oracle.max_threads(),
                                   routers=[routers[l]])
                assert_parity(bf16_bits_to_f64(tr[l + 1]), bf16_bits_to_f64(ref), ulps=1.0,
                              what=f"{shape.name} step {s} layer {l}")
    finally:
        moe.moe_destroy(h)


def test_missing_router_is_not_loaded(moe):
    shape = SHAPES[0]
    h = create_handle(shape, layers=2)
    try:
        for l in range(2):
            load_layer(h, l, synth.layer_tensors(shape, l))
        moe.moe_load_router(h, 0, *synth.router_tensors(shape, 0))
        x, r, lg = synth.step_inputs(shape, 0, M=1)
        for call in (lambda: _forward(moe, h, 1, x, r, None, 1, shape.top_k),
                     lambda: moe.moe_forward_stack(h, to_dev_bf16(r), None, 1, shape.top_k)):
            with pytest.raises(moe.MoeError) as ei:
                call()
            assert ei.value.status == moe.MOE_ERR_NOT_LOADED
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_load_router(h, 2, *synth.router_tensors(shape, 0))
        assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    finally:
        moe.moe_destroy(h)

"""GPU parity at the numeric edges of the formats, through the kernels that
serve each size: the tensor-core decode layer (M <= 4), the batched path
(M > 4) and the int4 layer.

The TinyTitan tracker (D108) records a GPU that flushed a denormal product to
zero where the CPU kept it; these cases make such a flush visible.  Every
layer here is one-hot (top_k = 1) or top-2 with no biases and a zero residual,
so the output is the expert path alone, and every token is checked against
its own max-norm: a token whose outputs sit near 2^-130 is not hidden behind
another one near 2^60.

* Weight exponents: 16 experts whose gate_up and down E8M0 bytes together
  cover 0 .. 254; each token's x is scaled by a power of two that keeps the
  gate sums finite, and the down bytes 0 .. 20 put the outputs (and the
  products behind them) in the fp32 subnormal range.
* Activation blocks: a token whose blocks peak near 2^120, one whose blocks
  peak near 2^-120 with whole blocks of bf16 subnormals, one with zero blocks,
  a block spanning 2^-40 .. 2^40 and a subnormal block among normal ones, and
  an all-zero token (its output must be exactly zero).
* int4: fp16 group scales that are subnormal (2^-24 .. 2^-15) or large
  (2^13 .. 65504).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from bit_moe_decode_02_gb300 import synth
from moe_testlib import (assert_parity, assert_parity_f32, create_handle, forward_both, load_layer,
                         oracle_layer)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_moe_decode_02_gb300 import build_ext
    build_ext.build()
    import bit_moe_decode_02_gb300 as m
    return m


def _bf16(v: np.ndarray) -> np.ndarray:
    return synth.bf16_bits_from_f32(np.asarray(v, np.float32))


def _check_rows(got, got32, ref, what):
    for m in range(ref.shape[0]):
        assert_parity(got[m], ref[m], what=f"{what} token {m}")
        assert_parity_f32(got32[m], ref[m], what=f"{what} token {m}")


def _one_hot_logits(experts, E):
    lg = np.zeros((len(experts), E), np.float32)
    for m, e in enumerate(experts):
        lg[m, e] = 8.0
    return lg


# ------------------------------------------------------- weight exponents

# (down E8M0 byte D, gate_up E8M0 byte G, x scale exponent X) per expert: with
# |gate| ~ 2^(G + X - 121.5) and |h| ~ 2^(2 (G + X) - 244), the outputs are
# near 2^(D + 2 (G + X) - 364.5): ~2^-130 for D <= 20, ~2^0 .. 2^34 above.
EXP_TABLE = [(0, 240, -123), (1, 220, -103), (3, 200, -84), (8, 180, -67), (20, 160, -53),
             (40, 254, -92), (70, 250, -103), (100, 127, 5), (127, 110, 9), (150, 90, 17),
             (180, 70, 22), (200, 50, 32), (220, 30, 42), (240, 10, 62), (250, 2, 70), (254, 0, 72)]


def _exponent_layer():
    H = I = 256
    E = len(EXP_TABLE)
    shape = synth.Shape("E8M0 edges H=I=256 E=16 top-1", H, I, E, 1, has_bias=False, seed=61)
    t = synth.layer_tensors(shape)
    for e, (D, G, _) in enumerate(EXP_TABLE):
        t.gu_scales[e] = G
        t.dn_scales[e] = D
    return shape, t


def _exponent_inputs(shape, experts, seed):
    rng = np.random.default_rng(seed)
    M, H = len(experts), shape.hidden
    xs = np.stack([np.ldexp(rng.standard_normal(H), EXP_TABLE[e][2]) for e in experts])
    x = _bf16(xs)
    r = np.zeros((M, H), np.uint16)
    return x, r, _one_hot_logits(experts, shape.experts)


@pytest.mark.parametrize("M", [1, 4])
def test_decode_weight_exponents_0_to_254(moe, M):
    shape, t = _exponent_layer()
    h = create_handle(shape, max_top_k=1)
    try:
        load_layer(h, 0, t)
        for c in range(0, len(EXP_TABLE), M):
            experts = list(range(c, c + M))
            x, r, lg = _exponent_inputs(shape, experts, 100 + c)
            got, got32 = forward_both(moe, h, 0, x, r, lg, 1)
            ref, idx, _ = oracle_layer(shape, t, x, lg, r, k=1)
            assert list(idx[:, 0]) == experts
            assert np.all(np.isfinite(ref)) and np.all(np.abs(ref).max(axis=1) > 0)
            _check_rows(got, got32, ref, f"experts {experts} (D, G, X) = {[EXP_TABLE[e] for e in experts]}")
    finally:
        moe.moe_destroy(h)


def _gpu_h(moe, h, Mk, I):
    codes = torch.zeros(Mk * I // 2, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(Mk * I // 32, dtype=torch.uint8, device="cuda")
    moe.moe_debug_batched_h(h, codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy().reshape(Mk, I // 2), scales.cpu().numpy().reshape(Mk, I // 32)


def _batched_check(moe, h, shape, t, x, r, lg, k, what):
    """The batched layer against the oracle fed the GPU's own MXFP4 h (the
    quantiser is bit-exact; fp32 and fp64 h may round to neighbouring codes),
    token by token, at both bars."""
    H, I, E = shape.hidden, shape.intermediate, shape.experts
    got, got32 = forward_both(moe, h, 0, x, r, lg, k)
    gh, gs = _gpu_h(moe, h, x.shape[0] * k, I)
    ref = oracle.layer_batched(H, I, E, k, t, x, lg, r, h_codes_in=gh, h_scales_in=gs,
                               nthreads=oracle.max_threads())
    _check_rows(got, got32, ref, what)


def test_batched_weight_exponents_0_to_254(moe):
    shape, t = _exponent_layer()
    h = moe.moe_create(shape.hidden, shape.intermediate, shape.experts, 1, 16, 1, moe.MOE_FMT_MXFP4, 32, 0)
    try:
        load_layer(h, 0, t)
        experts = list(range(16))
        x, r, lg = _exponent_inputs(shape, experts, 7)
        _batched_check(moe, h, shape, t, x, r, lg, 1, "batched E8M0 edges")
    finally:
        moe.moe_destroy(h)


# ------------------------------------------------------- activation blocks

def _activation_layer():
    """Experts 0-3 scaled for huge x (gate_up byte 4), 4-7 for tiny x (250),
    8-11 for ordinary x (125); every down byte 120."""
    H, I, E = 512, 256, 12
    shape = synth.Shape("activation edges H=512 I=256 E=12 top-2", H, I, E, 2, has_bias=False, seed=62)
    t = synth.layer_tensors(shape)
    for e in range(E):
        t.gu_scales[e] = 4 if e < 4 else (250 if e < 8 else 125)
        t.dn_scales[e] = 120
    return shape, t


def _activation_inputs(shape):
    rng = np.random.default_rng(5)
    H, nb = shape.hidden, shape.hidden // 32
    blk = lambda X: np.ldexp(rng.standard_normal(32), X)
    huge = np.concatenate([blk(118) if b % 3 else np.zeros(32) for b in range(nb)])
    tiny = np.concatenate([blk(-122) if b % 4 else (np.zeros(32) if b == 4 else blk(-130)) for b in range(nb)])
    mixed = []
    for b in range(nb):
        if b == 0:
            mixed.append(np.zeros(32))
        elif b == 1:     # one block spanning 2^-40 .. 2^40
            v = blk(0)
            v[::2] = np.ldexp(v[::2], 40)
            v[1::2] = np.ldexp(v[1::2], -40)
            mixed.append(v)
        elif b == 2:     # bf16 subnormals among normal blocks
            mixed.append(blk(-131))
        else:
            mixed.append(blk(0))
    mixed = np.concatenate(mixed)
    zero = np.zeros(H)
    x = _bf16(np.stack([huge, tiny, mixed, zero]))
    assert np.any((x[1] & 0x7f80) == 0) and np.any((x[1] & 0x7fff) != 0)   # has bf16 subnormals
    lg = np.full((4, shape.experts), -4.0, np.float32)
    for m, (e0, e1) in enumerate([(0, 1), (4, 5), (8, 9), (10, 11)]):
        lg[m, e0], lg[m, e1] = 3.0, 2.5
    r = np.zeros((4, H), np.uint16)
    return x, r, lg


def test_decode_activation_blocks(moe):
    shape, t = _activation_layer()
    x, r, lg = _activation_inputs(shape)
    h = create_handle(shape)
    try:
        load_layer(h, 0, t)
        got, got32 = forward_both(moe, h, 0, x, r, lg, 2)
        ref, _, _ = oracle_layer(shape, t, x, lg, r)
        assert np.all(ref[3] == 0) and np.all(got32[3] == 0) and np.all(got[3] == 0)
        _check_rows(got[:3], got32[:3], ref[:3], "activation edges M=4")
        for m in range(3):   # one token at a time (the M = 1 kernel configuration)
            g1, g132 = forward_both(moe, h, 0, x[m:m + 1], r[m:m + 1], lg[m:m + 1], 2)
            _check_rows(g1, g132, ref[m:m + 1], f"activation edges M=1 token {m}")
    finally:
        moe.moe_destroy(h)


def test_batched_activation_blocks(moe):
    shape, t = _activation_layer()
    x, r, lg = _activation_inputs(shape)
    x, r, lg = np.concatenate([x, x]), np.concatenate([r, r]), np.concatenate([lg, lg])
    h = moe.moe_create(shape.hidden, shape.intermediate, shape.experts, 1, 8, 2, moe.MOE_FMT_MXFP4, 32, 0)
    try:
        load_layer(h, 0, t)
        got, got32 = forward_both(moe, h, 0, x, r, lg, 2)
        assert np.all(got32[3] == 0) and np.all(got32[7] == 0)
        keep = [0, 1, 2, 4, 5, 6]
        gh, gs = _gpu_h(moe, h, 16, shape.intermediate)
        ref = oracle.layer_batched(shape.hidden, shape.intermediate, shape.experts, 2, t, x, lg, r,
                                   h_codes_in=gh, h_scales_in=gs, nthreads=oracle.max_threads())
        _check_rows(got[keep], got32[keep], ref[keep], "batched activation edges")
    finally:
        moe.moe_destroy(h)


# ------------------------------------------------------- int4 scales

def test_int4_subnormal_and_large_scales(moe):
    H, I, E = 256, 128, 8
    shape = synth.Shape("int4 scale edges H=256 I=128 E=8 top-1", H, I, E, 1, fmt=synth.FMT_INT4, group=32,
                        has_bias=False, seed=63)
    t = synth.layer_tensors(shape)
    rng = np.random.default_rng(8)
    for e in range(E):
        for a in (t.gu_scales, t.dn_scales):
            n = a[e].size
            if e < 4:   # subnormal fp16: exponent field 0, mantissa 1 .. 1023
                a[e] = rng.integers(1, 1024, n).astype(np.uint16).reshape(a[e].shape)
            else:       # large: exponent fields 28 .. 30 (2^13 .. 65504)
                a[e] = ((rng.integers(28, 31, n) << 10) | rng.integers(0, 1024, n)).astype(np.uint16).reshape(a[e].shape)
    h = create_handle(shape, max_top_k=1)
    try:
        load_layer(h, 0, t)
        for M in (1, 4):
            for c in range(0, E, M):
                experts = list(range(c, c + M))
                x = _bf16(rng.standard_normal((M, H)))
                r = np.zeros((M, H), np.uint16)
                lg = _one_hot_logits(experts, E)
                got, got32 = forward_both(moe, h, 0, x, r, lg, 1)
                ref, _, _ = oracle_layer(shape, t, x, lg, r, k=1)
                assert np.all(np.isfinite(ref))
                _check_rows(got, got32, ref, f"int4 scale edges M={M} experts {experts}")
    finally:
        moe.moe_destroy(h)

"""GPU parity of the batched path (M > 4: grouped GEMMs on tcgen05 kind::mxf4).

The batched layer quantises x and h to MXFP4 (OCP MX v1.0) so that both MMA
operands are FP4; the oracle applies the same quantiser in fp64.  Checks:
  * the GPU quantiser is bit-exact against the oracle's on the same fp32
    inputs (the decision is taken in the same precision on both sides);
  * x quantisation is therefore exact, and h -- computed in fp32 on the GPU and
    in fp64 by the oracle -- may land on the other side of an E2M1 rounding
    boundary: the share of differing h codes must stay below 0.1%;
  * the layer output matches the oracle fed the GPU's own quantised h within
    2e-3 of the output's max-norm plus half a bf16 ulp.
Full-size 512-token layers are checked on sampled tokens (the oracle's cost).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from bit_moe_decode_02_gb300 import synth
from moe_testlib import assert_parity, assert_parity_f32, forward_both, load_layer

pytestmark = pytest.mark.gpu

FLIP_RATE = 1e-3


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_moe_decode_02_gb300 import build_ext
    build_ext.build()
    import bit_moe_decode_02_gb300 as m
    return m


def _quantize_gpu(moe, v32: np.ndarray):
    n = v32.size
    x = torch.from_numpy(np.ascontiguousarray(v32, np.float32)).cuda()
    codes = torch.zeros(n // 2, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(n // 32, dtype=torch.uint8, device="cuda")
    moe.moe_debug_mx_quantize(x, n, codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy()


def _quantizer_cases() -> np.ndarray:
    rng = np.random.default_rng(11)
    blocks = []
    # every E2M1 rounding tie and its neighbours at several shared exponents
    grid = np.arange(0, 25) * 0.25
    for X in (-127, -100, -3, 0, 5, 100, 125):
        for sign in (1.0, -1.0):
            v = np.concatenate([grid, grid[:7] + 0.125]) * sign
            v[0] = 6.0 * sign   # amax = 6 * 2^X fixes the shared exponent at X
            blocks.append(np.ldexp(v, X)[:32])
    blocks.append(np.zeros(32))
    blocks.append(-np.zeros(32))
    blocks.append(np.full(32, 1e-45))                   # smallest fp32 subnormal
    blocks.append(np.linspace(-1e-39, 1e-39, 32))       # subnormal block
    blocks.append(np.linspace(-3.3e38, 3.3e38, 32))     # near fp32 max
    blocks.append(np.array([7.9, -7.9, 6.5, 5.5, 0.2, -0.2] + [0.0] * 26))
    for _ in range(400):                                 # random magnitudes
        e = rng.integers(-140, 120)
        blocks.append(rng.standard_normal(32) * 2.0 ** e * rng.random(32) ** rng.integers(0, 4))
    v = np.concatenate(blocks).astype(np.float32)
    return v


def test_mx_quantizer_bitexact_vs_oracle(moe):
    v = _quantizer_cases()
    gc, gs = _quantize_gpu(moe, v)
    oc, osc = oracle.mx_quantize(v.astype(np.float64))
    bad_s = np.flatnonzero(gs != osc)
    assert bad_s.size == 0, f"scale bytes differ in blocks {bad_s[:8]}: gpu {gs[bad_s[:8]]} oracle {osc[bad_s[:8]]}"
    bad_c = np.flatnonzero(gc != oc)
    assert bad_c.size == 0, (f"code bytes differ at {bad_c[:8]}: gpu {gc[bad_c[:8]]} oracle {oc[bad_c[:8]]}, "
                             f"inputs {v[2 * bad_c[0]:2 * bad_c[0] + 2]}")


def _create(moe, shape, M, k=None):
    return moe.moe_create(shape.hidden, shape.intermediate, shape.experts, 1, M, k or shape.top_k,
                          moe.MOE_FMT_MXFP4, 32, 1 if shape.has_bias else 0)


def _forward(moe, h, x, r, logits, k, want_f32=False):
    got, got32 = forward_both(moe, h, 0, x, r, logits, k)
    return (got, got32) if want_f32 else got


def _gpu_h(moe, h, Mk, I):
    codes = torch.zeros(Mk * I // 2, dtype=torch.uint8, device="cuda")
    scales = torch.zeros(Mk * I // 32, dtype=torch.uint8, device="cuda")
    moe.moe_debug_batched_h(h, codes, scales)
    torch.cuda.synchronize()
    return codes.cpu().numpy().reshape(Mk, I // 2), scales.cpu().numpy().reshape(Mk, I // 32)


def _nibbles(c: np.ndarray) -> np.ndarray:
    return np.stack([c & 15, c >> 4], axis=-1).reshape(c.shape[0], -1)


def _check_layer(moe, shape, t, x, r, logits, k, h, tokens=None):
    """Run one batched forward on all tokens; compare `tokens` (all if None)."""
    H, I, E = shape.hidden, shape.intermediate, shape.experts
    M = x.shape[0]
    got, got32 = _forward(moe, h, x, r, logits, k, want_f32=True)
    gh, gs = _gpu_h(moe, h, M * k, I)
    sel = np.arange(M) if tokens is None else np.asarray(tokens)
    slots = (sel[:, None] * k + np.arange(k)[None, :]).ravel()
    nt = oracle.max_threads()
    _, oh, os_ = oracle.layer_batched(H, I, E, k, t, x[sel], logits[sel], r[sel], want_h=True, nthreads=nt)
    # (i) h codes: same decisions except across a rounding boundary
    gn = _nibbles(gh[slots])
    on = _nibbles(oh.reshape(len(slots), I // 2))
    flips = np.count_nonzero(gn != on) / gn.size
    assert flips < FLIP_RATE, f"h code flip rate {flips:.2e}"
    scale_diff = np.count_nonzero(gs[slots] != os_.reshape(len(slots), -1)) / gs[slots].size
    assert scale_diff < FLIP_RATE, f"h scale byte difference rate {scale_diff:.2e}"
    # (ii) the layer on the GPU's own h
    ref = oracle.layer_batched(H, I, E, k, t, x[sel], logits[sel], r[sel],
                               h_codes_in=np.ascontiguousarray(gh[slots]),
                               h_scales_in=np.ascontiguousarray(gs[slots]), nthreads=nt)
    rel = assert_parity(got[sel], ref, what=f"batched {shape.name} M={M}")
    assert_parity_f32(got32[sel], ref, what=f"batched {shape.name} M={M}")
    return got, rel, flips


SMALL = [
    # name, H, I, E, k, M, bias, hot experts
    ("square H=I=256 E=8 top-2 M=64", 256, 256, 8, 2, 64, True, ()),
    ("ragged H=320 I=192 E=4 top-2 M=300 (token tiles > 1 per expert)", 320, 192, 4, 2, 300, True, ()),
    ("smallest batch M=5 H=I=128 E=8 top-4", 128, 128, 8, 4, 5, True, ()),
    ("no bias H=384 I=640 E=16 top-4 M=96", 384, 640, 16, 4, 96, False, ()),
    ("skewed E=16 top-2 M=200, +2 on experts 0..3", 256, 320, 16, 2, 200, True, (0, 1, 2, 3)),
    ("single expert top-1 E=1 M=130", 192, 256, 1, 1, 130, True, ()),
]


@pytest.mark.parametrize("case", SMALL, ids=[c[0] for c in SMALL])
def test_batched_layer_small(moe, case):
    name, H, I, E, k, M, bias, hot = case
    shape = synth.Shape(name, H, I, E, k, has_bias=bias, e8m0_lo=117, e8m0_hi=124, seed=21,
                        tokens=M, hot_experts=hot, hot_bias=2.0 if hot else 0.0)
    t = synth.layer_tensors(shape)
    x, r, logits = synth.step_inputs(shape, 0, M=M, layers=1)
    h = _create(moe, shape, M)
    try:
        load_layer(h, 0, t)
        got, rel, flips = _check_layer(moe, shape, t, x, r, logits[0], k, h)
        # deterministic: a second call gives the same bits
        again = _forward(moe, h, x, r, logits[0], k)
        assert np.array_equal(np.nan_to_num(got), np.nan_to_num(again))
        # algorithmic bytes: every expert with at least one token, once
        distinct = len(set(np.argsort(-logits[0], axis=1, kind="stable")[:, :k].ravel().tolist()))
        assert moe.moe_last_bytes(h) == distinct * moe.moe_expert_bytes(h)
    finally:
        moe.moe_destroy(h)


def test_decode_and_batched_paths_share_one_handle(moe):
    """A handle created with max_tokens 8 runs M <= 4 on the decode kernel
    (exact activations) and M > 4 on the tensor-core path, on the same loaded
    weights; each is checked against its own oracle."""
    shape = synth.Shape("both paths H=I=256 E=8 top-2", 256, 256, 8, 2, e8m0_lo=117, e8m0_hi=124, seed=5)
    t = synth.layer_tensors(shape)
    x, r, logits = synth.step_inputs(shape, 3, M=8, layers=1)
    h = _create(moe, shape, 8)
    try:
        load_layer(h, 0, t)
        got4 = _forward(moe, h, x[:4], r[:4], logits[0][:4], 2)
        ref4, _, _ = oracle.layer(oracle.FMT_MXFP4, 256, 256, 8, 2, t, x[:4], logits[0][:4], r[:4])
        assert_parity(got4, ref4, what="decode path on a batched handle")
        _check_layer(moe, shape, t, x, r, logits[0], 2, h)
    finally:
        moe.moe_destroy(h)


@pytest.mark.parametrize("shape", [synth.BATCHED, synth.BATCHED_SKEWED], ids=["uniform", "skewed"])
def test_batched_full_size_sampled(moe, shape):
    """H=I=2880, 128 experts, top-4, M=512: every output of sampled tokens,
    chosen to include tokens routed to the busiest experts."""
    t = synth.layer_tensors(shape)
    x, r, logits = synth.step_inputs(shape, 0)
    lg = logits[0]
    M, k = x.shape[0], shape.top_k
    h = _create(moe, shape, M)
    try:
        load_layer(h, 0, t)
        top = np.argsort(-lg, axis=1, kind="stable")[:, :k]
        counts = np.bincount(top.ravel(), minlength=shape.experts)
        busiest = int(np.argmax(counts))
        sample = sorted({0, M - 1, 137, int(np.flatnonzero((top == busiest).any(axis=1))[0]),
                         int(np.flatnonzero((top == busiest).any(axis=1))[-1])})
        _check_layer(moe, shape, t, x, r, lg, k, h, tokens=sample)
        nb = moe.moe_last_bytes(h)
        assert nb == np.count_nonzero(counts) * moe.moe_expert_bytes(h)
    finally:
        moe.moe_destroy(h)

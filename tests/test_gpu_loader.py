"""Checkpoint-layout loader flags (moe_load_experts_ex): a layer given with
gate and up rows alternating, and/or with both projections in the transposed
[K][N] orientation, must hold the same resident weights as the same layer
given in the caller layout -- every dequantised element bit for bit (read
back from the bytes the kernels stream) -- and give the same outputs.

The checkpoint layouts are built here from the caller-layout tensors by
re-indexing bytes and nibbles only (no arithmetic of the method).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from bit_moe_decode_02_gb300 import synth
from moe_testlib import create_handle, dev_to_bits, load_layer, to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_moe_decode_02_gb300 import build_ext
    build_ext.build()
    import bit_moe_decode_02_gb300 as m
    return m


def _interleave_rows(a, I):
    """[E][2I][...] gate rows then up rows -> row 2j gate j, row 2j+1 up j."""
    out = np.empty_like(a)
    out[:, 0::2] = a[:, :I]
    out[:, 1::2] = a[:, I:]
    return out


def _transpose_codes(c):
    """[E][N][K/2] nibbles (even K index low) -> [E][K][N/2] (even N index low)."""
    E, N, K2 = c.shape
    el = np.empty((E, N, 2 * K2), np.uint8)
    el[:, :, 0::2] = c & 0xF
    el[:, :, 1::2] = c >> 4
    t = np.ascontiguousarray(el.transpose(0, 2, 1))   # [E][K][N]
    return (t[:, :, 0::2] | (t[:, :, 1::2] << 4)).astype(np.uint8)


def _checkpoint(t, I, flags, moe):
    gu_c, gu_s, gu_b = t.gu_codes, t.gu_scales, t.gu_bias
    dn_c, dn_s = t.dn_codes, t.dn_scales
    if flags & moe.MOE_LOAD_GATE_UP_INTERLEAVED:
        gu_c, gu_s = _interleave_rows(gu_c, I), _interleave_rows(gu_s, I)
        gu_b = None if gu_b is None else _interleave_rows(gu_b, I)
    if flags & moe.MOE_LOAD_TRANSPOSED:
        gu_c, dn_c = _transpose_codes(gu_c), _transpose_codes(dn_c)
        gu_s = np.ascontiguousarray(gu_s.transpose(0, 2, 1))
        dn_s = np.ascontiguousarray(dn_s.transpose(0, 2, 1))
    return [np.ascontiguousarray(a) if a is not None else None for a in (gu_c, gu_s, gu_b, dn_c, dn_s, t.dn_bias)]


def _dequant(moe, h, e, proj, N, K):
    out = torch.empty((N, K), dtype=torch.float32, device="cuda")
    moe.moe_debug_dequant(h, 0, e, proj, out)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint32)


SHAPES = [
    synth.Shape("loader MXFP4 H=256 I=192 E=4 top-2", 256, 192, 4, 2, bias_sigma=0.02, seed=91),
    synth.Shape("loader int4 H=256 I=128 E=4 top-2 g64", 256, 128, 4, 2, fmt=synth.FMT_INT4, group=64,
                has_bias=False, seed=92),
    synth.Shape("loader int4 H=128 I=128 E=3 top-2 g32 bias", 128, 128, 3, 2, fmt=synth.FMT_INT4, group=32,
                bias_sigma=0.02, seed=93),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
@pytest.mark.parametrize("flags", [1, 2, 3], ids=["interleaved", "transposed", "both"])
def test_flagged_load_equals_caller_layout(moe, shape, flags):
    H, I, E = shape.hidden, shape.intermediate, shape.experts
    t = synth.layer_tensors(shape, 0)
    ha, hb = create_handle(shape), create_handle(shape)
    try:
        load_layer(ha, 0, t)
        moe.moe_load_experts_ex(hb, 0, *_checkpoint(t, I, flags, moe), flags)
        for e in range(E):
            for proj, (N, K) in enumerate([(2 * I, H), (H, I)]):
                assert np.array_equal(_dequant(moe, ha, e, proj, N, K), _dequant(moe, hb, e, proj, N, K)), \
                    f"expert {e} proj {proj}"
        for M in (1, 3):
            x, r, lg = synth.step_inputs(shape, 10 + M, M=M, layers=1)
            outs = []
            for h in (ha, hb):
                od = to_dev_bf16(r)
                moe.moe_forward(h, 0, to_dev_bf16(x), torch.from_numpy(np.ascontiguousarray(lg[0])).cuda(), M,
                                shape.top_k, od)
                torch.cuda.synchronize()
                assert moe.moe_get_status(h) == 0
                outs.append(dev_to_bits(od))
            assert np.array_equal(outs[0], outs[1]), f"M={M}"
        with pytest.raises(moe.MoeError) as ei:
            moe.moe_load_experts_ex(hb, 0, *_checkpoint(t, I, 0, moe), 4)
        assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    finally:
        moe.moe_destroy(ha)
        moe.moe_destroy(hb)

"""The streaming-floor measurement call: argument checks, and a read of every
resident layer that completes with a clean status."""
import pytest

torch = pytest.importorskip("torch")

from bit_moe_decode_02_gb300 import synth
from moe_testlib import create_handle, load_layer

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_moe_decode_02_gb300 import build_ext
    build_ext.build()
    import bit_moe_decode_02_gb300 as m
    return m


def test_stream_weights(moe):
    shape = synth.Shape("probe tiny", 256, 256, 8, 2, layers=3, bias_sigma=0.02, seed=95)
    h = create_handle(shape, layers=3)
    try:
        for l in range(3):
            load_layer(h, l, synth.layer_tensors(shape, l))
        for n, nbytes in [(1, 16), (3, 4096), (3, 40960), (2, 100000)]:
            moe.moe_debug_stream_weights(h, 0, n, nbytes)
            torch.cuda.synchronize()
            assert moe.moe_get_status(h) == 0
        for args in [(0, 4, 4096), (-1, 1, 4096), (0, 1, 8), (0, 1, 4100), (1, 3, 4096), (0, 1, 1 << 40)]:
            with pytest.raises(moe.MoeError) as ei:
                moe.moe_debug_stream_weights(h, *args)
            assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    finally:
        moe.moe_destroy(h)

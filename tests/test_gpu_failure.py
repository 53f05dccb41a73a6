"""Failure detection on the GPU without a fault: a wait that can never be
satisfied (an mbarrier phase nothing completes, a word nothing writes) runs
out its bounded limit, the status word reports the timeout, the status clears,
and the same context still computes the layer correctly."""
import pytest

from tests import gpu_parity as gp
from w4a16_compact_expert_gb300 import moe_w4a16 as M, synth

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("which", [0, 1])
def test_bounded_wait_times_out_and_the_context_survives(which):
    import torch
    layer = synth.tiny_layer()
    m = gp.make_handle(layer, 16)
    try:
        assert m.get_status() == (M.OK, 0)
        m.selftest_timeout(which, 2_000_000)       # about a millisecond of SM cycles
        torch.cuda.synchronize()
        st, _ = m.get_status()
        assert st == M.ERR_TIMEOUT
        assert m.get_status() == (M.OK, 0)         # reported once, then cleared
        gp.check_full(layer, synth.draw_x(31, 13, layer.shape.hidden), m=m)
    finally:
        m.close()


def test_selftest_argument_errors():
    layer = synth.tiny_layer()
    m = gp.make_handle(layer, 4)
    try:
        for which, limit in ((2, 10_000), (-1, 10_000), (0, 10), (1, 1 << 40)):
            with pytest.raises(M.MoEError) as ex:
                m.selftest_timeout(which, limit)
            assert ex.value.status == M.ERR_INVALID_ARG
    finally:
        m.close()

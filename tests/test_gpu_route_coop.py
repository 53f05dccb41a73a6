"""The cooperative router (one launch: logits, top-k, the stable permutation
and, on the grouped-GEMM path, the copy of the x rows into sorted-row order)
against the oracle router and layer; for 8 < T <= 64 the same phases run on
one thread-block cluster.

One handle runs several token counts in turn, on both grid sizes (and
barrier counters) of the router; a timeout there would show as a non-OK
status."""
import numpy as np
import pytest

from tests import gpu_parity as gp
from w4a16_compact_expert_gb300 import moe_w4a16 as M, synth

pytestmark = pytest.mark.gpu


def test_route_coop_token_counts_on_one_handle():
    layer = synth.olmoe_prefill_layer(1)
    m = gp.make_handle(layer, 2048)
    try:
        for i, (T, flags) in enumerate([(65, 0), (2048, 0), (300, M.PRENORM | M.RESIDUAL), (1001, 0), (65, 0)]):
            x = synth.draw_x(5200 + i, T, layer.shape.hidden)
            rows = np.unique(np.r_[0, T - 1, np.random.default_rng(i).choice(T, size=6, replace=False)])
            gp.check_sampled(layer, x, rows, flags=flags | M.FORCE_GEMM, m=m)
            path, launches = m.last_path()
            assert (path, launches) == (M.PATH_GEMM, 4)
    finally:
        m.close()


@pytest.mark.parametrize("T,flags", [(9, 0), (33, M.PRENORM), (64, M.RESIDUAL), (64, M.PRENORM | M.RESIDUAL)])
@pytest.mark.parametrize("force", [M.FORCE_GEMM, M.FORCE_GEMV | M.UNFUSED])
def test_route_cluster_phases_full_parity(T, flags, force):
    """8 < T <= 64: the router's phases on one 8-CTA cluster (cluster barriers
    between them), on the grouped-GEMM path (which also gathers the x rows)
    and on the separate-launch decode path; every token against the oracle,
    and the same forward twice bit-identical."""
    layer = synth.olmoe_decode_layer()
    x = synth.draw_x(5400 + T, T, layer.shape.hidden)
    m = gp.make_handle(layer, 64)
    try:
        gp.check_full(layer, x, flags | force, m=m)
        a, da = gp.gpu_forward(m, layer, x, flags | force)
        b, db = gp.gpu_forward(m, layer, x, flags | force)
        assert np.array_equal(a, b)
        assert all(np.array_equal(da[k], db[k]) for k in da)
        assert m.last_path()[0] == (M.PATH_GEMM if force == M.FORCE_GEMM else M.PATH_DECODE)
    finally:
        m.close()


def test_route_coop_tiny_full_parity():
    """Tiny layer above the single-launch router's range: every token."""
    layer = synth.tiny_layer()
    T = 200
    x = synth.draw_x(5300, T, layer.shape.hidden)
    m = gp.make_handle(layer, T)
    try:
        gp.check_full(layer, x, M.FORCE_GEMM, m=m)
        assert m.last_path() == (M.PATH_GEMM, 4)
        # the same forward twice: bit-identical
        a, da = gp.gpu_forward(m, layer, x, M.FORCE_GEMM)
        b, db = gp.gpu_forward(m, layer, x, M.FORCE_GEMM)
        assert np.array_equal(a, b)
        assert all(np.array_equal(da[k], db[k]) for k in da)
    finally:
        m.close()

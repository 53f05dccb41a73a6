"""The offload-qpacked comparison path on the GPU: each batch of active
experts is expanded into bounded FP16 execution slots, then the grouped GEMM
runs on the FP16 copies.  Its outputs must match the oracle, and be
bit-identical to the compact grouped-GEMM path: both multiply the same FP16
values (q * s rounded once) with the same tiles and summation order."""
import numpy as np
import pytest

from tests import gpu_parity as gp
from w4a16_compact_expert_gb300 import moe_w4a16 as M, synth

pytestmark = pytest.mark.gpu


def _forward(m, layer, x, flags):
    out, _ = gp.gpu_forward(m, layer, x, flags)
    st, miss = m.get_status()
    assert st == M.OK, st
    return out


@pytest.mark.parametrize("T,slots", [(4, 3), (33, 3), (64, 8)])
def test_tiny_offload_matches_oracle_and_compact_gemm(T, slots):
    layer = synth.tiny_layer()
    x = synth.draw_x(3000 + T, T, layer.shape.hidden)
    m = gp.make_handle(layer, 64)
    try:
        m.offload_enable(slots)
        out = _forward(m, layer, x, M.OFFLOAD)
        path, launches = m.last_path()
        assert path == M.PATH_OFFLOAD
        ref = gp.oracle_layer(layer, x)
        gp.assert_output(out, ref.out, ~ref.near_tie)
        compact = _forward(m, layer, x, M.FORCE_GEMM)
        assert np.array_equal(out, compact)
    finally:
        m.close()


def test_offload_flag_errors():
    layer = synth.tiny_layer()
    m = gp.make_handle(layer, 8)
    try:
        x = synth.draw_x(11, 2, layer.shape.hidden)
        with pytest.raises(M.MoEError):   # not enabled
            gp.gpu_forward(m, layer, x, M.OFFLOAD)
        m.offload_enable(2)
        with pytest.raises(M.MoEError):   # exclusive with FORCE_GEMV
            gp.gpu_forward(m, layer, x, M.OFFLOAD | M.FORCE_GEMV)
        with pytest.raises(M.MoEError):
            m.offload_enable(0)
        m.offload_enable(4)               # replaces the slots
        _forward(m, layer, x, M.OFFLOAD)
    finally:
        m.close()


def test_qwen_partial_offload():
    layer = synth.qwen_partial_layer()
    T = 32
    x = synth.draw_x(4100, T, layer.shape.hidden)
    m = gp.make_handle(layer, T)
    try:
        m.offload_enable(8)
        out = _forward(m, layer, x, M.OFFLOAD)
        ref = gp.oracle_layer(layer, x)
        gp.assert_output(out, ref.out, ~ref.near_tie)
        assert np.array_equal(out, _forward(m, layer, x, M.FORCE_GEMM))
    finally:
        m.close()


def test_olmoe_prefill_offload_sampled():
    layer = synth.olmoe_prefill_layer(2)
    T = 2048
    x = synth.draw_x(synth.SEED_OLMOE_PREFILL_SKEW, T, layer.shape.hidden)
    m = gp.make_handle(layer, T)
    try:
        m.offload_enable(16)
        rows = np.random.default_rng(7).choice(T, size=24, replace=False)
        gp.check_sampled(layer, x, rows, flags=M.OFFLOAD, m=m)
        assert m.last_path()[0] == M.PATH_OFFLOAD
        a = _forward(m, layer, x, M.OFFLOAD)
        b = _forward(m, layer, x, M.FORCE_GEMM)
        assert np.array_equal(a, b)
    finally:
        m.close()

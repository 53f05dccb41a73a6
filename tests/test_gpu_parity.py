"""CUDA path vs the CPU oracle on the seeded workloads (element-wise)."""
import numpy as np
import pytest

from tests import gpu_parity as gp
from w4a16_compact_expert_gb300 import moe_w4a16, synth

pytestmark = pytest.mark.gpu

F = moe_w4a16


@pytest.fixture(scope="module")
def tiny():
    return synth.tiny_layer()


@pytest.fixture(scope="module")
def olmoe():
    return synth.olmoe_decode_layer()


@pytest.fixture(scope="module")
def qwen():
    return synth.qwen_partial_layer()


@pytest.mark.parametrize("T", [4, 1, 3, 8, 9, 13, 37, 64, 100, 257])
@pytest.mark.parametrize("force", [0, F.FORCE_GEMV | F.UNFUSED, F.FORCE_GEMM])
def test_tiny(tiny, T, force):
    x = synth.draw_x(synth.SEED_TINY, T, tiny.shape.hidden)
    err, nflag = gp.check_full(tiny, x, flags=force, max_tokens=max(T, 8))
    print(f"tiny T={T} rel={err:.2e} flagged={nflag}")


@pytest.mark.parametrize("T", [12, 20])
@pytest.mark.parametrize("flags", [F.RESIDUAL, F.PRENORM, F.RESIDUAL | F.PRENORM])
@pytest.mark.parametrize("force", [0, F.FORCE_GEMV | F.UNFUSED, F.FORCE_GEMM])
def test_tiny_flags(tiny, flags, force, T):
    """T = 12 with force = 0 runs the single-launch decode kernel; T = 20 the
    separate-launch decode path."""
    x = synth.draw_x(synth.SEED_TINY, T, tiny.shape.hidden)
    m = gp.make_handle(tiny, 32)
    try:
        gp.check_full(tiny, x, flags=flags | force, m=m)
        if force == 0:
            assert m.last_path()[0] == (F.PATH_DECODE_FUSED if T <= 16 else F.PATH_DECODE)
    finally:
        m.close()


def test_tiny_gemm_large_groups():
    """Experts with more than 256 tokens (several token chunks per expert)."""
    shape = synth.LayerShape(hidden=256, inter=128, num_experts=4, top_k=2)
    layer = synth.make_layer(shape, 77)
    x = synth.draw_x(77, 700, 256)
    gp.check_full(layer, x, flags=F.FORCE_GEMM, max_tokens=700)


@pytest.mark.parametrize("T,tile", [(64, 32), (65, 128), (256, 128), (257, 256)])
def test_tiny_gemm_token_tiles(T, tile):
    """Every token tile of the grouped GEMM on one skewed layer, each at its
    first or last T for 8 experts x top-2: the 32-token tile (weights through
    tensor memory) up to 16 pairs per expert on average, the 128-token tile
    (two accumulators) up to 64, the 256-token tile above.  The logit bias
    piles pairs onto a few experts, so some expert holds more than one tile
    where T allows (asserted) and every chunk boundary is crossed."""
    layer = synth.make_layer(synth.TINY, 91, bias_sigma=2.0)
    x = synth.draw_x(91, T, synth.TINY.hidden)
    m = gp.make_handle(layer, T)
    try:
        _, dbg = gp.gpu_forward(m, layer, x, F.FORCE_GEMM)
        counts = np.diff(dbg["offsets"])
        if T > tile:   # the skew puts more than one tile on some expert
            assert counts.max() > tile, counts
        gp.check_full(layer, x, flags=F.FORCE_GEMM, m=m)
        assert m.last_path()[0] == F.PATH_GEMM
    finally:
        m.close()


@pytest.mark.parametrize("T", [1, 4, 16])
@pytest.mark.parametrize("force", [0, F.UNFUSED, F.FORCE_GEMM])
def test_olmoe_decode(olmoe, T, force):
    x = synth.draw_x(synth.SEED_OLMOE_DECODE, T, olmoe.shape.hidden)
    err, nflag = gp.check_full(olmoe, x, flags=force, max_tokens=2048)
    print(f"olmoe T={T} rel={err:.2e} flagged={nflag}")


@pytest.mark.parametrize("T", [1, 4, 16])
@pytest.mark.parametrize("flags", [F.PRENORM, F.RESIDUAL | F.PRENORM])
def test_olmoe_decode_prenorm_fused(olmoe, T, flags):
    """PRENORM on the single-launch decode kernel with real routing: 1/rms is
    folded into the router logits (it can change the top-k) and into the
    gate/up epilogue."""
    x = synth.draw_x(synth.SEED_OLMOE_DECODE + 50, T, olmoe.shape.hidden)
    x = (x.astype(np.float32) * np.float32(3.0)).astype(np.float16)   # rms far from 1
    m = gp.make_handle(olmoe, 16)
    try:
        err, nflag = gp.check_full(olmoe, x, flags=flags, m=m)
        assert m.last_path() == (F.PATH_DECODE_FUSED, 1)
    finally:
        m.close()
    print(f"olmoe prenorm T={T} flags={flags} rel={err:.2e} flagged={nflag}")


@pytest.mark.parametrize("T", [1, 8, 32])
@pytest.mark.parametrize("force", [0, F.UNFUSED, F.FORCE_GEMM])
def test_qwen_partial(qwen, T, force):
    x = synth.draw_x(synth.SEED_QWEN_PARTIAL, T, qwen.shape.hidden)
    err, nflag = gp.check_full(qwen, x, flags=force, max_tokens=64)
    print(f"qwen T={T} rel={err:.2e} flagged={nflag}")


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("force", [0, F.FORCE_GEMV])
def test_olmoe_prefill_sampled(variant, force):
    layer = synth.olmoe_prefill_layer(variant)
    seed = synth.SEED_OLMOE_PREFILL if variant == 1 else synth.SEED_OLMOE_PREFILL_SKEW
    T = 2048
    x = synth.draw_x(seed, T, layer.shape.hidden)
    rows = np.random.default_rng(variant).choice(T, size=40, replace=False)
    rows = np.concatenate([rows, [0, T - 1]])
    err, nflag = gp.check_sampled(layer, x, rows, flags=force)
    print(f"prefill v{variant} sampled rel={err:.2e} flagged={nflag}")


@pytest.mark.parametrize("variant", [1, 2])
def test_olmoe_prefill_every_row(variant):
    """T = 2048 prefill, every output row against the oracle (grouped-GEMM
    path, and the decode kernels forced), one oracle evaluation for both."""
    layer = synth.olmoe_prefill_layer(variant)
    seed = synth.SEED_OLMOE_PREFILL if variant == 1 else synth.SEED_OLMOE_PREFILL_SKEW
    x = synth.draw_x(seed, 2048, layer.shape.hidden)
    m = gp.make_handle(layer, 2048)
    try:
        got = [gp.gpu_forward(m, layer, x, force) for force in (0, F.FORCE_GEMV)]
        assert m.get_status() == (F.OK, 0)
    finally:
        m.close()
    ref = gp.oracle_layer(layer, x, 0)
    assert not ref.overflow.any()
    for out, dbg in got:
        gp.assert_routing(dbg, ref.ids, ref.weights, ref.near_tie, layer.shape.num_experts, ref.perm)
        err = gp.assert_output(out, ref.out, ~ref.near_tie)
        print(f"prefill v{variant} every row rel={err:.2e} flagged={int(ref.near_tie.sum())}")

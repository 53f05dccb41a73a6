"""Exact routing ties on every router the library has.

The router rule is: top-k by the largest logit, equal logits ordered by the
lower expert index (landing page, "06 / Follow a token": routing selects the
experts; the tie rule is the reading this library takes).  The other parity
tests exclude near ties, so here the inputs are built to make ties exact in
every summation order: x holds small integers and the router weights are
integers / 64, so every product and every partial sum of a logit is a
multiple of 1/64 below 2^15 in magnitude, exact in FP16 x FP16 -> FP32 and
in FP64.  Many experts then share a logit exactly, and the GPU's ids must
equal the oracle's stable top-k on every token (nothing excluded).

Routers reached: the single-launch decode kernel's routing phase (T <= 16),
the one-cluster router (separate launches, T <= 8) and the cooperative router
(T > 8, both of its grid sizes).  The allocation-free router has the same
check in its own test file.
"""
import numpy as np
import pytest

from oracle import moe_oracle
from tests import gpu_parity as gp
from w4a16_compact_expert_gb300 import moe_w4a16 as F, synth

pytestmark = pytest.mark.gpu


def _dyadic_layer(shape, seed, bias_kind):
    layer = synth.make_layer(shape, seed)
    rng = np.random.default_rng(seed)
    E, H = shape.num_experts, shape.hidden
    if bias_kind == "zero_router":
        layer.router_w = np.zeros((E, H), np.float16)
        layer.bias = None
    else:
        layer.router_w = (rng.integers(-4, 5, size=(E, H)) / 64.0).astype(np.float16)
        layer.bias = None
        if bias_kind == "grouped_bias":
            # three bias levels: many experts tie on the bias alone
            layer.bias = (((np.arange(E) * 5) % 3) / 64.0).astype(np.float32)
    return layer


def _dyadic_x(seed, T, H):
    return np.random.default_rng(seed + 7).integers(-3, 4, size=(T, H)).astype(np.float16)


def _exact_route(layer, x, flags):
    """The oracle's routing with the exact logits.  PRENORM multiplies every
    logit of a token by the same positive 1/rms, so the order is that of
    x W^T (no bias in the PRENORM cases); the weights are the oracle's."""
    k = layer.shape.top_k
    exact = moe_oracle.router_logits(x, layer.router_w, layer.bias)
    ids = moe_oracle.topk_ids(exact, k)
    xin = moe_oracle.rms_prenorm(x) if flags & F.PRENORM else x
    _, probs, _, _ = moe_oracle.route(xin, layer.router_w, layer.bias, k)
    return exact, ids, np.take_along_axis(probs, ids, axis=-1)


CASES = [
    # (T, forced family, router the library takes)
    (3, 0, "fused"),
    (12, 0, "fused"),
    (3, F.FORCE_GEMV | F.UNFUSED, "cluster"),
    (12, F.FORCE_GEMV | F.UNFUSED, "cooperative phases on one cluster"),
    (70, F.FORCE_GEMV, "cooperative"),
    (3, F.FORCE_GEMM, "cluster"),
    (40, F.FORCE_GEMM, "cooperative phases on one cluster, x rows gathered"),
    (70, F.FORCE_GEMM, "cooperative"),
    (600, F.FORCE_GEMM, "cooperative, two CTAs per SM"),
]


@pytest.mark.parametrize("kind", ["zero_router", "dyadic", "grouped_bias"])
@pytest.mark.parametrize("shape", [synth.TINY, synth.LayerShape(hidden=256, inter=128, num_experts=64, top_k=8),
                                   synth.LayerShape(hidden=512, inter=128, num_experts=16, top_k=3)],
                         ids=["E8k2", "E64k8", "E16k3"])
def test_exact_ties_all_routers(shape, kind):
    layer = _dyadic_layer(shape, 31 + shape.num_experts, kind)
    m = gp.make_handle(layer, 600)
    k, E = shape.top_k, shape.num_experts
    ties = 0
    try:
        for T, force, _ in CASES:
            x = _dyadic_x(T, T, shape.hidden)
            exact, ids_ref, w_ref = _exact_route(layer, x, 0)
            s = -np.sort(-exact, axis=-1)[:, : k + 1]
            ties += int((np.diff(s, axis=-1) == 0).any(axis=-1).sum())
            out, dbg = gp.gpu_forward(m, layer, x, force)
            assert m.get_status() == (F.OK, 0)
            assert np.array_equal(dbg["ids"], ids_ref), (T, force)
            assert np.abs(dbg["weights"] - w_ref).max() <= gp.TOL_W
            if kind == "zero_router":
                assert np.array_equal(dbg["ids"], np.tile(np.arange(k), (T, 1)))
                assert np.abs(dbg["weights"] - 1.0 / E).max() <= gp.TOL_W
            perm = moe_oracle.permutation(ids_ref, E)
            assert np.array_equal(dbg["sorted_pairs"], perm.sorted_pairs)
            assert np.array_equal(dbg["offsets"], perm.offsets)
            if T <= 70:
                # routing is exact, so the layer output is compared on every token
                ref = gp.oracle_layer(layer, x, 0)
                assert np.array_equal(ref.ids, ids_ref)
                gp.assert_output(out, ref.out, np.ones(T, bool))
    finally:
        m.close()
    assert ties > 0, "the inputs should produce exact ties among the k+1 largest logits"


@pytest.mark.parametrize("T,force", [(5, 0), (5, F.FORCE_GEMV | F.UNFUSED), (40, F.FORCE_GEMM)])
def test_exact_ties_under_prenorm(T, force):
    """PRENORM scales a token's logits by one positive factor: exact ties stay
    ties and are broken to the lower index."""
    shape = synth.LayerShape(hidden=256, inter=128, num_experts=64, top_k=8)
    layer = _dyadic_layer(shape, 77, "dyadic")
    x = _dyadic_x(5 + T, T, shape.hidden)
    _, ids_ref, w_ref = _exact_route(layer, x, F.PRENORM)
    m = gp.make_handle(layer, 64)
    try:
        _, dbg = gp.gpu_forward(m, layer, x, F.PRENORM | force)
        assert m.get_status() == (F.OK, 0)
    finally:
        m.close()
    assert np.array_equal(dbg["ids"], ids_ref)
    assert np.abs(dbg["weights"] - w_ref).max() <= gp.TOL_W
    assert np.array_equal(dbg["sorted_pairs"], moe_oracle.permutation(ids_ref, 64).sorted_pairs)


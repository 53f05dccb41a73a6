"""moe_w4a16_route_noalloc: routing without any device allocation.

Some callers cannot call cudaMalloc -- a runtime whose allocator already owns
all device memory, a path that must not risk an allocation's implicit
synchronisation, code running while allocation is forbidden -- and creating a
handle allocates.  This entry point routes a layer using only a fixed device
array inside the library.  The tests call it through the C ABI:
  * twice in a row, each result checked against the oracle's routing and
    against moe_w4a16_forward's cooperative router (bit for bit);
  * at the limits of its scratch array (T * E * ceil(H / 256) equal to the
    maximum; 256 experts with top-32), with and without PRENORM;
  * on exact routing ties;
  * with every argument check, each of which must leave the outputs
    untouched (nothing is enqueued).
This file is collected last, so a run that stops at the first failure has
run every other test before it.
"""
import ctypes

import numpy as np
import pytest

from oracle import moe_oracle
from tests import gpu_parity as gp
from w4a16_compact_expert_gb300 import build_ext, moe_w4a16, synth

pytestmark = pytest.mark.gpu
SENT = -7
MAX_LOGITS = 786432   # MOE_W4A16_NOALLOC_MAX_LOGITS


@pytest.fixture(scope="module")
def lib():
    build_ext.build()
    lib = moe_w4a16.load_library()
    vp, i32, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32
    lib.moe_w4a16_route_noalloc.argtypes = [vp, i32, i32, i32, i32, vp, vp, u32, vp, vp, vp, vp, vp]
    return lib


def _outputs(T, E, k):
    import torch
    return (torch.full((T, k), SENT, dtype=torch.int32, device="cuda"),
            torch.full((T, k), float(SENT), dtype=torch.float32, device="cuda"),
            torch.full((T * k,), SENT, dtype=torch.int32, device="cuda"),
            torch.full((E + 1,), SENT, dtype=torch.int32, device="cuda"))


def _call(lib, x, T, H, E, k, rw, bias, flags, outs, x_off=0, rw_off=0):
    import torch
    ids, w, sp, off = outs
    return lib.moe_w4a16_route_noalloc(x.data_ptr() + x_off, T, H, E, k, rw.data_ptr() + rw_off,
                                       None if bias is None else bias.data_ptr(), flags, ids.data_ptr(),
                                       w.data_ptr(), sp.data_ptr(), off.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)


def _route_noalloc(lib, x, rw, bias, E, k, flags):
    import torch
    T, H = x.shape
    outs = _outputs(T, E, k)
    st = _call(lib, x, T, H, E, k, rw, bias, flags, outs)
    assert st == moe_w4a16.OK, lib.moe_w4a16_last_error(None)
    torch.cuda.synchronize()
    ids, w, sp, off = (t.cpu().numpy() for t in outs)
    return {"ids": ids, "weights": w, "sorted_pairs": sp, "offsets": off}


def _check_against_oracle(got, x, router_w, bias, E, k, flags):
    """ids bit-exact and weights within 1e-5 on tokens that are not near ties;
    the permutation bit-exact against the oracle's permutation of the ids
    returned, and of the oracle's own ids when no token is a near tie."""
    xin = moe_oracle.rms_prenorm(x) if flags & moe_oracle.FLAG_PRENORM else x
    logits, _, ids, w = moe_oracle.route(xin, router_w, bias, k)
    flagged = moe_oracle.near_tie_flags(logits, k)
    gp.assert_routing(got, ids, w, flagged, E, moe_oracle.permutation(ids, E))
    return int(flagged.sum())


def test_route_noalloc_twice_matches_oracle_and_forward(lib):
    shape = synth.LayerShape(hidden=256, inter=128, num_experts=64, top_k=8)
    layer = synth.make_layer(shape, 4242, bias_sigma=0.5)
    m = gp.make_handle(layer, 256)
    try:
        for T, flags in ((200, 0), (37, moe_w4a16.PRENORM)):
            x = synth.draw_x(4242, T, 256)
            # the forward's cooperative router (every T > 8 on the grouped-GEMM path)
            _, ref = gp.gpu_forward(m, layer, x, flags | moe_w4a16.FORCE_GEMM)
            got = _route_noalloc(lib, gp.to_dev(x), gp.to_dev(layer.router_w), gp.to_dev(layer.bias), 64, 8, flags)
            _check_against_oracle(got, x, layer.router_w, layer.bias, 64, 8, flags)
            for key in ("ids", "weights", "sorted_pairs", "offsets"):
                assert np.array_equal(got[key], ref[key]), key
    finally:
        m.close()


@pytest.mark.parametrize("flags", [0, moe_w4a16.PRENORM])
@pytest.mark.parametrize("T,H,E,k", [(1536, 2048, 64, 8), (8, 512, 256, 32), (3, 2048, 256, 32)],
                         ids=["max_logits", "E256k32", "E256k32_T3"])
def test_route_noalloc_at_the_limits(lib, T, H, E, k, flags):
    """T * E * ceil(H / 256) = 786,432 (the maximum: the logits region full and
    the block-count region at its end used), and 256 experts with top-32
    (several 64-expert logits tiles, 32 K slices summed by the top-k kernel)."""
    rng = np.random.Generator(np.random.PCG64(900 + E))
    router_w = (rng.standard_normal((E, H)) * 0.02).astype(np.float16)
    bias = (rng.standard_normal(E) * 0.3).astype(np.float32) if not flags else None
    x = synth.draw_x(900 + T, T, H)
    if flags:
        x = (x.astype(np.float32) * 3).astype(np.float16)
    assert T * E * -(-H // 256) <= MAX_LOGITS
    for _ in range(2):   # twice in a row: the shared array keeps the last call's contents
        got = _route_noalloc(lib, gp.to_dev(x), gp.to_dev(router_w), gp.to_dev(bias), E, k, flags)
        nflag = _check_against_oracle(got, x, router_w, bias, E, k, flags)
    print(f"route_noalloc T={T} H={H} E={E} k={k} flags={flags}: near ties {nflag}")


@pytest.mark.parametrize("flags", [0, moe_w4a16.PRENORM])
def test_route_noalloc_exact_ties(lib, flags):
    """Integer x and integer/64 router weights make every logit exact in any
    summation order, so many experts tie exactly; ties go to the lower index
    (PRENORM scales a token's logits by one positive factor and keeps ties)."""
    E, k, H = 64, 8, 256
    rng = np.random.default_rng(91)
    router_w = (rng.integers(-4, 5, size=(E, H)) / 64.0).astype(np.float16)
    bias = None if flags else (((np.arange(E) * 5) % 3) / 64.0).astype(np.float32)
    for T in (7, 300):
        x = np.random.default_rng(T).integers(-3, 4, size=(T, H)).astype(np.float16)
        exact = moe_oracle.router_logits(x, router_w, bias)
        ids_ref = moe_oracle.topk_ids(exact, k)
        xin = moe_oracle.rms_prenorm(x) if flags else x
        _, probs, _, _ = moe_oracle.route(xin, router_w, bias, k)
        s = -np.sort(-exact, axis=-1)[:, : k + 1]
        assert (np.diff(s, axis=-1) == 0).any()
        got = _route_noalloc(lib, gp.to_dev(x), gp.to_dev(router_w), gp.to_dev(bias), E, k, flags)
        perm = moe_oracle.permutation(ids_ref, E)
        assert np.array_equal(got["ids"], ids_ref)
        assert np.abs(got["weights"] - np.take_along_axis(probs, ids_ref, axis=-1)).max() <= gp.TOL_W
        assert np.array_equal(got["sorted_pairs"], perm.sorted_pairs)
        assert np.array_equal(got["offsets"], perm.offsets)


REJECTIONS = [
    # (T, H, E, k, flags, x byte offset, router_w byte offset, message fragment)
    (5000, 256, 64, 8, 0, 0, 0, b"MAX_TOKENS"),
    (4096, 256, 256, 8, 0, 0, 0, b"MAX_LOGITS"),
    (8, 8192, 64, 8, 0, 0, 0, b"MAX_HIDDEN"),
    (4096, 256, 32, 32, 0, 0, 0, b"MAX_PAIRS"),
    (8, 256, 64, 33, 0, 0, 0, b"top_k"),
    (8, 256, 16, 17, 0, 0, 0, b"top_k"),
    (8, 200, 64, 8, 0, 0, 0, b"multiple of 64"),
    (8, 256, 300, 8, 0, 0, 0, b"num_experts"),
    (8, 256, 64, 8, moe_w4a16.RESIDUAL, 0, 0, b"PRENORM"),
    (8, 256, 64, 8, 64, 0, 0, b"PRENORM"),
    (8, 256, 64, 8, 0, 8, 0, b"16-byte aligned"),
    (8, 256, 64, 8, 0, 0, 8, b"16-byte aligned"),
]


@pytest.mark.parametrize("T,H,E,k,flags,xo,ro,msg", REJECTIONS)
def test_route_noalloc_rejects_and_enqueues_nothing(lib, T, H, E, k, flags, xo, ro, msg):
    import torch
    x = torch.zeros(64, 512, dtype=torch.float16, device="cuda")
    rw = torch.zeros(64, 512, dtype=torch.float16, device="cuda")
    outs = _outputs(8, 300, 33)
    st = _call(lib, x, T, H, E, k, rw, None, flags, outs, x_off=xo, rw_off=ro)
    assert st == moe_w4a16.ERR_INVALID_ARG
    assert msg in lib.moe_w4a16_last_error(None)
    torch.cuda.synchronize()
    for t in outs:
        assert bool((t == SENT).all()), "a rejected call wrote its outputs"

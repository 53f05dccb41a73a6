"""moe_w4a16_route_noalloc: routing without any device allocation.

Some callers cannot call cudaMalloc -- a runtime whose allocator already owns
all device memory, a path that must not risk an allocation's implicit
synchronisation, code running while allocation is forbidden -- and creating a
handle allocates.  This entry point routes a layer using only a fixed device
array inside the library.  The test calls it twice in a row through the C ABI
and checks both results against the routing outputs of moe_w4a16_forward.
"""
import ctypes

import numpy as np
import pytest

from oracle import moe_oracle
from tests import gpu_parity as gp
from w4a16_compact_expert_gb300 import build_ext, moe_w4a16, synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    build_ext.build()
    lib = moe_w4a16.load_library()
    vp, i32, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32
    lib.moe_w4a16_route_noalloc.argtypes = [vp, i32, i32, i32, i32, vp, vp, u32, vp, vp, vp, vp, vp]
    return lib


def _route_noalloc(lib, x, rw, bias, E, k, flags):
    import torch
    T, H = x.shape
    ids = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, k), -7.0, dtype=torch.float32, device="cuda")
    sp = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    off = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    st = lib.moe_w4a16_route_noalloc(x.data_ptr(), T, H, E, k, rw.data_ptr(),
                                     None if bias is None else bias.data_ptr(), flags, ids.data_ptr(),
                                     w.data_ptr(), sp.data_ptr(), off.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)
    assert st == moe_w4a16.OK, lib.moe_w4a16_last_error(None)
    torch.cuda.synchronize()
    return {"ids": ids.cpu().numpy(), "weights": w.cpu().numpy(), "sorted_pairs": sp.cpu().numpy(),
            "offsets": off.cpu().numpy()}


def test_route_noalloc_matches_forward_twice(lib):
    shape = synth.LayerShape(hidden=256, inter=128, num_experts=64, top_k=8)
    layer = synth.make_layer(shape, 4242, bias_sigma=0.5)
    m = gp.make_handle(layer, 256)
    try:
        for T, flags in ((200, 0), (37, moe_w4a16.PRENORM)):
            x = synth.draw_x(4242, T, 256)
            _, ref = gp.gpu_forward(m, layer, x, flags)
            got = _route_noalloc(lib, gp.to_dev(x), gp.to_dev(layer.router_w), gp.to_dev(layer.bias), 64, 8, flags)
            xin = moe_oracle.rms_prenorm(x) if flags & moe_oracle.FLAG_PRENORM else x
            logits = moe_oracle.router_logits(xin, layer.router_w, layer.bias)
            keep = ~moe_oracle.near_tie_flags(logits, 8)
            assert np.array_equal(got["ids"][keep], ref["ids"][keep])
            assert np.abs(got["weights"][keep] - ref["weights"][keep]).max() <= gp.TOL_W
            own = moe_oracle.permutation(got["ids"], 64)
            assert np.array_equal(got["sorted_pairs"], own.sorted_pairs)
            assert np.array_equal(got["offsets"], own.offsets)
            if T > 64:   # the forward took the same routing kernels: identical results
                assert np.array_equal(got["ids"], ref["ids"])
                assert np.array_equal(got["weights"], ref["weights"])
                assert np.array_equal(got["sorted_pairs"], ref["sorted_pairs"])
    finally:
        m.close()


def test_route_noalloc_rejects_sizes_beyond_the_limit(lib):
    import torch
    x = torch.zeros(8, 256, dtype=torch.float16, device="cuda")
    rw = torch.zeros(64, 256, dtype=torch.float16, device="cuda")
    ids = torch.empty(8, 8, dtype=torch.int32, device="cuda")
    w = torch.empty(8, 8, dtype=torch.float32, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    st = lib.moe_w4a16_route_noalloc(x.data_ptr(), 5000, 256, 64, 8, rw.data_ptr(), None, 0, ids.data_ptr(),
                                     w.data_ptr(), None, None, s)
    assert st == moe_w4a16.ERR_INVALID_ARG and b"MAX_TOKENS" in lib.moe_w4a16_last_error(None)
    st = lib.moe_w4a16_route_noalloc(x.data_ptr(), 4096, 256, 256, 8, rw.data_ptr(), None, 0, ids.data_ptr(),
                                     w.data_ptr(), None, None, s)
    assert st == moe_w4a16.ERR_INVALID_ARG and b"MAX_LOGITS" in lib.moe_w4a16_last_error(None)
    st = lib.moe_w4a16_route_noalloc(x.data_ptr(), 8, 8192, 64, 8, rw.data_ptr(), None, 0, ids.data_ptr(),
                                     w.data_ptr(), None, None, s)
    assert st == moe_w4a16.ERR_INVALID_ARG and b"MAX_HIDDEN" in lib.moe_w4a16_last_error(None)

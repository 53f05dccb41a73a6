"""The expert cache's miss path on the GPU: routing on the device, the routed
group acquired through the cache (misses copied from the immutable host
backing through pinned staging into spare rows, a new generation published,
least recently used experts discarded), then the layer forward, which must
match the oracle over the full expert set."""
import ctypes

import numpy as np
import pytest

from oracle import moe_oracle
from tests import gpu_parity as gp
from w4a16_compact_expert_gb300 import moe_w4a16 as M, synth

pytestmark = pytest.mark.gpu


def _route_ids(lib, x, rw, bias, E, k):
    import torch
    T, H = x.shape
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    sp = torch.empty((T * k,), dtype=torch.int32, device="cuda")
    off = torch.empty((E + 1,), dtype=torch.int32, device="cuda")
    st = lib.moe_w4a16_route_noalloc(x.data_ptr(), T, H, E, k, rw.data_ptr(),
                                     None if bias is None else bias.data_ptr(), 0, ids.data_ptr(), w.data_ptr(),
                                     sp.data_ptr(), off.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert st == M.OK
    return ids.cpu().numpy()


def test_cache_miss_path_matches_the_oracle():
    import torch
    lib = M.load_library()
    vp, i32, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32
    lib.moe_w4a16_route_noalloc.argtypes = [vp, i32, i32, i32, i32, vp, vp, u32, vp, vp, vp, vp, vp]
    layer = synth.tiny_layer()
    s = layer.shape
    backing = layer.experts.arrays()          # all E experts, canonical, host: the immutable source
    expert_bytes = s.packed_bytes_per_expert()
    m = M.MoELayer(s.hidden, s.inter, s.num_experts, s.top_k, num_slots=8, max_tokens=8)
    cache = M.ExpertCache(m, backing, staging_experts=2, spare_slots=4, max_group=4, initial=[0, 1, 2])
    try:
        with pytest.raises(M.MoEError):
            m.set_slot_table(list(range(8)))  # the cache owns the table
        rw, bias = gp.to_dev(layer.router_w), gp.to_dev(layer.bias)
        for i in range(16):
            x = synth.draw_x(500 + i, 2, s.hidden)
            xd = gp.to_dev(x)
            group = sorted(set(_route_ids(lib, xd, rw, bias, s.num_experts, s.top_k).ravel().tolist()))
            lease = cache.acquire(group)
            assert all(cache.slot_of(e) >= 0 for e in group)
            out = m.forward(xd, rw, bias, 0)
            cache.release(lease)
            torch.cuda.synchronize()
            ref = moe_oracle.moe_layer(x, layer.router_w, layer.bias, backing, s.top_k)
            gp.assert_output(out.float().cpu().numpy().astype(np.float64), ref.out, ~ref.near_tie)
        st, miss = m.get_status()
        assert st == M.OK and miss == 0
        stats = cache.stats()
        assert stats["misses"] > 0 and stats["evictions"] > 0 and stats["transactions"] > 0
        assert stats["d2h_bytes"] == 0
        assert stats["h2d_bytes"] == expert_bytes * (3 + stats["misses"])
        assert stats["resident"] <= 8 - 4
        last = [cache.slot_of(e) for e in range(s.num_experts)]
    finally:
        cache.close()
    try:
        # detached: the handle keeps serving the last published generation
        group = [e for e in range(s.num_experts) if last[e] >= 0][:2]
        x = synth.draw_x(999, 1, s.hidden)
        bias = np.full(s.num_experts, -np.inf, np.float32)
        bias[group] = 0.0                       # route only to experts of the last generation
        out = m.forward(gp.to_dev(x), gp.to_dev(layer.router_w), gp.to_dev(bias), 0)
        torch.cuda.synchronize()
        ref = moe_oracle.moe_layer(x, layer.router_w, bias, backing, s.top_k)
        gp.assert_output(out.float().cpu().numpy().astype(np.float64), ref.out, ~ref.near_tie)
        st, miss = m.get_status()
        assert st == M.OK and miss == 0
    finally:
        m.close()

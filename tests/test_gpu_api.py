"""Library behaviour on the GPU: edge cases, invariants, misses, errors."""
import numpy as np
import pytest

from oracle import moe_oracle
from tests import gpu_parity as gp
from w4a16_compact_expert_gb300 import moe_w4a16, synth

pytestmark = pytest.mark.gpu
F = moe_w4a16


@pytest.fixture(scope="module")
def tiny():
    return synth.tiny_layer()


def test_t0_is_noop(tiny):
    import torch
    m = gp.make_handle(tiny, 8)
    try:
        x = torch.empty(0, 256, dtype=torch.float16, device="cuda")
        out = m.forward(x, gp.to_dev(tiny.router_w))
        assert out.shape == (0, 256)
    finally:
        m.close()


@pytest.mark.parametrize("flags", [0, F.UNFUSED, F.FORCE_GEMM])
def test_deterministic_and_slot_relabel_invariant(tiny, flags):
    x = synth.draw_x(7, 33, 256)
    m = gp.make_handle(tiny, 64)
    out1, d1 = gp.gpu_forward(m, tiny, x, flags)
    out2, d2 = gp.gpu_forward(m, tiny, x, flags)
    m.close()
    assert np.array_equal(out1, out2) and np.array_equal(d1["sorted_pairs"], d2["sorted_pairs"])
    # same experts at a permuted set of slot rows (and two spare rows never used)
    perm = np.array([5, 9, 0, 3, 7, 1, 8, 2])
    s = tiny.shape
    m2 = moe_w4a16.MoELayer(s.hidden, s.inter, s.num_experts, s.top_k, num_slots=10, max_tokens=64)
    try:
        ex = tiny.experts.arrays()
        for e in range(8):
            m2.pack_experts(int(perm[e]), *(a[e:e + 1] for a in ex))
        m2.pack_experts(4, *(a[:1] for a in ex))
        m2.pack_experts(6, *(a[1:2] for a in ex))
        m2.set_slot_table(perm)
        out3, _ = gp.gpu_forward(m2, tiny, x, flags)
    finally:
        m2.close()
    assert np.array_equal(out1, out3)


def test_zero_input_gives_zero(tiny):
    x = np.zeros((5, 256), np.float16)
    m = gp.make_handle(tiny, 8)
    try:
        out, _ = gp.gpu_forward(m, tiny, x)
    finally:
        m.close()
    assert np.all(out == 0)


def test_all_routed_experts_absent(tiny):
    """Only two experts resident and none of them routed: out = x (RESIDUAL) or 0."""
    x = synth.draw_x(12, 6, 256)
    m = gp.make_handle(tiny, 8)
    try:
        m.set_slot_table([-1, -1, -1, -1, -1, -1, 6, 7])
        bias = np.zeros(8, np.float32)
        bias[6:] = -1e4          # never routed
        for flags in (0, F.RESIDUAL, F.UNFUSED, F.RESIDUAL | F.UNFUSED, F.FORCE_GEMM | F.RESIDUAL):
            out, _ = m.forward(gp.to_dev(x), gp.to_dev(tiny.router_w), gp.to_dev(bias), flags, debug=True)
            got = out.float().cpu().numpy()
            expect = x.astype(np.float32) if flags & F.RESIDUAL else np.zeros_like(got)
            assert np.array_equal(got, expect), flags
        st, miss = m.get_status()
        assert st == F.ERR_NOT_RESIDENT and miss == 5 * 6 * 2
    finally:
        m.close()


@pytest.mark.parametrize("flags", [0, F.UNFUSED, F.FORCE_GEMM])
def test_routed_absent_expert_counts_misses(tiny, flags):
    x = synth.draw_x(11, 24, 256)
    table = tiny.expert_to_slot.copy()
    table[3] = -1
    table[6] = -1
    m = gp.make_handle(tiny, 32)
    try:
        m.set_slot_table(table)
        out, dbg = gp.gpu_forward(m, tiny, x, flags)
        st, miss = m.get_status()
        st2, miss2 = m.get_status()
    finally:
        m.close()
    ref = moe_oracle.moe_layer(x, tiny.router_w, tiny.bias, tiny.slot_experts().arrays(), 2,
                               expert_to_slot=table)
    expected_miss = int(np.isin(ref.ids, [3, 6]).sum())
    assert expected_miss > 0
    assert st == F.ERR_NOT_RESIDENT and miss == expected_miss
    assert st2 == F.OK and miss2 == 0   # cleared by the read
    keep = ~ref.near_tie
    gp.assert_output(out, ref.out, keep)


@pytest.mark.parametrize("name,T,absent", [("tiny", 6, (3, 6)), ("olmoe", 8, tuple(range(0, 64, 5))),
                                           ("olmoe", 16, tuple(range(2, 64, 5)))])
@pytest.mark.parametrize("flags", [0, F.RESIDUAL])
def test_fused_kernel_routed_absent_experts(name, T, absent, flags):
    """Routed experts without a slot on the single-launch decode kernel, in
    both of its unit orders: TINY at T = 6 and OLMoE at T = 8 run the
    interleaved order (OLMoE with 30 active experts, past the lag, so down
    items and gate/up items alternate), OLMoE at T = 16 the phase order.  The
    pairs routed to absent experts count as misses and add nothing; the rest
    matches the oracle."""
    layer = synth.tiny_layer() if name == "tiny" else synth.olmoe_decode_layer()
    x = synth.draw_x(31 + T, T, layer.shape.hidden)
    table = layer.expert_to_slot.copy()
    table[list(absent)] = -1
    m = gp.make_handle(layer, 16)
    try:
        m.set_slot_table(table)
        out, _ = gp.gpu_forward(m, layer, x, flags)
        path = m.last_path()
        st, miss = m.get_status()
    finally:
        m.close()
    ref = moe_oracle.moe_layer(x, layer.router_w, layer.bias, layer.slot_experts().arrays(), layer.shape.top_k,
                               flags, expert_to_slot=table)
    expected_miss = int(np.isin(ref.ids, absent).sum())
    assert expected_miss > 0
    assert path == (F.PATH_DECODE_FUSED, 1)
    assert st == F.ERR_NOT_RESIDENT and miss == expected_miss
    gp.assert_output(out, ref.out, ~ref.near_tie)


def test_dense_single_expert_and_k_equals_e():
    shape = synth.LayerShape(hidden=128, inter=64, num_experts=1, top_k=1)
    layer = synth.make_layer(shape, 5)
    x = synth.draw_x(5, 9, 128)
    gp.check_full(layer, x, max_tokens=16)
    shape = synth.LayerShape(hidden=192, inter=128, num_experts=4, top_k=4)
    layer = synth.make_layer(shape, 6, bias_sigma=0.5)
    x = synth.draw_x(6, 9, 192)
    gp.check_full(layer, x, max_tokens=16)


def test_forward_host_matches_forward(tiny):
    x = synth.draw_x(3, 12, 256)
    m = gp.make_handle(tiny, 16)
    try:
        out, _ = gp.gpu_forward(m, tiny, x, F.RESIDUAL)
        oh = m.forward_host(x, gp.to_dev(tiny.router_w), None, F.RESIDUAL)
    finally:
        m.close()
    assert np.array_equal(out, oh.astype(np.float64))


def test_forward_host_async_two_streams():
    """Two handles (OLMoE-shaped decode layers, single-launch cooperative
    kernel) enqueued alternately on two streams with host buffers, as the
    benchmark's end-to-end leg does: outputs equal the device forwards and no
    bounded wait gave up."""
    import torch
    layers = [synth.olmoe_decode_layer(), synth.tiny_layer()]
    T = 4
    ms = [gp.make_handle(layer, 16) for layer in layers]
    try:
        streams = [torch.cuda.Stream(), torch.cuda.Stream()]
        xs = [[synth.draw_x(60 + 10 * j + r, T, layer.shape.hidden) for r in range(3)]
              for j, layer in enumerate(layers)]
        rws = [gp.to_dev(layer.router_w) for layer in layers]
        outs = [[torch.empty(T, layer.shape.hidden, dtype=torch.float16).pin_memory() for _ in range(3)]
                for layer in layers]
        xh = [[torch.from_numpy(x).pin_memory() for x in row] for row in xs]
        for r in range(3):
            for j, m in enumerate(ms):
                m.forward_host_async(xh[j][r], rws[j], outs[j][r], None, 0, stream=streams[j])
        torch.cuda.synchronize()
        for j, (m, layer) in enumerate(zip(ms, layers)):
            for r in range(3):
                ref, _ = gp.gpu_forward(m, layer, xs[j][r], 0)
                assert np.array_equal(outs[j][r].numpy().astype(np.float64), ref)
            assert m.get_status() == (F.OK, 0)
    finally:
        for m in ms:
            m.close()


def test_forward_host_async_chain_matches_forward(tiny):
    """Three enqueued host-buffer forwards on one handle and one stream, each
    reading the previous one's host output (stream order), then one
    synchronisation: equal to the device forwards chained the same way."""
    import torch
    x = synth.draw_x(4, 12, 256)
    m = gp.make_handle(tiny, 16)
    try:
        rw = gp.to_dev(tiny.router_w)
        hosts = [torch.from_numpy(x).pin_memory()] + [torch.empty(12, 256, dtype=torch.float16).pin_memory()
                                                      for _ in range(3)]
        for i in range(3):
            m.forward_host_async(hosts[i], rw, hosts[i + 1], None, F.RESIDUAL)
        torch.cuda.synchronize()
        ref = x
        for i in range(3):
            out, _ = gp.gpu_forward(m, tiny, ref.astype(np.float16), F.RESIDUAL)
            ref = out
    finally:
        m.close()
    assert np.array_equal(hosts[3].numpy().astype(np.float64), ref)


def test_argument_errors(tiny):
    import torch
    m = gp.make_handle(tiny, 8)
    try:
        x = gp.to_dev(synth.draw_x(1, 9, 256))
        rw = gp.to_dev(tiny.router_w)
        with pytest.raises(F.MoEError) as e:
            m.forward(x, rw)                    # T = 9 > max_tokens = 8
        assert e.value.status == F.ERR_INVALID_ARG
        with pytest.raises(F.MoEError) as e:
            m.forward(x[:2], rw, flags=F.FORCE_GEMM | F.FORCE_GEMV)
        assert e.value.status == F.ERR_INVALID_ARG
        with pytest.raises(F.MoEError) as e:
            m.forward(x[:2], rw, flags=64)
        assert e.value.status == F.ERR_INVALID_ARG
        with pytest.raises(F.MoEError) as e:
            m.set_slot_table([0, 1, 2, 3, 4, 5, 6, 6])
        assert e.value.status == F.ERR_INVALID_ARG
        with pytest.raises(F.MoEError) as e:
            m.set_slot_table([0, 1, 2, 3, 4, 5, 6, 8])
        assert e.value.status == F.ERR_INVALID_ARG
        with pytest.raises(F.MoEError) as e:
            m.pack_experts(7, *(a[:2] for a in tiny.experts.arrays()))
        assert e.value.status == F.ERR_INVALID_ARG
        torch.cuda.synchronize()
    finally:
        m.close()
    s = tiny.shape
    m2 = moe_w4a16.MoELayer(s.hidden, s.inter, s.num_experts, s.top_k, num_slots=9, max_tokens=8)
    try:
        m2.pack_experts(0, *tiny.experts.arrays())
        with pytest.raises(F.MoEError) as e:
            m2.set_slot_table([0, 1, 2, 3, 4, 5, 6, 8])   # slot 8 never packed
        assert e.value.status == F.ERR_NOT_PACKED
        with pytest.raises(F.MoEError) as e:
            m2.forward(gp.to_dev(synth.draw_x(1, 2, 256)), gp.to_dev(tiny.router_w))   # no table yet
        assert e.value.status == F.ERR_INVALID_ARG
    finally:
        m2.close()


def test_device_source_pack_matches_host_pack(tiny):
    import torch
    x = synth.draw_x(4, 6, 256)
    m = gp.make_handle(tiny, 8)
    s = tiny.shape
    m2 = moe_w4a16.MoELayer(s.hidden, s.inter, s.num_experts, s.top_k, max_tokens=8)
    try:
        m2.pack_experts(0, *(torch.from_numpy(a).cuda() for a in tiny.experts.arrays()))
        m2.set_slot_table(tiny.expert_to_slot)
        o1, _ = gp.gpu_forward(m, tiny, x)
        o2, _ = gp.gpu_forward(m2, tiny, x)
    finally:
        m.close()
        m2.close()
    assert np.array_equal(o1, o2)


@pytest.mark.parametrize("T,flags,path,launches", [
    (4, 0, F.PATH_DECODE_FUSED, 1),
    (4, F.UNFUSED, F.PATH_DECODE, 3),
    (4, F.FORCE_GEMM, F.PATH_GEMM, 5),
    (100, F.FORCE_GEMM, F.PATH_GEMM, 4),
    (100, F.FORCE_GEMV, F.PATH_DECODE, 3),
    (12, F.UNFUSED, F.PATH_DECODE, 3),
])
def test_last_path_reports_kernels(tiny, T, flags, path, launches):
    """The reported path and launch count follow the dispatch rules: one
    cooperative kernel for small T, a one-kernel cluster router up to 8
    tokens, a one-kernel cooperative router above (which also gathers the x
    rows on the grouped-GEMM path)."""
    m = gp.make_handle(tiny, 128)
    try:
        assert m.last_path() == (F.PATH_NONE, 0)
        gp.gpu_forward(m, tiny, synth.draw_x(3, T, 256), flags)
        assert m.last_path() == (path, launches)
    finally:
        m.close()

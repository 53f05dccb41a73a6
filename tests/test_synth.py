"""Seeded input generator: determinism, format and distributions."""
import numpy as np

from w4a16_compact_expert_gb300 import synth


def test_tiny_layer_is_deterministic():
    a, b = synth.tiny_layer(), synth.tiny_layer()
    for x, y in zip(a.experts.arrays(), b.experts.arrays()):
        assert np.array_equal(x, y)
    assert np.array_equal(a.router_w, b.router_w)
    assert np.array_equal(synth.draw_x(1000, 4, 256), synth.draw_x(1000, 4, 256))
    assert not np.array_equal(synth.draw_x(1000, 4, 256)[:1], synth.draw_x(1000, 1, 256))


def test_shapes_and_ranges():
    L = synth.tiny_layer()
    E, H, I = 8, 256, 128
    ex = L.experts
    assert ex.gate_q.shape == (E, I, H // 2) and ex.gate_q.dtype == np.uint8
    assert ex.gate_s.shape == (E, I, 1) and ex.gate_s.dtype == np.uint16
    assert ex.down_q.shape == (E, H, I // 2) and ex.down_s.shape == (E, H, 1)
    s = ex.gate_s.view(np.float16).astype(np.float64)
    assert s.min() >= 0.00199 and s.max() <= 0.02001
    # every nibble value occurs with frequency close to 1/16
    lo = np.bincount((ex.gate_q & 15).ravel(), minlength=16) / ex.gate_q.size
    assert np.all(np.abs(lo - 1 / 16) < 0.01)
    rw = L.router_w.astype(np.float64)
    assert 0.015 < rw.std() < 0.025
    assert list(L.expert_to_slot) == list(range(E))


def test_per_expert_bytes():
    assert synth.OLMOE.packed_bytes_per_expert() == 3_194_880
    assert synth.QWEN.packed_bytes_per_expert() == 4_395_008
    assert synth.TINY.packed_bytes_per_expert() == 50_176


def test_partial_residency_layout():
    shape = synth.LayerShape(hidden=256, inter=128, num_experts=60, top_k=4)
    L = synth.make_layer(shape, 77, num_resident=39)
    e2s = L.expert_to_slot
    res = e2s >= 0
    assert res.sum() == 39
    assert sorted(e2s[res].tolist()) == list(range(39))
    assert np.all(np.isneginf(L.bias[~res])) and np.all(L.bias[res] == 0)
    pool = L.slot_experts()
    for e in np.nonzero(res)[0]:
        assert np.array_equal(pool.gate_q[e2s[e]], L.experts.gate_q[e])

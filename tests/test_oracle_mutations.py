"""Planted mistakes in the oracle (on the CPU) must each trip at least one pin.

Every mutant below is a plausible slip in restating the layer: a swapped
nibble order, a wrong sign convention, a wrong scale block, a renormalised
or mis-ordered top-k, a wrong activation, swapped operands, a dropped term.
"""
import numpy as np
import pytest

from oracle import moe_oracle as o
from tests import oracle_pins

_orig = {name: getattr(o, name) for name in dir(o) if callable(getattr(o, name))}


def _unpack_hi_first(packed):
    q = _orig["unpack_int4"](packed)
    out = q.copy()
    out[..., 0::2], out[..., 1::2] = q[..., 1::2], q[..., 0::2]
    return out


def _unpack_unsigned(packed):
    q = _orig["unpack_int4"](packed)
    return np.where(q < 0, q + 16, q)


def _unpack_sign_magnitude(packed):
    q = _orig["unpack_int4"](packed)
    n = np.where(q < 0, q + 16, q)
    return np.where(n >= 8, -(n - 8), n)


def _dequant_one_scale(q_packed, scale_bits):
    q = o.unpack_int4(q_packed).astype(np.float64)
    s = o.fp16_bits_to_f64(scale_bits)
    return q * s[..., :1]


def _dequant_block128(q_packed, scale_bits):
    q = o.unpack_int4(q_packed).astype(np.float64)
    s = o.fp16_bits_to_f64(scale_bits)
    idx = np.minimum(np.arange(q.shape[-1]) // 128, s.shape[-1] - 1)
    return q * s[..., idx]


def _route_renorm(x, rw, bias, k):
    logits, probs, ids, w = _orig["route"](x, rw, bias, k)
    return logits, probs, ids, w / w.sum(axis=-1, keepdims=True)


def _route_no_bias(x, rw, bias, k):
    return _orig["route"](x, rw, None, k)


def _topk_high_tie(logits, k):
    E = logits.shape[-1]
    order = np.argsort(-logits[:, ::-1], axis=-1, kind="stable")
    return (E - 1 - order)[:, :k]


def _topk_ascending(logits, k):
    return _orig["topk_ids"](logits, k)[:, ::-1]


def _softmax_no_shift_wrong(logits):
    z = np.exp(logits)
    return z / np.sum(z, axis=0, keepdims=True)      # normalised over tokens


def _ffn_swapped(x, wg, wu, wd):
    return _orig["expert_ffn"](x, wu, wg, wd)


def _ffn_sigmoid(x, wg, wu, wd):
    g = x @ wg.T
    return ((1 / (1 + np.exp(-g))) * (x @ wu.T)) @ wd.T


def _ffn_relu(x, wg, wu, wd):
    g = x @ wg.T
    return (np.maximum(g, 0) * (x @ wu.T)) @ wd.T


def _perm_unstable(ids, E):
    p = _orig["permutation"](ids, E)
    for e in range(E):
        a, b = p.offsets[e], p.offsets[e + 1]
        p.sorted_pairs[a:b] = p.sorted_pairs[a:b][::-1].copy()
    p.pair_to_row[p.sorted_pairs] = np.arange(p.sorted_pairs.size)
    return p


def _prenorm_over_tokens(x, eps=1e-6):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=0, keepdims=True) + eps)


def _near_tie_k_only(logits, k, gap=o.NEAR_TIE_GAP):
    s = -np.sort(-logits, axis=-1)
    return (s[:, k - 1] - s[:, k]) < gap


MUTANTS = {
    "nibble_hi_first": ("unpack_int4", _unpack_hi_first),
    "nibble_unsigned": ("unpack_int4", _unpack_unsigned),
    "nibble_sign_magnitude": ("unpack_int4", _unpack_sign_magnitude),
    "one_scale_per_row": ("dequantize", _dequant_one_scale),
    "scale_block_128": ("dequantize", _dequant_block128),
    "topk_renormalised": ("route", _route_renorm),
    "bias_dropped": ("route", _route_no_bias),
    "tie_to_higher_index": ("topk_ids", _topk_high_tie),
    "topk_ascending": ("topk_ids", _topk_ascending),
    "softmax_wrong_axis": ("softmax", _softmax_no_shift_wrong),
    "gate_up_swapped": ("expert_ffn", _ffn_swapped),
    "sigmoid_not_silu": ("expert_ffn", _ffn_sigmoid),
    "relu_not_silu": ("expert_ffn", _ffn_relu),
    "unstable_permutation": ("permutation", _perm_unstable),
    "prenorm_over_tokens": ("rms_prenorm", _prenorm_over_tokens),
    "near_tie_boundary_only": ("near_tie_flags", _near_tie_k_only),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(o, attr, fn)
    assert oracle_pins.failing_pins(o), f"mutant {name} passed every pin"


def test_unmutated_oracle_passes_everything():
    assert oracle_pins.failing_pins(o) == []

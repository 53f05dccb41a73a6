"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each pin is a plain function taking the oracle module and raising
AssertionError (or any exception) when the oracle disagrees.  The test files
run every pin against the real oracle (all must pass) and against oracles
with planted mistakes (each mistake must be caught by at least one pin).

Independent sources used here:
  * exhaustive byte tables written out by hand (format);
  * hand-worked closed forms (tests/golden/*.json);
  * a dense brute force written with different formulas: nibbles by integer
    division, signs by modular arithmetic, scales by np.repeat, top-k by a
    Python sort on (-logit, index), every expert evaluated for every token
    and masked;
  * closed forms and invariants of the definition.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ------------------------------------------------------------ hand builders

def _rows_bytes(n_rows, n_bytes, row0_byte=None, other_byte=0x00):
    a = np.full((n_rows, n_bytes), other_byte, np.uint8)
    if row0_byte is not None:
        a[0, :] = row0_byte
    return a


def example_expert(gate_row0_byte, up_row0_byte, down_byte0, H=256, I=64):
    """Canonical arrays of one hand-built expert (see tests/golden)."""
    gq = _rows_bytes(I, H // 2, gate_row0_byte)
    uq = _rows_bytes(I, H // 2, up_row0_byte)
    gs = np.full((I, math.ceil(H / 256)), 0x1C00, np.uint16)   # 2^-8
    us = gs.copy()
    dq = np.zeros((H, I // 2), np.uint8)
    dq[:, 0] = down_byte0
    ds = np.full((H, math.ceil(I / 256)), 0x3800, np.uint16)   # 0.5
    return gq, gs, uq, us, dq, ds


def stack_experts(*experts):
    return tuple(np.stack(parts) for parts in zip(*experts))


# ------------------------------------------------------------------ format

def pin_nibble_table(o):
    """All 256 bytes: low nibble = even index, two's complement."""
    signed = [0, 1, 2, 3, 4, 5, 6, 7, -8, -7, -6, -5, -4, -3, -2, -1]
    table = np.array([[signed[b & 15], signed[b >> 4]] for b in range(256)])
    got = o.unpack_int4(np.arange(256, dtype=np.uint8)[:, None])
    assert got.shape == (256, 2)
    assert np.array_equal(got, table)


def pin_pack_examples(o):
    assert o.pack_int4(np.array([1, -2]))[0] == 0xE1
    assert o.pack_int4(np.array([-8, 7]))[0] == 0x78
    assert o.pack_int4(np.array([0, -1]))[0] == 0xF0
    every = np.array([[a, b] for a in range(-8, 8) for b in range(-8, 8)])
    assert np.array_equal(o.unpack_int4(o.pack_int4(every)), every)
    assert np.array_equal(o.pack_int4(o.unpack_int4(np.arange(256, dtype=np.uint8)[:, None]))[:, 0],
                          np.arange(256))


def pin_block_scales(o):
    """K = 1408 (five full 256-blocks and one 128-wide block): with every
    int4 = +1 and scale 2^-b on block b, each weight equals 2^-(k // 256)."""
    K = 1408
    q = np.full((2, K // 2), 0x11, np.uint8)
    s = np.array([[0x3C00, 0x3800, 0x3400, 0x3000, 0x2C00, 0x2800]] * 2, np.uint16)  # 1, .5, ..., 1/32
    w = o.dequantize(q, s)
    assert w.shape == (2, K)
    expect = np.concatenate([np.full(256, 2.0 ** -b) for b in range(5)] + [np.full(128, 2.0 ** -5)])
    assert np.array_equal(w[0], expect) and np.array_equal(w[1], expect)
    assert w[0].sum() == 500.0
    # a single -8 at K index 600 (block 2) under scale 0.25
    q2 = np.zeros((1, K // 2), np.uint8)
    q2[0, 300] = 0x08
    w2 = o.dequantize(q2, s[:1])
    assert w2[0, 600] == -2.0 and np.count_nonzero(w2) == 1


# ---------------------------------------------------------- hand examples

def _run_example(o, experts, bias, k, H=256):
    E = experts[0].shape[0]
    x = np.ones((1, H), np.float16)
    rw = np.zeros((E, H), np.float16)
    return o.moe_layer(x, rw, bias, experts, k)


def pin_example_a(o):
    g = load_golden("example_a.json")
    ex = stack_experts(example_expert(0x11, 0x11, 0x02))
    r = _run_example(o, ex, None, 1)
    assert np.allclose(r.out, g["expected_out_every_h"], rtol=0, atol=1e-14)
    assert r.ids[0, 0] == 0 and r.weights[0, 0] == 1.0


def pin_example_b(o):
    g = load_golden("example_b.json")
    ex = stack_experts(example_expert(0xFF, 0x11, 0x02))
    r = _run_example(o, ex, None, 1)
    assert np.allclose(r.out, g["expected_out_every_h"], rtol=0, atol=1e-14)


def pin_example_c(o):
    g = load_golden("example_c.json")
    ex = stack_experts(example_expert(0x11, 0x11, 0x02), example_expert(0x11, 0x11, 0x0E))
    bias = np.array([0.0, np.log(3.0)], np.float32)
    r = _run_example(o, ex, bias, 2)
    assert list(r.ids[0]) == g["expected_ids"]
    assert np.allclose(r.weights[0], g["expected_weights"], rtol=0, atol=1e-7)
    assert np.allclose(r.out, g["expected_out_every_h"], rtol=0, atol=g["tolerance_abs"])
    # the weights are the softmax entries: they sum to 1 when k = E
    assert abs(r.weights.sum() - 1.0) < 1e-12


def pin_residual_prenorm(o):
    """RESIDUAL adds x; PRENORM feeds x / rms(x): with x = c (constant), rms = |c|
    (eps aside), so the expert sees ones and example A's output is unchanged."""
    g = load_golden("example_a.json")
    ex = stack_experts(example_expert(0x11, 0x11, 0x02))
    x = np.full((1, 256), 4.0, np.float16)
    rw = np.zeros((1, 256), np.float16)
    r = o.moe_layer(x, rw, None, ex, 1, flags=o.FLAG_RESIDUAL | o.FLAG_PRENORM)
    expect = 4.0 + g["expected_out_every_h"]
    assert np.allclose(r.out, expect, rtol=0, atol=1e-6)     # eps = 1e-6 shifts it by ~1e-7
    r2 = o.moe_layer(x, rw, None, ex, 1, flags=o.FLAG_RESIDUAL)
    # without PRENORM the expert sees 4s: g = u = 4, y = SiLU(4) * 4
    s4 = 4.0 / (1.0 + math.exp(-4.0)) * 4.0
    assert np.allclose(r2.out, 4.0 + s4, rtol=0, atol=1e-12)


def pin_overflow(o):
    """Example A with down q = +-7 at scale 65504 (0x7BFF, the largest finite
    FP16 value): y = +-7 * 65504 * SiLU(1) = +-335,208.6..., beyond FP16 range
    on both signs; example A itself (out = SiLU(1)) is flagged nowhere."""
    g = load_golden("example_a.json")
    for byte, sign in ((0x07, 1.0), (0x09, -1.0)):
        ex = list(stack_experts(example_expert(0x11, 0x11, byte)))
        ex[5] = np.full_like(ex[5], 0x7BFF)
        r = _run_example(o, tuple(ex), None, 1)
        assert np.allclose(r.out, sign * 7.0 * 65504.0 * g["expected_out_every_h"], rtol=1e-14, atol=0)
        assert r.overflow.shape == r.out.shape and r.overflow.all()
    ok = _run_example(o, stack_experts(example_expert(0x11, 0x11, 0x02)), None, 1)
    assert not ok.overflow.any()


# ------------------------------------------------------- routing specifics

def pin_router_rules(o):
    """Ties go to the lower index, ids are in descending logit order, -inf
    experts are never chosen and weigh 0, weights are unrenormalised."""
    logits = np.array([[1.0, 3.0, 3.0, 2.0, -np.inf],
                       [0.0, 0.0, 0.0, 0.0, 0.0]])
    ids = o.topk_ids(logits, 3)
    assert ids.tolist() == [[1, 2, 3], [0, 1, 2]]
    p = o.softmax(logits)
    assert p[0, 4] == 0.0
    e = np.exp([1.0, 3.0, 3.0, 2.0])
    assert np.allclose(p[0, :4], e / e.sum(), rtol=1e-15)
    assert np.allclose(p[1], 0.2, rtol=1e-15)
    # route(): weights equal the full-softmax probabilities of the chosen ids
    x = np.array([[1.0, 0.0], [0.0, 1.0]], np.float16)
    rw = np.array([[0.5, 0.0], [0.25, 0.0], [0.0, 0.75], [0.0, 0.125]], np.float16)
    logits2, probs, ids2, w = o.route(x, rw, np.array([0.0, 0.0, 0.0, 1.0], np.float32), 2)
    assert np.array_equal(logits2, [[0.5, 0.25, 0.0, 1.0], [0.0, 0.0, 0.75, 1.125]])
    assert ids2.tolist() == [[3, 0], [3, 2]]
    ex0 = np.exp([0.5, 0.25, 0.0, 1.0])
    assert np.allclose(w[0], [ex0[3] / ex0.sum(), ex0[0] / ex0.sum()], rtol=1e-15)
    assert (w.sum(axis=1) < 1.0).all()


def pin_near_tie(o):
    logits = np.array([[5.0, 4.0, 3.0, 2.0],
                       [5.0, 4.0, 4.00005, 1.0],     # tie at the k=2 boundary
                       [5.0, 5.00001, 1.0, 0.0],      # tie inside the top-2
                       [5.0, 4.0, 1.0, 0.99995]])     # tie below the k+1 window: not flagged
    assert o.near_tie_flags(logits, 2).tolist() == [False, True, True, False]


def pin_permutation(o):
    ids = np.array([[2, 0], [0, 3], [2, 3], [1, 0]])
    perm = o.permutation(ids, 5)
    assert perm.counts.tolist() == [3, 1, 2, 2, 0]
    assert perm.offsets.tolist() == [0, 3, 4, 6, 8, 8]
    # expert 0 gets pairs 1 (t0 j1), 2 (t1 j0), 7 (t3 j1); expert 1: 6; expert 2: 0, 4; expert 3: 3, 5
    assert perm.sorted_pairs.tolist() == [1, 2, 7, 6, 0, 4, 3, 5]
    assert np.array_equal(perm.pair_to_row[perm.sorted_pairs], np.arange(8))


# ------------------------------------------------------------ brute force

def _bf_unpack(packed):
    b = packed.astype(np.int64)
    lo, hi = b % 16, b // 16
    lo = (lo + 8) % 16 - 8
    hi = (hi + 8) % 16 - 8
    out = np.empty(packed.shape[:-1] + (2 * packed.shape[-1],), np.int64)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def _bf_dense(qp, sb):
    q = _bf_unpack(qp).astype(np.float64)
    K = q.shape[-1]
    s = sb.view(np.float16).astype(np.float64)
    return q * np.repeat(s, 256, axis=-1)[..., :K]


def brute_force_layer(x, router_w, bias, experts, k, residual=False, prenorm=False, expert_to_slot=None):
    gq, gs, uq, us, dq, ds = experts
    x = x.astype(np.float64)
    T, H = x.shape
    E = router_w.shape[0]
    xin = x
    if prenorm:
        xin = x / np.sqrt((x ** 2).sum(axis=1, keepdims=True) / H + 1e-6)
    logits = np.einsum("th,eh->te", xin, router_w.astype(np.float64))
    if bias is not None:
        logits = logits + bias.astype(np.float64)
    out = x.copy() if residual else np.zeros_like(x)
    for t in range(T):
        finite = np.isfinite(logits[t])
        m = logits[t][finite].max()
        den = sum(math.exp(l - m) for l in logits[t][finite])
        chosen = sorted(range(E), key=lambda e: (-logits[t, e], e))[:k]
        for e in range(E):
            slot = e if expert_to_slot is None else expert_to_slot[e]
            if slot < 0:
                continue
            Wg, Wu, Wd = _bf_dense(gq[slot], gs[slot]), _bf_dense(uq[slot], us[slot]), _bf_dense(dq[slot], ds[slot])
            gz = np.einsum("ih,h->i", Wg, xin[t])
            uz = np.einsum("ih,h->i", Wu, xin[t])
            hz = gz * (1.0 / (1.0 + np.exp(-gz))) * uz
            yz = np.einsum("hi,i->h", Wd, hz)
            mask = 1.0 if e in chosen else 0.0
            p = math.exp(logits[t, e] - m) / den if finite[e] else 0.0
            out[t] += mask * p * yz
    return out


def _small_random_layer(seed, H=256, I=128, E=6, k=2, T=5, bias=True):
    rng = np.random.default_rng(seed)
    experts = (rng.integers(0, 256, (E, I, H // 2), dtype=np.uint8),
               rng.uniform(0.002, 0.02, (E, I, H // 256)).astype(np.float16).view(np.uint16),
               rng.integers(0, 256, (E, I, H // 2), dtype=np.uint8),
               rng.uniform(0.002, 0.02, (E, I, H // 256)).astype(np.float16).view(np.uint16),
               rng.integers(0, 256, (E, H, I // 2), dtype=np.uint8),
               rng.uniform(0.002, 0.02, (E, H, math.ceil(I / 256))).astype(np.float16).view(np.uint16))
    x = (rng.standard_normal((T, H)) * 3).astype(np.float16)
    rw = (rng.standard_normal((E, H)) * 0.05).astype(np.float16)
    b = rng.standard_normal(E).astype(np.float32) if bias else None
    return x, rw, b, experts


def pin_brute_force(o):
    for seed, flags in ((1, 0), (2, 3), (3, 1)):
        x, rw, b, ex = _small_random_layer(seed)
        r = o.moe_layer(x, rw, b, ex, 2, flags=flags)
        ref = brute_force_layer(x, rw, b, ex, 2, residual=bool(flags & 1), prenorm=bool(flags & 2))
        err = np.abs(r.out - ref).max() / np.abs(ref).max()
        assert err < 1e-12, err


def pin_brute_force_slots(o):
    """A permuted slot table with an absent (masked) expert."""
    x, rw, b, ex = _small_random_layer(7, E=5, k=2, T=6)
    e2s = np.array([3, -1, 0, 2, 1])           # expert 1 absent
    slots = [None] * 4
    for e, s in enumerate(e2s):
        if s >= 0:
            slots[s] = e
    pool = tuple(a[slots] for a in ex)
    b = b.copy()
    b[1] = -np.inf
    r = o.moe_layer(x, rw, b, pool, 2, expert_to_slot=e2s)
    assert not (r.ids == 1).any()
    ref = brute_force_layer(x, rw, b, pool, 2, expert_to_slot=e2s)
    assert np.abs(r.out - ref).max() <= 1e-12 * np.abs(ref).max()


def pin_closed_forms(o):
    x, rw, b, ex = _small_random_layer(11)
    # x = 0 -> out = 0
    z = o.moe_layer(np.zeros_like(x), rw, b, ex, 2)
    assert np.all(z.out == 0.0)
    # k = E -> weights sum to 1 for every token
    r = o.moe_layer(x, rw, b, ex, ex[0].shape[0])
    assert np.allclose(r.weights.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    # E = 1 -> plain dense SwiGLU FFN on x
    one = tuple(a[:1] for a in ex)
    r1 = o.moe_layer(x, rw[:1], None, one, 1)
    Wg, Wu, Wd = _bf_dense(one[0][0], one[1][0]), _bf_dense(one[2][0], one[3][0]), _bf_dense(one[4][0], one[5][0])
    xf = x.astype(np.float64)
    gz = xf @ Wg.T
    dense = ((gz / (1 + np.exp(-gz))) * (xf @ Wu.T)) @ Wd.T
    assert np.abs(r1.out - dense).max() <= 1e-12 * np.abs(dense).max()
    # an expert biased to -inf is never selected
    b2 = np.zeros(ex[0].shape[0], np.float32)
    b2[[0, 3]] = -np.inf
    r2 = o.moe_layer(x, rw, b2, ex, 2)
    assert not np.isin(r2.ids, [0, 3]).any()
    # linearity in the down projection: doubling every down scale doubles out
    ex2 = list(ex)
    ex2[5] = (ex[5].view(np.float16) * np.float16(2)).view(np.uint16)
    r3 = o.moe_layer(x, rw, b, tuple(ex2), 2)
    r0 = o.moe_layer(x, rw, b, ex, 2)
    assert np.allclose(r3.out, 2 * r0.out, rtol=1e-13, atol=0)


def pin_invariants(o):
    x, rw, b, ex = _small_random_layer(5, E=8, k=3, T=9)
    r = o.moe_layer(x, rw, b, ex, 3)
    T, k = r.ids.shape
    for t in range(T):
        assert len(set(r.ids[t].tolist())) == k
        assert np.all(np.diff(r.logits[t, r.ids[t]]) <= 0)
    assert np.all(r.weights.sum(axis=1) <= 1.0 + 1e-15)
    p = o.softmax(r.logits)
    assert np.array_equal(r.weights, np.take_along_axis(p, r.ids, axis=1))
    perm = r.perm
    assert perm.offsets[-1] == T * k
    assert np.array_equal(np.diff(perm.offsets), np.bincount(r.ids.ravel(), minlength=8))
    assert np.array_equal(perm.pair_to_row[perm.sorted_pairs], np.arange(T * k))
    flat = r.ids.ravel()
    for e in range(8):
        grp = perm.sorted_pairs[perm.offsets[e]:perm.offsets[e + 1]]
        assert np.all(flat[grp] == e) and np.all(np.diff(grp) > 0)


ALL_PINS = [pin_nibble_table, pin_pack_examples, pin_block_scales, pin_example_a, pin_example_b,
            pin_example_c, pin_residual_prenorm, pin_router_rules, pin_near_tie, pin_permutation,
            pin_brute_force, pin_brute_force_slots, pin_closed_forms, pin_invariants, pin_overflow]


def failing_pins(o):
    bad = []
    for pin in ALL_PINS:
        try:
            pin(o)
        except Exception:   # noqa: BLE001 - any exception means the pin caught the oracle
            bad.append(pin.__name__)
    return bad

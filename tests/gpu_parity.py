"""Helpers for the GPU-vs-oracle parity tests (imported by -m gpu tests only)."""
from __future__ import annotations

import numpy as np

from oracle import moe_oracle
from w4a16_compact_expert_gb300 import moe_w4a16

# Acceptance bars of the layer output (float): normwise relative error and
# max-abs error relative to max |ref|, over tokens whose routing is not a
# near tie.  Router weights: absolute error.
TOL_NORM = 2e-3
TOL_MAX = 1e-2
TOL_W = 1e-5


def make_handle(layer, max_tokens, device=0):
    s = layer.shape
    m = moe_w4a16.MoELayer(s.hidden, s.inter, s.num_experts, s.top_k, num_slots=layer.num_slots,
                           max_tokens=max_tokens, device=device)
    m.pack_experts(0, *layer.slot_experts().arrays())
    m.set_slot_table(layer.expert_to_slot)
    return m


def to_dev(a):
    import torch
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def gpu_forward(m, layer, x, flags=0):
    import torch
    out, dbg = m.forward(to_dev(x), to_dev(layer.router_w), to_dev(layer.bias), flags, debug=True)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64), {k: v.cpu().numpy() for k, v in dbg.items()}


def oracle_layer(layer, x, flags=0):
    return moe_oracle.moe_layer(x, layer.router_w, layer.bias, layer.slot_experts().arrays(), layer.shape.top_k,
                                flags, expert_to_slot=layer.expert_to_slot)


def assert_routing(dbg, ids_ref, w_ref, flagged, E, perm_ref=None):
    keep = ~flagged
    ids = dbg["ids"]
    assert np.array_equal(ids[keep], ids_ref[keep]), "expert ids differ on unflagged tokens"
    assert np.abs(dbg["weights"][keep] - w_ref[keep]).max(initial=0) <= TOL_W
    own = moe_oracle.permutation(ids, E)   # permutation of the GPU's own ids: always bit-exact
    assert np.array_equal(dbg["offsets"], own.offsets)
    assert np.array_equal(dbg["sorted_pairs"], own.sorted_pairs)
    if perm_ref is not None and not flagged.any():
        assert np.array_equal(dbg["sorted_pairs"], perm_ref.sorted_pairs)


def assert_output(out, ref_out, keep):
    d = out[keep] - ref_out[keep]
    nref = np.linalg.norm(ref_out[keep])
    assert np.isfinite(out).all()
    assert np.linalg.norm(d) <= TOL_NORM * nref, (np.linalg.norm(d) / nref)
    assert np.abs(d).max(initial=0) <= TOL_MAX * np.abs(ref_out[keep]).max(initial=0)
    return float(np.linalg.norm(d) / max(nref, 1e-300))


def check_full(layer, x, flags=0, m=None, max_tokens=None):
    """Whole-layer parity on every token (sizes the oracle finishes in seconds)."""
    own = m is None
    if own:
        m = make_handle(layer, max_tokens or x.shape[0])
    try:
        out, dbg = gpu_forward(m, layer, x, flags)
        st, miss = m.get_status()
        assert st == moe_w4a16.OK and miss == 0, (st, miss)
    finally:
        if own:
            m.close()
    ref = oracle_layer(layer, x, flags)
    assert_routing(dbg, ref.ids, ref.weights, ref.near_tie, layer.shape.num_experts, ref.perm)
    return assert_output(out, ref.out, ~ref.near_tie), int(ref.near_tie.sum())


def check_sampled(layer, x, rows, flags=0, m=None):
    """Large-T parity: routing of every token against the oracle router, the
    layer output on the sampled token rows (each computed by the oracle on its own)."""
    own = m is None
    if own:
        m = make_handle(layer, x.shape[0])
    try:
        out, dbg = gpu_forward(m, layer, x, flags)
        st, miss = m.get_status()
        assert st == moe_w4a16.OK and miss == 0, (st, miss)
    finally:
        if own:
            m.close()
    k, E = layer.shape.top_k, layer.shape.num_experts
    xin = moe_oracle.rms_prenorm(x) if flags & moe_oracle.FLAG_PRENORM else x
    logits, probs, ids, w = moe_oracle.route(xin, layer.router_w, layer.bias, k)
    flagged = moe_oracle.near_tie_flags(logits, k)
    assert_routing(dbg, ids, w, flagged, E, moe_oracle.permutation(ids, E))
    rows = np.asarray(rows)
    ref = oracle_layer(layer, x[rows], flags)
    return assert_output(out[rows], ref.out, ~flagged[rows]), int(flagged.sum())

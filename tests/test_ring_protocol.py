"""Host-side model of the weight ring of the single-launch decode kernel.

The first half models the phase order (each CTA: a share of the gate/up
items, then a share of the down items).  The kernel's producer issues
entries in order into slot e % NS once the
slot's previous entry has been released; consumer groups take items
q, q + NG, ... in order (a gate/up item consumes two entries, a down item
one), and a down item may only start once every gate/up item of the CTA has
finished (the model's stand-in for the cross-CTA readiness counters: the
strongest dependency a down item can have).  A consumer first checks that
the slot holds its entry (the published sequence number), so it never waits
on a stale phase.  Random interleavings of these moves must always finish.

The second half models the interleaved order (gate/up and down items of all
active experts in one sequence, two ring entries per unit) with several
CTAs, each with its own ring: unit x belongs to CTA x % G, whose producer
issues its units in order and whose group q takes its units q, q + NG, ...
The real dependency holds: a down item of expert u waits for every gate/up
item of u, wherever it runs.
"""
import random

import pytest


def run_ring(m1, m2, ns, ng, seed):
    rnd = random.Random(seed)
    ne = 2 * m1 + m2
    seq = [-1] * ns
    released = set()
    issued = 0
    groups = [{"items": list(range(q, m1 + m2, ng)), "pos": 0, "sub": 0} for q in range(ng)]
    gate_up_done = 0
    for _ in range(100_000):
        moves = []
        if issued < ne and (issued - ns < 0 or (issued - ns) in released):
            moves.append(("produce",))
        for q, g in enumerate(groups):
            if g["pos"] >= len(g["items"]):
                continue
            i = g["items"][g["pos"]]
            if i < m1:
                e = 2 * i + g["sub"]
            else:
                if gate_up_done < m1:
                    continue
                e = 2 * m1 + (i - m1)
            if seq[e % ns] == e:
                moves.append(("consume", q, e))
        if not moves:
            return issued == ne and all(g["pos"] >= len(g["items"]) for g in groups)
        mv = rnd.choice(moves)
        if mv[0] == "produce":
            seq[issued % ns] = issued
            issued += 1
        else:
            _, q, e = mv
            g = groups[q]
            released.add(e)
            i = g["items"][g["pos"]]
            if i < m1 and g["sub"] == 0:
                g["sub"] = 1
            else:
                if i < m1:
                    gate_up_done += 1
                g["pos"] += 1
                g["sub"] = 0
    return False


@pytest.mark.parametrize("ng", [2, 3])
def test_ring_never_deadlocks(ng):
    for m1 in range(0, 9):
        for m2 in range(0, 7):
            for ns in range(1, 7):
                for seed in range(3):
                    assert run_ring(m1, m2, ns, ng, seed), (m1, m2, ns, ng, seed)


def test_stale_parity_is_possible_without_the_sequence_check():
    """Why the sequence check exists: with 2 slots and 3 groups, group 0 can reach
    entry 4 (slot 0, phase 2, parity 0) while slot 0 still holds entry 2, whose
    phase 1 is pending; a bare parity-0 wait would then see phase 0 (entry 0)
    as complete."""
    ns = 2
    e_wanted, e_held = 4, 2
    assert e_wanted % ns == e_held % ns
    assert (e_wanted // ns) % 2 == ((e_held // ns) - 1) % 2   # same parity as the last completed phase


# ---------------------------------------------------------------- unit order

def unit_order_lag(G, NG, t1, t2, lag_q=6):
    """Blocks of lag: the gate/up items of L - 1 experts span lag_q quarters
    of one step of the grid's groups."""
    return 1 + (lag_q * G * NG + 4 * t1 - 1) // (4 * t1)


def unit_at(U, L, t1, t2, x):
    """The kernel's closed form of the order (kind, expert, index)."""
    r1 = min(L, U) * t1
    if x < r1:
        return (0, x // t1, x % t1)
    x -= r1
    nmix, bs = max(U - L, 0), t1 + t2
    if x < nmix * bs:
        jj, r = divmod(x, bs)
        return (1, jj, r) if r < t2 else (0, L + jj, r - t2)
    x -= nmix * bs
    return (1, nmix + x // t2, x % t2)


def order_by_blocks(U, L, t1, t2):
    """The order written out from its definition: block j holds the down items
    of expert j - L, then the gate/up items of expert j."""
    out = []
    for j in range(U + L):
        if 0 <= j - L < U:
            out += [(1, j - L, i) for i in range(t2)]
        if j < U:
            out += [(0, j, i) for i in range(t1)]
    return out


@pytest.mark.parametrize("U,L,t1,t2", [(1, 1, 4, 4), (3, 1, 2, 3), (5, 2, 4, 2), (2, 6, 3, 5),
                                         (26, 5, 64, 64), (60, 4, 88, 64), (8, 12, 64, 64)])
def test_unit_order_closed_form_matches_blocks(U, L, t1, t2):
    ref = order_by_blocks(U, L, t1, t2)
    assert len(ref) == U * (t1 + t2)
    assert [unit_at(U, L, t1, t2, x) for x in range(len(ref))] == ref
    # every item exactly once; every down item after all gate/up items of its expert
    assert len(set(ref)) == len(ref)
    last_gu = {u: max(x for x, v in enumerate(ref) if v[:2] == (0, u)) for u in range(U)}
    for x, (d, u, _) in enumerate(ref):
        if d:
            assert x > last_gu[u]
            if u + L - 1 < U:   # the blocks between hold the gate/up items of L - 1 experts
                assert x - last_gu[u] >= (L - 1) * t1 + 1


@pytest.mark.parametrize("NG,U", [(3, 26), (2, 56), (6, 8)])
def test_unit_order_lag_covers_a_step(NG, U):
    # OLMoE-shaped decode on 152 CTAs: 64 + 64 items per expert.  Units at
    # positions < G NG start together; a down item sits at least 1.5 steps
    # of the grid's groups after the first gate/up item of its expert.
    G, t1, t2 = 152, 64, 64
    L = unit_order_lag(G, NG, t1, t2)
    ref = order_by_blocks(U, L, t1, t2)
    if L >= U:   # too few experts for the lag (one token): every gate/up item first
        assert all(d == 0 for d, _, _ in ref[:U * t1])
        return
    first_gu = {}
    for x, (d, u, _) in enumerate(ref):
        if not d:
            first_gu.setdefault(u, x)
        else:
            assert x - first_gu[u] >= 1.5 * G * NG


def run_grid(U, t1, t2, G, NG, NS, L, seed):
    rnd = random.Random(seed)
    order = order_by_blocks(U, L, t1, t2)
    ctas = []
    for b in range(G):
        units = order[b::G]
        ctas.append({"units": units, "seq": [-1] * NS, "released": set(), "issued": 0,
                     "groups": [{"js": list(range(q, len(units), NG)), "pos": 0, "sub": 0} for q in range(NG)]})
    done_gu = [0] * U
    for _ in range(400_000):
        moves = []
        for b, c in enumerate(ctas):
            i = c["issued"]
            if i < 2 * len(c["units"]) and (i - NS < 0 or (i - NS) in c["released"]):
                moves.append(("produce", b))
            for q, g in enumerate(c["groups"]):
                if g["pos"] >= len(g["js"]):
                    continue
                j = g["js"][g["pos"]]
                d, u, _ = c["units"][j]
                if d and done_gu[u] < t1:
                    continue
                e = 2 * j + g["sub"]
                if c["seq"][e % NS] == e:
                    moves.append(("consume", b, q, e))
        if not moves:
            return all(c["issued"] == 2 * len(c["units"]) and all(g["pos"] >= len(g["js"]) for g in c["groups"])
                       for c in ctas)
        mv = rnd.choice(moves)
        c = ctas[mv[1]]
        if mv[0] == "produce":
            c["seq"][c["issued"] % NS] = c["issued"]
            c["issued"] += 1
        else:
            _, b, q, e = mv
            g = c["groups"][q]
            c["released"].add(e)
            d, u, _ = c["units"][g["js"][g["pos"]]]
            if g["sub"] == 0:
                g["sub"] = 1
            else:
                if not d:
                    done_gu[u] += 1
                g["pos"] += 1
                g["sub"] = 0
    return False


@pytest.mark.parametrize("G,NG", [(1, 2), (2, 2), (3, 3), (4, 2)])
def test_grid_unit_order_never_deadlocks(G, NG):
    for U in (1, 2, 3, 5):
        for t1, t2 in ((1, 1), (2, 1), (2, 3)):
            for NS in (1, 2, 4):
                for L in (1, 2, unit_order_lag(G, NG, t1, t2)):
                    for seed in range(2):
                        assert run_grid(U, t1, t2, G, NG, NS, L, seed), (U, t1, t2, G, NG, NS, L, seed)

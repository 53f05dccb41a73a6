"""Host-side model of the weight ring of the single-launch decode kernel.

The kernel's producer issues entries in order into slot e % NS once the
slot's previous entry has been released; consumer groups take items
q, q + NG, ... in order (a gate/up item consumes two entries, a down item
one), and a down item may only start once every gate/up item of the CTA has
finished (the model's stand-in for the cross-CTA readiness counters: the
strongest dependency a down item can have).  A consumer first checks that
the slot holds its entry (the published sequence number), so it never waits
on a stale phase.  Random interleavings of these moves must always finish.
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

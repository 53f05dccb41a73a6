"""The expert cache's lifecycle on the host-only simulated transport (no GPU):
admission, canonical initial placement, hits and misses, LRU discard
eviction, lease-gated reuse of evicted rows, serialised generations, the two
failure modes and the byte counters."""
import pytest

from w4a16_compact_expert_gb300 import build_ext, moe_w4a16 as M


@pytest.fixture(scope="module", autouse=True)
def lib():
    build_ext.build()
    return M.load_library()


def make(E=8, S=6, spare=2, group=2, staging=1, initial=(0, 1, 2, 3), eb=1000):
    return M.ExpertCache.sim(E, S, expert_bytes=eb, staging_experts=staging, spare_slots=spare, max_group=group,
                             initial=initial)


@pytest.mark.parametrize("kw", [
    dict(spare=1, group=2),                 # spares cannot hold a group's misses
    dict(staging=0),                        # no staging
    dict(S=5, initial=(0, 1, 2, 3)),        # initial + spares exceed the pool
    dict(group=0),
    dict(group=9),                          # larger than E
    dict(initial=(0, 0)),                   # duplicate initial ids
    dict(initial=(0, 8)),                   # out of range
    dict(S=3, spare=2, group=2, initial=()),  # published rows cannot hold a group
])
def test_admission_rejects_insufficient_capacity(kw):
    with pytest.raises(M.MoEError) as ex:
        make(**kw)
    assert ex.value.status == M.ERR_INVALID_ARG


def test_canonical_initial_placement():
    c = make()
    assert [c.slot_of(e) for e in range(8)] == [0, 1, 2, 3, -1, -1, -1, -1]
    s = c.stats()
    assert s["generation"] == 1 and s["resident"] == 4 and s["free_spares"] == 2
    assert s["h2d_bytes"] == 4 * 1000 and s["d2h_bytes"] == 0
    c.close()


def test_all_hits_publish_nothing():
    c = make()
    lease = c.acquire([1, 3])
    s = c.stats()
    assert s["generation"] == 1 and s["hits"] == 2 and s["misses"] == 0 and s["transactions"] == 0
    c.release(lease)
    c.sim_complete(lease)
    assert c.stats()["active_leases"] == 0
    c.close()


def test_miss_takes_a_spare_row_and_evicts_lru():
    c = make()
    l1 = c.acquire([0, 1])          # experts 0, 1 used at tick 1; 2, 3 never used (tick 0)
    c.release(l1)
    c.sim_complete(l1)
    l2 = c.acquire([5])             # miss: lowest spare row 4; LRU victim among {2, 3} -> 2 (tie, lower id)
    assert c.slot_of(5) == 4
    assert c.slot_of(2) == -1 and c.slot_of(3) == 3
    s = c.stats()
    assert s["generation"] == 2 and s["misses"] == 1 and s["evictions"] == 1
    assert s["resident"] == 4 and s["h2d_bytes"] == 5 * 1000 and s["d2h_bytes"] == 0
    c.release(l2)
    c.sim_complete(l2)
    c.close()


def test_evicted_row_is_not_reused_while_an_older_lease_is_held():
    c = make(S=6, spare=2, group=2)
    old = c.acquire([0])                     # lease on generation 1, where expert 1 lives in row 1
    la = c.acquire([4, 5])                   # misses fill rows 4, 5; evicts 1, 2 (LRU, not in group)
    assert c.stats()["generation"] == 2
    c.release(la)
    c.sim_complete(la)
    assert c.stats()["free_spares"] == 0 and c.stats()["retiring"] == 2
    # a new miss needs a row: rows 1 and 2 must wait for the generation-1 lease
    with pytest.raises(M.MoEError) as ex:
        c.acquire([6])
    assert ex.value.status == M.ERR_TIMEOUT
    assert c.stats()["generation"] == 2 and c.slot_of(6) == -1     # previous generation kept
    c.release(old)
    with pytest.raises(M.MoEError):                                 # released but its event not complete
        c.acquire([6])
    c.sim_complete(old)
    lb = c.acquire([6])
    assert c.slot_of(6) in (1, 2) and c.stats()["generation"] == 3
    c.release(lb)
    c.sim_complete(lb)
    c.close()


def test_failure_before_publication_keeps_the_generation():
    c = make()
    c.sim_fail(1)
    with pytest.raises(M.MoEError) as ex:
        c.acquire([6, 7])
    assert ex.value.status == M.ERR_CUDA
    s = c.stats()
    assert s["generation"] == 1 and s["faulted"] == 0 and s["misses"] == 0
    assert [c.slot_of(e) for e in range(8)] == [0, 1, 2, 3, -1, -1, -1, -1]
    lease = c.acquire([6, 7])                # the next transaction succeeds
    assert c.stats()["generation"] == 2 and c.slot_of(6) >= 0 and c.slot_of(7) >= 0
    c.release(lease)
    c.sim_complete(lease)
    c.close()


def test_failure_at_publication_faults_the_cache():
    c = make()
    c.sim_fail(2)
    with pytest.raises(M.MoEError) as ex:
        c.acquire([6])
    assert ex.value.status == M.ERR_CUDA
    assert c.stats()["faulted"] == 1
    with pytest.raises(M.MoEError) as ex2:
        c.acquire([0])                       # even an all-hit acquire fails once faulted
    assert ex2.value.status == M.ERR_CUDA
    c.close()


def test_argument_errors():
    c = make()
    for ids in ([0, 0], [8], [-1], [0, 1, 2]):   # duplicate, out of range, negative, over max_group
        with pytest.raises(M.MoEError) as ex:
            c.acquire(ids)
        assert ex.value.status == M.ERR_INVALID_ARG
    lease = c.acquire([0])
    c.release(lease)
    with pytest.raises(M.MoEError):
        c.release(lease)                     # twice
    with pytest.raises(M.MoEError):
        c.release(12345)                     # unknown
    c.sim_complete(lease)
    c.close()


def test_many_transactions_keep_the_invariants():
    """Random groups: the published table stays a partial injection of
    experts into rows, resident <= slots - spares, every group is resident
    after its acquire, and the byte counters add up."""
    import random
    rnd = random.Random(5)
    E, S, spare, group = 16, 10, 4, 4
    c = make(E=E, S=S, spare=spare, group=group, staging=2, initial=tuple(range(6)), eb=7)
    held = []
    for it in range(300):
        ids = rnd.sample(range(E), rnd.randint(1, group))
        try:
            lease = c.acquire(ids)
        except M.MoEError as ex:
            assert ex.status == M.ERR_TIMEOUT
            for l in held:
                c.sim_complete(l)
            held.clear()
            lease = c.acquire(ids)
        slots = [c.slot_of(e) for e in range(E)]
        assert all(slots[e] >= 0 for e in ids)
        used = [s for s in slots if s >= 0]
        assert len(used) == len(set(used)) and all(0 <= s < S for s in used)
        st = c.stats()
        assert st["resident"] <= S - spare and st["d2h_bytes"] == 0
        assert st["h2d_bytes"] == 7 * (6 + st["misses"])
        c.release(lease)
        held.append(lease)
        if rnd.random() < 0.5:
            for l in held:
                c.sim_complete(l)
            held.clear()
    c.close()

"""Pins of the oracle's prefetch model (SeqMoE tags, HybriMoE priority), CPU only."""
import numpy as np
import pytest

from oracle.cache import EVICT_CORE, EVICT_LRU, EVICT_MRS, SlotPoolSim
from oracle.prefetch import PrefetchSim, pending_owner


@pytest.mark.parametrize("policy", [EVICT_CORE, EVICT_MRS, EVICT_LRU])
def test_without_prefetch_it_is_the_pinned_simulator(policy):
    """per_step = 0: identical tables, owners, tags, scores and counters to cache.SlotPoolSim."""
    rng = np.random.default_rng(policy)
    L, E, S, k = 3, 10, 8, 2
    a = SlotPoolSim(L, E, S, policy, window=4)
    b = PrefetchSim(L, E, S, policy, window=4, per_step=0)
    lut = np.full((L, E), -1, np.int32)
    lut[0, :3], lut[1, 3:6], lut[2, 1:3] = [0, 1, 2], [3, 4, 5], [6, 7]
    a.set_lut(lut)
    b.set_lut(lut)
    for step in range(60):
        l = step % L
        T = int(rng.integers(1, 4))
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
        p = rng.random((T, E)).astype(np.float32)
        sa, sb = a.update_scores(l, ids, p), b.update_scores(l, ids, p)
        a.plan(l, ids)
        b.plan(l, ids, sb)
        for n in ("lut", "owner", "tag", "score"):
            np.testing.assert_array_equal(getattr(a, n), getattr(b, n))
        assert (a.hits, a.misses, a.bypass, a.evictions) == (b.hits, b.misses, b.bypass, b.evictions)


def _two_layer_pool(per_step=1):
    sim = PrefetchSim(2, 4, 4, EVICT_LRU, window=4, per_step=per_step)
    lut = np.full((2, 4), -1, np.int32)
    lut[0, 0], lut[0, 1], lut[1, 0], lut[1, 1] = 0, 1, 2, 3
    sim.set_lut(lut)                   # every slot's tag is 1
    return sim


def _step(sim, l, e, s):
    ids = np.array([[e]])
    sc = sim.update_scores(l, ids, np.array([s], np.float32))
    return sim.plan(l, ids, sc)


def test_prefetch_lands_is_committed_and_then_hits():
    """Layer 0 needs expert 0 (a hit, no miss: budget 1).  The highest router score among the
    experts it neither needs nor holds is expert 2 (0.3 > 0.2): its prefetch takes the lowest-score
    slot of layer 0 that the step does not need (slot 1, expert 1 evicted), the slot turns pending
    with tag 2.  Once the host has written that tag back, the next plan (layer 1) commits it, and
    layer 0's next step finds expert 2 resident."""
    sim = _two_layer_pool()
    r = _step(sim, 0, 0, [0.4, 0.1, 0.3, 0.2])
    assert (r["hits"], r["misses"]) == (1, 0)
    assert sim.owner[1] == pending_owner(2) and sim.pf_expert[1] == 2 and sim.tag[1] == 2 and sim.lut[0, 1] == -1
    assert sim.lut[0, 2] == -1 and sim.pf_issued == 1 and sim.evictions == 1
    sim.drain()
    _step(sim, 1, 0, [0.4, 0.3, 0.2, 0.1])          # layer 1's plan commits layer 0's prefetch
    assert sim.lut[0, 2] == 1 and sim.owner[1] == 2 and sim.pf_committed == 1
    r = _step(sim, 0, 2, [0.1, 0.1, 0.7, 0.1])
    assert (r["hits"], r["misses"]) == (1, 0)


def test_a_wrong_tag_is_never_committed_and_demand_takes_the_slot():
    sim = _two_layer_pool()
    _step(sim, 0, 0, [0.4, 0.1, 0.3, 0.2])
    sim.corrupt(1)
    sim.drain()
    for _ in range(3):
        _step(sim, 1, 0, [0.4, 0.3, 0.2, 0.1])
    assert sim.owner[1] == pending_owner(2) and sim.lut[0, 2] == -1 and sim.pf_committed == 0
    r = _step(sim, 0, 2, [0.1, 0.1, 0.7, 0.1])     # demand: a miss, served into the pending slot
    assert r["misses"] == 1 and sim.lut[0, 2] == 1 and sim.owner[1] == 2 and sim.tag[1] == 3
    # evictions: expert 1 of layer 0 (its prefetch) and expert 1 of layer 1 (layer 1's own prefetch of
    # expert 2 on its first step; on later steps its only evictable slot is pending)
    assert sim.pf_demanded == 1 and sim.evictions == 2


def test_demand_before_the_copy_lands_is_a_miss_into_the_same_slot():
    sim = _two_layer_pool()
    _step(sim, 0, 0, [0.4, 0.1, 0.3, 0.2])
    r = _step(sim, 0, 2, [0.1, 0.1, 0.7, 0.1])     # no drain: the copy has not landed
    assert r["misses"] == 1 and sim.lut[0, 2] == 1 and sim.pf_demanded == 1
    sim.drain()                                     # the late write-back names tag 2; the slot has 3 now
    _step(sim, 1, 0, [0.4, 0.3, 0.2, 0.1])
    assert sim.owner[1] == 2 and sim.pf_committed == 0


def test_misses_use_the_budget():
    """A step with a miss and per_step = 1 issues no prefetch (the demand copy already takes the link)."""
    sim = _two_layer_pool()
    r = _step(sim, 0, 3, [0.1, 0.2, 0.3, 0.4])
    assert r["misses"] == 1 and sim.pf_issued == 0
    sim2 = _two_layer_pool(per_step=2)
    _step(sim2, 0, 3, [0.1, 0.2, 0.3, 0.4])
    assert sim2.pf_issued == 1 and sim2.pf_expert[sim2.pending[0]] == 2     # expert 2: the best remaining


def test_a_demanded_slot_is_not_a_victim_until_its_prefetch_has_landed():
    """Expert 2 is demanded before its prefetch landed (slot 1, tag 3 now, prefetch tag 2).  Until
    the host writes tag 2 back, slot 1 is not evictable, so layer 0's next miss takes slot 0."""
    sim = _two_layer_pool()
    _step(sim, 0, 0, [0.4, 0.1, 0.3, 0.2])
    _step(sim, 0, 2, [0.1, 0.1, 0.7, 0.1])          # demanded: slot 1 holds expert 2, copy in flight
    assert sim._busy(1)
    r = _step(sim, 0, 3, [0.1, 0.1, 0.1, 0.7])      # expert 3 misses; slot 1 (lower LRU score?) is busy
    assert r["misses"] == 1 and sim.lut[0, 3] == 0 and sim.lut[0, 2] == 1
    sim.drain()
    assert not sim._busy(1)

"""MoE-CORE offline cache shaping: hit-rate replay, nonuniform quotas and the profile fill.

The oracle (oracle/quota.py) is pinned by closed forms on hand-made traces; the
library's host implementation (moe_plan_quotas, moe_profile_lut) must then give
exactly the oracle's quotas, hit rates and tables on random traces under all
three eviction policies.  CPU only.
"""
import numpy as np
import pytest

import expert_offload_slot_gb300 as moe
from oracle import quota as oq
from oracle.cache import EVICT_CORE, EVICT_LRU, EVICT_MRS


def _cyclic(steps, experts, E):
    """One token per step selecting experts[step % len], uniform probabilities."""
    ids = np.array([[[experts[s % len(experts)]]] for s in range(steps)], np.int32)     # [steps, T=1, k=1]
    probs = np.full((steps, 1, E), 1.0 / E, np.float32)
    return ids, probs


def test_lru_cyclic_trace_closed_forms():
    """A cycle over 5 experts through an LRU cache: with K >= 5 every step hits (the profile fill,
    ties to the lower id, holds experts 0..4); with K = 4 the first 4 steps hit and every later step
    misses (each miss evicts the expert needed next).  K = 0 has hit rate 0."""
    E, steps = 6, 40
    ids, probs = _cyclic(steps, [0, 1, 2, 3, 4], E)
    for K, expect in ((5, 1.0), (6, 1.0), (4, 4 / steps), (0, 0.0)):
        h, hits, needed = oq.layer_hit_rate(ids, probs, E, K, EVICT_LRU, 16, 0.9, (0.25,) * 4)
        assert needed == steps
        assert h == expect, (K, h)


def test_profile_order_by_mean_probability_ties_lower_id():
    probs = np.zeros((3, 2, 4), np.float32)
    probs[..., 2] = 0.5
    probs[..., 0] = 0.25
    probs[..., 3] = 0.25          # ties with 0: the lower id first
    assert oq.profile_order(probs) == [2, 0, 3, 1]


def test_plan_moves_slots_from_a_saturated_layer_to_a_thrashing_one():
    """Layer 0 only ever needs expert 0 (hit rate 1 at any K >= 1); layer 1 cycles over 5 experts
    (LRU: 3/steps at K = 3, 1 at K = 5).  Budget 6, delta-K 2: the uniform 3/3 split moves one step
    to 1/5 (donor layer 0 loses nothing, layer 1 gains 1 - 3/steps); then layer 1 at K = 3 would fall
    below the median, so no donor is left and the plan stops."""
    E, steps = 6, 30
    ids0, p0 = _cyclic(steps, [0], E)
    ids1, p1 = _cyclic(steps, [0, 1, 2, 3, 4], E)
    ids = np.stack([ids0, ids1], axis=1)               # [steps, L, T, k]
    probs = np.stack([p0, p1], axis=1)
    K, h, moves = oq.plan_quotas(ids, probs, E, 6, 2, 0.1, EVICT_LRU)
    assert K.tolist() == [1, 5] and moves == 1
    assert h.tolist() == [1.0, 1.0]
    # the same trace with tau_low above the gap: no receiver, uniform split kept
    K2, _, moves2 = oq.plan_quotas(ids, probs, E, 6, 2, 0.99, EVICT_LRU)
    assert K2.tolist() == [3, 3] and moves2 == 0


def test_no_move_when_the_receiver_gains_less_than_the_donor_loses():
    """Two layers cycling over 4 and 5 experts: shrinking either one from K = 4 costs more than
    growing the other by one slot gains (LRU cyclic: all hits at K >= cycle, 4/steps below)."""
    E, steps = 8, 40
    ids0, p0 = _cyclic(steps, [0, 1, 2, 3], E)
    ids1, p1 = _cyclic(steps, [0, 1, 2, 3, 4], E)
    ids = np.stack([ids0, ids1], axis=1)
    probs = np.stack([p0, p1], axis=1)
    # h0(4) = 1, h0(3) = 3/40; h1(4) = 4/40, h1(5) = 1.  median = (1 + 0.1)/2; donor layer 0 would
    # fall to 0.075 < median: not a donor.  No move.
    K, h, moves = oq.plan_quotas(ids, probs, E, 8, 1, 0.05, EVICT_LRU)
    assert K.tolist() == [4, 4] and moves == 0
    assert h.tolist() == [1.0, 4 / steps]


def test_profile_lut_fills_each_quota_with_the_highest_mean_experts():
    rng = np.random.default_rng(3)
    probs = rng.random((5, 3, 2, 6)).astype(np.float32)
    lut = oq.profile_lut(probs, [2, 0, 3], 6)
    assert (lut >= 0).sum() == 5 and sorted(lut[lut >= 0].tolist()) == list(range(5))
    for l, q in enumerate([2, 0, 3]):
        order = oq.profile_order(probs[:, l])
        assert set(np.nonzero(lut[l] >= 0)[0].tolist()) == set(order[:q])


def _random_trace(rng, steps, L, T, E, k, zipf):
    """Biased, drifting routing: a per-layer Zipf preference plus noise, top-k of it."""
    rank = np.stack([rng.permutation(E) + 1 for _ in range(L)])
    bias = -zipf * np.log(rank.astype(np.float64))
    ids = np.empty((steps, L, T, k), np.int32)
    probs = np.empty((steps, L, T, E), np.float32)
    z = rng.standard_normal((L, T, E))
    for s in range(steps):
        z = 0.8 * z + 0.6 * rng.standard_normal((L, T, E))
        logits = (z + bias[:, None, :]).astype(np.float32)
        ex = np.exp(logits - logits.max(-1, keepdims=True))
        probs[s] = ex / ex.sum(-1, keepdims=True)
        ids[s] = np.argsort(-logits, axis=-1, kind="stable")[..., :k]
    return ids, probs


@pytest.mark.parametrize("policy", [EVICT_CORE, EVICT_MRS, EVICT_LRU])
def test_library_plan_equals_the_oracle(policy):
    rng = np.random.default_rng(10 + policy)
    L, E, k, T, steps = 4, 16, 2, 3, 30
    ids, probs = _random_trace(rng, steps, L, T, E, k, zipf=0.3)
    # layers differ in how concentrated their routing is: one layer with a much stronger preference
    ids2, probs2 = _random_trace(rng, steps, L, T, E, k, zipf=2.0)
    ids[:, 1], probs[:, 1] = ids2[:, 1], probs2[:, 1]
    budget, dk, tau = 20, 1, 0.02
    cfg = moe.make_config(L, E, k, 256, 128, budget, moe.MOE_F32, moe.MOE_F32, evict=policy, window=4)
    q_lib, h_lib = moe.moe_plan_quotas(cfg, ids, probs, budget, dk, tau)
    q_ref, h_ref, moves = oq.plan_quotas(ids, probs, E, budget, dk, tau, policy, 4, np.float32(0.9),
                                         tuple(np.float32(v) for v in (0.25,) * 4))
    np.testing.assert_array_equal(q_lib, q_ref)
    np.testing.assert_array_equal(h_lib, h_ref)
    assert q_lib.sum() == budget and moves > 0            # the trace is uneven enough to move slots
    lut_lib = moe.moe_profile_lut(cfg, probs, q_lib)
    np.testing.assert_array_equal(lut_lib, oq.profile_lut(probs, q_ref, E))


def test_library_rejects_bad_traces_and_quotas():
    cfg = moe.make_config(2, 8, 2, 256, 128, 6, moe.MOE_F32, moe.MOE_F32)
    ids = np.zeros((3, 2, 1, 2), np.int32)
    probs = np.full((3, 2, 1, 8), 0.125, np.float32)
    ids[1, 1, 0, 0] = 8                                 # out of range
    with pytest.raises(moe.MoeError):
        moe.moe_plan_quotas(cfg, ids, probs, 6, 1, 0.0)
    with pytest.raises(moe.MoeError):
        moe.moe_profile_lut(cfg, probs, [4, 4])         # 8 > num_slots

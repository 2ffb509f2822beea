"""Pins for the oracle's slot-pool simulator and permutation (CPU only)."""
import itertools
import os

import numpy as np
import pytest

from oracle.cache import EVICT_CORE, EVICT_LRU, EVICT_MRS, SlotPoolSim, permute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_trace():
    steps, expect = [], {}
    with open(os.path.join(GOLDEN, "evict_trace.txt")) as f:
        for ln in f:
            if ln.startswith("#") or not ln.strip():
                continue
            if ln.startswith("step"):
                probs, sel = ln.split(":", 1)[1].split(";")
                steps.append(([float(v) for v in probs.split()], int(sel)))
            elif ln.startswith("expect"):
                pol, rest = ln[len("expect "):].split(":", 1)
                toks = rest.split()
                expect[pol.strip()] = {toks[i]: float(toks[i + 1]) for i in range(0, len(toks), 2)}
    return steps, expect


@pytest.mark.parametrize("name,policy", [("lru", EVICT_LRU), ("mrs", EVICT_MRS), ("core", EVICT_CORE)])
def test_hand_trace_victims(name, policy):
    steps, expect = _read_trace()
    sim = SlotPoolSim(L=1, E=4, S=2, policy=policy, window=4, ema_decay=0.5)
    sim.set_lut(np.array([[0, 1, -1, -1]]))
    last = None
    for probs, sel in steps:
        ids = np.array([[sel]])
        sim.update_scores(0, ids, np.array([probs], np.float32))
        last = sim.plan(0, ids)
    ex = expect[name]
    assert sim.score[0, 0] == ex["score_e0"] and sim.score[0, 1] == ex["score_e1"]
    (e, slot, old), = last["events"]
    assert e == 3 and slot == int(ex["victim_slot"]) and old == int(ex["evicted_expert"])
    assert sim.lut[0, 3] == slot and sim.lut[0, old] == -1


def test_ema_and_count_closed_forms():
    lam = 0.9
    sim = SlotPoolSim(L=1, E=3, S=3, policy=EVICT_CORE, window=16, ema_decay=lam)
    p = np.array([[0.5, 0.25, 0.25]], np.float32)
    for n in range(1, 40):
        sim.update_scores(0, np.array([[0]]), p)
        assert abs(float(sim.ema[0, 0]) - (1 - lam ** n)) <= 1e-6 * n
        assert sim.hist_sel[0].sum(axis=0)[0] == min(n, 16)
        assert sim.ema[0, 1] == 0 and sim.last_sel[0, 0] == n - 1 and sim.last_sel[0, 1] == -1


def test_mrs_closed_forms():
    W = 16
    sim = SlotPoolSim(L=1, E=2, S=2, policy=EVICT_MRS, window=W)
    s = 0.3
    for n in range(1, 3 * W):
        sim.update_scores(0, np.array([[0]]), np.array([[s, 0.0]], np.float32))
        expect = (min(n, W) - 1) * np.float32(s)
        assert abs(float(sim.score[0, 0]) - expect) <= 1e-6 * W
    # an expert scored only at the latest step has MRS exactly 0 (HybriMoE "Mechanism")
    sim.update_scores(0, np.array([[1]]), np.array([[0.0, 0.9]], np.float32))
    assert sim.score[0, 1] == 0.0
    assert abs(float(sim.score[0, 0]) - (W - 1) * 0.3) < 1e-5


def test_lru_score_is_last_selection_step():
    sim = SlotPoolSim(L=1, E=4, S=2, policy=EVICT_LRU)
    for t, e in enumerate([2, 0, 2, 3]):
        sim.update_scores(0, np.array([[e]]), np.full((1, 4), 0.25, np.float32))
    assert list(sim.score[0]) == [1.0, -1.0, 2.0, 3.0]


def test_free_slots_first_then_lowest_score_with_tie_to_lowest_slot():
    sim = SlotPoolSim(L=1, E=6, S=4, policy=EVICT_LRU)
    sim.set_lut(np.array([[0, -1, 2, -1, -1, -1]]))       # slots 1, 3 free
    sim.update_scores(0, np.array([[1, 3]]), np.full((1, 6), 1 / 6, np.float32))
    r = sim.plan(0, np.array([[1, 3]]))
    assert [(e, s) for e, s, _ in r["events"]] == [(1, 1), (3, 3)]
    # all full now; experts 0 and 2 both last used never (-1): tie -> lowest slot (0)
    sim.update_scores(0, np.array([[4, 1]]), np.full((1, 6), 1 / 6, np.float32))
    r = sim.plan(0, np.array([[4, 1]]))
    assert r["events"] == [(4, 0, 0)] and r["hits"] == 1


def test_needed_experts_are_never_evicted_and_bypass_when_all_needed():
    sim = SlotPoolSim(L=1, E=8, S=2, policy=EVICT_MRS, window=4)
    sim.set_lut(np.array([[0, 1, -1, -1, -1, -1, -1, -1]]))
    ids = np.array([[0, 1], [2, 3]])
    sim.update_scores(0, ids, np.full((2, 8), 0.125, np.float32))
    r = sim.plan(0, ids)
    assert r["hits"] == 2 and r["misses"] == 2 and r["bypass"] == 2
    assert r["slot_of"] == {0: 0, 1: 1, 2: -1, 3: -1}
    assert list(sim.lut[0, :2]) == [0, 1]


def test_victim_from_other_layer_when_own_layer_exhausted():
    sim = SlotPoolSim(L=2, E=4, S=3, policy=EVICT_LRU)
    sim.set_lut(np.array([[0, 1, -1, -1], [2, -1, -1, -1]]))
    for l in range(2):
        sim.update_scores(l, np.array([[0]]), np.full((1, 4), 0.25, np.float32))
    ids = np.array([[0, 1, 2]])
    sim.update_scores(0, ids, np.full((1, 4), 0.25, np.float32))
    r = sim.plan(0, ids)
    # layer 0 needs 0, 1 (resident) and 2 (miss); its own slots are protected -> slot 2 of layer 1
    assert r["events"] == [(2, 2, 1 * 4 + 0)]
    assert sim.lut[1, 0] == -1 and sim.lut[0, 2] == 2


def test_table_stays_a_bijection_on_a_long_random_trace():
    rng = np.random.default_rng(0)
    L, E, S, k = 3, 16, 20, 4
    for policy in (EVICT_CORE, EVICT_MRS, EVICT_LRU):
        sim = SlotPoolSim(L, E, S, policy=policy, window=8)
        lut = np.full((L, E), -1, np.int32)
        perm = rng.permutation(L * E)[:S]
        for s, le in enumerate(perm):
            lut[le // E, le % E] = s
        sim.set_lut(lut)
        for step in range(200):
            for l in range(L):
                T = int(rng.integers(1, 5))
                z = rng.standard_normal((T, E))
                ids = np.argsort(-z, axis=1)[:, :k]
                p = np.exp(z) / np.exp(z).sum(1, keepdims=True)
                sim.update_scores(l, ids, p.astype(np.float32))
                r = sim.plan(l, ids)
                for e in r["U"]:
                    assert sim.lut[l, e] >= 0 or r["slot_of"][e] == -1
                occ = sim.owner[sim.owner >= 0]
                assert np.unique(occ).size == occ.size
                for s in range(S):
                    o = sim.owner[s]
                    if o >= 0:
                        assert sim.lut[o // E, o % E] == s
                assert (sim.lut >= 0).sum() == (sim.owner >= 0).sum()
        assert sim.hits + sim.misses > 0


def test_brute_force_lru_victims_small():
    """LRU victims against an independent brute force on every 3-step trace of E=4, S=2, top-1."""
    E, S = 4, 2
    for seq in itertools.product(range(E), repeat=3):
        sim = SlotPoolSim(L=1, E=E, S=S, policy=EVICT_LRU)
        sim.set_lut(np.array([[0, 1, -1, -1]]))
        resident = {0: 0, 1: 1}             # expert -> slot
        last = {e: -1 for e in range(E)}
        for t, e in enumerate(seq):
            sim.update_scores(0, np.array([[e]]), np.full((1, E), 0.25, np.float32))
            sim.plan(0, np.array([[e]]))
            last[e] = t
            if e not in resident:
                # evict the resident expert used least recently (ties: lower slot)
                cand = sorted(resident.items(), key=lambda kv: (last[kv[0]], kv[1]))
                old, slot = cand[0]
                del resident[old]
                resident[e] = slot
        for ex, slot in resident.items():
            assert sim.lut[0, ex] == slot, (seq, resident, sim.lut)


def test_permutation_properties_and_python_sorted():
    rng = np.random.default_rng(7)
    for T, k, E in ((1, 8, 128), (4, 2, 8), (16, 8, 128), (37, 3, 11), (0, 2, 4)):
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]) if T else np.zeros((0, k), np.int64)
        counts, offs, perm, inv = permute(ids, E)
        assert counts.sum() == T * k and offs[0] == 0 and offs[-1] == T * k
        assert np.all(np.diff(offs) == counts)
        assert sorted(perm.tolist()) == list(range(T * k))
        assert np.all(inv[perm] == np.arange(T * k))
        ref = [i for _, _, _, i in sorted((int(ids.reshape(-1)[i]), i // k, i % k, i) for i in range(T * k))]
        assert perm.tolist() == ref
        for e in range(E):
            rows = perm[offs[e]:offs[e + 1]]
            assert np.all(ids.reshape(-1)[rows] == e)
            assert np.all(np.diff(rows // k) > 0)          # stable: ascending tokens within an expert


def test_token_average_sums_tokens_in_ascending_order():
    """s_e(t) is the fp32 sum of the probabilities in ascending token order, / T.

    The values are chosen so that every other order gives another float32:
    1 followed by 99 copies of 2^-24 rounds back to 1 at every add (a tie to
    even), while the small values first sum exactly to 99 * 2^-24.
    """
    tiny = 2.0 ** -24
    T = 100
    # expert 0: the large value first; expert 1: the large value last;
    # expert 2: every token equal (exact in any order)
    p = np.zeros((T, 3), np.float32)
    p[:, 0] = tiny
    p[0, 0] = 1.0
    p[:, 1] = tiny
    p[T - 1, 1] = 1.0
    p[:, 2] = 0.5
    sim = SlotPoolSim(L=1, E=3, S=2, policy=EVICT_MRS, window=2)
    s = sim.update_scores(0, np.zeros((T, 1), np.int64), p)
    assert s[0] == np.float32(1.0) / np.float32(T)
    large_last = np.float32(99 * tiny) + np.float32(1.0)     # 99 * 2^-24 is exact in fp32
    assert large_last == np.float32(1.0 + 50 * 2.0 ** -23)   # 49.5 ulps rounds to even
    assert s[1] == large_last / np.float32(T)
    assert s[2] == np.float32(0.5)
    # a blocked or reversed order would change expert 0: 32-token blocks give
    # 1 + 68 * 2^-24 before the division
    assert np.float32(1.0) + np.float32(68 * tiny) != np.float32(1.0)


def test_token_average_short_steps_match_float64_mean():
    rng = np.random.default_rng(5)
    for T in (1, 7, 32, 33, 100):
        p = rng.random((T, 6)).astype(np.float32)
        sim = SlotPoolSim(L=1, E=6, S=2, policy=EVICT_MRS, window=2)
        s = sim.update_scores(0, np.zeros((T, 1), np.int64), p)
        np.testing.assert_allclose(s, p.astype(np.float64).mean(0), rtol=1e-5)

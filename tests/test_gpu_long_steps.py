"""Cache decisions of steps with more than 32 tokens, bit for bit against the oracle.

A multi-token step scores each expert by its token-averaged probability
(RapidMoE §4.3), summed in ascending token order; the history, the eviction
scores (MoE-CORE score, Minus Recent Score, LRU), the table, owners, tags and
the permutation of token rows (SeqMoE "Mechanism") must equal the oracle's
simulator after every step.  Covered here for the plan kernel with supplied
routing (dense tensor-core and gather expert paths), for decode calls with the
pool's own router, for staged prefill calls (MoE-CORE "Mechanism": history
updated, table untouched) and for moe_update_scores alone.
"""
import numpy as np
import pytest
import torch

import expert_offload_slot_gb300 as moe
from oracle.cache import EVICT_CORE, EVICT_LRU, EVICT_MRS, permute
from synth import gen, get_workload
from tests.gpu_harness import Rig, act_to_f64, check_output, check_routing, synthetic_routing, variant

pytestmark = pytest.mark.gpu

LONG_T = (33, 100, 300, 1024, 2048)
POLICIES = (EVICT_CORE, EVICT_MRS, EVICT_LRU)


def _wl(E=32, k=4, L=2, **kw):
    return variant(get_workload("qwen3_decode"), name=f"long_steps_E{E}", L=L, E=E, k=k, H=256, I=128,
                   zipf_s=0.5, **kw)


def _check_state(rig):
    st = rig.pool.state()
    np.testing.assert_array_equal(st["score"], rig.sim.score)
    np.testing.assert_array_equal(st["lut"], rig.sim.lut)
    np.testing.assert_array_equal(st["owner"], rig.sim.owner)
    np.testing.assert_array_equal(st["tag"], rig.sim.tag)


def _check_perm(g, ids, E):
    _, offs, perm, _ = permute(ids, E)
    np.testing.assert_array_equal(g["offs"], offs)
    np.testing.assert_array_equal(g["perm"], perm)


@pytest.mark.parametrize("policy", POLICIES)
@pytest.mark.parametrize("E,k", [(32, 4), (128, 8)])
def test_supplied_routing_long_steps(policy, E, k):
    """moe_forward_routed: the plan kernel at T > 32, then the dense (T <= 256) or gather expert path."""
    wl = _wl(E=E, k=k)
    S = E // 2
    rig = Rig(wl, S=S, lut=gen.initial_lut(wl, S=S), policy=policy, window=4, max_tokens=max(LONG_T))
    rng = np.random.default_rng(1000 + 10 * policy + E)
    try:
        for rep in range(2):
            for T in LONG_T:
                for l in range(wl.L):
                    ids, w, probs = synthetic_routing(rng, T, wl.E, wl.k)
                    xs = gen.store_act(wl, rng.standard_normal((T, wl.H)).astype(np.float32))
                    x = torch.from_numpy(xs.view(np.int16)).cuda()
                    out = torch.empty_like(x)
                    rig.pool.forward_routed(l, x, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(),
                                            torch.from_numpy(probs).cuda(), out)
                    rig.sim.update_scores(l, ids, probs)
                    plan = rig.sim.plan(l, ids)
                    _check_state(rig)
                    g = rig.pool.routing(max(LONG_T))
                    _check_perm(g, ids, wl.E)
                    np.testing.assert_array_equal(g["slots"], np.vectorize(plan["slot_of"].get)(ids))
                    if rep == 0 and l == 0 and T in (100, 2048):
                        sample = np.arange(0, T, max(1, T // 64))
                        ref = rig.oracle_routed(l, xs[sample], ids[sample], w[sample])
                        check_output(wl, act_to_f64(wl, out)[sample], ref)
        s = rig.pool.stats()
        assert (s["hits"], s["misses"], s["bypass"], s["evictions"]) == \
               (rig.sim.hits, rig.sim.misses, rig.sim.bypass, rig.sim.evictions)
        assert rig.sim.evictions > 0
        assert rig.pool.status() == moe.MOE_OK
    finally:
        rig.close()


@pytest.mark.parametrize("policy", POLICIES)
def test_own_router_decode_calls_long_steps(policy):
    """moe_forward(DECODE) at T > 32 (router, gate, plan kernel, experts): the oracle's simulator is
    replayed on the GPU's own routing, as the parity protocol's second tier says."""
    wl = _wl()
    S = 12
    rig = Rig(wl, S=S, lut=gen.initial_lut(wl, S=S), policy=policy, window=4, max_tokens=300)
    try:
        for T in (33, 100, 300, 64):
            for l in range(wl.L):
                xs = gen.store_act(wl, gen.prefill_hidden(wl, l, T))
                out = rig.forward(l, xs)
                g = rig.pool.routing(300)
                rig.sim.update_scores(l, g["ids"], g["probs"])
                plan = rig.sim.plan(l, g["ids"])
                _check_state(rig)
                _check_perm(g, g["ids"], wl.E)
                np.testing.assert_array_equal(g["slots"], np.vectorize(plan["slot_of"].get)(g["ids"]))
                ref, r = rig.oracle_forward(l, xs)
                ok = check_routing(g, r, wl.k)
                check_output(wl, out, ref, ok)
        assert rig.pool.status() == moe.MOE_OK
    finally:
        rig.close()


@pytest.mark.parametrize("policy", POLICIES)
def test_staged_prefill_long_steps(policy):
    """Staged prefill (whole layers from the staging regions): scores bit-exact, table, owners and
    tags untouched, permutation bit-exact, output against the oracle on sampled tokens."""
    wl = _wl(L=3)
    S = 20
    rig = Rig(wl, S=S, lut=gen.initial_lut(wl, S=S), policy=policy, window=4, max_tokens=2048, staging=2)
    try:
        for T in (100, 300, 1024, 2048):
            for l in range(wl.L):
                xs = gen.store_act(wl, gen.prefill_hidden(wl, l, T))
                out = rig.forward(l, xs, mode=moe.MOE_MODE_PREFILL_STAGED)
                g = rig.pool.routing(2048)
                assert np.all(g["slots"] == -2)
                rig.sim.update_scores(l, g["ids"], g["probs"])
                _check_state(rig)
                _check_perm(g, g["ids"], wl.E)
                if l == 1:
                    sample = np.arange(0, T, max(1, T // 48))
                    ref, r = rig.oracle_forward(l, xs[sample])
                    g_s = {n: g[n][sample] for n in ("ids", "w", "probs")}
                    ok = check_routing(g_s, r, wl.k)
                    check_output(wl, out[sample], ref, ok)
        s = rig.pool.stats()
        assert s["misses"] == 0 and s["staged_layers"] >= wl.L
        assert rig.pool.status() == moe.MOE_OK
    finally:
        rig.close()


def test_update_scores_alone_long_steps():
    wl = _wl(E=64, k=8)
    for policy in POLICIES:
        rig = Rig(wl, S=16, policy=policy, window=16, max_tokens=2048)
        rng = np.random.default_rng(21 + policy)
        try:
            for step, T in enumerate((33, 2048, 100, 1024, 300, 64, 2047)):
                l = step % 2
                ids, _, probs = synthetic_routing(rng, T, wl.E, wl.k)
                rig.pool.update_scores(l, torch.from_numpy(ids).cuda(), torch.from_numpy(probs).cuda())
                rig.sim.update_scores(l, ids, probs)
                np.testing.assert_array_equal(rig.pool.state()["score"], rig.sim.score)
            np.testing.assert_array_equal(rig.pool.state()["lut"], rig.lut0)
        finally:
            rig.close()

"""Approximate expert substitution (MoE-CORE "Mechanism"), opt-in, against the oracle.

The gate rewrites a token's low-score misses (not resident at the step's start,
logit within alpha of the rank-(k+1) boundary) into its best resident
unselected experts, keeping their weights.  Checked on every gate path (decode
layer kernel at one and four tokens, the warp gate after the tensor-core
router at 40 tokens): the rewritten routing equals oracle.aes on the oracle's
own routing and the same resident set (tokens at a near tie or within 1e-4 of
the alpha bound excluded: the two sides' logits round differently), the cache
decisions equal the oracle's simulator replayed on that routing, and the
output equals the oracle layer evaluated on it.
"""
import numpy as np
import pytest

import expert_offload_slot_gb300 as moe
from oracle import layer as olayer
from oracle.aes import aes_substitute, rank_order
from oracle.numerics import decode_act
from synth import gen, get_workload
from tests.gpu_harness import NEAR_TIE, Rig, check_output, variant

pytestmark = pytest.mark.gpu

ALPHA = np.float32(0.3)


@pytest.mark.parametrize("T", [1, 4, 40])
def test_aes_routing_cache_and_output_match_oracle(T):
    wl = variant(get_workload("qwen3_decode"), name="aes", L=2, E=32, k=4, H=512, I=256, zipf_s=0.5,
                 residency=0.3)
    rig = Rig(wl, max_tokens=64)
    rig.pool.set_aes(1, float(ALPHA))
    try:
        subs = 0
        for step in range(6):
            for l in range(wl.L):
                xs = gen.store_act(wl, gen.decode_hidden(wl, l, T, 6, base_seed=31)[step])
                resident = rig.sim.lut[l] >= 0                  # the table at the step's start
                out = rig.forward(l, xs)
                g = rig.pool.routing(64)
                x = decode_act(xs, wl.act_dtype)
                r = olayer.route(x, decode_act(rig.w_r[l], wl.act_dtype), rig.b[l], wl.k, wl.gating)
                ref_ids, n = aes_substitute(r["z"], r["ids"], resident, ALPHA)
                subs += n
                z32 = r["z"].astype(np.float32)
                ok = np.ones(T, bool)
                for t in range(T):
                    order = rank_order(z32[t])
                    bnd = z32[t, order[wl.k]]
                    edge = any(abs(float(z32[t, e] - bnd) - float(ALPHA)) < 1e-4 for e in order[:wl.k])
                    # the ranks that decide the rewrite: the top-k and the resident unselected ones it
                    # may draw on; the two sides' logits round differently, so near-equal ones are skipped
                    res_uns = [i for i in range(wl.k, wl.E) if resident[order[i]]][:wl.k + 1]
                    last = max([wl.k] + res_uns)
                    zz = z32[t, order[:last + 1]]
                    close = np.any(np.abs(np.diff(zz)) < 1e-4)
                    if r["gap"][t] < NEAR_TIE or edge or close:
                        ok[t] = False
                        continue
                    # same experts, and each keeps the weight of the position it took
                    assert sorted(g["ids"][t].tolist()) == sorted(ref_ids[t].tolist()), (step, l, t)
                    gw = dict(zip(g["ids"][t].tolist(), g["w"][t].tolist()))
                    for e, wv in zip(ref_ids[t].tolist(), r["w"][t].tolist()):
                        assert abs(gw[e] - wv) <= 1e-5, (step, l, t, e)
                rig.sim.update_scores(l, g["ids"], g["probs"])
                rig.sim.plan(l, g["ids"])
                st = rig.pool.state()
                for n_ in ("lut", "owner", "tag", "score"):
                    np.testing.assert_array_equal(st[n_], getattr(rig.sim, n_))
                ref = olayer.moe_layer(x, {"ids": g["ids"], "w": r["w"]}, lambda e: rig.mats(l, e), None)
                check_output(wl, out, ref, ok)
        s = rig.pool.stats()
        assert subs > 0 and s["aes_substitutions"] > 0
        assert rig.pool.status() == moe.MOE_OK
    finally:
        rig.close()


def test_aes_is_off_by_default_and_rejects_bad_alpha():
    wl = variant(get_workload("qwen3_decode"), name="aes_off", L=1, E=16, k=2, H=256, I=128, residency=0.25)
    rig = Rig(wl, max_tokens=8)
    try:
        for step in range(4):
            rig.forward(0, gen.store_act(wl, gen.decode_hidden(wl, 0, 4, 4)[step]))
        assert rig.pool.stats()["aes_substitutions"] == 0
        with pytest.raises(moe.MoeError):
            rig.pool.set_aes(1, -1.0)
        rig.pool.set_aes(0)
    finally:
        rig.close()

"""RapidMoE residual-split experts under UMIA (RapidMoE §4.3-4.4), on the GPU through the C ABI.

Each step's critical set is decided on the step's token-averaged router
probability; the oracle's simulator replays the GPU's own routing, so its
score s is bit-identical to the device's and the critical sets must agree
exactly.  The output must equal the oracle layer with every expert at the
precision UMIA chose (W^Q + W^R and W^H_down, or W^Q and W^L_down), within the
bf16 tolerance; decode calls and staged prefill calls (their own gamma).
"""
import numpy as np
import pytest

import expert_offload_slot_gb300 as moe
from oracle import layer as olayer
from oracle.numerics import decode_act
from oracle.resplit import resplit_mats, umia_critical
from synth import gen, get_workload
from synth.configs import RESPLIT_Q4R4
from tests.gpu_harness import Rig, check_output, check_routing, variant

pytestmark = pytest.mark.gpu

THETA, BETA, G_DEC, G_PRE = 0.06, (1.0, 0.6), 1.0, 0.8


def _wl(shared):
    return variant(get_workload("qwen3_decode"), name=f"resplit_{int(shared)}", L=2, E=16, k=4, H=512, I=256,
                   weight_dtype=RESPLIT_Q4R4, residency=0.5, zipf_s=0.7, shared=shared)


def _shared_mats(rig, l):
    if rig.shared_np is None:
        return None
    st = gen.record_to_stored(rig.wl, rig.shared_np[l * rig.rec:(l + 1) * rig.rec])
    return resplit_mats(st, rig.wl.I, True)


@pytest.mark.parametrize("shared", [False, True])
def test_resplit_umia_decode_and_staged_prefill(shared):
    wl = _wl(shared)
    rig = Rig(wl, max_tokens=64, staging=2)
    rig.pool.set_umia(THETA, BETA, G_DEC, G_PRE)
    try:
        crit_total = n_crit_lo = 0
        for mode, Ts, gamma in ((moe.MOE_MODE_DECODE, (1, 4, 40), G_DEC), (moe.MOE_MODE_PREFILL_STAGED, (64,), G_PRE)):
            for T in Ts:
                for step in range(3):
                    for l in range(wl.L):
                        xs = gen.store_act(wl, gen.decode_hidden(wl, l, T, 3, base_seed=17)[step])
                        out = rig.forward(l, xs, mode=mode)
                        g = rig.pool.routing(64)
                        s = rig.sim.update_scores(l, g["ids"], g["probs"])
                        if mode == moe.MOE_MODE_DECODE:
                            rig.sim.plan(l, g["ids"])
                        crit = umia_critical(s, THETA, BETA[l], gamma)
                        used = sorted(set(int(e) for e in g["ids"].reshape(-1)))
                        crit_total += sum(1 for e in used if crit[e]) + (1 if shared else 0)
                        n_crit_lo += sum(1 for e in used if not crit[e])
                        x = decode_act(xs, wl.act_dtype)
                        r = olayer.route(x, decode_act(rig.w_r[l], wl.act_dtype), rig.b[l], wl.k, wl.gating)
                        ok = check_routing(g, r, wl.k)
                        ref = olayer.moe_layer(x, {"ids": g["ids"], "w": g["w"]},
                                               lambda e: resplit_mats(rig.stored(l, e), wl.I, bool(crit[e])),
                                               _shared_mats(rig, l))
                        check_output(wl, out, ref, ok)
        st = rig.pool.stats()
        assert st["critical_entries"] == crit_total
        assert crit_total > 0 and n_crit_lo > 0            # both precisions were exercised
        assert st["misses"] > 0                             # copies beside the resident entries' gate/up
        assert rig.pool.status() == moe.MOE_OK
    finally:
        rig.close()


def test_resplit_precision_changes_the_output_as_the_codec_says():
    """All critical (theta 0) vs none critical (theta above every score): the two outputs differ, and
    the high-precision one is closer to the unquantized bf16 layer of the same drawn weights."""
    wl = _wl(False)
    rig = Rig(wl, max_tokens=8)
    try:
        xs = gen.store_act(wl, gen.decode_hidden(wl, 0, 4, 1, base_seed=5)[0])
        rig.pool.set_umia(0.0)
        hi = rig.forward(0, xs)
        rig.pool.set_umia(10.0)
        lo = rig.forward(0, xs)
        x = decode_act(xs, wl.act_dtype)
        r = olayer.route(x, decode_act(rig.w_r[0], wl.act_dtype), rig.b[0], wl.k, wl.gating)
        exact = olayer.moe_layer(x, r, lambda e: tuple(np.asarray(m, np.float64) for m in gen.expert_fp32(wl, 0, e)))
        assert not np.array_equal(hi, lo)
        assert np.abs(hi - exact).max() < np.abs(lo - exact).max()
    finally:
        rig.close()

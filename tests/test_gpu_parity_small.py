"""GPU parity on small cases: the CUDA path through the C ABI against the oracle.

Tiers (the parity protocol):
  1. routing: top-k sets bit-exact except near ties (oracle gap < 1e-4), weights
     and probabilities within fp32 rounding;
  2. cache decisions: bit-exact table/owner/tag/score when both sides get the
     same routing (moe_forward_routed with seeded synthetic ids and probs);
     with each side's own router, identical until a rounding-level near tie;
  3. output: max|out - ref| <= 1e-5 (fp32), 2e-2 (bf16), 5e-2 (fp8) * max|ref|.
"""
import numpy as np
import pytest
import torch

import expert_offload_slot_gb300 as moe
from oracle.cache import EVICT_CORE, EVICT_LRU, EVICT_MRS, permute
from synth import gen, get_workload
from synth.configs import BF16, F32, FP8_E4M3_B128, GATE_SIGMOID_RENORM
from tests.gpu_harness import Rig, check_output, check_routing, synthetic_routing, variant

pytestmark = pytest.mark.gpu


def _compare_cache(rig, l):
    st = rig.pool.state()
    sim = rig.sim
    np.testing.assert_allclose(st["score"][l], sim.score[l], rtol=1e-5, atol=1e-6)
    same = (np.array_equal(st["lut"], sim.lut) and np.array_equal(st["owner"], sim.owner)
            and np.array_equal(st["tag"], sim.tag))
    return same


def _run_trace(rig, steps, T, layers=None):
    """Returns (worst relative error, cache outcome).

    The outcome is "same" while GPU and oracle tables agree bit for bit after every
    step, "near_tie" once a token's top-k set differed at a near tie (the two
    sides then legitimately hold different tables), and "diverged" otherwise.
    """
    wl = rig.wl
    layers = range(wl.L) if layers is None else layers
    outcome = "same"
    worst = 0.0
    for l in layers:
        xs = gen.store_act(wl, gen.decode_hidden(wl, l, T, steps))
        for t in range(steps):
            out = rig.forward(l, xs[t])
            ref, r = rig.oracle_forward(l, xs[t])
            g = rig.pool.routing(T)
            ok = check_routing(g, r, wl.k)
            worst = max(worst, check_output(wl, out, ref, ok))
            if outcome == "same" and not ok.all():
                outcome = "near_tie"
            if outcome == "same":
                rig.sim.update_scores(l, r["ids"], r["probs"].astype(np.float32))
                rig.sim.plan(l, r["ids"])
                if not _compare_cache(rig, l):
                    outcome = "diverged"
    return worst, outcome


def test_tiny_workload_decode_trace():
    wl = get_workload("tiny")
    rig = Rig(wl)
    try:
        worst, outcome = _run_trace(rig, steps=wl.decode_steps, T=4)
        assert outcome == "same", outcome
        assert rig.pool.status() == moe.MOE_OK
        s = rig.pool.stats()
        assert s["steps"] == wl.decode_steps and s["hits"] + s["misses"] > 0
        assert (s["hits"], s["misses"], s["bypass"]) == (rig.sim.hits, rig.sim.misses, rig.sim.bypass)
    finally:
        rig.close()


@pytest.mark.parametrize("gating", [0, 1])
@pytest.mark.parametrize("policy", [EVICT_CORE, EVICT_MRS, EVICT_LRU])
def test_bf16_multilayer_trace(gating, policy):
    wl = variant(get_workload("qwen3_decode"), name="small_bf16", L=3, E=32, k=4, H=512, I=256,
                 residency=0.3, gating=gating, zipf_s=1.0)
    rig = Rig(wl, policy=policy, window=8)
    try:
        for T in (1, 3, 8):
            worst, outcome = _run_trace(rig, steps=6, T=T)
            assert outcome != "diverged"
        assert rig.pool.status() == moe.MOE_OK
    finally:
        rig.close()


_synthetic_routing = synthetic_routing


@pytest.mark.parametrize("policy", [EVICT_CORE, EVICT_MRS, EVICT_LRU])
@pytest.mark.parametrize("S,fill", [(12, True), (40, False), (5, True)])
def test_cache_decisions_bit_exact_with_shared_routing(policy, S, fill):
    """Same routing in -> identical table, owners, tags, scores, permutation and counters, every step."""
    wl = variant(get_workload("qwen3_decode"), name="routed_small", L=3, E=16, k=4, H=256, I=256, zipf_s=0.5)
    lut = gen.initial_lut(wl, S=S) if fill else np.full((wl.L, wl.E), -1, np.int32)
    rig = Rig(wl, S=S, lut=lut, policy=policy, window=4, ema=0.9)
    rng = np.random.default_rng(policy * 100 + S)
    try:
        for step in range(40):
            for l in range(wl.L):
                T = int(rng.choice([1, 2, 5, 9]))
                ids, w, probs = _synthetic_routing(rng, T, wl.E, wl.k)
                xs = gen.store_act(wl, rng.standard_normal((T, wl.H)).astype(np.float32))
                x = torch.from_numpy(xs.view(np.int16)).cuda()
                out = torch.empty_like(x)
                rig.pool.forward_routed(l, x, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(),
                                        torch.from_numpy(probs).cuda(), out)
                rig.sim.update_scores(l, ids, probs)
                plan = rig.sim.plan(l, ids)
                st = rig.pool.state()
                np.testing.assert_array_equal(st["score"], rig.sim.score)
                np.testing.assert_array_equal(st["lut"], rig.sim.lut)
                np.testing.assert_array_equal(st["owner"], rig.sim.owner)
                np.testing.assert_array_equal(st["tag"], rig.sim.tag)
                g = rig.pool.routing(T)
                counts, offs, perm, inv = permute(ids, wl.E)
                np.testing.assert_array_equal(g["offs"], offs)
                np.testing.assert_array_equal(g["perm"], perm)
                exp_slots = np.array([[plan["slot_of"][int(e)] for e in row] for row in ids])
                np.testing.assert_array_equal(g["slots"], exp_slots)
                if step % 10 == 0:
                    ref = rig.oracle_routed(l, xs, ids, w)
                    from tests.gpu_harness import act_to_f64
                    check_output(wl, act_to_f64(wl, out), ref)
        s = rig.pool.stats()
        assert (s["hits"], s["misses"], s["bypass"], s["evictions"]) == \
               (rig.sim.hits, rig.sim.misses, rig.sim.bypass, rig.sim.evictions)
        assert s["bytes_copied"] == rig.sim.misses * rig.rec      # slot fills + one-step copies
        assert rig.pool.status() == moe.MOE_OK
    finally:
        rig.close()


def test_update_scores_alone_matches_oracle():
    wl = variant(get_workload("qwen3_decode"), name="scores_only", L=2, E=64, k=8, H=256, I=256)
    for policy in (EVICT_CORE, EVICT_MRS, EVICT_LRU):
        rig = Rig(wl, S=16, policy=policy, window=16)
        rng = np.random.default_rng(11)
        try:
            for step in range(30):
                l = step % 2
                ids, w, probs = _synthetic_routing(rng, 16, wl.E, wl.k)
                rig.pool.update_scores(l, torch.from_numpy(ids).cuda(), torch.from_numpy(probs).cuda())
                rig.sim.update_scores(l, ids, probs)
            np.testing.assert_array_equal(rig.pool.state()["score"], rig.sim.score)
            np.testing.assert_array_equal(rig.pool.state()["lut"], rig.lut0)
        finally:
            rig.close()


def test_fp8_block_scaled_with_shared_expert():
    wl = variant(get_workload("dsv3"), name="small_fp8", L=2, E=32, k=4, H=512, I=256, residency=0.4)
    assert wl.weight_dtype == FP8_E4M3_B128 and wl.shared and wl.gating == GATE_SIGMOID_RENORM
    rig = Rig(wl)
    try:
        worst, outcome = _run_trace(rig, steps=4, T=5)
        assert outcome != "diverged"
    finally:
        rig.close()


@pytest.mark.parametrize("T", [1, 17, 257, 600])
def test_bf16_dense_and_gather_paths_with_shared_expert(T):
    """T = 1 takes the CUDA-core streaming path, T <= 256 the dense tensor-core path, larger T the
    expert-grouped (gather) path; I = 320 leaves the last 128-row tile of I partly padding."""
    wl = variant(get_workload("qwen3_decode"), name="gather_bf16", L=2, E=32, k=4, H=512, I=320,
                 residency=0.5, shared=True, zipf_s=0.5)
    rig = Rig(wl, max_tokens=640)
    try:
        for l in range(wl.L):
            xs = gen.store_act(wl, gen.prefill_hidden(wl, l, T))
            out = rig.forward(l, xs)
            ref, r = rig.oracle_forward(l, xs)
            ok = check_routing(rig.pool.routing(640), r, wl.k)
            check_output(wl, out, ref, ok)
        assert rig.pool.status() == moe.MOE_OK
    finally:
        rig.close()


@pytest.mark.parametrize("T", [24, 300])
def test_fp8_dense_and_gather_paths_with_shared_expert(T):
    """fp8 e4m3 with 128x128 block scales on the tensor cores: T <= 256 on the dense path,
    larger T on the gather path; the shared expert is streamed by every call."""
    wl = variant(get_workload("dsv3"), name="gather_fp8", L=2, E=32, k=4, H=512, I=256, residency=0.5)
    assert wl.weight_dtype == FP8_E4M3_B128 and wl.shared
    rig = Rig(wl, max_tokens=320)
    try:
        for l in range(wl.L):
            xs = gen.store_act(wl, gen.prefill_hidden(wl, l, T))
            out = rig.forward(l, xs)
            ref, r = rig.oracle_forward(l, xs)
            ok = check_routing(rig.pool.routing(320), r, wl.k)
            check_output(wl, out, ref, ok)
        assert rig.pool.status() == moe.MOE_OK
    finally:
        rig.close()


@pytest.mark.parametrize("wname,I", [("qwen3_decode", 320), ("dsv3", 256)])
def test_gather_path_with_256_row_token_tiles(wname, I):
    """Few experts and many tokens (routed rows average >= 192 per expert): the gather path's token
    tiles are 256 rows, one weight tile serving every row of a tile; experts whose rows are not a
    multiple of 256 end in a ragged tile, and the shared expert's T rows span three tiles."""
    wl = variant(get_workload(wname), name="gather256_" + wname, L=2, E=4, k=2, H=512, I=I, residency=0.5,
                 shared=True, zipf_s=0.5)
    rig = Rig(wl, max_tokens=640)
    try:
        for l in range(wl.L):
            xs = gen.store_act(wl, gen.prefill_hidden(wl, l, 600))
            out = rig.forward(l, xs)
            ref, r = rig.oracle_forward(l, xs)
            ok = check_routing(rig.pool.routing(640), r, wl.k)
            check_output(wl, out, ref, ok)
        assert rig.pool.status() == moe.MOE_OK
    finally:
        rig.close()


@pytest.mark.parametrize("wname", ["qwen3_decode", "dsv3"])
def test_pool_from_library_packed_records_matches_oracle(wname):
    """A caller with plain row-major weights packs its host pool with moe_pack_expert_record; the
    oracle gets the row-major matrices themselves (no record parsing on its side)."""
    from oracle import layer as olayer
    from oracle.numerics import decode_act
    from tests.gpu_harness import act_to_f64, to_device_act
    wl = variant(get_workload(wname), name=f"packed_{wname}", L=2, E=16, k=4, H=256 if wname != "dsv3" else 512,
                 I=192 if wname != "dsv3" else 256, residency=0.5, shared=False)
    cfg = moe.make_config(wl.L, wl.E, wl.k, wl.H, wl.I, wl.S, wl.weight_dtype, wl.act_dtype, wl.gating, False,
                          wl.evict, wl.window, 0.9, (0.25,) * 4, 0, 16)
    rec = moe.moe_expert_layout(cfg)[4]
    host = moe.HostPool(wl.L * wl.E * rec)
    stored = {}
    I = wl.I
    for l in range(wl.L):
        for e in range(wl.E):
            st = gen.expert_stored(wl, l, e)
            stored[l, e] = st
            kw = {}
            if "s13" in st:
                kw = dict(s_gate=st["s13"][:I // 128], s_up=st["s13"][I // 128:], s_down=st["s2"])
            off = (l * wl.E + e) * rec
            host.numpy()[off:off + rec] = moe.moe_pack_expert_record(cfg, st["w13"][:I], st["w13"][I:], st["w2"],
                                                                     **kw)
    w_r, b = gen.routers(wl)
    wr_dev = torch.from_numpy(np.ascontiguousarray(w_r.view(np.int16))).cuda()
    b_dev = torch.from_numpy(b).cuda()
    pool = moe.Pool(cfg, host.ptr, host.nbytes, wr_dev, b_dev)
    try:
        pool.set_lut(gen.initial_lut(wl))
        for T in (1, 4, 16):
            for l in range(wl.L):
                xs = gen.store_act(wl, gen.decode_hidden(wl, l, T, 1)[0])
                x = to_device_act(wl, xs)
                out = torch.empty_like(x)
                pool.forward(l, x, out)
                torch.cuda.synchronize()
                xf = decode_act(xs, wl.act_dtype)
                r = olayer.route(xf, decode_act(w_r[l], wl.act_dtype), b[l], wl.k, wl.gating)
                ref = olayer.moe_layer(xf, r, lambda e: olayer.expert_mats(stored[l, e], wl.weight_dtype, I), None)
                ok = check_routing(pool.routing(16), r, wl.k)
                check_output(wl, act_to_f64(wl, out), ref, ok)
        assert pool.status() == moe.MOE_OK and pool.stats()["misses"] > 0
    finally:
        pool.close()
        host.free()

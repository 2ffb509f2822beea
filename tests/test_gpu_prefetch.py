"""Asynchronous prefetch with per-slot tags (SeqMoE "Mechanism"), on the GPU through the C ABI.

* Deterministic: the host thread is drained after every call (every request has
  landed and its tag is written back before the next call), so the table,
  owners, tags, scores and the prefetch counters must equal the oracle's
  simulator (oracle/prefetch.py) bit for bit, on the decode layer kernel
  (one and four tokens) and on the plan kernel (caller routing).
* Wrong tags: the thread writes back wrong tags; no prefetched slot is ever
  committed, and the state still equals the simulator's.
* Asynchronous: steps replayed from a CUDA graph while the thread copies in the
  background; outputs are bit-identical to a pool without prefetch (the output
  never depends on which experts are resident), and afterwards every owned slot
  holds its owner's host record.
"""
import numpy as np
import pytest
import torch

import expert_offload_slot_gb300 as moe
from oracle.cache import EVICT_CORE, EVICT_LRU, EVICT_MRS
from oracle.prefetch import PrefetchSim
from synth import gen, get_workload
from tests.gpu_harness import Rig, act_to_f64, check_output, check_routing, synthetic_routing, variant

pytestmark = pytest.mark.gpu


def _wl(**kw):
    return variant(get_workload("qwen3_decode"), name="prefetch", L=3, E=16, k=2, H=512, I=256, zipf_s=0.7, **kw)


def _rig(wl, S, policy, per_step, max_tokens=16):
    rig = Rig(wl, S=S, policy=policy, window=4, max_tokens=max_tokens)
    rig.sim = PrefetchSim(wl.L, wl.E, S, policy, 4, 0.9, (0.25,) * 4, per_step=per_step)
    rig.sim.set_lut(rig.lut0)
    rig.pool.prefetch_enable(per_step)
    return rig


def _check(rig):
    st = rig.pool.state()
    sim = rig.sim
    np.testing.assert_array_equal(st["lut"], sim.lut)
    np.testing.assert_array_equal(st["owner"], sim.owner)
    np.testing.assert_array_equal(st["tag"], sim.tag)
    np.testing.assert_array_equal(st["score"], sim.score)
    s = rig.pool.stats()
    assert (s["hits"], s["misses"], s["evictions"]) == (sim.hits, sim.misses, sim.evictions)
    assert (s["prefetch_issued"], s["prefetch_committed"], s["prefetch_demanded"]) == \
           (sim.pf_issued, sim.pf_committed, sim.pf_demanded)


@pytest.mark.parametrize("policy", [EVICT_CORE, EVICT_MRS, EVICT_LRU])
def test_prefetch_state_matches_oracle_when_drained(policy):
    wl = _wl()
    rig = _rig(wl, S=12, policy=policy, per_step=2)
    rng = np.random.default_rng(40 + policy)
    try:
        for T in (1, 4):
            xs = [gen.store_act(wl, gen.decode_hidden(wl, l, T, 8, base_seed=5 + T)) for l in range(wl.L)]
            for step in range(8):
                for l in range(wl.L):
                    out = rig.forward(l, xs[l][step])
                    rig.pool.prefetch_drain()
                    g = rig.pool.routing(16)
                    sc = rig.sim.update_scores(l, g["ids"], g["probs"])
                    rig.sim.plan(l, g["ids"], sc)
                    rig.sim.drain()
                    _check(rig)
                    if step == 7:
                        ref, r = rig.oracle_forward(l, xs[l][step])
                        check_output(wl, out, ref, check_routing(g, r, wl.k))
        # caller routing: the plan kernel
        for step in range(10):
            for l in range(wl.L):
                T = int(rng.choice([3, 9]))
                ids, w, probs = synthetic_routing(rng, T, wl.E, wl.k)
                x = torch.from_numpy(gen.store_act(wl, rng.standard_normal((T, wl.H)).astype(np.float32))
                                     .view(np.int16)).cuda()
                out = torch.empty_like(x)
                rig.pool.forward_routed(l, x, torch.from_numpy(ids).cuda(), torch.from_numpy(w).cuda(),
                                        torch.from_numpy(probs).cuda(), out)
                rig.pool.prefetch_drain()
                sc = rig.sim.update_scores(l, ids, probs)
                rig.sim.plan(l, ids, sc)
                rig.sim.drain()
                _check(rig)
        assert rig.sim.pf_issued > 0 and rig.sim.pf_committed > 0
        assert rig.pool.status() == moe.MOE_OK
    finally:
        rig.close()


def test_wrong_tags_are_never_committed():
    wl = _wl()
    rig = _rig(wl, S=12, policy=EVICT_MRS, per_step=2)
    try:
        rig.pool.prefetch_inject_wrong_tags(1 << 20)
        rig.sim.corrupt(1 << 20)
        xs = [gen.store_act(wl, gen.decode_hidden(wl, l, 4, 10, base_seed=77)) for l in range(wl.L)]
        for step in range(10):
            for l in range(wl.L):
                rig.forward(l, xs[l][step])
                rig.pool.prefetch_drain()
                g = rig.pool.routing(16)
                sc = rig.sim.update_scores(l, g["ids"], g["probs"])
                rig.sim.plan(l, g["ids"], sc)
                rig.sim.drain()
                _check(rig)
        s = rig.pool.stats()
        assert s["prefetch_issued"] > 0 and s["prefetch_committed"] == 0
        assert rig.pool.status() == moe.MOE_OK
    finally:
        rig.close()


@pytest.mark.parametrize("T", [1, 16])
def test_async_prefetch_in_graph_replay_keeps_outputs_and_slots(T):
    wl = variant(get_workload("qwen3_decode"), name="prefetch_async", L=4, E=64, k=8, H=1024, I=512, zipf_s=1.0)
    S = int(0.45 * wl.L * wl.E)
    rigs = [Rig(wl, S=S, max_tokens=16), Rig(wl, S=S, max_tokens=16)]
    rigs[1].pool.prefetch_enable(1)
    try:
        steps = 12
        xs = gen.torch_decode_hidden(wl, T, steps, "cuda", base_seed=3)
        outs = []
        for rig in rigs:
            torch.cuda.synchronize()
            s = torch.cuda.Stream()
            x_in = torch.empty_like(xs[0])
            out = torch.empty_like(x_in)
            with torch.cuda.stream(s):
                x_in.copy_(xs[0])
                for l in range(wl.L):
                    rig.pool.forward(l, x_in[l], out[l], moe.MOE_MODE_DECODE)
            s.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                for l in range(wl.L):
                    rig.pool.forward(l, x_in[l], out[l], moe.MOE_MODE_DECODE)
            res = []
            for i in range(1, steps):
                with torch.cuda.stream(s):
                    x_in.copy_(xs[i])
                    g.replay()
                    res.append(out.clone())
            s.synchronize()
            del g
            outs.append(torch.stack(res).cpu())
        assert torch.equal(outs[0], outs[1])
        p = rigs[1].pool
        p.prefetch_drain()
        st = p.state()
        host = rigs[1].host.numpy()
        rec = rigs[1].rec
        for slot in range(S):
            o = int(st["owner"][slot])
            if o >= 0:
                assert np.array_equal(p.read_slot(slot), host[o * rec:(o + 1) * rec]), (slot, o)
        s = p.stats()
        assert s["prefetch_issued"] > 0 and s["prefetch_bytes"] == s["prefetch_issued"] * rec
        assert p.status() == moe.MOE_OK and rigs[0].pool.status() == moe.MOE_OK
    finally:
        for rig in rigs:
            rig.close()


def test_prefetch_arguments_and_load_slot_refusal():
    wl = _wl()
    rig = _rig(wl, S=12, policy=EVICT_LRU, per_step=1)
    try:
        with pytest.raises(moe.MoeError):
            rig.pool.prefetch_enable(9)
        with pytest.raises(moe.MoeError):
            rig.pool.load_slot(0, 1, 0)
        rig.pool.prefetch_enable(0)
        rig.pool.prefetch_drain()
    finally:
        rig.close()

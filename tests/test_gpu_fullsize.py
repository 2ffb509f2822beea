"""Full-size parity of the Qwen3-30B-A3B-shaped decode in the benchmark's launch configuration.

48 layers, 128 experts, top-8, hidden 2048, intermediate 768, bf16, a pool of
round(0.45 * 48 * 128) = 2765 slots, T = 16 tokens per step (and the
benchmark's other decode batches, 1 and 4 tokens: the one-token streaming FFN
and the four-token tensor-core FFN); the 48 moe_forward calls of a step are
captured in one CUDA graph and replayed.

* Outputs: sampled layers of the last replayed step against the oracle layer
  function evaluated on the same stored bytes (tokens at an oracle near tie,
  gap < 1e-4, excluded: their expert set may legitimately differ).
* Cache decisions: eager steps through all 48 layers, the oracle's simulator
  replayed on the GPU's own routing; table, owners, tags and scores must agree
  bit for bit after every step (SeqMoE "Mechanism"; MoE-CORE "Mechanism").
"""
import numpy as np
import pytest
import torch

import expert_offload_slot_gb300 as moe
from oracle import layer as olayer
from oracle.cache import SlotPoolSim
from oracle.numerics import decode_act
from synth import gen, get_workload
from tests.gpu_harness import NEAR_TIE, act_to_f64, check_output

pytestmark = pytest.mark.gpu

T = 16


@pytest.fixture(scope="module")
def qwen3():
    wl = get_workload("qwen3_decode")
    rec = wl.expert_layout()[4]
    host = moe.HostPool(wl.L * wl.E * rec)
    gen.fill_host_pool(wl, host.torch(), device="cuda")
    w_r, b = gen.routers(wl)
    wr_dev = torch.from_numpy(np.ascontiguousarray(w_r.view(np.int16))).cuda()
    b_dev = torch.from_numpy(b).cuda()
    yield wl, rec, host, w_r, b, wr_dev, b_dev
    host.free()


def _pool(wl, host, wr_dev, b_dev, max_T=T):
    cfg = moe.make_config(wl.L, wl.E, wl.k, wl.H, wl.I, wl.S, wl.weight_dtype, wl.act_dtype, wl.gating, False,
                          wl.evict, wl.window, 0.9, (0.25, 0.25, 0.25, 0.25), 0, max_T)
    pool = moe.Pool(cfg, host.ptr, host.nbytes, wr_dev, b_dev)
    lut0 = gen.initial_lut(wl)
    pool.set_lut(lut0)
    # set_lut fills the slots asynchronously on the current stream; the graph test runs its steps on
    # a stream of its own, which must not start before every slot holds its record
    torch.cuda.synchronize()
    return pool, lut0


def _expert_mats(wl, host, rec, l, e):
    off = (l * wl.E + e) * rec
    st = gen.record_to_stored(wl, host.numpy()[off:off + rec])
    return olayer.expert_mats(st, wl.weight_dtype, wl.I)


@pytest.mark.parametrize("Tb", [16, 4, 1])
def test_graph_replayed_steps_sampled_layers(qwen3, Tb):
    wl, rec, host, w_r, b, wr_dev, b_dev = qwen3
    pool, _ = _pool(wl, host, wr_dev, b_dev, Tb)
    try:
        steps = 4
        xs = gen.torch_decode_hidden(wl, Tb, steps, "cuda")      # [steps, L, T, H] bf16
        s = torch.cuda.Stream()
        x_in = torch.empty_like(xs[0])
        out = torch.empty_like(x_in)
        with torch.cuda.stream(s):
            x_in.copy_(xs[0])
            for l in range(wl.L):
                pool.forward(l, x_in[l], out[l], moe.MOE_MODE_DECODE)
        s.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for l in range(wl.L):
                pool.forward(l, x_in[l], out[l], moe.MOE_MODE_DECODE)
        for i in range(1, steps):
            with torch.cuda.stream(s):
                x_in.copy_(xs[i])
                g.replay()
        s.synchronize()
        assert pool.status() == 0
        st = pool.stats()
        assert st["misses"] > 0 and st["hits"] > 0
        got = act_to_f64(wl, out.view(torch.int16))
        x_last = xs[steps - 1].view(torch.int16).cpu().numpy().view(np.uint16)
        for l in (0, 23, 47):
            x = decode_act(x_last[l], wl.act_dtype)
            r = olayer.route(x, decode_act(w_r[l], wl.act_dtype), b[l], wl.k, wl.gating)
            ref = olayer.moe_layer(x, r, lambda e: _expert_mats(wl, host, rec, l, e), None)
            ok = r["gap"] >= NEAR_TIE
            assert ok.sum() >= Tb - 2
            check_output(wl, got[l], ref, ok)
        del g
    finally:
        pool.close()


def test_eager_steps_cache_decisions_bit_exact(qwen3):
    wl, rec, host, w_r, b, wr_dev, b_dev = qwen3
    pool, lut0 = _pool(wl, host, wr_dev, b_dev)
    try:
        sim = SlotPoolSim(wl.L, wl.E, wl.S, wl.evict, wl.window)
        sim.set_lut(lut0)
        steps = 2
        xs = gen.torch_decode_hidden(wl, T, steps, "cuda", base_seed=7)
        out = torch.empty_like(xs[0, 0])
        misses = 0
        for t in range(steps):
            for l in range(wl.L):
                pool.forward(l, xs[t, l], out, moe.MOE_MODE_DECODE)
                r = pool.routing(T)
                sim.update_scores(l, r["ids"], r["probs"])
                misses += sim.plan(l, r["ids"])["misses"]
                slot_of = sim.lut[l][r["ids"]]
                np.testing.assert_array_equal(r["slots"], slot_of)
            state = pool.state()
            np.testing.assert_array_equal(state["lut"], sim.lut)
            np.testing.assert_array_equal(state["owner"], sim.owner)
            np.testing.assert_array_equal(state["tag"], sim.tag)
            np.testing.assert_array_equal(state["score"], sim.score)
        assert misses > 0
        assert pool.stats()["misses"] == misses
        assert pool.status() == 0
    finally:
        pool.close()

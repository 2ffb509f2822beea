"""GPU invariants and edge cases of the slot-pool layer (through the C ABI).

* Offloading is lossless (HybriMoE notes: no quantisation or approximation of
  experts; MoE-CORE: exact host-to-device copy path): the output is
  bit-identical under every slot assignment, with an empty table (every
  expert copied or read from the host), and with an all-resident pool.
* The table is transparent to the expert kernel (SeqMoE "Mechanism").
* Edge cases: T = 0, T = max_tokens, ragged H/I, k = E, k = 1, E = 1, E = 256,
  out-of-range ids (device status, no fault), argument errors.
"""
import itertools

import numpy as np
import pytest
import torch

import expert_offload_slot_gb300 as moe
from synth import gen, get_workload
from tests.gpu_harness import Rig, act_to_f64, check_output, check_routing, to_device_act, variant

pytestmark = pytest.mark.gpu


def _fresh_forward(rig, lut, l, x_stored):
    rig.pool.set_lut(lut)
    return rig.forward(l, x_stored)


def test_tiny_output_bit_identical_under_every_slot_assignment():
    wl = get_workload("tiny")
    rig = Rig(wl)
    try:
        x = gen.store_act(wl, gen.decode_hidden(wl, 0, 4, 1)[0])
        base = _fresh_forward(rig, np.full((1, 8), -1, np.int32), 0, x)
        n = 0
        for experts in itertools.combinations(range(8), 4):
            for slots in itertools.permutations(range(4)):
                lut = np.full((1, 8), -1, np.int32)
                lut[0, list(experts)] = slots
                out = _fresh_forward(rig, lut, 0, x)
                assert np.array_equal(out, base), (experts, slots)
                n += 1
        assert n == 1680
        ref, r = rig.oracle_forward(0, x)
        check_output(wl, base, ref)
    finally:
        rig.close()


def test_all_resident_pool_equals_offloaded_pool():
    wl = variant(get_workload("qwen3_decode"), name="resident", L=2, E=32, k=4, H=512, I=256)
    full = Rig(wl, S=wl.L * wl.E, lut=np.arange(wl.L * wl.E, dtype=np.int32).reshape(wl.L, wl.E))
    part = Rig(wl, S=7)
    more = Rig(wl, S=wl.L * wl.E + 13)
    try:
        for l in range(wl.L):
            xs = gen.store_act(wl, gen.decode_hidden(wl, l, 6, 5))
            for t in range(5):
                a, b, c = full.forward(l, xs[t]), part.forward(l, xs[t]), more.forward(l, xs[t])
                assert np.array_equal(a, b) and np.array_equal(a, c)
        assert full.pool.stats()["misses"] == 0
        assert part.pool.stats()["misses"] > 0
    finally:
        for r in (full, part, more):
            r.close()


def test_tensor_core_output_independent_of_resident_set():
    """bf16 tensor-core path, sizes where many entries share the grid: the output of a step is the
    same bits whether all, some or few of its experts were resident (misses copied in-kernel)."""
    wl = variant(get_workload("qwen3_decode"), name="resident_set", L=2, E=64, k=8, H=1024, I=512)
    rigs = [Rig(wl, S=wl.L * wl.E, lut=np.arange(wl.L * wl.E, dtype=np.int32).reshape(wl.L, wl.E)),
            Rig(wl, S=wl.L * wl.E // 3), Rig(wl, S=6)]
    try:
        for l in range(wl.L):
            xs = gen.store_act(wl, gen.decode_hidden(wl, l, 16, 4))
            for t in range(4):
                outs = [r.forward(l, xs[t]) for r in rigs]
                for o in outs[1:]:
                    assert np.array_equal(outs[0], o)
            ref, _ = rigs[0].oracle_forward(l, xs[3])
            check_output(wl, outs[0], ref)
        assert rigs[0].pool.stats()["misses"] == 0
        assert rigs[1].pool.stats()["misses"] > 0 and rigs[2].pool.stats()["bypass"] > 0
    finally:
        for r in rigs:
            r.close()


@pytest.mark.parametrize("T", [1, 2, 4])
def test_streaming_output_independent_of_resident_set(T):
    """One-token calls take the bf16 streaming path, two and four tokens the tensor-core path: on
    either, the output of a step is the same bits whether all, a third or six of the layer's
    experts were resident (misses copied in-kernel, bypass records), and it matches the oracle."""
    wl = variant(get_workload("qwen3_decode"), name="resident_set_stream", L=2, E=64, k=8, H=1024, I=512)
    rigs = [Rig(wl, S=wl.L * wl.E, lut=np.arange(wl.L * wl.E, dtype=np.int32).reshape(wl.L, wl.E)),
            Rig(wl, S=wl.L * wl.E // 3), Rig(wl, S=6)]
    try:
        for l in range(wl.L):
            xs = gen.store_act(wl, gen.decode_hidden(wl, l, T, 4))
            for t in range(4):
                outs = [r.forward(l, xs[t]) for r in rigs]
                for o in outs[1:]:
                    assert np.array_equal(outs[0], o)
                ref, _ = rigs[0].oracle_forward(l, xs[t])
                check_output(wl, outs[0], ref)
        assert rigs[0].pool.stats()["misses"] == 0
        assert rigs[1].pool.stats()["misses"] > 0 and rigs[2].pool.stats()["misses"] > 0
        assert all(r.pool.status() == moe.MOE_OK for r in rigs)
    finally:
        for r in rigs:
            r.close()


@pytest.mark.parametrize("shape", ["bf16_small", "bf16_qwen3_layer", "fp8"])
def test_slots_hold_their_owners_records_after_decode_steps(shape):
    """After decode steps whose misses were copied in-kernel (landing record, then slot), every owned
    slot holds exactly the host record of its owner (SeqMoE "Mechanism": a miss fills the slot the
    table points at), and the table agrees with the oracle's simulator."""
    if shape == "fp8":
        wl = variant(get_workload("dsv3"), name="slots_fp8", L=2, E=32, k=4, H=512, I=256)
        S, Ts = 20, (1, 8, 24)
    elif shape == "bf16_small":
        wl = variant(get_workload("qwen3_decode"), name="slots_bf16", L=2, E=64, k=8, H=1024, I=512)
        S, Ts = 40, (1, 4, 16)
    else:
        wl = variant(get_workload("qwen3_decode"), name="slots_qwen3", L=2, E=128, k=8, H=2048, I=768)
        S, Ts = 110, (16,)
    rig = Rig(wl, S=S, max_tokens=32)
    try:
        host = rig.host.numpy()
        misses = 0
        for T in Ts:
            for step in range(3):
                for l in range(wl.L):
                    x = gen.store_act(wl, gen.decode_hidden(wl, l, T, 1, base_seed=97 * T + step)[0])
                    rig.forward(l, x)
                    r = rig.pool.routing(T)
                    rig.sim.update_scores(l, r["ids"], r["probs"])
                    misses += rig.sim.plan(l, r["ids"])["misses"]
            st = rig.pool.state()
            np.testing.assert_array_equal(st["lut"], rig.sim.lut)
            np.testing.assert_array_equal(st["owner"], rig.sim.owner)
            for slot in range(S):
                o = int(st["owner"][slot])
                if o >= 0:
                    got = rig.pool.read_slot(slot)
                    assert np.array_equal(got, host[o * rig.rec:(o + 1) * rig.rec]), (T, slot, o)
        assert misses > 0 and rig.pool.status() == 0
    finally:
        rig.close()


def test_load_slot_matches_oracle_and_keeps_output():
    wl = variant(get_workload("qwen3_decode"), name="loadslot", L=2, E=16, k=2, H=256, I=256)
    rig = Rig(wl, S=6)
    try:
        x = gen.store_act(wl, gen.decode_hidden(wl, 1, 3, 1)[0])
        base = rig.forward(1, x)
        rig.sim.update_scores(1, *_oracle_ids_probs(rig, 1, x))
        rig.sim.plan(1, _oracle_ids_probs(rig, 1, x)[0])
        for (l, e, s) in ((0, 3, 2), (1, 5, 2), (1, 5, 4), (0, 15, 0), (0, 15, 0)):
            rig.pool.load_slot(l, e, s)
            rig.sim.load_slot(l, e, s)
            st = rig.pool.state()
            np.testing.assert_array_equal(st["lut"], rig.sim.lut)
            np.testing.assert_array_equal(st["owner"], rig.sim.owner)
            np.testing.assert_array_equal(st["tag"], rig.sim.tag)
        rig.pool.set_lut(rig.sim.lut)
        assert np.array_equal(rig.forward(1, x), base)
    finally:
        rig.close()


def _oracle_ids_probs(rig, l, x):
    _, r = rig.oracle_forward(l, x)
    return r["ids"], r["probs"].astype(np.float32)


def test_staged_prefill_equals_slot_path_and_leaves_table_alone():
    wl = variant(get_workload("qwen3_decode"), name="staged", L=4, E=16, k=4, H=256, I=256)
    a = Rig(wl, S=10, staging=2, max_tokens=128)
    b = Rig(wl, S=10, max_tokens=128)
    try:
        lut_before = a.pool.state()["lut"].copy()
        for l in range(wl.L):
            xs = gen.store_act(wl, gen.prefill_hidden(wl, l, 100))
            o1 = a.forward(l, xs, mode=moe.MOE_MODE_PREFILL_STAGED)
            o2 = b.forward(l, xs, mode=moe.MOE_MODE_DECODE)
            assert np.array_equal(o1, o2)
            ref, r = a.oracle_forward(l, xs)
            ok = check_routing(a.pool.routing(128), r, wl.k)
            check_output(wl, o1, ref, ok)
        st = a.pool.state()
        np.testing.assert_array_equal(st["lut"], lut_before)
        s = a.pool.stats()
        assert s["steps"] == wl.L and s["staged_layers"] >= wl.L and s["misses"] == 0
        # AUTO: T >= floor(K_l / k) stages, smaller prefills take the slot path
        xs = gen.store_act(wl, gen.prefill_hidden(wl, 0, 64))
        assert np.array_equal(a.forward(0, xs, mode=moe.MOE_MODE_AUTO), b.forward(0, xs))
    finally:
        a.close()
        b.close()


@pytest.mark.parametrize("shape", [
    dict(E=8, k=8, H=256, I=128),        # k == E: no gap, every expert active
    dict(E=8, k=1, H=256, I=128),        # k == 1: weight 1
    dict(E=1, k=1, H=256, I=128),        # a single expert: plain SwiGLU FFN
    dict(E=256, k=8, H=256, I=128),      # widest router
    dict(E=24, k=3, H=272, I=144),       # ragged H, I (not multiples of the warp width)
])
def test_shape_edge_cases(shape):
    wl = variant(get_workload("qwen3_decode"), name=f"edge{shape['E']}_{shape['k']}", L=1, **shape)
    rig = Rig(wl, S=max(1, wl.E // 2), max_tokens=40)
    try:
        for T in (1, 7, 40):
            xs = gen.store_act(wl, gen.prefill_hidden(wl, 0, T))
            out = rig.forward(0, xs)
            ref, r = rig.oracle_forward(0, xs)
            ok = check_routing(rig.pool.routing(40), r, wl.k)
            check_output(wl, out, ref, ok)
            if wl.k == wl.E:
                assert np.all(np.isinf(rig.pool.routing(40)["gap"]))
        assert rig.pool.status() == moe.MOE_OK
    finally:
        rig.close()


def test_empty_and_oversized_calls():
    wl = variant(get_workload("tiny"), name="empty")
    rig = Rig(wl, max_tokens=4)
    try:
        x = torch.zeros((0, wl.H), dtype=torch.float32, device="cuda")
        rig.pool.forward(0, x, torch.zeros_like(x), T=0)
        assert rig.pool.stats()["steps"] == 0
        x5 = torch.zeros((5, wl.H), dtype=torch.float32, device="cuda")
        with pytest.raises(moe.MoeError) as ei:
            rig.pool.forward(0, x5, torch.zeros_like(x5))
        assert ei.value.status == moe.MOE_ERR_CAPACITY
        with pytest.raises(moe.MoeError) as ei:
            rig.pool.forward(3, x5[:2], torch.zeros_like(x5[:2]))
        assert ei.value.status == moe.MOE_ERR_INVALID
        with pytest.raises(moe.MoeError):
            rig.pool.forward(0, x5[:2], x5[:2])                         # out aliases x
        with pytest.raises(moe.MoeError):
            rig.pool.set_lut(np.array([[0, 0, -1, -1, -1, -1, -1, -1]]))  # slot twice
        with pytest.raises(moe.MoeError):
            rig.pool.load_slot(0, 8, 0)
        with pytest.raises(moe.MoeError):
            rig.pool.forward(0, x5[:2], torch.zeros_like(x5[:2]), mode=moe.MOE_MODE_PREFILL_STAGED)
    finally:
        rig.close()


def test_out_of_range_expert_id_sets_device_status_without_fault():
    wl = variant(get_workload("tiny"), name="bounds")
    rig = Rig(wl)
    try:
        ids = torch.tensor([[0, 9], [1, 2]], dtype=torch.int32, device="cuda")     # 9 >= E
        w = torch.full((2, 2), 0.5, device="cuda")
        probs = torch.full((2, 8), 0.125, device="cuda")
        x = torch.randn((2, wl.H), device="cuda")
        out = torch.empty_like(x)
        rig.pool.forward_routed(0, x, ids, w, probs, out)
        assert rig.pool.status() == moe.MOE_ERR_BOUNDS
        rig.pool.clear_status()
        assert rig.pool.status() == moe.MOE_OK
    finally:
        rig.close()


def test_pool_rejects_unpinned_host_memory():
    wl = get_workload("tiny")
    cfg = moe.make_config(wl.L, wl.E, wl.k, wl.H, wl.I, wl.S, wl.weight_dtype, wl.act_dtype)
    rec = moe.moe_expert_layout(cfg)[4]
    pageable = np.zeros(wl.E * rec, np.uint8)
    wr = torch.zeros((wl.E, wl.H), device="cuda")
    b = torch.zeros(wl.E, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.Pool(cfg, pageable.ctypes.data, pageable.nbytes, wr, b)
    assert ei.value.status == moe.MOE_ERR_INVALID and "pinned" in str(ei.value)

"""moe_route_topk_noalloc: routing without any device allocation.

Callers that cannot allocate device memory where they route tokens (code that
runs while a CUDA graph is captured in global capture mode, or hosts whose
framework owns the device memory budget) use this entry point instead of a
pool.  It must give the same routing as the pool path (moe_forward ->
moe_get_routing) on the same inputs, call after call, although every call
reuses one static scratch array.  This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import expert_offload_slot_gb300 as moe
from synth import gen, get_workload
from tests.gpu_harness import Rig, to_device_act, variant

pytestmark = pytest.mark.gpu


def _noalloc(rig, x, T):
    wl = rig.wl
    ids = torch.empty((T, wl.k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, wl.k), dtype=torch.float32, device="cuda")
    probs = torch.empty((T, wl.E), dtype=torch.float32, device="cuda")
    gap = torch.empty(T, dtype=torch.float32, device="cuda")
    moe.moe_route_topk_noalloc(wl.E, wl.k, wl.H, wl.act_dtype, wl.gating, x, rig.w_r_dev[0], rig.b_dev[0],
                               ids, w, probs, gap)
    torch.cuda.synchronize()
    return {"ids": ids.cpu().numpy(), "w": w.cpu().numpy(), "probs": probs.cpu().numpy(), "gap": gap.cpu().numpy()}


@pytest.mark.parametrize("name,T", [("tiny", 4), ("qwen3_decode", 16)])
def test_noalloc_routing_matches_pool_routing_on_consecutive_calls(name, T):
    wl = get_workload(name)
    if name != "tiny":
        wl = variant(wl, name="noalloc_qwen3", L=1)
    rig = Rig(wl, max_tokens=T)
    try:
        xs = gen.store_act(wl, gen.decode_hidden(wl, 0, T, 2))
        for step in range(2):                       # two calls in a row share the static scratch
            x = to_device_act(wl, xs[step])
            out = torch.empty_like(x)
            rig.pool.forward(0, x, out)
            ref = rig.pool.routing(T)
            got = _noalloc(rig, x, T)
            np.testing.assert_array_equal(got["ids"], ref["ids"])
            np.testing.assert_allclose(got["w"], ref["w"], rtol=0, atol=1e-6)
            np.testing.assert_allclose(got["probs"], ref["probs"], rtol=0, atol=1e-6)
            np.testing.assert_allclose(got["gap"], ref["gap"], rtol=0, atol=1e-6)
    finally:
        rig.close()


def test_noalloc_rejects_sizes_beyond_its_scratch():
    E, H = 256, 256
    T = moe.MOE_NOALLOC_MAX_LOGITS // E + 1
    x = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    wr = torch.zeros((E, H), dtype=torch.float32, device="cuda")
    b = torch.zeros(E, dtype=torch.float32, device="cuda")
    ids = torch.empty((T, 8), dtype=torch.int32, device="cuda")
    w = torch.empty((T, 8), dtype=torch.float32, device="cuda")
    probs = torch.empty((T, E), dtype=torch.float32, device="cuda")
    gap = torch.empty(T, dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_route_topk_noalloc(E, 8, H, moe.MOE_F32, moe.MOE_GATE_SOFTMAX_RENORM, x, wr, b, ids, w, probs, gap)
    assert ei.value.status == moe.MOE_ERR_CAPACITY and "MOE_NOALLOC_MAX_LOGITS" in str(ei.value)

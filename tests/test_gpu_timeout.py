"""Bounded device waits: a wait that runs out reports MOE_ERR_TIMEOUT and the pool recovers.

Every wait a kernel makes on another CTA of its grid is bounded (1 s by
default).  Here the pool's limit is cut to 1 us with moe_set_wait_limit, so the
real readiness waits of a call with miss copies (routing published, miss
records landed, h tiles finished, final arrival before the combine) run out.
Nothing is broken on purpose: the waits are the kernels' ordinary ones and
every one of them still ends.  The test checks that the call returns, that the
sticky status says MOE_ERR_TIMEOUT, that moe_clear_status, the default limit
and moe_set_lut give back a pool whose next calls match the oracle.
Paths: one token (decode layer kernel, streaming FFN), 16 tokens (decode layer
kernel, tensor-core FFN), 100 tokens (plan kernel + cooperative fused FFN).
"""
import time

import numpy as np
import pytest
import torch

import expert_offload_slot_gb300 as moe
from synth import gen, get_workload
from tests.gpu_harness import Rig, check_output, check_routing, variant

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T", [1, 16, 100])
def test_wait_that_runs_out_reports_timeout_and_pool_recovers(T):
    wl = variant(get_workload("qwen3_decode"), name=f"timeout_T{T}", L=2, E=32, k=4, H=512, I=256,
                 residency=0.25, zipf_s=0.3)
    rig = Rig(wl, max_tokens=max(T, 16))
    try:
        xs = gen.store_act(wl, gen.decode_hidden(wl, 0, T, 6))
        # an ordinary call first
        out = rig.forward(0, xs[0])
        ref, r = rig.oracle_forward(0, xs[0])
        check_output(wl, out, ref, check_routing(rig.pool.routing(T), r, wl.k))
        assert rig.pool.status() == moe.MOE_OK
        misses0 = rig.pool.stats()["misses"]
        # 1 us: the call's cross-CTA waits give up
        rig.pool.set_wait_limit(1000)
        t0 = time.time()
        rig.forward(1, xs[1])
        assert time.time() - t0 < 30.0
        assert rig.pool.status() == moe.MOE_ERR_TIMEOUT
        # recovery: clear the status, default limit, table re-applied (slots refilled from the host pool)
        rig.pool.clear_status()
        rig.pool.set_wait_limit(0)
        assert rig.pool.status() == moe.MOE_OK
        rig.pool.set_lut(rig.pool.state()["lut"])
        torch.cuda.synchronize()
        for step in range(2, 6):
            for l in range(wl.L):
                out = rig.forward(l, xs[step])
                ref, r = rig.oracle_forward(l, xs[step])
                check_output(wl, out, ref, check_routing(rig.pool.routing(T), r, wl.k))
        assert rig.pool.status() == moe.MOE_OK
        assert rig.pool.stats()["misses"] > misses0
    finally:
        rig.close()


def test_wait_limit_argument_checks():
    wl = variant(get_workload("qwen3_decode"), name="timeout_args", L=1, E=8, k=2, H=256, I=128, residency=0.5)
    rig = Rig(wl, max_tokens=4)
    try:
        for bad in (1, 999, 10_000_000_001):
            with pytest.raises(moe.MoeError) as ei:
                rig.pool.set_wait_limit(bad)
            assert ei.value.status == moe.MOE_ERR_INVALID
        rig.pool.set_wait_limit(1000)
        rig.pool.set_wait_limit(0)
    finally:
        rig.close()

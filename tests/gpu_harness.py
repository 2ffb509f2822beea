"""Shared set-up for the GPU parity tests: a pool built from the seeded inputs,
and the oracle evaluated on exactly the same stored bytes.

The CUDA side is reached only through the C-ABI binding; the oracle side only
through oracle/; both read the inputs that synth/ draws.
"""
import dataclasses

import numpy as np
import torch

import expert_offload_slot_gb300 as moe
from oracle import layer as olayer
from oracle.cache import SlotPoolSim
from oracle.numerics import bf16_to_f64, decode_act
from synth import gen
from synth.configs import BF16, F32, FP8_E4M3_B128, RESPLIT_Q4R4

# max|out - ref| <= TOL * max|ref|; residual-split weights are compared with the oracle at the same
# quantized precision, so only the bf16 activations and outputs round: the bf16 bound
TOL = {F32: 1e-5, BF16: 2e-2, FP8_E4M3_B128: 5e-2, RESPLIT_Q4R4: 2e-2}
NEAR_TIE = 1e-4


def variant(wl, **kw):
    return dataclasses.replace(wl, **kw)


def to_device_act(wl, x_stored):
    if wl.act_dtype == BF16:
        return torch.from_numpy(np.ascontiguousarray(x_stored).view(np.int16)).cuda()
    return torch.from_numpy(np.ascontiguousarray(x_stored, np.float32)).cuda()


def act_to_f64(wl, t):
    a = t.cpu().numpy()
    if wl.act_dtype == BF16:
        return bf16_to_f64(a.view(np.uint16))
    return a.astype(np.float64)


class Rig:
    def __init__(self, wl, S=None, lut=None, max_tokens=64, zipf_s=None, device_fill=False, staging=0,
                 policy=None, window=None, ema=0.9, core_w=(0.25, 0.25, 0.25, 0.25)):
        self.wl = wl
        self.S = wl.S if S is None else S
        self.policy = wl.evict if policy is None else policy
        self.window = wl.window if window is None else window
        self.rec = wl.expert_layout()[4]
        self.cfg = moe.make_config(wl.L, wl.E, wl.k, wl.H, wl.I, self.S, wl.weight_dtype, wl.act_dtype,
                                   wl.gating, wl.shared, self.policy, self.window, ema, core_w,
                                   staging, max_tokens)
        assert moe.moe_expert_layout(self.cfg)[4] == self.rec
        self.host = moe.HostPool(wl.L * wl.E * self.rec)
        if device_fill:
            gen.fill_host_pool(wl, self.host.torch(), device="cuda")
        else:
            gen.fill_host_pool(wl, self.host.numpy())
        self.w_r, self.b = gen.routers(wl, zipf_s)
        wr = self.w_r.view(np.int16) if wl.act_dtype == BF16 else self.w_r
        self.w_r_dev = torch.from_numpy(np.ascontiguousarray(wr)).cuda()
        self.b_dev = torch.from_numpy(self.b).cuda()
        self.shared_np = gen.shared_records(wl) if wl.shared else None
        self.shared_dev = torch.from_numpy(self.shared_np).cuda() if wl.shared else None
        self.pool = moe.Pool(self.cfg, self.host.ptr, self.host.nbytes, self.w_r_dev, self.b_dev, self.shared_dev)
        self.lut0 = gen.initial_lut(wl, S=self.S) if lut is None else np.asarray(lut, np.int32)
        self.pool.set_lut(self.lut0)
        self.sim = SlotPoolSim(wl.L, wl.E, self.S, self.policy, self.window, ema, core_w)
        self.sim.set_lut(self.lut0)
        self._mats = {}
        self._shared = {}

    # ------------------------------------------------------------- oracle side
    def stored(self, l, e):
        off = (l * self.wl.E + e) * self.rec
        return gen.record_to_stored(self.wl, self.host.numpy()[off:off + self.rec])

    def mats(self, l, e):
        key = (l, e)
        if key not in self._mats:
            self._mats[key] = olayer.expert_mats(self.stored(l, e), self.wl.weight_dtype, self.wl.I)
        return self._mats[key]

    def shared_mats(self, l):
        if self.shared_np is None:
            return None
        key = ("shared", l)
        if key not in self._shared:
            st = gen.record_to_stored(self.wl, self.shared_np[l * self.rec:(l + 1) * self.rec])
            self._shared[key] = olayer.expert_mats(st, self.wl.weight_dtype, self.wl.I)
        return self._shared[key]

    def oracle_forward(self, l, x_stored):
        wl = self.wl
        x = decode_act(x_stored, wl.act_dtype)
        w_r = decode_act(self.w_r[l], wl.act_dtype)
        r = olayer.route(x, w_r, self.b[l], wl.k, wl.gating)
        out = olayer.moe_layer(x, r, lambda e: self.mats(l, e), self.shared_mats(l))
        return out, r

    def oracle_routed(self, l, x_stored, ids, w):
        x = decode_act(x_stored, self.wl.act_dtype)
        r = {"ids": np.asarray(ids), "w": np.asarray(w, np.float64)}
        return olayer.moe_layer(x, r, lambda e: self.mats(l, e), self.shared_mats(l))

    # ---------------------------------------------------------------- GPU side
    def forward(self, l, x_stored, mode=moe.MOE_MODE_DECODE):
        x = to_device_act(self.wl, x_stored)
        out = torch.empty_like(x)
        self.pool.forward(l, x, out, mode)
        torch.cuda.synchronize()
        return act_to_f64(self.wl, out)

    def close(self):
        self.pool.close()
        self.host.free()


def check_output(wl, out, ref, ok_tokens=None):
    if ok_tokens is not None:
        out, ref = out[ok_tokens], ref[ok_tokens]
    if ref.size == 0:
        return 0.0
    err = np.max(np.abs(out - ref))
    scale = np.max(np.abs(ref))
    assert err <= TOL[wl.weight_dtype] * scale, f"max err {err:.3e} > {TOL[wl.weight_dtype]} * {scale:.3e}"
    return err / scale


def check_routing(gpu, ref, k):
    """Top-k sets must agree except at near ties (oracle gap < 1e-4); returns the tokens that agree."""
    T = ref["ids"].shape[0]
    ok = np.ones(T, bool)
    for t in range(T):
        a, b = sorted(gpu["ids"][t].tolist()), sorted(ref["ids"][t].tolist())
        if a != b:
            assert ref["gap"][t] < NEAR_TIE, f"token {t}: ids {a} vs {b}, gap {ref['gap'][t]}"
            ok[t] = False
            continue
        # weights, matched by expert id
        gw = dict(zip(gpu["ids"][t].tolist(), gpu["w"][t].tolist()))
        rw = dict(zip(ref["ids"][t].tolist(), ref["w"][t].tolist()))
        for e in rw:
            assert abs(gw[e] - rw[e]) <= 1e-5, (t, e, gw[e], rw[e])
    np.testing.assert_allclose(gpu["probs"], ref["probs"], atol=2e-6, rtol=1e-4)
    return ok


def synthetic_routing(rng, T, E, k):
    """Seeded routing for the cache-decision tests: distinct ids per token, softmax-like probs."""
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    z = rng.standard_normal((T, E)).astype(np.float32) * 2
    p = np.exp(z - z.max(1, keepdims=True))
    probs = (p / p.sum(1, keepdims=True)).astype(np.float32)
    w = np.take_along_axis(probs, ids.astype(np.int64), axis=1)
    w = (w / w.sum(1, keepdims=True)).astype(np.float32)
    return ids, w, probs

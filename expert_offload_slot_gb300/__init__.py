"""Python binding of libmoeslot, the GB300 slot-pool MoE layer.

Argument marshalling only: every step of the layer runs in the CUDA kernels of
libmoeslot.so, reached through ctypes with the C names of include/moeslot.h.
Tensors are passed as raw device pointers (``tensor.data_ptr()``) and streams
as ``torch.cuda.Stream.cuda_stream``.  There is no fallback: if the library has
not been built, importing this package raises.
"""
import ctypes
import os

import numpy as np

from ._build import LIB, build  # noqa: F401

if not os.path.exists(LIB):
    raise ImportError(f"{LIB} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")

_lib = ctypes.CDLL(LIB)

MOE_OK, MOE_ERR_INVALID, MOE_ERR_OOM, MOE_ERR_CUDA, MOE_ERR_CAPACITY = 0, 1, 2, 3, 4
MOE_ERR_TIMEOUT, MOE_ERR_TAG, MOE_ERR_BOUNDS = 5, 6, 7
MOE_F32, MOE_BF16, MOE_FP8_E4M3_B128, MOE_RESPLIT_Q4R4 = 0, 1, 2, 3
MOE_GATE_SOFTMAX_RENORM, MOE_GATE_SIGMOID_RENORM = 0, 1
MOE_EVICT_CORE, MOE_EVICT_MRS, MOE_EVICT_LRU = 0, 1, 2
MOE_MODE_AUTO, MOE_MODE_DECODE, MOE_MODE_PREFILL_STAGED = 0, 1, 2
STAGES = ("route", "plan", "copy", "ffn")
MOE_NUM_STAGES = len(STAGES)

STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID", 2: "MOE_ERR_OOM", 3: "MOE_ERR_CUDA", 4: "MOE_ERR_CAPACITY",
                5: "MOE_ERR_TIMEOUT", 6: "MOE_ERR_TAG", 7: "MOE_ERR_BOUNDS"}


class moe_config(ctypes.Structure):
    _fields_ = [("num_layers", ctypes.c_int32), ("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("hidden", ctypes.c_int32), ("inter", ctypes.c_int32), ("num_slots", ctypes.c_int32),
                ("weight_dtype", ctypes.c_int32), ("act_dtype", ctypes.c_int32), ("gating", ctypes.c_int32),
                ("has_shared_expert", ctypes.c_int32), ("evict_policy", ctypes.c_int32),
                ("window", ctypes.c_int32), ("ema_decay", ctypes.c_float), ("core_w", ctypes.c_float * 4),
                ("staging_regions", ctypes.c_int32), ("max_tokens", ctypes.c_int32)]


class moe_stats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in ("steps", "hits", "misses", "bypass", "evictions",
                                               "bytes_copied", "near_ties", "staged_layers", "prefetch_issued",
                                               "prefetch_committed", "prefetch_demanded", "prefetch_bytes",
                                               "aes_substitutions", "critical_entries")]


_vp, _i32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
_P = ctypes.POINTER
_sig = {
    "moe_expert_layout": (_i32, [_P(moe_config), _P(_sz), _P(_sz), _P(_sz), _P(_sz), _P(_sz)]),
    "moe_pack_expert_record": (_i32, [_P(moe_config), _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz]),
    "moe_plan_quotas": (_i32, [_P(moe_config), _vp, _vp, _i32, _i32, _i32, _i32, ctypes.c_double, _vp, _vp]),
    "moe_profile_lut": (_i32, [_P(moe_config), _vp, _i32, _i32, _vp, _vp]),
    "moe_host_alloc": (_i32, [_sz, _P(_vp)]),
    "moe_host_free": (_i32, [_vp]),
    "moe_pool_create": (_i32, [_P(moe_config), _vp, _sz, _vp, _vp, _vp, ctypes.c_int, _P(_vp)]),
    "moe_pool_destroy": (_i32, [_vp]),
    "moe_set_lut": (_i32, [_vp, _vp, _vp]),
    "moe_load_slot": (_i32, [_vp, _i32, _i32, _i32, _vp]),
    "moe_forward": (_i32, [_vp, _i32, _vp, _i32, _vp, _i32, _vp]),
    "moe_forward_routed": (_i32, [_vp, _i32, _vp, _i32, _vp, _vp, _vp, _vp, _vp]),
    "moe_update_scores": (_i32, [_vp, _i32, _vp, _vp, _i32, _vp]),
    "moe_set_wait_limit": (_i32, [_vp, ctypes.c_uint64]),
    "moe_prefetch_enable": (_i32, [_vp, _i32]),
    "moe_set_aes": (_i32, [_vp, _i32, ctypes.c_float]),
    "moe_set_umia": (_i32, [_vp, ctypes.c_float, _vp, ctypes.c_float, ctypes.c_float]),
    "moe_prefetch_drain": (_i32, [_vp]),
    "moe_prefetch_inject_wrong_tags": (_i32, [_vp, ctypes.c_uint32]),
    "moe_get_status": (_i32, [_vp]),
    "moe_clear_status": (_i32, [_vp]),
    "moe_get_routing": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _P(_i32)]),
    "moe_get_state": (_i32, [_vp, _vp, _vp, _vp, _vp]),
    "moe_read_slot": (_i32, [_vp, _i32, _vp, _sz]),
    "moe_get_stats": (_i32, [_vp, _P(moe_stats)]),
    "moe_launch_count": (ctypes.c_uint64, [_vp]),
    "moe_profile_enable": (_i32, [_vp, _i32]),
    "moe_profile_read": (_i32, [_vp, _i32, _P(ctypes.c_float)]),
    "moe_last_error": (ctypes.c_char_p, []),
    "moe_route_topk_noalloc": (_i32, [_i32, _i32, _i32, _i32, _i32, _vp, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
}
for _name, (_res, _args) in _sig.items():
    _f = getattr(_lib, _name)
    _f.restype = _res
    _f.argtypes = _args

EXPORTED = tuple(_sig)


class MoeError(RuntimeError):
    def __init__(self, status, where):
        msg = _lib.moe_last_error().decode(errors="replace")
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _check(status, where):
    if status != MOE_OK:
        raise MoeError(status, where)


def _ptr(t):
    """Device/host address of a tensor, numpy array or int; None -> NULL."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, np.ndarray):
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_config(L, E, k, H, I, S, weight_dtype, act_dtype, gating=MOE_GATE_SOFTMAX_RENORM, shared=False,
                evict=MOE_EVICT_CORE, window=16, ema_decay=0.9, core_w=(0.25, 0.25, 0.25, 0.25),
                staging_regions=0, max_tokens=64):
    c = moe_config()
    c.num_layers, c.num_experts, c.top_k, c.hidden, c.inter, c.num_slots = L, E, k, H, I, S
    c.weight_dtype, c.act_dtype, c.gating, c.has_shared_expert = weight_dtype, act_dtype, gating, int(shared)
    c.evict_policy, c.window, c.ema_decay = evict, window, ema_decay
    c.core_w = (ctypes.c_float * 4)(*core_w)
    c.staging_regions, c.max_tokens = staging_regions, max_tokens
    return c


def moe_expert_layout(cfg):
    v = [_sz() for _ in range(5)]
    _check(_lib.moe_expert_layout(ctypes.byref(cfg), *[ctypes.byref(x) for x in v]), "moe_expert_layout")
    return tuple(x.value for x in v)   # (w13_off, w2_off, s13_off, s2_off, record_bytes)


def moe_pack_expert_record(cfg, w_gate, w_up, w_down, s_gate=None, s_up=None, s_down=None):
    """One record (uint8 numpy array) from row-major numpy matrices in the weight dtype's storage."""
    rec = moe_expert_layout(cfg)[4]
    out = np.zeros(rec, np.uint8)
    mats = [np.ascontiguousarray(m) for m in (w_gate, w_up, w_down)]
    scales = [None if v is None else np.ascontiguousarray(v, np.float32) for v in (s_gate, s_up, s_down)]
    _check(_lib.moe_pack_expert_record(ctypes.byref(cfg), *(m.ctypes.data for m in mats),
                                       *(None if v is None else v.ctypes.data for v in scales),
                                       out.ctypes.data, rec), "moe_pack_expert_record")
    return out


def moe_plan_quotas(cfg, ids, probs, budget, delta_k, tau_low):
    """Per-layer slot quotas from a profiling trace (ids int32 [steps,L,T,k], probs float32
    [steps,L,T,E], host numpy).  Returns (quota int32 [L], hit rate float64 [L])."""
    ids = np.ascontiguousarray(ids, np.int32)
    probs = np.ascontiguousarray(probs, np.float32)
    steps, L, T = ids.shape[:3]
    quota = np.zeros(L, np.int32)
    hit = np.zeros(L, np.float64)
    _check(_lib.moe_plan_quotas(ctypes.byref(cfg), ids.ctypes.data, probs.ctypes.data, steps, T, budget, delta_k,
                                float(tau_low), quota.ctypes.data, hit.ctypes.data), "moe_plan_quotas")
    return quota, hit


def moe_profile_lut(cfg, probs, quota):
    """Initial table [L, E] from a profiling trace's probabilities (host numpy) and per-layer quotas."""
    probs = np.ascontiguousarray(probs, np.float32)
    steps, L, T, E = probs.shape
    q = np.ascontiguousarray(quota, np.int32)
    lut = np.zeros((L, E), np.int32)
    _check(_lib.moe_profile_lut(ctypes.byref(cfg), probs.ctypes.data, steps, T, q.ctypes.data, lut.ctypes.data),
           "moe_profile_lut")
    return lut


MOE_NOALLOC_MAX_LOGITS = 65536


def moe_route_topk_noalloc(E, k, H, act_dtype, gating, x, router_w, router_b, ids, w, probs, gap, stream=None):
    """Router + top-k without any device allocation (scratch in a static device array).

    For callers that cannot allocate device memory where they route tokens; see
    include/moeslot.h.  All outputs are caller-owned device tensors.
    """
    _check(_lib.moe_route_topk_noalloc(E, k, H, act_dtype, gating, _ptr(x), x.shape[0], _ptr(router_w),
                                       _ptr(router_b), _ptr(ids), _ptr(w), _ptr(probs), _ptr(gap),
                                       _stream(stream)), "moe_route_topk_noalloc")


class HostPool:
    """Pinned, mapped host memory from moe_host_alloc, viewable as a uint8 numpy array."""

    def __init__(self, nbytes):
        p = _vp()
        _check(_lib.moe_host_alloc(nbytes, ctypes.byref(p)), "moe_host_alloc")
        self.ptr, self.nbytes = p.value, nbytes

    def numpy(self):
        return np.ctypeslib.as_array((ctypes.c_uint8 * self.nbytes).from_address(self.ptr))

    def torch(self):
        import torch
        return torch.frombuffer((ctypes.c_uint8 * self.nbytes).from_address(self.ptr), dtype=torch.uint8)

    def free(self):
        if self.ptr:
            _lib.moe_host_free(self.ptr)
            self.ptr = 0

    def __del__(self):
        try:
            self.free()
        except Exception:
            pass


class Pool:
    """One slot pool (moe_pool_create ... moe_pool_destroy)."""

    def __init__(self, cfg, host_pool_ptr, host_pool_bytes, router_w, router_b, shared_w=None, device=0):
        self.cfg = cfg
        self._keep = (router_w, router_b, shared_w)
        h = _vp()
        _check(_lib.moe_pool_create(ctypes.byref(cfg), host_pool_ptr, host_pool_bytes, _ptr(router_w),
                                    _ptr(router_b), _ptr(shared_w), device, ctypes.byref(h)), "moe_pool_create")
        self.h = h.value
        self.record_bytes = moe_expert_layout(cfg)[4]

    def close(self):
        if self.h:
            _lib.moe_pool_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_lut(self, lut, stream=None):
        a = np.ascontiguousarray(lut, dtype=np.int32).reshape(-1)
        _check(_lib.moe_set_lut(self.h, a.ctypes.data, _stream(stream)), "moe_set_lut")

    def load_slot(self, layer, expert, slot, stream=None):
        _check(_lib.moe_load_slot(self.h, layer, expert, slot, _stream(stream)), "moe_load_slot")

    def forward(self, layer, x, out, mode=MOE_MODE_DECODE, stream=None, T=None):
        T = x.shape[0] if T is None else T
        _check(_lib.moe_forward(self.h, layer, _ptr(x), T, _ptr(out), mode, _stream(stream)), "moe_forward")

    def forward_routed(self, layer, x, ids, w, probs, out, stream=None):
        _check(_lib.moe_forward_routed(self.h, layer, _ptr(x), x.shape[0], _ptr(ids), _ptr(w), _ptr(probs),
                                       _ptr(out), _stream(stream)), "moe_forward_routed")

    def update_scores(self, layer, ids, probs, stream=None):
        _check(_lib.moe_update_scores(self.h, layer, _ptr(ids), _ptr(probs), ids.shape[0], _stream(stream)),
               "moe_update_scores")

    def set_umia(self, theta, beta=None, gamma_decode=1.0, gamma_prefill=1.0):
        b = None if beta is None else np.ascontiguousarray(beta, np.float32)
        _check(_lib.moe_set_umia(self.h, float(theta), None if b is None else b.ctypes.data, float(gamma_decode),
                                 float(gamma_prefill)), "moe_set_umia")

    def set_aes(self, on, alpha=0.0):
        _check(_lib.moe_set_aes(self.h, int(on), float(alpha)), "moe_set_aes")

    def prefetch_enable(self, per_step):
        _check(_lib.moe_prefetch_enable(self.h, int(per_step)), "moe_prefetch_enable")

    def prefetch_drain(self):
        _check(_lib.moe_prefetch_drain(self.h), "moe_prefetch_drain")

    def prefetch_inject_wrong_tags(self, n):
        _check(_lib.moe_prefetch_inject_wrong_tags(self.h, int(n)), "moe_prefetch_inject_wrong_tags")

    def set_wait_limit(self, ns):
        _check(_lib.moe_set_wait_limit(self.h, int(ns)), "moe_set_wait_limit")

    def status(self):
        return _lib.moe_get_status(self.h)

    def clear_status(self):
        _check(_lib.moe_clear_status(self.h), "moe_clear_status")

    def routing(self, cap_T):
        c = self.cfg
        k, E = c.top_k, c.num_experts
        out = {"ids": np.zeros((cap_T, k), np.int32), "w": np.zeros((cap_T, k), np.float32),
               "probs": np.zeros((cap_T, E), np.float32), "gap": np.zeros(cap_T, np.float32),
               "slots": np.zeros((cap_T, k), np.int32), "perm": np.zeros(cap_T * k, np.int32),
               "offs": np.zeros(E + 1, np.int32)}
        T = _i32()
        _check(_lib.moe_get_routing(self.h, *(out[n].ctypes.data for n in ("ids", "w", "probs", "gap", "slots",
                                                                           "perm", "offs")),
                                    cap_T, ctypes.byref(T)), "moe_get_routing")
        T = T.value
        for n in ("ids", "w", "probs", "gap", "slots"):
            out[n] = out[n][:T]
        out["perm"] = out["perm"][:T * k]
        out["T"] = T
        return out

    def state(self):
        c = self.cfg
        LE, S = c.num_layers * c.num_experts, c.num_slots
        lut, owner = np.zeros(LE, np.int32), np.zeros(S, np.int32)
        tag, score = np.zeros(S, np.uint32), np.zeros(LE, np.float32)
        _check(_lib.moe_get_state(self.h, lut.ctypes.data, owner.ctypes.data, tag.ctypes.data, score.ctypes.data),
               "moe_get_state")
        return {"lut": lut.reshape(c.num_layers, c.num_experts), "owner": owner, "tag": tag,
                "score": score.reshape(c.num_layers, c.num_experts)}

    def read_slot(self, slot):
        """The record bytes slot `slot` holds (host copy, blocking)."""
        rec = moe_expert_layout(self.cfg)[4]
        buf = np.zeros(rec, np.uint8)
        _check(_lib.moe_read_slot(self.h, int(slot), buf.ctypes.data, rec), "moe_read_slot")
        return buf

    def stats(self):
        s = moe_stats()
        _check(_lib.moe_get_stats(self.h, ctypes.byref(s)), "moe_get_stats")
        return {n: getattr(s, n) for n, _ in moe_stats._fields_}

    def profile_enable(self, on=True):
        _check(_lib.moe_profile_enable(self.h, int(on)), "moe_profile_enable")

    def profile_read(self, layer):
        v = (ctypes.c_float * MOE_NUM_STAGES)()
        _check(_lib.moe_profile_read(self.h, layer, v), "moe_profile_read")
        return list(v)

    def launch_count(self):
        return int(_lib.moe_launch_count(self.h))

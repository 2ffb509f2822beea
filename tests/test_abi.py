"""The C-ABI library loads and exports every symbol include/moeslot.h declares (CPU only: no compute calls)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moeslot.h")


def declared_symbols():
    src = open(HEADER).read()
    return sorted(set(re.findall(r"MOE_API\s+[\w\s\*]+?\b(moe_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for n in ("moe_pool_create", "moe_set_lut", "moe_load_slot", "moe_forward", "moe_update_scores",
              "moe_pool_destroy", "moe_get_status", "moe_get_stats", "moe_get_routing"):
        assert n in names


def test_library_loads_and_exports_every_declared_symbol():
    import __graft_entry__
    b = __graft_entry__._build_module()
    b.build()
    lib = ctypes.CDLL(b.LIB)
    for n in declared_symbols():
        assert hasattr(lib, n), n


def test_binding_binds_every_declared_symbol():
    import expert_offload_slot_gb300 as moe
    assert sorted(moe.EXPORTED) == declared_symbols()


def test_host_side_argument_errors_need_no_gpu():
    import expert_offload_slot_gb300 as moe
    bad = moe.make_config(1, 300, 2, 256, 128, 4, moe.MOE_F32, moe.MOE_F32)     # E > 256
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_expert_layout(bad)
    assert ei.value.status == moe.MOE_ERR_INVALID and "num_experts" in str(ei.value)
    mixed = moe.make_config(1, 8, 2, 256, 128, 4, moe.MOE_BF16, moe.MOE_F32)     # unsupported pair
    with pytest.raises(moe.MoeError):
        moe.moe_expert_layout(mixed)
    ragged = moe.make_config(1, 8, 2, 260, 128, 4, moe.MOE_BF16, moe.MOE_BF16)   # H not a multiple of 8
    with pytest.raises(moe.MoeError):
        moe.moe_expert_layout(ragged)


def test_record_layout_matches_the_generator():
    import expert_offload_slot_gb300 as moe
    from synth import WORKLOADS
    for wl in WORKLOADS.values():
        cfg = moe.make_config(wl.L, wl.E, wl.k, wl.H, wl.I, wl.S, wl.weight_dtype, wl.act_dtype)
        assert moe.moe_expert_layout(cfg) == wl.expert_layout(), wl.name


def test_noalloc_rejects_misaligned_pointers_before_any_launch():
    """The router reads x and W_r 16 bytes at a time: a misaligned view must be refused on the host
    (MOE_ERR_INVALID), never reach a kernel.  The addresses are never dereferenced."""
    import expert_offload_slot_gb300 as moe
    lib = moe._lib
    E, k, H, T = 8, 2, 256, 4
    good, odd8 = 1 << 20, (1 << 20) + 8
    args = dict(x=good, wr=good, b=good, ids=good, w=good, probs=good, gap=good)
    for name, bad in (("x", odd8), ("wr", odd8), ("x", good + 2), ("b", good + 2), ("probs", good + 1)):
        a = dict(args, **{name: bad})
        st = lib.moe_route_topk_noalloc(E, k, H, moe.MOE_BF16, moe.MOE_GATE_SOFTMAX_RENORM, a["x"], T, a["wr"],
                                        a["b"], a["ids"], a["w"], a["probs"], a["gap"], None)
        assert st == moe.MOE_ERR_INVALID, name
        assert b"aligned" in lib.moe_last_error()

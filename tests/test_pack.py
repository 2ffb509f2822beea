"""moe_pack_expert_record: the record format the header documents, checked on the host (no GPU).

The header states each byte position; these tests place element-coded
matrices with the library and check every element against that statement,
written out here from the header's words, and against the generator that
fills the host pools of the GPU tests.
"""
import numpy as np
import pytest

import expert_offload_slot_gb300 as moe
from synth import gen, get_workload
from tests.gpu_harness import variant


def _cfg(wl):
    return moe.make_config(wl.L, wl.E, wl.k, wl.H, wl.I, wl.S, wl.weight_dtype, wl.act_dtype)


def _documented_bf16_offset(kind, i, j, H, I, w13_off, w2_off):
    """Byte of element (i, j) as include/moeslot.h words it."""
    r, c = i % 128, j % 64
    in_tile = r * 128 + ((c // 8) ^ (r % 8)) * 16 + (c % 8) * 2
    if kind == "down":
        return w2_off + ((i // 128) * -(-I // 64) + j // 64) * 16384 + in_tile
    g = 0 if kind == "gate" else 1
    return w13_off + (((i // 128) * -(-H // 64) + j // 64) * 2 + g) * 16384 + in_tile


def test_bf16_record_places_every_element_where_the_header_says():
    H, I = 136, 136            # ragged in both directions: partial tiles of rows and columns
    wl = variant(get_workload("qwen3_decode"), name="pack", L=1, E=2, k=1, H=H, I=I)
    cfg = _cfg(wl)
    w13_off, w2_off, _, _, rec = moe.moe_expert_layout(cfg)
    n = I * H
    gate = (np.arange(n, dtype=np.uint32) + 1).astype(np.uint16).reshape(I, H)           # codes 1..n
    up = (np.arange(n, dtype=np.uint32) + 1 + n).astype(np.uint16).reshape(I, H)
    down = (np.arange(n, dtype=np.uint32) + 1 + 2 * n).astype(np.uint16).reshape(H, I)
    assert 3 * n < 65536
    out = moe.moe_pack_expert_record(cfg, gate, up, down)
    assert out.size == rec
    seen = np.zeros(rec, bool)
    for kind, m in (("gate", gate), ("up", up), ("down", down)):
        R, C = m.shape
        for i in range(R):
            for j in range(C):
                o = _documented_bf16_offset(kind, i, j, H, I, w13_off, w2_off)
                assert out[o:o + 2].view(np.uint16)[0] == m[i, j], (kind, i, j)
                seen[o:o + 2] = True
    assert not out[~seen].any()          # everything else (tile padding, record padding) is zero
    assert rec % 4096 == 0


@pytest.mark.parametrize("name", ["tiny", "qwen3_decode", "dsv3"])
def test_library_packing_equals_the_generators_records(name):
    base = get_workload(name)
    shape = dict(H=512, I=256) if name != "tiny" else {}
    wl = variant(base, name=f"pack_{name}", L=1, E=2, k=1, **shape)
    cfg = _cfg(wl)
    for e in range(wl.E):
        st = gen.expert_stored(wl, 0, e)
        I = wl.I
        kw = {}
        if "s13" in st:
            kw = dict(s_gate=st["s13"][:I // 128], s_up=st["s13"][I // 128:], s_down=st["s2"])
        got = moe.moe_pack_expert_record(cfg, st["w13"][:I], st["w13"][I:], st["w2"], **kw)
        np.testing.assert_array_equal(got, gen.expert_record_bytes(wl, st))


def test_row_major_formats_and_argument_errors():
    wl = variant(get_workload("dsv3"), name="pack_fp8", L=1, E=2, k=1, H=256, I=128)
    cfg = _cfg(wl)
    w13_off, w2_off, s13_off, s2_off, rec = moe.moe_expert_layout(cfg)
    rng = np.random.default_rng(0)
    g, u = rng.integers(0, 256, (128, 256), np.uint8), rng.integers(0, 256, (128, 256), np.uint8)
    d = rng.integers(0, 256, (256, 128), np.uint8)
    sg, su, sd = (rng.random(s).astype(np.float32) for s in ((1, 2), (1, 2), (2, 1)))
    out = moe.moe_pack_expert_record(cfg, g, u, d, sg, su, sd)
    np.testing.assert_array_equal(out[w13_off:w13_off + g.size], g.ravel())
    np.testing.assert_array_equal(out[w13_off + g.size:w13_off + 2 * g.size], u.ravel())
    np.testing.assert_array_equal(out[w2_off:w2_off + d.size], d.ravel())
    np.testing.assert_array_equal(out[s13_off:s13_off + 16].view(np.float32), np.concatenate([sg, su]).ravel())
    np.testing.assert_array_equal(out[s2_off:s2_off + 8].view(np.float32), sd.ravel())
    with pytest.raises(moe.MoeError) as ei:
        moe.moe_pack_expert_record(cfg, g, u, d)          # fp8 without scales
    assert ei.value.status == moe.MOE_ERR_INVALID
    st = moe._lib.moe_pack_expert_record(moe.ctypes.byref(cfg), g.ctypes.data, u.ctypes.data, d.ctypes.data,
                                         sg.ctypes.data, su.ctypes.data, sd.ctypes.data, out.ctypes.data, rec - 1)
    assert st == moe.MOE_ERR_INVALID                     # buffer one byte short


def test_a_row_major_bf16_record_is_not_the_packed_record():
    """The bf16 record is tiled: bytes laid out row-major differ from it (the header's warning)."""
    wl = variant(get_workload("qwen3_decode"), name="pack_rm", L=1, E=2, k=1, H=256, I=128)
    st = gen.expert_stored(wl, 0, 0)
    packed = moe.moe_pack_expert_record(_cfg(wl), st["w13"][:128], st["w13"][128:], st["w2"])
    row_major = np.concatenate([st["w13"].view(np.uint8).ravel(), st["w2"].view(np.uint8).ravel()])
    assert not np.array_equal(packed[:row_major.size], row_major)
    # same multiset of elements: a permutation, not a re-encoding
    np.testing.assert_array_equal(np.sort(packed[:row_major.size].view(np.uint16)),
                                  np.sort(row_major.view(np.uint16)))


def test_residual_split_records_equal_the_generators():
    """The library's residual-split encoder (fp32 in) writes the generator's record byte for byte."""
    from synth.configs import RESPLIT_Q4R4
    wl = variant(get_workload("dsv3"), name="pack_resplit", L=1, E=2, k=1, H=512, I=256,
                 weight_dtype=RESPLIT_Q4R4, shared=False)
    cfg = _cfg(wl)
    assert moe.moe_expert_layout(cfg) == wl.expert_layout()
    for e in range(wl.E):
        wg, wu, wd = gen.expert_fp32(wl, 0, e)
        got = moe.moe_pack_expert_record(cfg, wg, wu, wd)
        np.testing.assert_array_equal(got, gen.expert_record_bytes(wl, gen.expert_stored(wl, 0, e)))

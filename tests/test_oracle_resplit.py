"""Pins of the residual-split codec and the UMIA critical set (RapidMoE §4.3-4.4), CPU only.

The decode is checked against the fp32 weights the generator drew, through the
error bounds that round-to-nearest quantization guarantees: at most half a step
of W^Q; with the residual W^R at most half a step of W^R, whose step is at
most 1/14 of W^Q's; the 8-bit down_proj at most half of its step.
"""
import numpy as np

from oracle.resplit import dequant_groups, resplit_mats, umia_critical, umia_threshold
from synth import gen
from synth.configs import BF16, RESPLIT_Q4R4, Workload


def _wl():
    return Workload(name="resplit_pin", L=1, E=2, k=1, H=384, I=256, weight_dtype=RESPLIT_Q4R4, act_dtype=BF16,
                    gating=0, residency=0.5, zipf_s=0.0)


def test_int4_nibbles_decode_as_twos_complement():
    codes = np.arange(-8, 8, dtype=np.int8).reshape(1, 16)
    packed = gen.pack_int4(codes)
    assert packed[0, 0] == 0x98 and packed[0, 4] == 0x10          # (-8, -7) and (0, 1)
    np.testing.assert_array_equal(gen.unpack_int4(packed, 16), codes)


def test_decode_error_bounds_against_the_drawn_weights():
    wl = _wl()
    wg, wu, wd = gen.expert_fp32(wl, 0, 0)
    st = gen.record_to_stored(wl, gen.expert_record_bytes(wl, gen.expert_stored(wl, 0, 0)))
    w13 = np.concatenate([wg, wu]).astype(np.float64)
    sq = np.repeat(st["sq13"].astype(np.float64), 128, axis=1)
    sr = np.repeat(st["sr13"].astype(np.float64), 128, axis=1)
    g_lo, u_lo, d_lo = resplit_mats(st, wl.I, False)
    g_hi, u_hi, d_hi = resplit_mats(st, wl.I, True)
    lo = np.concatenate([g_lo, u_lo])
    hi = np.concatenate([g_hi, u_hi])
    tol = 1e-6 * np.abs(w13).max()                 # fp32 rounding of the generator's own arithmetic
    assert np.all(np.abs(w13 - lo) <= sq / 2 + tol)
    assert np.all(np.abs(w13 - hi) <= sr / 2 + tol)
    assert np.all(sr <= sq / 14 + tol)
    assert np.abs(w13 - hi).max() < np.abs(w13 - lo).max() / 5
    sh = np.repeat(st["sh2"].astype(np.float64), 128, axis=1)
    sl = np.repeat(st["sl2"].astype(np.float64), 128, axis=1)
    assert np.all(np.abs(wd - d_hi) <= sh / 2 + tol)
    assert np.all(np.abs(wd - d_lo) <= sl / 2 + tol)
    assert np.abs(st["q13"]).max() <= 7 and np.abs(st["h2"]).max() <= 127


def test_dequant_is_code_times_group_scale():
    codes = np.array([[1, -2] * 128], np.int8)
    scales = np.array([[0.5, 0.25]], np.float32)
    w = dequant_groups(codes, scales)
    assert w[0, 0] == 0.5 and w[0, 1] == -1.0 and w[0, 128] == 0.25 and w[0, 129] == -0.5


def test_umia_threshold_and_critical_set():
    thr = umia_threshold(0.1, 0.5, 1.5)
    assert thr == np.float32(np.float32(np.float32(0.1) * np.float32(0.5)) * np.float32(1.5))
    s = np.array([0.2, 0.07, thr, 0.0], np.float32)
    assert umia_critical(s, 0.1, 0.5, 1.5).tolist() == [True, False, True, False]
    assert not umia_critical(s, 10.0, 1.0, 1.0).any()
    assert umia_critical(s, 0.0, 1.0, 1.0).all()            # threshold 0: every expert is critical

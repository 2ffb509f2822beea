"""Pins for the oracle's number-format decoding (CPU only)."""
import os

import numpy as np
import pytest
import torch

from oracle.numerics import bf16_to_f64, e4m3_to_f64, dequant_fp8_blocks

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_bf16_all_codes_match_torch():
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = bf16_to_f64(codes)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[ok], ref[ok])


def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = e4m3_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(np.isnan(ours), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(ours[ok], ref[ok])
    # sign of zero survives
    assert np.signbit(ours[0x80]) and not np.signbit(ours[0x00])


def test_e4m3_spec_points():
    with open(os.path.join(GOLDEN, "e4m3_codes.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for code, val in rows:
        got = e4m3_to_f64(np.array([int(code, 16)], np.uint8))[0]
        if val == "nan":
            assert np.isnan(got)
        else:
            assert got == float(val), (code, got, val)


def test_fp8_block_dequant_uses_the_right_block_scale():
    # 256 x 384 codes all equal to 1.0 (0x38); scales distinct per block -> W equals its block's scale.
    codes = np.full((256, 384), 0x38, np.uint8)
    scales = np.array([[1.0, 2.0, 4.0], [0.5, 0.25, 8.0]], np.float32)
    w = dequant_fp8_blocks(codes, scales)
    for bi in range(2):
        for bj in range(3):
            blk = w[bi * 128:(bi + 1) * 128, bj * 128:(bj + 1) * 128]
            assert np.all(blk == scales[bi, bj])
    # a transposed use of the scale grid would fail here: (0, 2) and (1, 0) differ
    assert w[0, 300] == 4.0 and w[200, 0] == 0.5


def test_fp8_dequant_is_one_exact_multiply():
    rng = np.random.default_rng(1)
    codes = rng.integers(0, 256, (128, 128), dtype=np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x10
    s = np.array([[0.0123]], np.float32)
    w = dequant_fp8_blocks(codes, s)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy() * np.float64(s[0, 0])
    np.testing.assert_array_equal(w, ref)

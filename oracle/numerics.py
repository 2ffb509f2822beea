"""Exact decoding of the stored number formats (oracle; test infrastructure only).

bf16: the upper 16 bits of an IEEE binary32 — widening is a 16-bit shift.
fp8 e4m3 (OCP 8-bit floating point, "E4M3"): 1 sign bit, 4 exponent bits with
bias 7, 3 mantissa bits; exponent field 0 encodes subnormals m/8 * 2^-6; the
all-ones pattern S.1111.111 is NaN; there is no infinity.  The largest finite
value is 0.1111.110 = 448.
Block-scaled fp8 (the DeepSeek-V3-shaped workload): one fp32 scale per 128x128
block, W[i, j] = e4m3(q[i, j]) * scale[i // 128, j // 128].
"""
import numpy as np


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def e4m3_to_f64(codes: np.ndarray) -> np.ndarray:
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = (c & 0x7).astype(np.float64)
    normal = (1.0 + man / 8.0) * np.exp2(exp.astype(np.float64) - 7.0)
    subnormal = (man / 8.0) * 2.0 ** -6
    val = np.where(exp == 0, subnormal, normal) * sign
    nan = (c & 0x7F) == 0x7F
    return np.where(nan, np.nan, val)


_E4M3_VALUES = None


def e4m3_value_table() -> np.ndarray:
    """e4m3_to_f64 of every one of the 256 codes, indexed by code."""
    global _E4M3_VALUES
    if _E4M3_VALUES is None:
        _E4M3_VALUES = e4m3_to_f64(np.arange(256, dtype=np.uint8))
    return _E4M3_VALUES


def dequant_fp8_blocks(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """W[i, j] = e4m3(codes[i, j]) * scales[i // 128, j // 128]  (float64, exact).

    Each code is decoded by looking up its value in e4m3_to_f64 of all 256 codes
    (the same values, without re-evaluating the formula per element); the rows
    and columns are multiplied by their block's scale.
    """
    c = np.asarray(codes, dtype=np.uint8)
    R, C = c.shape
    w = e4m3_value_table()[c]
    s = np.asarray(scales, dtype=np.float32).astype(np.float64)
    if R % 128 == 0 and C % 128 == 0:
        blocks = w.reshape(R // 128, 128, C // 128, 128)
        blocks *= s[:, None, :, None]
        return w
    s_full = np.repeat(np.repeat(s, 128, axis=0), 128, axis=1)
    return w * s_full[:R, :C]


def decode_weight(stored, key: str, dtype: int) -> np.ndarray:
    """Decode stored[key] ("w13" or "w2") of one expert to float64.

    dtype: 0 = fp32, 1 = bf16 bits, 2 = fp8 e4m3 codes + stored["s13"/"s2"].
    """
    a = stored[key]
    if dtype == 0:
        return np.asarray(a, np.float32).astype(np.float64)
    if dtype == 1:
        return bf16_to_f64(a)
    scale_key = {"w13": "s13", "w2": "s2"}[key]
    return dequant_fp8_blocks(a, stored[scale_key])


def decode_act(a: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == 1:
        return bf16_to_f64(a)
    return np.asarray(a, np.float32).astype(np.float64)

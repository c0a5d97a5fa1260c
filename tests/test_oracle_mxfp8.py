"""Pins for the MXFP8 oracle (CPU only): brute-force nearest code, closed forms, library cast.

Brute force: every finite positive E4M3 code is decoded and the nearest one is picked, ties to
the code with an even mantissa, anything above 448 clamped to 448. Values are handled in
float64, which is exact here: a BF16 value scaled by 2^-X keeps its 8 significant bits, and
every difference that can decide a rounding (|q| below 2^10, codes at or above 2^-9) needs
fewer than 53 bits; far-away values are decided without ties.
"""
import numpy as np
import pytest
import torch

from oracle import mxfp8 as M
from oracle import coracle as C

X_VALUES = (-127, -20, -9, -1, 0, 1, 3, 8, 40, 119)


def _codes_table():
    codes = [c for c in range(0x7F) if M.e4m3_value(c) is not None]
    vals = np.array([float(M.e4m3_value(c)) for c in codes])
    return np.array(codes), vals


def brute_e4m3(q: np.ndarray) -> np.ndarray:
    codes, vals = _codes_table()
    a = np.minimum(np.abs(q), 448.0)
    diff = np.abs(a[:, None] - vals[None, :])
    best = diff.min(axis=1, keepdims=True)
    cand = diff == best
    # ties: prefer the even mantissa (code LSB 0)
    even = (codes[None, :] & 1) == 0
    pick = np.where((cand & even).any(axis=1), np.argmax(cand & even, axis=1), np.argmax(cand, axis=1))
    out = codes[pick].astype(np.int64)
    return np.where(np.signbit(q), out | 0x80, out)


def _bf16_as_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _finite_bf16():
    b = np.arange(65536, dtype=np.uint32)
    return b[(b & 0x7F80) != 0x7F80]


def check_elements(convert, stride=1, xs=X_VALUES):
    bits = _finite_bf16()[::stride]
    for x in xs:
        q = _bf16_as_f64(bits) / (2.0 ** x)
        want = brute_e4m3(q)
        got = np.array([convert(int(b), x) for b in bits])
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, (x, [hex(int(bits[i])) for i in bad[:5]], got[bad[:5]], want[bad[:5]])


def test_c_oracle_all_bf16_patterns_brute_force():
    check_elements(C.e4m3)


def test_python_oracle_bf16_subsample_brute_force():
    check_elements(M.convert_element, stride=13, xs=(-127, -9, 0, 5, 119))


def test_codes_round_trip():
    for c in range(256):
        v = M.e4m3_value(c)
        if v is None:
            continue
        assert M.e4m3_encode(v, bool(c & 0x80)) == c


def test_torch_float8_cast_agrees_in_range():
    """torch's float8_e4m3fn cast (RNE) is a library pin for |q| <= 448."""
    bits = _finite_bf16()
    for x in (-3, 0, 2):
        q = _bf16_as_f64(bits) / (2.0 ** x)
        keep = np.abs(q) <= 448
        tq = torch.from_numpy(q[keep].astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        got = np.array([C.e4m3(int(b), x) for b in bits[keep]])
        assert np.array_equal(got, tq.astype(np.int64)), x


def _bits(vals):
    return [int(b) for b in (np.asarray(vals, np.float32).view(np.uint32) >> 16)]


def check_block_closed_forms(quantize_block):
    # amax = 2^k exactly -> X = k - 8, and that element becomes 2^8 = 256 (code 0x78)
    for k in (-100, -6, 0, 1, 7, 8, 9, 100, 127):
        vals = [0.0] * 31 + [2.0 ** k]
        codes, scale = quantize_block(_bits(vals))
        assert scale == max(-127, k - 8) + 127, k
        if k - 8 >= -127:
            assert codes[31] == 0x78, (k, hex(codes[31]))
    # amax in [448, 512) * 2^X saturates to 448 (0x7E); 480 rounds up and still clamps
    codes, scale = quantize_block(_bits([500.0, -470.0, 448.0, 449.0] + [1.0] * 28))
    assert scale == 127 and codes[:4] == [0x7E, 0xFE, 0x7E, 0x7E]
    # all-zero block: X = -127 (byte 0), signs kept
    codes, scale = quantize_block(_bits([0.0] * 16 + [-0.0] * 16))
    assert scale == 0 and codes == [0x00] * 16 + [0x80] * 16
    # Inf / NaN anywhere: scale 0xFF, elements 0x7F
    for bad in (np.inf, -np.inf, np.nan):
        codes, scale = quantize_block(_bits([1.0] * 31 + [bad]))
        assert scale == 0xFF and codes == [0x7F] * 32
    # subnormal bf16 amax: X clamps at -127
    codes, scale = quantize_block([0x0001] * 32)
    assert scale == 0
    # a midpoint: with X = 0, 1.0625 lies halfway between 1.0 (0x38) and 1.125 (0x39): even wins
    codes, scale = quantize_block(_bits([256.0, 1.0625, 1.1875, -1.0625] + [0.0] * 28))
    assert scale == 127 and codes[1:4] == [0x38, 0x3A, 0xB8]
    # negative values that round to zero keep the sign bit
    codes, scale = quantize_block(_bits([256.0, -2.0 ** -11] + [0.0] * 30))
    assert codes[1] == 0x80


def test_block_closed_forms_python():
    check_block_closed_forms(M.quantize_block)


def test_block_closed_forms_c():
    check_block_closed_forms(C.mxfp8_block)


def test_random_blocks_c_vs_python():
    rng = np.random.Generator(np.random.PCG64(4))
    for _ in range(300):
        scale = 2.0 ** rng.integers(-30, 30)
        vals = (rng.standard_normal(32) * scale).astype(np.float32)
        if rng.random() < 0.2:
            vals[rng.integers(0, 32, size=5)] = 0.0
        b = _bits(vals)
        assert M.quantize_block(b) == tuple(C.mxfp8_block(b))

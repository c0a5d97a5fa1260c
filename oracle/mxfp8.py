"""BF16 -> MXFP8 (E4M3 elements + E8M0 scale per 32-element block), exact Python reference.

TEST INFRASTRUCTURE (see the package docstring): only tests, smoke() and the bench's
CPU-baseline leg use it.

The NeMo-RL design doc "NCCL Reshard Refit (Experimental)", section "Enabling It", says only
that the generation ranks quantize each received BF16 shard into MXFP8 before installing it.
The rule itself is the published OCP Microscaling Formats (MX) v1.0 conversion, with the
element encoding of the OCP 8-bit floating point (OFP8) E4M3 format:

- a block is 32 consecutive elements along the destination shard's last dim;
- shared scale X = floor(log2(max_i |v_i|)) - 8, where 8 is the exponent of E4M3's largest
  normal (448 = 1.75 * 2^8); X is stored as an E8M0 byte X + 127, clamped to [-127, 127];
- each element is v_i / 2^X rounded to nearest-even into E4M3, saturating at +-448.

Readings where the specs leave a choice (each is listed in the design notes):
- an all-zero block (log2(0) undefined) takes X = -127 (scale byte 0x00); its elements keep
  their sign: +0 -> 0x00, -0 -> 0x80;
- a block holding NaN or Inf gets the E8M0 NaN scale 0xFF and every element 0x7F (E4M3 NaN);
- a negative element that rounds to zero encodes as 0x80 (sign kept).

Parity: pinned by brute-force nearest-code enumeration over all BF16 patterns, exact powers
of two, rounding midpoints, saturation, subnormals and the zero/NaN policies (tests).
"""
from __future__ import annotations

from fractions import Fraction
from typing import List, Optional, Sequence, Tuple

E4M3_MAX = Fraction(448)
E4M3_EMAX = 8           # exponent of the largest normal, 448 = 1.75 * 2^8
E4M3_MIN_NORMAL = Fraction(1, 64)    # 2^-6
E4M3_SUB_QUANTUM = Fraction(1, 512)  # 2^-9, the subnormal step


def bf16_fields(bits: int) -> Tuple[int, int, int]:
    """(sign, biased exponent, 7-bit mantissa) of a BF16 bit pattern."""
    return (bits >> 15) & 1, (bits >> 7) & 0xFF, bits & 0x7F


def bf16_value(bits: int) -> Optional[Fraction]:
    """Exact value of a finite BF16 pattern as a Fraction; None for Inf/NaN.

    BF16 is the top half of IEEE binary32: bias 127, 7 stored mantissa bits.
    """
    s, e, m = bf16_fields(bits)
    if e == 0xFF:
        return None
    if e == 0:
        mag = Fraction(m, 1 << 7) * Fraction(1, 1 << 126)
    else:
        mag = Fraction(128 + m, 128) * (Fraction(2) ** (e - 127))
    return -mag if s else mag


def floor_log2(x: Fraction) -> int:
    """floor(log2 x) for x > 0, exactly."""
    assert x > 0
    e = x.numerator.bit_length() - x.denominator.bit_length()
    # now 2^(e-1) < x < 2^(e+1); fix up to the exact floor
    while Fraction(2) ** e > x:
        e -= 1
    while Fraction(2) ** (e + 1) <= x:
        e += 1
    return e


def shared_exponent(block_bits: Sequence[int]) -> Optional[int]:
    """The block's E8M0 exponent X, or None when the block holds Inf/NaN."""
    amax = Fraction(0)
    for b in block_bits:
        v = bf16_value(b)
        if v is None:
            return None
        amax = max(amax, abs(v))
    if amax == 0:
        return -127
    return max(-127, min(127, floor_log2(amax) - E4M3_EMAX))


def e4m3_encode(q: Fraction, negative: bool) -> int:
    """Round |q| to nearest-even E4M3 magnitude, saturate at 448, attach the sign bit."""
    a = abs(q)
    if a == 0:
        return 0x80 if negative else 0x00
    if a < E4M3_MIN_NORMAL:
        quantum = E4M3_SUB_QUANTUM
    else:
        quantum = Fraction(2) ** (floor_log2(a) - 3)   # 3 mantissa bits
    n = a / quantum
    k = n.numerator // n.denominator
    rem = n - k
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and k % 2 == 1):
        k += 1
    val = k * quantum
    if val > E4M3_MAX:
        val = E4M3_MAX
    sign = 0x80 if negative else 0x00
    if val == 0:
        return sign
    if val < E4M3_MIN_NORMAL:
        return sign | int(val / E4M3_SUB_QUANTUM)          # subnormal: m * 2^-9
    e = floor_log2(val)
    m = int(val / (Fraction(2) ** (e - 3))) - 8            # normal: (8 + m) * 2^(e-3)
    return sign | ((e + 7) << 3) | m


def e4m3_value(code: int) -> Optional[Fraction]:
    """Exact value of an E4M3 code (bias 7, no Inf; S.1111.111 is NaN)."""
    s = (code >> 7) & 1
    e = (code >> 3) & 0xF
    m = code & 7
    if e == 0xF and m == 7:
        return None
    if e == 0:
        mag = m * E4M3_SUB_QUANTUM
    else:
        mag = Fraction(8 + m, 8) * (Fraction(2) ** (e - 7))
    return -mag if s else mag


def convert_element(bits: int, x: int) -> int:
    """One BF16 element into E4M3 under shared exponent X: v / 2^X, RNE, saturating."""
    v = bf16_value(bits)
    assert v is not None
    return e4m3_encode(v / (Fraction(2) ** x), bool(bits >> 15))


def quantize_block(block_bits: Sequence[int]) -> Tuple[List[int], int]:
    """32 BF16 patterns -> (32 E4M3 codes, E8M0 scale byte)."""
    assert len(block_bits) == 32
    x = shared_exponent(block_bits)
    if x is None:
        return [0x7F] * 32, 0xFF
    return [convert_element(b, x) for b in block_bits], x + 127


def quantize_rows(bits_rows: Sequence[Sequence[int]]) -> Tuple[List[List[int]], List[List[int]]]:
    """Row-major quantization: every row split into 32-element blocks along its length."""
    codes, scales = [], []
    for row in bits_rows:
        assert len(row) % 32 == 0
        rc, rs = [], []
        for b in range(0, len(row), 32):
            c, s = quantize_block(row[b:b + 32])
            rc.extend(c)
            rs.append(s)
        codes.append(rc)
        scales.append(rs)
    return codes, scales

"""Storage codecs of the oracle, written from the number-format definitions.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The DeepSeek-V4 report (§2.3.4 "efficiency discussion") stores the content
dimensions of every compressed KV entry in FP8 and the 64 RoPE dimensions in
BF16, and runs the lightning indexer's QK path in FP4 (§5.2.1 "FP4
quantization-aware training").  The report names MXFP4; the workload
definitions fix e2m1 elements with one e4m3 scale per 16 elements, which is the
reading taken here.

Every encoder below works by the definition: build the sorted list of finite
values a format can hold, pick the nearest one, break an exact tie toward the
code whose last mantissa bit is zero (round-to-nearest-even), and saturate to
the largest finite value.  No bit tricks are shared with the CUDA path.
"""
from __future__ import annotations

import numpy as np

# ---------------------------------------------------------------- e4m3 (OCP FP8 E4M3, "fn": no infinities)
# sign(1) exponent(4, bias 7) mantissa(3); exponent field 15 with mantissa 7 is NaN.


def _e4m3_positive_values() -> np.ndarray:
    """Values of codes 0x00..0x7E in code order (monotonic), float64."""
    vals = []
    for code in range(0x7F):
        e = code >> 3
        mant = code & 7
        if e == 0:
            vals.append(mant / 8.0 * 2.0 ** (1 - 7))
        else:
            vals.append((1.0 + mant / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, dtype=np.float64)


E4M3_VALUES = _e4m3_positive_values()
E4M3_MAX = float(E4M3_VALUES[-1])  # 448


def _encode_by_table(x: np.ndarray, table: np.ndarray) -> np.ndarray:
    """Nearest entry of the sorted non-negative ``table`` for |x| (float64),
    exact ties to the even index, saturating at the last entry.  Returns the
    index (the magnitude code) as int64."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    if np.isnan(a).any():
        raise ValueError("NaN has no finite code")
    a = np.minimum(a, table[-1])
    hi = np.searchsorted(table, a, side="left")  # first index with table[hi] >= a
    hi = np.clip(hi, 0, len(table) - 1)
    lo = np.clip(hi - 1, 0, len(table) - 1)
    d_lo = a - table[lo]
    d_hi = table[hi] - a
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(table[hi] == a, hi, code)  # exact hits
    return code.astype(np.int64)


def e4m3_encode(x) -> np.ndarray:
    """float -> uint8 e4m3 code, round-to-nearest-even, saturating to +-448.
    The input is taken as the exact value of its float (float32 values are
    exact in float64)."""
    x = np.asarray(x, dtype=np.float64)
    mag = _encode_by_table(x, E4M3_VALUES)
    sign = np.signbit(x)  # a negative value that rounds to zero keeps its sign (-0)
    return (mag | (sign.astype(np.int64) << 7)).astype(np.uint8)


def e4m3_decode(code) -> np.ndarray:
    code = np.asarray(code, dtype=np.int64)
    mag = code & 0x7F
    if (mag == 0x7F).any():
        raise ValueError("e4m3 NaN code")
    v = E4M3_VALUES[mag]
    return np.where(code & 0x80, -v, v)


# ---------------------------------------------------------------- bf16
# The upper half of an IEEE binary32: sign(1) exponent(8) mantissa(7).


def bf16_decode(bits) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint32)
    with np.errstate(invalid="ignore"):
        return (bits << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_encode(x) -> np.ndarray:
    """float32 value -> uint16 bf16 bits, round-to-nearest-even on the value.

    The two candidates are the bf16 values that bracket x: the one obtained by
    dropping the low 16 bits (toward zero) and the next one away from zero.
    The nearer one wins; an exact tie goes to the even mantissa.  Values past
    the bf16 range round to infinity, as IEEE rounding does."""
    x32 = np.asarray(x, dtype=np.float32)
    u = x32.view(np.uint32).astype(np.uint64)
    toward0 = (u >> 16).astype(np.uint64)  # bits of the truncated value
    away = toward0 + 1                      # next magnitude up (same sign)
    v = np.abs(x32.astype(np.float64))
    v0 = np.abs(bf16_decode(toward0.astype(np.uint32)))
    with np.errstate(over="ignore", invalid="ignore"):
        v1 = np.abs(bf16_decode(away.astype(np.uint32)))
    # past the largest finite bf16 the next step up is 2^128 (infinity's slot)
    v1 = np.where(np.isinf(v1), 2.0 ** 128, v1)
    d0 = v - v0
    d1 = v1 - v
    take_away = (d1 < d0) | ((d1 == d0) & (toward0 % 2 == 1))
    take_away &= d0 != 0  # exact values stay
    out = np.where(take_away, away, toward0)
    return out.astype(np.uint16)


def bf16_round(x) -> np.ndarray:
    """float -> nearest bf16 value (float64)."""
    return bf16_decode(bf16_encode(np.asarray(x, dtype=np.float32)))


# ---------------------------------------------------------------- e2m1 (FP4)
# sign(1) exponent(2, bias 1) mantissa(1): magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6.

E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
E2M1_MAX = 6.0


def e2m1_encode(x) -> np.ndarray:
    """float -> 4-bit code (uint8 0..15), RNE, saturating to +-6."""
    x = np.asarray(x, dtype=np.float64)
    mag = _encode_by_table(x, E2M1_VALUES)
    sign = np.signbit(x)  # as for e4m3: -0 for negatives that round to zero
    return (mag | (sign.astype(np.int64) << 3)).astype(np.uint8)


def e2m1_decode(code) -> np.ndarray:
    code = np.asarray(code, dtype=np.int64)
    v = E2M1_VALUES[code & 7]
    return np.where(code & 8, -v, v)


def pack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[..., 2n] 4-bit codes -> [..., n] bytes; the even element sits in the
    low nibble."""
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[..., 0::2] | (codes[..., 1::2] << 4)).astype(np.uint8)


def unpack_nibbles(packed: np.ndarray) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


# ---------------------------------------------------------------- composite formats

def kv_entry_encode(v, d_content: int = 512):
    """One compressed KV entry -> (content e4m3 codes, fp32 scale, rope bf16 bits).

    Content dims: per-entry scale = amax / 448 as an IEEE float32 division
    (1 when amax is 0 or the quotient underflows to 0); code = e4m3(c / scale)
    with the division also in float32.  RoPE dims: bf16 of the float32 value.
    ``v`` is a float32 array [..., d_content + d_rope]."""
    v = np.asarray(v, dtype=np.float32)
    c = v[..., :d_content]
    r = v[..., d_content:]
    amax = np.max(np.abs(c), axis=-1)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    scale = np.where(scale == 0, np.float32(1.0), scale).astype(np.float32)
    quot = (c / scale[..., None]).astype(np.float32)
    return e4m3_encode(quot), scale, bf16_encode(r)


def kv_entry_decode(codes, scale, rope_bits) -> np.ndarray:
    """Inverse of ``kv_entry_encode`` (exact, float64)."""
    c = e4m3_decode(codes) * np.asarray(scale, dtype=np.float64)[..., None]
    return np.concatenate([c, bf16_decode(rope_bits)], axis=-1)


def fp4_block_encode(x, block: int = 16):
    """float32 [..., K] -> (e2m1 codes [..., K], e4m3 scale codes [..., K/block]).

    Per block of 16: s = e4m3(amax / 6) with the division in float32; the
    elements are e2m1(x / s) with s the decoded scale, division in float32.
    A block whose scale rounds to zero (or whose amax is zero) stores scale
    code 0 and all-zero elements."""
    x = np.asarray(x, dtype=np.float32)
    K = x.shape[-1]
    assert K % block == 0
    xb = x.reshape(x.shape[:-1] + (K // block, block))
    amax = np.max(np.abs(xb), axis=-1)
    s_code = e4m3_encode((amax / np.float32(E2M1_MAX)).astype(np.float32))
    s_val = e4m3_decode(s_code).astype(np.float32)
    safe = np.where(s_val == 0, np.float32(1.0), s_val).astype(np.float32)
    quot = (xb / safe[..., None]).astype(np.float32)
    codes = e2m1_encode(quot)
    codes = np.where((s_val == 0)[..., None], np.uint8(0), codes).astype(np.uint8)
    return codes.reshape(x.shape), s_code


def fp4_block_decode(codes, s_code, block: int = 16) -> np.ndarray:
    codes = np.asarray(codes)
    K = codes.shape[-1]
    v = e2m1_decode(codes).reshape(codes.shape[:-1] + (K // block, block))
    s = e4m3_decode(s_code)[..., None]
    return (v * s).reshape(codes.shape)

"""MX FP8 quantisation for the oracle: e4m3 elements, one power-of-two scale
per block of 32 consecutive elements along the contraction axis.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: nothing in the product
package imports it, and it shares no code with the CUDA path.

Source.  "AI-Research-SKILLs MoE 训练实战…全指南" §9.2 (inference optimisation)
compares FP8 with FP16 serving of an MoE model (higher throughput, about half
the memory, under 1 % accuracy loss); the pages fix neither the FP8 format nor
its scaling.  Reading (R22): the OCP Microscaling form the B300 tensor cores
consume natively -- elements in FP8 E4M3 (1 sign, 4 exponent bits with bias 7,
3 mantissa bits, subnormals, largest finite value 448 = 1.75 * 2^8, no
infinities), one shared scale X = 2^s per block of 32 elements stored as an
8-bit biased exponent (s + 127), s = floor(log2(max |v|)) - 8 (8 being the
exponent of E4M3's largest normal), clamped to [-127, 127]; an all-zero block
takes s = -127.  Each element is v / X rounded to the nearest E4M3 value, ties
to the even mantissa, and values beyond 448 in magnitude saturate to +-448.

The quantised value of v is decode(code) * X.  Everything here is float64
arithmetic on the exact values (divisions by powers of two are exact), except
that the inputs are taken as float32 numbers: the quantisation decisions are
made on the float32 values the kernels hold.
"""

from __future__ import annotations

import math

import numpy as np

BLOCK = 32              # elements per shared scale
E4M3_MAX = 448.0        # largest finite E4M3 magnitude: 1.75 * 2^8
E4M3_EMAX = 8           # exponent of the largest normal E4M3 value
E4M3_EMIN = -6          # exponent of the smallest normal (exponent field 1, bias 7)
E4M3_MBITS = 3
SCALE_BIAS = 127        # the scale byte is s + 127 (E8M0)


def e4m3_decode(code) -> np.ndarray:
    """Value of each E4M3 code (uint8): exponent field 0 is subnormal,
    m * 2^-9; otherwise (1 + m/8) * 2^(e - 7).  Code 0x7F / 0xFF (NaN) is not
    produced by the quantiser and decodes to NaN."""
    c = np.asarray(code, np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    sub = m * 2.0 ** (E4M3_EMIN - E4M3_MBITS)
    nor = (1.0 + m / 8.0) * np.exp2(e - 7.0)
    v = sign * np.where(e == 0, sub, nor)
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


def e4m3_round(v) -> np.ndarray:
    """v (float64) rounded to the nearest E4M3 value, ties to even, saturating
    at +-448.  The quantum is 2^(e - 3) for |v| in [2^e, 2^(e+1)), e >= -6, and
    2^-9 below 2^-6 (the subnormals)."""
    v = np.asarray(v, np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)                       # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, E4M3_EMIN)         # floor(log2 a), at least the normal minimum
    q = np.exp2(e - E4M3_MBITS)
    r = np.round(a / q) * q                   # numpy rounds half to even
    r = np.minimum(r, E4M3_MAX)
    return np.copysign(r, v)


def e4m3_encode(v) -> np.ndarray:
    """Code of e4m3_round(v) (uint8)."""
    r = e4m3_round(v)
    a = np.abs(r)
    sign = np.signbit(r).astype(np.int64) << 7
    _, ex = np.frexp(a)
    e = ex - 1
    normal = a >= 2.0 ** E4M3_EMIN
    m_sub = np.round(a / 2.0 ** (E4M3_EMIN - E4M3_MBITS)).astype(np.int64)
    e_field = np.where(normal, e + 7, 0)
    m_nor = np.round((a / np.exp2(np.where(normal, e, 0)) - 1.0) * 8.0).astype(np.int64)
    m = np.where(normal, m_nor, m_sub)
    return (sign | (e_field.astype(np.int64) << 3) | m).astype(np.uint8)


def block_scale_exponent(amax) -> np.ndarray:
    """s = floor(log2(amax)) - 8 clamped to [-127, 127]; -127 for amax = 0."""
    a = np.asarray(amax, np.float64)
    _, ex = np.frexp(a)
    s = np.where(a > 0, ex - 1 - E4M3_EMAX, -SCALE_BIAS)
    return np.clip(s, -SCALE_BIAS, SCALE_BIAS).astype(np.int64)


def quantize(a, block: int = BLOCK):
    """MX-quantise the rows of a [rows, K] along K.

    Returns (codes uint8 [rows, K], scale bytes uint8 [rows, ceil(K / block)]).
    A last partial block is scaled by its own maximum."""
    a32 = np.asarray(a, np.float32).astype(np.float64)
    rows, K = a32.shape
    nb = -(-K // block)
    pad = np.zeros((rows, nb * block), np.float64)
    pad[:, :K] = a32
    blocks = pad.reshape(rows, nb, block)
    s = block_scale_exponent(np.abs(blocks).max(axis=-1))
    scaled = blocks / np.exp2(s)[:, :, None]
    codes = e4m3_encode(scaled).reshape(rows, nb * block)[:, :K]
    return codes, (s + SCALE_BIAS).astype(np.uint8)


def dequantize(codes, scales, block: int = BLOCK) -> np.ndarray:
    """float64 values of MX-quantised rows."""
    codes = np.asarray(codes, np.uint8)
    rows, K = codes.shape
    s = np.asarray(scales, np.uint8).astype(np.int64) - SCALE_BIAS
    X = np.repeat(np.exp2(s.astype(np.float64)), block, axis=1)[:, :K]
    return e4m3_decode(codes) * X


def fake_quant(a, block: int = BLOCK) -> np.ndarray:
    """dequantize(quantize(a)): the values an MX FP8 operand stands for."""
    return dequantize(*quantize(a, block), block)


def finite_values() -> np.ndarray:
    """Every finite E4M3 value (both signs), ascending, for brute-force pins."""
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    return np.unique(e4m3_decode(codes))


_TABLE = None


def _table():
    """(value, code) of every finite E4M3 code, decoded once."""
    global _TABLE
    if _TABLE is None:
        codes = [c for c in range(256) if (c & 0x7F) != 0x7F]
        vals = e4m3_decode(np.array(codes, np.uint8))
        _TABLE = [(float(v), c) for v, c in zip(vals, codes)]
    return _TABLE


def nearest_by_search(v: float) -> float:
    """The E4M3 value nearest to v by exhaustive search over every finite
    value, ties to the one with an even mantissa field, beyond +-448
    saturating: an independent restatement of e4m3_round for the pins."""
    if math.isnan(v):
        return math.nan
    if abs(v) >= E4M3_MAX:
        return math.copysign(E4M3_MAX, v)
    best, best_d, best_even = None, math.inf, False
    for val, c in _table():
        if val == 0.0 and math.copysign(1.0, val) != math.copysign(1.0, v):
            continue
        dd = abs(val - v)
        even = (c & 1) == 0
        if dd < best_d or (dd == best_d and even and not best_even):
            best, best_d, best_even = val, dd, even
    return best

"""Number formats used by the MoE layer, decoded and encoded exactly in float64.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this
module; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` use it.

Formats (the pages name them; the bit layouts are the public OCP / IEEE ones):

* E2M1 (FP4): 1 sign, 2 exponent (bias 1), 1 mantissa bit; no inf/NaN.
  Weight storage of the MXFP4 and NVFP4 schemes ("DeepSeek V4 MegaMoE Kernel
  深度解析", 五、为什么能这么高效 item 5, and the CUDA tag page's MXFP4 vs
  NVFP4 teaser).  Two codes per byte, element 2j in the low nibble (reading:
  the pages do not say which nibble comes first).
* E4M3 (FP8, OCP "FN" flavour): 1 sign, 4 exponent (bias 7), 3 mantissa
  bits, no inf, NaN = S.1111.111, max 448.  Activation format of the
  block-scaled GEMMs (MegaMoE page, 二、阶段 2 and 三、数据流图).
* UE8M0: unsigned power of two 2**(b-127); b = 255 is NaN.  The per-block
  scale of MXFP4 weights (per 32) and of FP8 activations (per 128).
* bfloat16: the top 16 bits of an IEEE binary32.
"""
import math

import numpy as np


def e2m1_value(code: int) -> float:
    """Value of one 4-bit E2M1 code, from its bit fields."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        mag = 0.5 * m  # subnormal: 2**(1-bias) * m/2 with bias 1
    else:
        mag = 2.0 ** (e - 1) * (1.0 + 0.5 * m)
    return -mag if s else mag


def e4m3_value(code: int) -> float:
    """Value of one 8-bit E4M3 code (OCP FN: no infinities)."""
    s = (code >> 7) & 1
    e = (code >> 3) & 15
    m = code & 7
    if e == 15 and m == 7:
        return math.nan
    if e == 0:
        mag = m * 2.0 ** -9  # subnormal: 2**(1-7) * m/8
    else:
        mag = 2.0 ** (e - 7) * (1.0 + m / 8.0)
    return -mag if s else mag


def ue8m0_value(code: int) -> float:
    """Value of one UE8M0 scale byte."""
    if code == 255:
        return math.nan
    return 2.0 ** (code - 127)


E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_value(c) for c in range(256)], dtype=np.float64)
UE8M0_TABLE = np.array([ue8m0_value(c) for c in range(256)], dtype=np.float64)


def decode_e2m1_packed(packed: np.ndarray) -> np.ndarray:
    """[..., n/2] uint8 (two codes per byte, element 2j low nibble) -> [..., n] float64."""
    packed = np.asarray(packed, dtype=np.uint8)
    lo = E2M1_TABLE[packed & 0x0F]
    hi = E2M1_TABLE[packed >> 4]
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.float64)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def decode_e4m3(codes: np.ndarray) -> np.ndarray:
    return E4M3_TABLE[np.asarray(codes, dtype=np.uint8)]


def decode_ue8m0(codes: np.ndarray) -> np.ndarray:
    return UE8M0_TABLE[np.asarray(codes, dtype=np.uint8)]


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bfloat16 stored as uint16 bit patterns -> float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


# ----------------------------------------------------------------------------
# Round-to-nearest-even encoders, written from the definition: list every
# finite non-negative value of the target format in increasing order, find the
# two neighbours of |x|, take the nearer, and on an exact tie the one whose
# code is even (its last mantissa bit is 0).  The sign bit is kept, so a
# negative value that rounds to zero becomes negative zero.

_E4M3_POS_CODES = np.arange(0, 127, dtype=np.int64)          # 0x00 .. 0x7E (0x7F is NaN)
_E4M3_POS_VALUES = E4M3_TABLE[_E4M3_POS_CODES]               # strictly increasing


def encode_e4m3_rne(x: np.ndarray) -> np.ndarray:
    """float64 array with |x| <= 448 -> E4M3 codes (uint8), round to nearest even.

    Callers scale first so that no value exceeds the largest finite E4M3
    value; anything beyond it is an error here rather than a silent clamp.
    """
    x = np.asarray(x, dtype=np.float64)
    if np.isnan(x).any():
        raise ValueError("NaN input to E4M3 encoder")
    a = np.abs(x)
    if (a > 448.0).any():
        raise ValueError("value beyond E4M3 range; scale before encoding")
    hi = np.searchsorted(_E4M3_POS_VALUES, a, side="left")    # first value >= a
    hi = np.minimum(hi, len(_E4M3_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    vhi = _E4M3_POS_VALUES[hi]
    vlo = _E4M3_POS_VALUES[lo]
    dhi = vhi - a
    dlo = a - vlo
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (_E4M3_POS_CODES[hi] % 2 == 0))
    exact = vhi == a
    code = np.where(exact | pick_hi, _E4M3_POS_CODES[hi], _E4M3_POS_CODES[lo])
    sign = np.signbit(x).astype(np.int64) << 7
    return (code | sign).astype(np.uint8)


def round_bf16_rne(x: np.ndarray) -> np.ndarray:
    """float64 -> nearest bfloat16 (ties to even), returned as uint16 bits.

    bfloat16 keeps 8 significant bits and binary32's exponent range:
    normal numbers m * 2**p with 1 <= m < 2 and -126 <= p <= 127, subnormals
    multiples of 2**-133.  The value is rounded once, directly from float64.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.float64)
    a = np.abs(x)
    finite = np.isfinite(x)
    nz = finite & (a > 0)
    # exponent p with 2**p <= a < 2**(p+1)
    _, p = np.frexp(np.where(nz, a, 1.0))
    p = p.astype(np.int64) - 1
    p = np.maximum(p, -126)                      # below 2**-126 the quantum stays 2**-133
    quantum = np.ldexp(1.0, (p - 7).astype(np.int64))
    q = a / quantum                              # exact: division by a power of two
    r = np.floor(q)
    frac = q - r
    up = (frac > 0.5) | ((frac == 0.5) & (np.fmod(r, 2.0) == 1.0))
    r = r + up
    mag = r * quantum
    mag = np.where(mag >= 2.0 ** 128, np.inf, mag)   # overflow after rounding
    out[:] = np.where(nz, np.copysign(mag, x), x)
    out = np.where(finite, out, x)
    f32 = out.astype(np.float32)                 # exact: every bf16 value is a binary32 value
    bits = (f32.view(np.uint32) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    bits = np.where(nan, np.uint16(0x7FC0), bits)
    return bits.astype(np.uint16)


def ue8m0_exponent_for_amax(amax: float, qmax: float = 448.0) -> int:
    """Smallest integer e with amax <= qmax * 2**e, clamped to [-127, 127]; 0 when amax == 0.

    This is the "amax -> UE8M0 scale" step of the FP8 requant (MegaMoE page,
    二、阶段 3): a power-of-two scale chosen so that no element saturates.
    Computed with exact power-of-two arithmetic only.
    """
    if not (amax >= 0.0):
        raise ValueError("amax must be a non-negative number")
    if amax == 0.0:
        return 0
    if math.isinf(amax):
        return 127
    e = math.frexp(amax / qmax)[1]               # amax/qmax < 2**e, and >= 2**(e-1)
    # exact search around the estimate (the division above may round)
    while amax > qmax * 2.0 ** e:
        e += 1
    while amax <= qmax * 2.0 ** (e - 1):
        e -= 1
    return max(-127, min(127, e))

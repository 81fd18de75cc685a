"""OCP FP8 E4M3 (the "e4m3fn" flavour) encode / decode, written from the format
definition: 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits, no
infinities, S.1111.111 is NaN, largest finite magnitude 448, subnormals
m/8 * 2^-6.

The fp8 KV cache of the pages ("KV Cache + Speculative Decoding" section 4.5,
FP8 KV; walkerchi "KV Cache" section 3.5, kv_cache_dtype='fp8') stores
code = e4m3(x / scale) with a per-(layer, kv-head) fp32 scale.

Reading adopted for the quantised code (an integer decided by floating point):
x / scale is formed in fp32 (IEEE division, the precision the kernel uses) and
then rounded to the nearest e4m3 value, ties to the even code, magnitudes above
448 saturated to 448 ("satfinite"), NaN kept as NaN.
"""
import numpy as np

NAN_CODE = 0x7F


def code_values() -> np.ndarray:
    """Value of each of the 256 codes as float64 (NaN for the two NaN codes)."""
    vals = np.empty(256, dtype=np.float64)
    for code in range(256):
        s = (code >> 7) & 1
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            v = np.nan
        elif e == 0:
            v = (m / 8.0) * 2.0 ** -6
        else:
            v = (1.0 + m / 8.0) * 2.0 ** (e - 7)
        vals[code] = -v if s else v
    return vals


_VALUES = code_values()
# codes 0x00..0x7E are the non-negative finite values in increasing order
_POS = _VALUES[:0x7F]


def decode(codes) -> np.ndarray:
    return _VALUES[np.asarray(codes, dtype=np.uint8)]


def encode(x32) -> np.ndarray:
    """Round float32 values to e4m3 codes (RNE, satfinite)."""
    x = np.asarray(x32, dtype=np.float32).astype(np.float64)
    out = np.empty(x.shape, dtype=np.uint8)
    nan = np.isnan(x)
    sign = np.signbit(x)
    a = np.minimum(np.abs(np.where(nan, 0.0, x)), 448.0)
    hi = np.searchsorted(_POS, a, side="left")          # first value >= a
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_hi = _POS[hi] - a
    d_lo = a - _POS[lo]
    exact = d_hi == 0.0
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    code = np.where(exact, hi, np.where(pick_hi, hi, lo)).astype(np.uint8)
    code = np.where(sign, code | 0x80, code).astype(np.uint8)
    code = np.where(nan, NAN_CODE, code).astype(np.uint8)
    out[...] = code
    return out


def quantize(x, scale) -> np.ndarray:
    """code = e4m3(fp32(x) / fp32(scale)) with the division done in fp32."""
    q = np.asarray(x, dtype=np.float32) / np.asarray(scale, dtype=np.float32)
    return encode(q.astype(np.float32))

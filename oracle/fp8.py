"""fp64 CPU oracle for an 8-bit KV cache: the E4M3 encoding and the per-head scaling that store
K and V in one byte per element.

TEST INFRASTRUCTURE ONLY (the same rule as llama_oracle.py).

The pages size the KV cache in bf16 and note that it dominates decode memory ("Llama
Architecture ...", Mathematical Foundations 4, KV cache scaling; "LLaMA-3 8B ...", section 七); they
give no 8-bit format.  Readings taken:
  * the format is OCP 8-bit floating point E4M3 ("e4m3fn"): sign, 4 exponent bits with bias 7,
    3 mantissa bits; exponent field 0 holds subnormals 2^-6 * m/8; S.1111.111 is NaN; there are
    no infinities; the largest finite magnitude is 448;
  * a cached element is x ~= code * s with one fp32 scale s per (layer, K or V, KV head);
  * encoding holds x in fp32 and divides in fp32 (q = fl32(fl32(x) / s)), rounds q to the nearest
    E4M3 value with ties to the even code, and saturates at +-448 -- so the integer decision is
    taken in the precision a GPU kernel takes it;
  * attention reads the decoded values code * s, including for the token being decoded, whose
    K and V are encoded before it attends to them.
"""
import numpy as np


def e4m3_decode(code) -> np.ndarray:
    """Value of each E4M3 code (uint8 array) as fp64."""
    c = np.asarray(code, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    val = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    val = np.where((e == 15) & (m == 7), np.nan, val)
    return sign * val


_POS_CODES = np.arange(0, 127, dtype=np.uint8)          # 0x00 .. 0x7E: every finite non-negative value
_POS_VALS = e4m3_decode(_POS_CODES)                      # increasing


def e4m3_encode(q) -> np.ndarray:
    """Nearest E4M3 code to each value of q (ties to the even code), saturating at +-448."""
    q = np.asarray(q, dtype=np.float64)
    a = np.minimum(np.abs(q), 448.0)
    hi = np.searchsorted(_POS_VALS, a, side="left")      # first value >= a
    hi = np.minimum(hi, 126)
    lo = np.maximum(hi - 1, 0)
    d_lo = a - _POS_VALS[lo]
    d_hi = _POS_VALS[hi] - a
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & ((_POS_CODES[hi] & 1) == 0))
    code = np.where(take_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.uint8)
    code = np.where(np.signbit(q), code | 0x80, code)
    return np.where(np.isnan(q), np.uint8(0x7F), code).astype(np.uint8)


def quantize(x, scale) -> np.ndarray:
    """Codes of x [..., n_kv, hd] with one scale per KV head (scale [n_kv]): the quotient is
    taken in fp32, then encoded."""
    x32 = np.asarray(x, dtype=np.float32)
    s32 = np.asarray(scale, dtype=np.float32)[:, None]
    return e4m3_encode((x32 / s32).astype(np.float64))


def dequantize(code, scale) -> np.ndarray:
    """code * s in fp64 for codes [..., n_kv, hd] and scale [n_kv]."""
    return e4m3_decode(code) * np.asarray(scale, dtype=np.float32).astype(np.float64)[:, None]


def kv_quant_fn(k_scale, v_scale):
    """(k_new, v_new) -> their stored values, for block_forward / stack_decode_step."""
    def f(k_new, v_new):
        return dequantize(quantize(k_new, k_scale), k_scale), dequantize(quantize(v_new, v_scale), v_scale)
    return f

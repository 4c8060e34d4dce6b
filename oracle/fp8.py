"""FP8 (E4M3) quantised base for the layer: the definition the GPU path is checked against.

TEST INFRASTRUCTURE (part of the oracle package).  Plain numpy, written from the format's
definition; it shares no code with the library.

"Multi-LoRA Serving 与 Adapter 隔离", section on quantisation, TP and loading: an INT4/FP8
base with an FP16 LoRA is the usual mixed precision; the quantised product X W_q and the
LoRA term must meet in an accumulator and epilogue the kernel supports, and a float delta
is never added in place to the packed quantised weights.  The reading taken (c17):

    y[i,n] = sx[i] sw[n] sum_k xq[i,k] wq[k,n]  +  delta[i,n]

- W is quantised once per output column n: sw[n] = max_k |W[k,n]| / 448 (fp32; 1 if the
  column is zero), wq[k,n] = e4m3(W[k,n] / sw[n]);
- x is quantised per row i each forward the same way: sx[i] = max_k |x[i,k]| / 448;
- e4m3 is the OCP 8-bit float with 4 exponent bits (bias 7) and 3 mantissa bits, largest
  finite 448, no infinities; values are rounded to nearest, ties to even, and saturated to
  +-448;
- the scales and the divisions are fp32 (IEEE, correctly rounded): the quantised codes are
  integers decided by floating point, so both sides decide them in the same precision;
- the LoRA delta is computed from the unquantised x (bf16) with the fp32 rank buffer, as
  in the plain layer.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL_EXP = -6   # smallest normal 2^-6
E4M3_MANT_BITS = 3


def e4m3_round(v) -> np.ndarray:
    """Round fp32 values to the nearest e4m3 value (ties to even), saturating at +-448.
    Returns the rounded values as float64 (exact)."""
    v = np.asarray(v, dtype=np.float32).astype(np.float64)
    a = np.abs(v)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, E4M3_MIN_NORMAL_EXP)          # subnormals share the quantum 2^-9
    q = np.exp2(e - E4M3_MANT_BITS)                 # spacing of e4m3 values near |v|
    r = np.rint(a / q) * q                           # a / q is exact (q a power of two)
    r = np.minimum(r, E4M3_MAX)                      # saturate (no infinities in e4m3)
    return np.copysign(r, v)


def _scales(amax) -> np.ndarray:
    amax = np.asarray(amax, dtype=np.float32)
    s = (amax / np.float32(E4M3_MAX)).astype(np.float32)
    return np.where(amax > 0, s, np.float32(1.0)).astype(np.float32)


def quantize_rows(x):
    """x [T,K] -> (xq [T,K] e4m3 values as float64, sx [T] fp32)."""
    x = np.asarray(x, dtype=np.float32)
    sx = _scales(np.abs(x).max(axis=1) if x.shape[1] else np.zeros(x.shape[0]))
    xq = e4m3_round((x / sx[:, None]).astype(np.float32))
    return xq, sx


def quantize_cols(W):
    """W [K,N] -> (wq [K,N] e4m3 values as float64, sw [N] fp32)."""
    W = np.asarray(W, dtype=np.float32)
    sw = _scales(np.abs(W).max(axis=0))
    wq = e4m3_round((W / sw[None, :]).astype(np.float32))
    return wq, sw


def base_w8a8(x, W) -> np.ndarray:
    """The quantised base product in fp64: sx[i] sw[n] (xq wq)[i,n]."""
    xq, sx = quantize_rows(x)
    wq, sw = quantize_cols(W)
    return (xq @ wq) * sx.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :]

"""FP8 rounding and per-block quantisation for the oracle (fp64 values).

TEST INFRASTRUCTURE, like the rest of this package (see oracle/attention.py).

The FlashAttentionScore operator doc (gitcode ops-transformer, parameter
table) takes FP8 query / key / value with full-quantisation scales d_scale_q,
d_scale_k, d_scale_v.  The FlashAttentionScoreGrad test write-up (section 5.1)
says how the golden forms them: along S in blocks of 128 rows, scale =
FP8_MAX / max |x| over the block (FP8_MAX 57344 for e5m2, 448 for e4m3fn; the
maximum floored at 1e-8), x_q = fp8(x * scale), and d_scale = 1 / scale; the
products then dequantise block by block while they accumulate, which in exact
arithmetic is attention on x_q * d_scale.

The two formats, from their bit layouts:
  e4m3fn  1 sign, 4 exponent (bias 7), 3 mantissa bits; normals 2^-6 .. 448,
          subnormals in steps of 2^-9; no infinity (overflow gives NaN)
  e5m2    1 sign, 5 exponent (bias 15), 2 mantissa bits; normals 2^-14 ..
          57344, subnormals in steps of 2^-16; overflow gives infinity
Rounding is to nearest, ties to even.
"""
from __future__ import annotations

import numpy as np

FORMATS = {
    # mantissa bits, smallest normal exponent, largest finite value, overflow value
    "e4m3fn": (3, -6, 448.0, np.nan),
    "e5m2": (2, -14, 57344.0, np.inf),
}
BLOCK = 128
EPSILON = 1e-8


def round_fp8(x: np.ndarray, fmt: str) -> np.ndarray:
    """Nearest fp8 value (ties to even) of every element, as float64."""
    mbits, emin, vmax, over = FORMATS[fmt]
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, emin)                       # subnormals share the smallest exponent's step
    ulp = np.exp2(e - mbits)
    r = np.round(a / ulp) * ulp                   # numpy rounds halves to even
    # the largest value representable before overflow: halfway to the next binade step
    limit = vmax + np.exp2(np.floor(np.log2(vmax)) - mbits) / 2
    out = np.where(a >= limit, over, r)
    if fmt == "e4m3fn":
        out = np.where((a > vmax) & (a < limit), vmax, out)
    return np.copysign(out, x)


def block_quant(x: np.ndarray, fmt: str, block: int = BLOCK):
    """Quantise x [..., S, D] per block of ``block`` rows along S.
    Returns (x_q [..., S, D] fp8 values as float64, d_scale [..., ceil(S/block)])."""
    mbits, emin, vmax, over = FORMATS[fmt]
    x = np.asarray(x, dtype=np.float64)
    S = x.shape[-2]
    nb = (S + block - 1) // block
    xq = np.empty_like(x)
    ds = np.empty(x.shape[:-2] + (nb,))
    for t in range(nb):
        blk = x[..., t * block:(t + 1) * block, :]
        mx = np.maximum(np.abs(blk).max(axis=(-2, -1)), EPSILON)
        scale = vmax / mx
        xq[..., t * block:(t + 1) * block, :] = round_fp8(blk * scale[..., None, None], fmt)
        ds[..., t] = 1.0 / scale
    return xq, ds


def dequant(xq: np.ndarray, d_scale: np.ndarray, block: int = BLOCK) -> np.ndarray:
    """x_q * d_scale of its block (the values the products consume)."""
    S = xq.shape[-2]
    rep = np.repeat(d_scale, block, axis=-1)[..., :S]
    return xq * rep[..., None]

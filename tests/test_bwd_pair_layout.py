"""Host checks of the backward's pair layout (no GPU).

fa_bwd writes P and dS as hi + lo pairs of the inputs' 16-bit type in place
over the fp32 S and dP: element j of a row becomes the 16-bit values 2j (hi)
and 2j + 1 (lo) of the same four bytes.  Read as 16-bit, a row is then 2 nc
interleaved values, and one GEMM per product takes both parts:
  dV2 = P2^T dO (row 2j + e: the hi (e = 0) or lo part of key j), dV = the
  row-pair sums; dQ = dS2 K2 with K2 every row of K twice.
These tests restate that bookkeeping in numpy with the same index
conventions and check it against the two-product form sum_e part_e^T dO and
sum_e part_e K, and the precision of the split itself.
"""
import numpy as np
import pytest

from attention_forward_fa_gb300 import workloads as W


def _split(x, dtype):
    """hi = round(x), lo = round(x - hi) in `dtype`, as bit patterns and values."""
    hb = W.to_bits(x, dtype)
    h = W.bits_to_f64(hb, dtype)
    lb = W.to_bits(x - h, dtype)
    return hb, lb, h, W.bits_to_f64(lb, dtype)


def _interleaved(hb, lb):
    """The fp32 words hi | lo << 16, read back as 16-bit: [..., 2 n]."""
    words = hb.astype(np.uint32) | (lb.astype(np.uint32) << 16)
    return words.view("<u2")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_pairs_in_place_read_as_interleaved_rows(dtype):
    rng = np.random.default_rng(5)
    x = rng.random((3, 40)) * rng.choice([1e-3, 1.0], size=(3, 40))
    hb, lb, _, _ = _split(x, dtype)
    u = _interleaved(hb, lb)
    assert u.shape == (3, 80)
    assert np.array_equal(u[:, 0::2], hb) and np.array_equal(u[:, 1::2], lb)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_one_gemm_per_product_equals_the_two_part_sums(dtype):
    rng = np.random.default_rng(6)
    nr, nc, D = 24, 40, 16
    p = rng.random((nr, nc))                       # P (or dS) of a row block
    k = W.bits_to_f64(W.to_bits(rng.standard_normal((nc, D)), dtype), dtype)
    do = W.bits_to_f64(W.to_bits(rng.standard_normal((nr, D)), dtype), dtype)
    hb, lb, h, lo = _split(p, dtype)
    p2 = W.bits_to_f64(_interleaved(hb, lb), dtype)   # [nr, 2 nc]
    k2 = np.repeat(k, 2, axis=0)                      # every row twice: [2 nc, D]
    # dQ-like: P2 K2 against hi K + lo K
    np.testing.assert_allclose(p2 @ k2, h @ k + lo @ k, rtol=0, atol=1e-12)
    # dV-like: P2^T dO with rows 2j + e, summed over e, against (hi + lo)^T dO
    dv2 = p2.T @ do
    np.testing.assert_allclose(dv2[0::2] + dv2[1::2], (h + lo).T @ do, rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv2[0::2], h.T @ do, rtol=0, atol=1e-12)


@pytest.mark.parametrize("dtype,bits,floor", [("bf16", 16, 0.0), ("fp16", 21, 2.0 ** -25)])
def test_pair_precision(dtype, bits, floor):
    """hi + lo carries about twice the type's significand: |x - (hi + lo)| <=
    2^-bits |x|.  fp16's lo part reaches the subnormals once |x| is below
    ~2^-3, which leaves an absolute floor of half the smallest subnormal
    spacing (2^-25); bf16 has fp32's exponent range and no such floor."""
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.random(4000) * 0.999 + 2.0 ** -10, rng.standard_normal(4000) * 30])
    _, _, h, lo = _split(x, dtype)
    err = np.abs(x - (h + lo))
    assert bool(np.all(err <= np.maximum(2.0 ** -bits * np.abs(x), floor)))
    big = np.abs(x) >= 0.125
    assert float(np.max(err[big] / np.abs(x[big]))) <= 2.0 ** -bits
    assert float(np.max(np.abs(x - h) / np.abs(x))) > 2.0 ** -(bits // 2 + 2)   # hi alone is not enough

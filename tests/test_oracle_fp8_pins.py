"""Pins of oracle/fp8.py (FP8 rounding and per-block quantisation).

* round_fp8 equals torch's float8_e4m3fn / float8_e5m2 casts (a library
  routine) on values across every magnitude, the subnormals, ties and the
  overflow region (e4m3fn: NaN, e5m2: inf);
* every finite e4m3fn and e5m2 value, enumerated from the bit layouts, rounds
  to itself, and the midpoint between two neighbours rounds to the even one;
* block_quant maps each 128-row block's largest magnitude to +-FP8_MAX,
  d_scale = max / FP8_MAX, and dequantised values are within half an fp8 step
  of the input.
"""
import numpy as np
import pytest

from oracle import fp8 as F

torch = pytest.importorskip("torch")
TORCH_DT = {"e4m3fn": "float8_e4m3fn", "e5m2": "float8_e5m2"}


def _all_finite(fmt):
    mbits, emin, vmax, _ = F.FORMATS[fmt]
    vals = [0.0]
    vals += [m * 2.0 ** (emin - mbits) for m in range(1, 2 ** mbits)]                    # subnormals
    e = emin
    while True:
        row = [(1 + m / 2 ** mbits) * 2.0 ** e for m in range(2 ** mbits)]
        row = [x for x in row if x <= vmax]
        if not row:
            break
        vals += row
        e += 1
    vals = np.array(sorted(set(vals)))
    return np.concatenate([-vals[::-1], vals])


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_rounding_equals_torch_casts(fmt):
    dt = getattr(torch, TORCH_DT[fmt], None)
    if dt is None:
        pytest.skip("torch without fp8 dtypes")
    vmax = F.FORMATS[fmt][2]
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(5000) * s for s in (1e-5, 1e-3, 0.1, 1, 20, vmax / 3, vmax)])
    x = x.astype(np.float32).astype(np.float64)           # torch casts from fp32
    ref = torch.from_numpy(x.astype(np.float32)).to(dt).float().double().numpy()
    got = F.round_fp8(x, fmt)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), (x[~same][:5], got[~same][:5], ref[~same][:5])


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_grid_values_and_midpoints(fmt):
    v = _all_finite(fmt)
    assert np.array_equal(F.round_fp8(v, fmt), v)
    assert v.max() == F.FORMATS[fmt][2]
    mid = (v[1:] + v[:-1]) / 2
    got = F.round_fp8(mid, fmt)
    lo, hi = v[:-1], v[1:]
    # ties go to the neighbour whose last mantissa bit is 0
    mbits = F.FORMATS[fmt][0]

    def even(x):
        a = np.abs(x)
        e = np.maximum(np.floor(np.log2(np.where(a > 0, a, 1.0))), F.FORMATS[fmt][1])
        return (np.round(a / 2.0 ** (e - mbits)).astype(np.int64) % 2) == 0
    want = np.where(even(lo), lo, hi)
    nz = (lo != 0) | (hi != 0)
    assert np.array_equal(got[nz], want[nz])


@pytest.mark.parametrize("fmt", ["e4m3fn", "e5m2"])
def test_block_quantisation(fmt):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2, 3, 300, 64)) * np.exp(rng.standard_normal((2, 3, 300, 1)))
    xq, ds = F.block_quant(x, fmt)
    assert ds.shape == (2, 3, 3)
    vmax = F.FORMATS[fmt][2]
    for t in range(3):
        blk = x[..., t * 128:(t + 1) * 128, :]
        qb = xq[..., t * 128:(t + 1) * 128, :]
        assert np.allclose(np.abs(qb).max(axis=(-2, -1)), vmax)
        assert np.allclose(ds[..., t], np.abs(blk).max(axis=(-2, -1)) / vmax, rtol=1e-15)
    back = F.dequant(xq, ds)
    mbits = F.FORMATS[fmt][0]
    # half a step of the scaled value, back in the input's units (normal range)
    rel = np.abs(back - x) / np.maximum(np.abs(x), 1e-300)
    scaled = np.abs(x) / np.repeat(ds, 128, axis=-1)[..., :300, None]
    normal = scaled >= 2.0 ** F.FORMATS[fmt][1]
    assert (rel[normal] <= 2.0 ** -(mbits + 1) * (1 + 1e-12)).all()

"""Error metrics of the sparse-MLA exact-max page (cf-1.com), section
"Measurement: magnitude of the coherent error" and "Meaning of the noise floor".

TEST INFRASTRUCTURE (see oracle/attention.py).

* row gain of one output row x against its reference r: <x - r, r> / <r, r>,
  the coherent (whole-row) component of the error;
* rel-L2: ||x - r|| / ||r|| over the whole output;
* bf16 output floor: the rel-L2 (or row-gain rms) of bf16(r) against r;
* noise floor of the difference of two outputs: elem_rms * sqrt(3 / D) with
  elem_rms the relative rms of the elementwise difference and D the output
  width; the coherent part of the difference is the rms row gain of
  (x_a - x_b) projected on r.

Reading: the page does not say how elem_rms is normalised.  It is taken per
row (rms of the row's difference over rms of the row's reference), then rms
over rows; with that reading the emulation in online.py reproduces the page's
ratios 1.05 (exact max) and 6.4 (lazy) to within a few percent, while a global
normalisation gives 2.6 and 8.4.
"""
from __future__ import annotations

import numpy as np

from .online import round_bf16


def row_gain(x: np.ndarray, ref: np.ndarray) -> np.ndarray:
    """Per-row <x - ref, ref> / <ref, ref> over the last axis (rows with
    ref == 0 give 0)."""
    num = ((x - ref) * ref).sum(axis=-1)
    den = (ref * ref).sum(axis=-1)
    return np.where(den > 0, num / np.where(den > 0, den, 1.0), 0.0)


def rms(a: np.ndarray) -> float:
    a = np.asarray(a, dtype=np.float64)
    return float(np.sqrt(np.mean(a * a))) if a.size else 0.0


def rel_l2(x: np.ndarray, ref: np.ndarray) -> float:
    return float(np.linalg.norm((x - ref).ravel()) / np.linalg.norm(ref.ravel()))


def bf16_output_floor(ref: np.ndarray) -> float:
    """rel-L2 of bf16(ref) against ref."""
    return rel_l2(round_bf16(ref), ref)


def bf16_row_gain_floor(ref: np.ndarray) -> float:
    """rms row gain of bf16(ref) against ref."""
    return rms(row_gain(round_bf16(ref), ref))


def order_difference(x_a: np.ndarray, x_b: np.ndarray, ref: np.ndarray):
    """(coherent, floor) for the difference of two outputs of the same problem.

    coherent = rms over rows of <x_a - x_b, ref> / <ref, ref>;
    floor    = elem_rms * sqrt(3 / D), elem_rms = sqrt(mean over rows of
               mean(d_row^2) / mean(ref_row^2)).
    """
    d = x_a - x_b
    den = (ref * ref).sum(axis=-1)
    ok = den > 0
    g = np.where(ok, (d * ref).sum(axis=-1) / np.where(ok, den, 1.0), 0.0)
    rel = np.where(ok, (d * d).sum(axis=-1) / np.where(ok, den, 1.0), 0.0)
    elem = float(np.sqrt(np.mean(rel[ok]))) if ok.any() else 0.0
    D = ref.shape[-1]
    return rms(g[ok]), elem * np.sqrt(3.0 / D)

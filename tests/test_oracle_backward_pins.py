"""Pins of the backward oracle (oracle/backward.py) against mathematics that
does not depend on it.

* Central finite differences of the forward oracle (itself pinned in
  test_oracle_pins.py) for L = sum(O * dO), on tiny problems covering every
  variant: dense, causal with per-batch lengths (padded rows and keys), GQA,
  block lists with invalid and duplicate slots and the diagonal-block mask,
  top-k lists with duplicates and invalid slots, and the shared MLA latent
  (V = the first Dv columns of K).
* A closed form: with one valid key per row, P = 1, so dQ = dK = 0 and dV of
  a key is the sum of dO over the rows that list it.
* An invariant: every row of dS sums to zero, so dK summed over the keys of a
  KV head is zero.
* Planted mistakes (dV scaled, d_row dropped, GQA sum replaced by the last
  head, scale missing on dK) must each fail the finite differences, which
  shows that the check can see them.
"""
import numpy as np
import pytest

from oracle import attention as A
from oracle import backward as BW

SCALE = 0.37


def _loss(q, k, v, do, **kw):
    o, _ = A.attention_fwd(q, k, v, SCALE, **kw)
    return float(np.nansum(np.where(np.isnan(o), 0.0, o) * do))


def _fd(x, f, eps=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        x0 = x[i]
        x[i] = x0 + eps
        fp = f()
        x[i] = x0 - eps
        fm = f()
        x[i] = x0
        g[i] = (fp - fm) / (2 * eps)
    return g


def _close(a, b):
    return np.allclose(a, b, rtol=1e-6, atol=1e-8)


def _problem(seed, B=1, Hq=2, Hkv=1, Sq=5, Skv=6, D=3, Dv=4):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, Hq, Sq, D))
    k = rng.standard_normal((B, Hkv, Skv, D))
    v = rng.standard_normal((B, Hkv, Skv, Dv))
    do = rng.standard_normal((B, Hq, Sq, Dv))
    return q, k, v, do


CASES = {
    "dense_gqa": dict(shape=dict(Hq=4, Hkv=2), kw={}),
    "causal_seqlens": dict(shape=dict(B=2, Sq=6, Skv=6),
                           kw=dict(mask=A.MASK_CAUSAL, seqlens=np.array([6, 4]))),
    "cross_lengths_causal": dict(shape=dict(Sq=4, Skv=7), kw=dict(mask=A.MASK_CAUSAL)),
    "block_lists": dict(
        shape=dict(Sq=6, Skv=8),
        kw=dict(mask=A.MASK_CAUSAL_DIAG_BLOCK, block=2,
                # [B, 1, ceil(Sq/2), max_sel]: invalid (-1, 9) and duplicate slots
                kv_block_idx=np.array([[[[0, -1, 0], [1, 0, 9], [2, 3, 1]]]]))),
    "topk": dict(
        shape=dict(Sq=5, Skv=6),
        kw=dict(topk_idx=np.array([[[0, 0, -1], [1, 0, 4], [2, 7, 1], [3, 3, 3], [5, 2, 0]]]))),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_backward_matches_finite_differences(case):
    c = CASES[case]
    q, k, v, do = _problem(11 + len(case), **c["shape"])
    kw = c["kw"]
    o, lse = A.attention_fwd(q, k, v, SCALE, **kw)
    dq, dk, dv = BW.attention_bwd(q, k, v, o, lse, do, SCALE, **kw)
    f = lambda: _loss(q, k, v, do, **kw)
    assert _close(dq, _fd(q, f))
    assert _close(dk, _fd(k, f))
    assert _close(dv, _fd(v, f))


def test_shared_latent_gradient_matches_finite_differences():
    # sparse MLA: V is the first Dv columns of the key latent (one KV head)
    q, k, _, do = _problem(5, Hq=3, Hkv=1, Sq=4, Skv=5, D=6, Dv=4)
    tk = np.array([[[0, 4, -1], [1, 1, 2], [3, 0, 2], [2, 4, 1]]])
    f = lambda: _loss(q, k, k[..., :4], do, topk_idx=tk)
    o, lse = A.attention_fwd(q, k, k[..., :4], SCALE, topk_idx=tk)
    dq, dk, dv = BW.attention_bwd(q, k, k[..., :4], o, lse, do, SCALE, topk_idx=tk)
    assert _close(BW.latent_grad(dk, dv), _fd(k, f))
    assert _close(dq, _fd(q, f))


def test_one_key_per_row_closed_form():
    q, k, v, do = _problem(7, Hq=2, Hkv=1, Sq=5, Skv=5)
    tk = np.array([[[2], [0], [2], [4], [-1]]])   # row 4 has no valid key
    o, lse = A.attention_fwd(q, k, v, SCALE, topk_idx=tk)
    dq, dk, dv = BW.attention_bwd(q, k, v, o, lse, do, SCALE, topk_idx=tk)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13
    want = np.zeros_like(dv)
    for i, j in enumerate(tk[0, :, 0]):
        if j >= 0:
            want[0, 0, j] += do[0, :, i].sum(axis=0)
    assert np.allclose(dv, want, rtol=0, atol=1e-13)


def test_key_gradients_sum_to_zero():
    q, k, v, do = _problem(9, B=2, Hq=4, Hkv=2, Sq=7, Skv=9, D=5, Dv=3)
    o, lse = A.attention_fwd(q, k, v, SCALE, mask=A.MASK_CAUSAL, seqlens=np.array([7, 5]))
    _, dk, _ = BW.attention_bwd(q, k, v, o, lse, do, SCALE, mask=A.MASK_CAUSAL,
                                seqlens=np.array([7, 5]))
    assert np.abs(dk.sum(axis=2)).max() < 1e-12


def test_planted_mistakes_fail_the_finite_differences():
    q, k, v, do = _problem(13, Hq=4, Hkv=2, Sq=5, Skv=6)
    kw = dict(mask=A.MASK_CAUSAL)
    o, lse = A.attention_fwd(q, k, v, SCALE, **kw)
    dq, dk, dv = BW.attention_bwd(q, k, v, o, lse, do, SCALE, **kw)
    f = lambda: _loss(q, k, v, do, **kw)
    fq, fk, fv = _fd(q, f), _fd(k, f), _fd(v, f)
    assert _close(dq, fq) and _close(dk, fk) and _close(dv, fv)
    assert not _close(SCALE * dv, fv)                       # dV scaled like dQ / dK
    # d_row dropped: dS = P * dP
    G = 2
    dq_bad = np.zeros_like(dq)
    dk_last = np.zeros_like(dk)
    for h in range(4):
        kh = h // G
        s = q[0, h] @ k[0, kh].T
        w = A._multiplicity(np.arange(5), 0, h, 5, 6, 6, 1, 128, A.MASK_CAUSAL, None, None)
        p = w * np.exp(SCALE * s - lse[0, h][:, None])
        dq_bad[0, h] = SCALE * ((p * (do[0, h] @ v[0, kh].T)) @ k[0, kh])
        ds = p * (do[0, h] @ v[0, kh].T - (do[0, h] * o[0, h]).sum(-1)[:, None])
        dk_last[0, kh] = SCALE * (ds.T @ q[0, h])          # last head only, no group sum
    assert not _close(dq_bad, fq)
    assert not _close(dk_last, fk)
    assert not _close(dk / SCALE, fk)                        # scale missing on dK

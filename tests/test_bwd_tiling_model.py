"""CPU model of the backward kernels' tiling (attention_forward_fa_gb300/csrc/
fa_bwd.cuh), written out step by step: which CTA owns which tile, which tiles
each step visits, the per-element masks, and which output rows each thread
writes.  It checks, before any GPU run, that

* the dK / dV kernel (one CTA per batch, KV head and 128-key tile, walking the
  query tiles of every head of the GQA group) and the dQ kernel (one CTA per
  batch, head and 128-row query tile, walking key tiles) each cover every
  valid (query, key) pair exactly once and no invalid pair;
* every output row is written exactly once, inside its tensor;
* TMA box coordinates address an existing plane (rows past the tensor are
  allowed: they read as zero);
* and, recomputing the products tile by tile from these pieces in float64,
  the result is the backward oracle's.
The model shares no code with the kernels; it follows their index arithmetic.
"""
import numpy as np
import pytest

from oracle import attention as A
from oracle import backward as BW

T = 128


def dense_tiles(qt, n_qt, q_len, kv_len, causal):
    q0 = qt * T
    if qt >= n_qt or q0 >= q_len or kv_len <= 0:
        return 0
    nkv = (kv_len + T - 1) // T
    if causal:
        nkv = min(nkv, min(q0 + T - 1, q_len - 1) // T + 1)
    return nkv


def dkdv_model(B, Hq, Hkv, Sq, Skv, causal, seqlens):
    """Yields (b, kvh, h, kt, qt, P-mask [128 keys x 128 queries], key rows written)."""
    G = Hq // Hkv
    n_kt = (Skv + T - 1) // T
    per_kt = B * Hkv
    for blk in range(n_kt * per_kt):
        kt, bk = divmod(blk, per_kt)
        b, kvh = divmod(bk, Hkv)
        q_len = Sq if seqlens is None else min(seqlens[b], Sq)
        kv_len = Skv if seqlens is None else min(seqlens[b], Skv)
        k0 = kt * T
        qt_hi = (q_len + T - 1) // T
        qt_lo = kt if causal else 0
        nq = qt_hi - qt_lo if (k0 < kv_len and qt_hi > qt_lo) else 0
        steps = []
        for n in range(nq * G):
            g, r = divmod(n, nq)
            qt = qt_lo + r
            h = kvh * G + g
            assert 0 <= b * Hq + h < B * Hq and 0 <= b * Hkv + kvh < B * Hkv   # TMA planes
            q0 = qt * T
            rows = np.arange(T)
            kj = k0 + rows[:, None]             # key of thread `row`
            qi = q0 + rows[None, :]             # query column i
            lim = kj - q0 if causal else -1
            mask = (kj < kv_len) & (rows[None, :] >= lim) & (qi < q_len)   # LSE +inf past q_len
            hilo = G > 1 or (min(q0 + 1, kv_len) if causal else kv_len) < 512
            steps.append((h, qt, mask, hilo))
        written = [k0 + r for r in range(T) if k0 + r < Skv]
        yield b, kvh, kt, steps, written


def dq_model(B, Hq, Hkv, Sq, Skv, causal, seqlens):
    G = Hq // Hkv
    n_qt = (Sq + T - 1) // T
    per_qt = B * Hq
    for blk in range(n_qt * per_qt):
        qt = n_qt - 1 - blk // per_qt
        b, h = divmod(blk % per_qt, Hq)
        kvh = h // G
        q_len = Sq if seqlens is None else min(seqlens[b], Sq)
        kv_len = Skv if seqlens is None else min(seqlens[b], Skv)
        q0 = qt * T
        nsteps = dense_tiles(qt, n_qt, q_len, kv_len, causal)
        steps = []
        for n in range(nsteps):
            kbase = n * T
            rows = np.arange(T)
            qi = q0 + rows[:, None]
            lim = np.minimum(kv_len - kbase, qi - kbase + 1 if causal else T)
            mask = (np.arange(T)[None, :] < lim) & (qi < q_len)
            steps.append((n, mask))
        written = [q0 + r for r in range(T) if q0 + r < Sq]
        yield b, h, kvh, qt, steps, written


def valid_pairs(b, Sq, Skv, causal, seqlens):
    q_len = Sq if seqlens is None else min(seqlens[b], Sq)
    kv_len = Skv if seqlens is None else min(seqlens[b], Skv)
    i = np.arange(Sq)[:, None]
    j = np.arange(Skv)[None, :]
    v = (i < q_len) & (j < kv_len)
    if causal:
        v &= j <= i
    return v


CASES = [
    dict(B=1, Hq=2, Hkv=2, Sq=384, Skv=384, causal=True, seqlens=None),
    dict(B=2, Hq=4, Hkv=2, Sq=300, Skv=300, causal=True, seqlens=[300, 129]),
    dict(B=1, Hq=3, Hkv=1, Sq=200, Skv=333, causal=False, seqlens=None),
    dict(B=1, Hq=2, Hkv=1, Sq=130, Skv=500, causal=True, seqlens=None),
    dict(B=2, Hq=2, Hkv=2, Sq=256, Skv=256, causal=False, seqlens=[1, 256]),
]


@pytest.mark.parametrize("c", CASES, ids=[f"case{i}" for i in range(len(CASES))])
def test_tiles_cover_every_valid_pair_once(c):
    B, Hq, Hkv, Sq, Skv, causal, sl = (c[k] for k in ("B", "Hq", "Hkv", "Sq", "Skv", "causal", "seqlens"))
    # dK / dV: per (b, query head) count how often each (query, key) pair is visited
    cover = np.zeros((B, Hq, Sq + T, Skv + T), int)
    rows_kv = np.zeros((B, Hkv, Skv), int)
    for b, kvh, kt, steps, written in dkdv_model(B, Hq, Hkv, Sq, Skv, causal, sl):
        for h, qt, mask, _ in steps:
            cover[b, h, qt * T:qt * T + T, kt * T:kt * T + T] += mask.T
        for r in written:
            rows_kv[b, kvh, r] += 1
    cover_q = np.zeros_like(cover)
    rows_q = np.zeros((B, Hq, Sq), int)
    for b, h, kvh, qt, steps, written in dq_model(B, Hq, Hkv, Sq, Skv, causal, sl):
        for n, mask in steps:
            cover_q[b, h, qt * T:qt * T + T, n * T:n * T + T] += mask
        for r in written:
            rows_q[b, h, r] += 1
    for b in range(B):
        want = valid_pairs(b, Sq, Skv, causal, sl)
        for h in range(Hq):
            assert np.array_equal(cover[b, h, :Sq, :Skv], want.astype(int))
            assert np.array_equal(cover_q[b, h, :Sq, :Skv], want.astype(int))
            assert not cover[b, h, Sq:].any() and not cover[b, h, :, Skv:].any()
            assert not cover_q[b, h, Sq:].any() and not cover_q[b, h, :, Skv:].any()
    assert (rows_kv == 1).all() and (rows_q == 1).all()


@pytest.mark.parametrize("c", CASES[:3], ids=[f"case{i}" for i in range(3)])
def test_tiled_products_equal_the_oracle(c):
    B, Hq, Hkv, Sq, Skv, causal, sl = (c[k] for k in ("B", "Hq", "Hkv", "Sq", "Skv", "causal", "seqlens"))
    rng = np.random.default_rng(5)
    q = rng.standard_normal((B, Hq, Sq, T))
    k = rng.standard_normal((B, Hkv, Skv, T))
    v = rng.standard_normal((B, Hkv, Skv, T))
    do = rng.standard_normal((B, Hq, Sq, T))
    scale = 0.09
    seqlens = None if sl is None else np.array(sl)
    mask = A.MASK_CAUSAL if causal else A.MASK_NONE
    o, lse = A.attention_fwd(q, k, v, scale, mask=mask, seqlens=seqlens)
    rq, rk, rv = BW.attention_bwd(q, k, v, o, lse, do, scale, mask=mask, seqlens=seqlens)
    o0 = np.nan_to_num(o)
    pad = lambda x, n: np.concatenate([x, np.zeros((n - x.shape[0],) + x.shape[1:])]) if x.shape[0] < n else x
    dk = np.zeros_like(rk)
    dv = np.zeros_like(rv)
    for b, kvh, kt, steps, written in dkdv_model(B, Hq, Hkv, Sq, Skv, causal, sl):
        K = pad(k[b, kvh, kt * T:kt * T + T], T)
        V = pad(v[b, kvh, kt * T:kt * T + T], T)
        acc_v = np.zeros((T, T))
        acc_k = np.zeros((T, T))
        for h, qt, m, _ in steps:
            Q = pad(q[b, h, qt * T:qt * T + T], T)
            dO = pad(do[b, h, qt * T:qt * T + T], T)
            L = pad(lse[b, h, qt * T:qt * T + T], T)
            D = pad((do[b, h] * o0[b, h]).sum(-1)[qt * T:qt * T + T], T)
            with np.errstate(over="ignore", invalid="ignore"):
                pt = np.where(m, np.exp(scale * (K @ Q.T) - np.where(np.isfinite(L), L, 0)[None, :]), 0.0)
            dst = pt * ((V @ dO.T) - D[None, :])
            acc_v += pt @ dO
            acc_k += dst @ Q
        for r in written:
            dv[b, kvh, r] = acc_v[r - kt * T] if r < (Skv if sl is None else min(sl[b], Skv)) else 0
            dk[b, kvh, r] = scale * acc_k[r - kt * T] if r < (Skv if sl is None else min(sl[b], Skv)) else 0
    dq = np.zeros_like(rq)
    for b, h, kvh, qt, steps, written in dq_model(B, Hq, Hkv, Sq, Skv, causal, sl):
        Q = pad(q[b, h, qt * T:qt * T + T], T)
        dO = pad(do[b, h, qt * T:qt * T + T], T)
        L = pad(lse[b, h, qt * T:qt * T + T], T)
        D = pad((do[b, h] * o0[b, h]).sum(-1)[qt * T:qt * T + T], T)
        acc = np.zeros((T, T))
        for n, m in steps:
            K = pad(k[b, kvh, n * T:n * T + T], T)
            V = pad(v[b, kvh, n * T:n * T + T], T)
            with np.errstate(over="ignore", invalid="ignore"):
                p = np.where(m, np.exp(scale * (Q @ K.T) - np.where(np.isfinite(L), L, 0)[:, None]), 0.0)
            acc += (p * ((dO @ V.T) - D[:, None])) @ K
        q_len = Sq if sl is None else min(sl[b], Sq)
        for r in written:
            dq[b, h, r] = scale * acc[r - qt * T] if r < q_len else 0
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        assert np.allclose(got, ref, rtol=1e-9, atol=1e-12)

"""Pins of the oracle's optional terms (oracle.attention.Extras: attention
mask, position bias, ALiBi, sparse-mode windows, dropout) and of the Philox
dropout generator, against results fixed independently of that code:

* masks and windows equal the plain causal oracle, or a boolean mask built
  element by element in pure Python;
* a per-row constant bias leaves O alone and moves LSE by the constant (scaled
  or not, by pse_type); a bias of ln 2 on one key equals duplicating that key;
* with zero scores, ALiBi rows are two-sided geometric (type 2) or decay as
  sqrt of the distance (type 3), with slopes in the ratio 2^(-8/Hq);
* dropout: O = (P * M / keep_prob) V from the oracle's own P, LSE unchanged;
* Philox4x32-10 reproduces the published known-answer vectors of its
  authors (Salmon et al., SC 2011), and its masks keep about keep_prob;
* the backward with every term matches central finite differences of the
  forward.
"""
import numpy as np
import pytest

from oracle import attention as A
from oracle import backward as BW
from oracle.attention import Extras

SCALE = 0.3


def _qkv(seed, B=1, Hq=2, Hkv=1, Sq=6, Skv=6, D=4, Dv=3):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, Hq, Sq, D)), rng.standard_normal((B, Hkv, Skv, D)),
            rng.standard_normal((B, Hkv, Skv, Dv)))


def _mask_py(Sq, Skv, visible):
    m = np.zeros((Sq, Skv))
    for i in range(Sq):
        for j in range(Skv):
            m[i, j] = 0.0 if visible(i, j) else 1.0
    return m


def _same(a, b):
    (o1, l1), (o2, l2) = a, b
    return np.allclose(o1, o2, rtol=1e-12, atol=1e-13) and np.allclose(l1, l2, rtol=1e-12, atol=1e-13)


def test_masks_and_windows():
    q, k, v = _qkv(1, Sq=7, Skv=7)
    causal = A.attention_fwd(q, k, v, SCALE, mask=A.MASK_CAUSAL)
    m = _mask_py(7, 7, lambda i, j: j <= i)
    assert _same(A.attention_fwd(q, k, v, SCALE, extras=Extras(atten_mask=m)), causal)
    assert _same(A.attention_fwd(q, k, v, SCALE, extras=Extras(sparse_mode=2)), causal)
    assert _same(A.attention_fwd(q, k, v, SCALE, extras=Extras(sparse_mode=3)), causal)
    assert _same(A.attention_fwd(q, k, v, SCALE, extras=Extras(sparse_mode=0, next_tokens=0)), causal)
    band = _mask_py(7, 7, lambda i, j: i - 2 <= j <= i + 1)
    assert _same(A.attention_fwd(q, k, v, SCALE, extras=Extras(sparse_mode=0, pre_tokens=2, next_tokens=1)),
                 A.attention_fwd(q, k, v, SCALE, extras=Extras(atten_mask=band)))
    q, k, v = _qkv(2, Sq=4, Skv=9)
    rd = _mask_py(4, 9, lambda i, j: j <= i + 5)
    assert _same(A.attention_fwd(q, k, v, SCALE, extras=Extras(sparse_mode=3)),
                 A.attention_fwd(q, k, v, SCALE, extras=Extras(atten_mask=rd)))


def test_bottom_right_causal_follows_each_batchs_lengths():
    """With per-batch lengths the bottom-right mask aligns each sequence's
    last query with its last key: batch b is the oracle on its own cropped
    problem, whose mask is built element by element."""
    q, k, v = _qkv(3, B=2, Sq=4, Skv=9)
    seq = np.array([9, 3])       # a length applies to queries and keys, up to Sq and Skv
    o, l = A.attention_fwd(q, k, v, SCALE, seqlens=seq, extras=Extras(sparse_mode=3))
    for b, n in enumerate(seq):
        ql, kl = min(n, 4), min(n, 9)
        m = _mask_py(ql, kl, lambda i, j: j <= i + (kl - ql))   # offsets 5 and 0
        oc, lc = A.attention_fwd(q[b:b + 1, :, :ql], k[b:b + 1, :, :kl], v[b:b + 1, :, :kl],
                                 SCALE, extras=Extras(atten_mask=m))
        assert np.allclose(o[b, :, :ql], oc[0], rtol=1e-12, atol=1e-14)
        assert np.allclose(l[b, :, :ql], lc[0], rtol=1e-12, atol=1e-14)
        assert np.all(np.isinf(l[b, :, ql:]))


@pytest.mark.parametrize("pse_type, moved", [(0, 1.0), (1, SCALE)])
def test_row_constant_bias(pse_type, moved):
    q, k, v = _qkv(3)
    c = np.arange(6, dtype=np.float64)[:, None] * np.ones((1, 6)) * 0.7 - 1.1   # per-row constant
    o0, l0 = A.attention_fwd(q, k, v, SCALE)
    o1, l1 = A.attention_fwd(q, k, v, SCALE, extras=Extras(pse=c, pse_type=pse_type))
    assert np.allclose(o1, o0, rtol=1e-12, atol=1e-13)
    assert np.allclose(l1 - l0, moved * c[:, 0][None, None], rtol=1e-12, atol=1e-12)


def test_ln2_bias_equals_a_duplicated_key():
    q, k, v = _qkv(4)
    pse = np.zeros((6, 6))
    pse[:, 2] = np.log(2.0)
    o1, l1 = A.attention_fwd(q, k, v, SCALE, extras=Extras(pse=pse, pse_type=0))
    k2 = np.concatenate([k, k[:, :, 2:3]], axis=2)
    v2 = np.concatenate([v, v[:, :, 2:3]], axis=2)
    o2, l2 = A.attention_fwd(q, k2, v2, SCALE)
    assert np.allclose(o1, o2, rtol=1e-12) and np.allclose(l1, l2, rtol=1e-12)


@pytest.mark.parametrize("pse_type", [2, 3])
def test_alibi_rows_with_zero_scores(pse_type):
    Hq, S = 4, 9
    q = np.zeros((1, Hq, S, 4))
    _, k, v = _qkv(5, Hq=Hq, Sq=S, Skv=S)
    *_, P = A.attention_fwd(q, k, v, SCALE, extras=Extras(pse_type=pse_type), return_p=True)
    slopes = []
    for h in range(Hq):
        p = P[(0, h, 0)]
        i = 4
        lp = np.log(p[i])
        d = np.abs(np.arange(S) - i).astype(float)
        prof = np.sqrt(d) if pse_type == 3 else d
        slope = (lp[i] - lp[i + 1]) / 1.0           # d = 1 either way
        assert np.allclose(lp[i] - lp, slope * prof, rtol=1e-10, atol=1e-12)
        slopes.append(slope)
    r = np.array(slopes[1:]) / np.array(slopes[:-1])
    assert np.allclose(r, 2.0 ** (-8.0 / Hq), rtol=1e-10)
    assert np.isclose(slopes[0], 2.0 ** (-8.0 / Hq), rtol=1e-10)


def test_dropout_from_the_oracles_own_p():
    q, k, v = _qkv(6, Hq=2, Sq=6, Skv=7)
    rng = np.random.default_rng(7)
    m = (rng.random((1, 2, 6, 7)) < 0.7).astype(np.float64)
    o0, l0, P = A.attention_fwd(q, k, v, SCALE, mask=A.MASK_CAUSAL, return_p=True)
    o1, l1 = A.attention_fwd(q, k, v, SCALE, mask=A.MASK_CAUSAL, extras=Extras(drop_mask=m, keep_prob=0.7))
    for h in range(2):
        want = (P[(0, h, 0)] * m[0, h] / 0.7) @ v[0, 0]
        assert np.allclose(o1[0, h], want, rtol=1e-12, atol=1e-13)
    assert np.array_equal(l1, l0)
    ones = A.attention_fwd(q, k, v, SCALE, mask=A.MASK_CAUSAL, extras=Extras(drop_mask=np.ones((6, 7))))
    assert _same(ones, (o0, l0))


def test_dropout_without_a_mask_is_refused():
    """keep_prob < 1 names a dropout, which drops elements: without the mask
    that says which, the oracle refuses rather than rescale every element by
    1 / keep_prob (the formula's O = (P * M / keep_prob) V has no such case)."""
    q, k, v = _qkv(6, Hq=2, Sq=6, Skv=7)
    with pytest.raises(ValueError):
        A.attention_fwd(q, k, v, SCALE, extras=Extras(keep_prob=0.5))
    with pytest.raises(ValueError):
        BW.attention_bwd(q, k, v, *A.attention_fwd(q, k, v, SCALE), np.ones_like(q), SCALE,
                         extras=Extras(keep_prob=0.5))
    # keep_prob 1 without a mask is no dropout at all
    assert _same(A.attention_fwd(q, k, v, SCALE, extras=Extras(keep_prob=1.0)),
                 A.attention_fwd(q, k, v, SCALE))


def test_philox_dropout_mask_byte_order_worked_example():
    """One Philox block worked by hand from the authors' published answer for
    counter (0, 0, 0, 0) and key (0, 0): words 0x6627E8D5, 0xE169C58D,
    0xBC57AC4C, 0x9B00DBD8.  Seed 0 and offset 0 select exactly that block;
    taken word by word, low byte first, its 16 bytes are
    D5 E8 27 66 | 8D C5 69 E1 | 4C AC 57 BC | D8 DB 00 9B, and with
    keep_prob 0.5 an element is kept when its byte is below 127.5."""
    bytes_ = [0xD5, 0xE8, 0x27, 0x66, 0x8D, 0xC5, 0x69, 0xE1,
              0x4C, 0xAC, 0x57, 0xBC, 0xD8, 0xDB, 0x00, 0x9B]
    want = [1 if b < 127.5 else 0 for b in bytes_]
    assert want == [0, 0, 1, 1, 0, 0, 1, 0, 1, 0, 1, 0, 0, 0, 1, 0]
    assert BW.philox_dropout_mask(seed=0, offset=0, n=16, keep_prob=0.5).tolist() == want
    # keep_prob 0.9: only the bytes above 229.5 (E8 = 232) are dropped
    assert BW.philox_dropout_mask(seed=0, offset=0, n=16, keep_prob=0.9).tolist() == \
        [1 if b < 229.5 else 0 for b in bytes_]
    # n not a multiple of 16 takes the block's first bytes
    assert BW.philox_dropout_mask(seed=0, offset=0, n=5, keep_prob=0.5).tolist() == want[:5]


def test_philox_known_answers():
    assert BW.philox4x32((0, 0, 0, 0), (0, 0)) == [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]
    assert BW.philox4x32((0xFFFFFFFF,) * 4, (0xFFFFFFFF, 0xFFFFFFFF)) == \
        [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]
    assert BW.philox4x32((0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344), (0xA4093822, 0x299F31D0)) == \
        [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]


def test_philox_dropout_masks():
    m = BW.philox_dropout_mask(seed=2024, offset=0, n=16000, keep_prob=0.9)
    assert set(np.unique(m)) <= {0, 1}
    assert abs(m.mean() - 0.9 * 255 / 256) < 0.01        # bytes below 229.5 of 0..255
    assert np.array_equal(m, BW.philox_dropout_mask(2024, 0, 16000, 0.9))
    shifted = BW.philox_dropout_mask(seed=2024, offset=32, n=160, keep_prob=0.9)
    assert np.array_equal(shifted, m[32:192])             # offset / 16 advances the counter
    assert not np.array_equal(BW.philox_dropout_mask(2025, 0, 160, 0.9), m[:160])


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


EXTRA_CASES = {
    "pse0": lambda rng: Extras(pse=rng.standard_normal((1, 2, 6, 6)), pse_type=0),
    "pse1": lambda rng: Extras(pse=rng.standard_normal((6, 6)), pse_type=1),
    "alibi2": lambda rng: Extras(pse_type=2, sparse_mode=2),
    "alibi3": lambda rng: Extras(pse_type=3),
    "atten_mask": lambda rng: Extras(atten_mask=(rng.random((1, 2, 6, 6)) < 0.3).astype(float)),
    "window": lambda rng: Extras(sparse_mode=0, pre_tokens=2, next_tokens=1),
    "dropout": lambda rng: Extras(drop_mask=(rng.random((1, 2, 6, 6)) < 0.8).astype(float), keep_prob=0.8,
                                  sparse_mode=2),
}


@pytest.mark.parametrize("case", sorted(EXTRA_CASES))
def test_backward_with_extras_matches_finite_differences(case):
    rng = np.random.default_rng(11)
    q, k, v = _qkv(12, Hq=2, Hkv=1)
    do = rng.standard_normal((1, 2, 6, 3))
    ex = EXTRA_CASES[case](rng)
    o, lse = A.attention_fwd(q, k, v, SCALE, extras=ex)
    dq, dk, dv = BW.attention_bwd(q, k, v, o, lse, do, SCALE, extras=ex)

    def loss():
        oo, _ = A.attention_fwd(q, k, v, SCALE, extras=ex)
        return float((np.nan_to_num(oo) * do).sum())
    for g, x in ((dq, q), (dk, k), (dv, v)):
        assert np.allclose(g, _fd(x, loss), rtol=1e-6, atol=1e-8), case

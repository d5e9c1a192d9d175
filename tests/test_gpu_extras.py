"""GPU parity of the operator's optional terms (fa_fwd_ext) against the fp64
oracle's Extras: the key window of sparse_mode 0 (pre_tokens / next_tokens),
the bottom-right causal mask of sparse_mode 3, an explicit attention mask, the
ALiBi position bias of pse_type 2, a pse bias tensor added after (pse_type
0) or before (pse_type 1) the scale, and dropout with the Philox mask of the
"FlashAttentionScoreGrad" write-up, section 5.3 ("FlashAttentionScore" operator doc,
gitcode ops-transformer, sections "Function description" and "Parameter
description").  Tolerances as every forward parity test: elementwise
|dO| <= 1e-4 + 7.8125e-3 |ref|, rel-L2 <= 3e-3, |dLSE| <= 2e-3, +inf rows
exact."""
import numpy as np
import pytest

from attention_forward_fa_gb300 import workloads as W
from oracle import attention as A
from oracle import backward as BW
from tests.parity import compare, to_device

pytestmark = pytest.mark.gpu


def _mask_bits(shape, frac, seed, full_rows=()):
    """Seeded boolean mask (True = masked) with about `frac` masked keys;
    rows in `full_rows` (index tuples over the leading axes and the row)
    masked entirely."""
    rng = np.random.Generator(np.random.PCG64(seed))
    m = rng.random(shape) < frac
    for r in full_rows:
        m[r] = True
    return m


def _bias(shape, dtype, seed, sigma=2.0):
    """Seeded bias tensor: N(0, sigma^2) rounded to the input type; returns
    (bits, float64 values)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    bits = W.to_bits((sigma * rng.standard_normal(shape)).astype(np.float32), dtype)
    return bits, W.bits_to_f64(bits, dtype)


def _run(p, causal=False, window=None, bottom_right=False, mask=None, alibi=False, thr=0.0,
         pse=None, pse_type=0, dropout=None):
    import torch
    import attention_forward_fa_gb300 as fa
    d = to_device(p)
    am = torch.from_numpy(mask).cuda() if mask is not None else None
    pse_t = None
    if pse is not None:
        tdt = torch.bfloat16 if p.dtype == "bf16" else torch.float16
        pse_t = torch.from_numpy(pse[0].view(np.int16).copy()).cuda().view(tdt)
    o, lse = fa.flash_attention_forward(d["q"], d["k"], d["v"], scale=p.scale, causal=causal,
                                        seqlens=d["seqlens"], window=window,
                                        bottom_right_causal=bottom_right, atten_mask=am,
                                        alibi=alibi, pse=pse_t, pse_type=pse_type,
                                        dropout=dropout, rescale_threshold=thr)
    code = fa.fa_check_status()
    assert code == 0, fa.fa_strerror(code)
    torch.cuda.synchronize()
    drop = {}
    if dropout is not None:
        keep, seed, offset = dropout
        # keep_prob is a float32 argument of the C ABI (as of the operator):
        # the byte bound keep_prob * 255 is taken from that value
        keep = float(np.float32(keep))
        mflat = BW.philox_dropout_mask(seed, offset, p.B * p.Hq * p.Sq * p.Skv, keep)
        drop = dict(drop_mask=mflat.reshape(p.B, p.Hq, p.Sq, p.Skv).astype(np.float64), keep_prob=keep)
    ex = A.Extras(**drop, atten_mask=None if mask is None else mask.astype(np.float64),
                  pse=None if pse is None else pse[1],
                  pse_type=(3 if alibi == 3 else 2) if alibi else (pse_type if pse is not None else 1),
                  sparse_mode=0 if window is not None else (3 if bottom_right else None),
                  pre_tokens=window[0] if window is not None else 2 ** 31 - 1,
                  next_tokens=window[1] if window is not None else 2 ** 31 - 1)
    Or, Lr = A.attention_fwd(p.q(), p.k(), p.v(), p.scale, mask=p.mask, seqlens=p.seqlens, extras=ex)
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy(), Or, Lr


@pytest.mark.parametrize("thr", [0.0, 8.0])
def test_sliding_window_causal(thr):
    """A causal band of 300 keys (pre_tokens 299, next_tokens 0) over 1024
    rows: each tile list starts inside the sequence."""
    p = W.dense(name="win", B=1, Hq=2, Sq=1024, D=128, mask=W.MASK_CAUSAL, seed=51)
    O, L, Or, Lr = _run(p, causal=True, window=(299, 0), thr=thr)
    compare(O, L, Or, Lr, f"window 299/0 thr {thr}")


def test_two_sided_window_fp16_d64_sq_ne_skv():
    """A two-sided band (pre 200, next 77) with Sq 384 != Skv 640, fp16, D 64,
    GQA 4:2: rows near the end see keys past their own index."""
    p = W.dense(name="win2", B=1, Hq=4, Hkv=2, Sq=384, Skv=640, D=64, dtype="fp16",
                mask=W.MASK_NONE, seed=52)
    O, L, Or, Lr = _run(p, window=(200, 77))
    compare(O, L, Or, Lr, "window 200/77")


def test_window_excluding_the_diagonal_leaves_empty_rows():
    """next_tokens -1 excludes each row's own key; with pre_tokens 40 the
    first row sees no key at all (O = 0, LSE = +inf)."""
    p = W.dense(name="win3", B=1, Hq=2, Sq=256, D=128, mask=W.MASK_NONE, seed=53)
    O, L, Or, Lr = _run(p, window=(40, -1))
    assert np.isinf(Lr[0, :, 0]).all()
    compare(O, L, Or, Lr, "window 40/-1")


def test_bottom_right_causal_sq_lt_skv():
    """sparse_mode 3 with Sq 200 < Skv 520: query i sees keys j <= i + 320."""
    p = W.dense(name="brc", B=2, Hq=2, Sq=200, Skv=520, D=128, mask=W.MASK_NONE, seed=54)
    O, L, Or, Lr = _run(p, bottom_right=True)
    compare(O, L, Or, Lr, "bottom-right causal 200 x 520")


def test_bottom_right_causal_with_lengths_equals_top_left():
    """With per-batch lengths applied to queries and keys alike the offset
    kv_len - q_len is 0, so sparse_mode 3 equals the top-left causal mask."""
    p = W.dense(name="brc_len", B=2, Hq=2, Sq=384, D=128, mask=W.MASK_NONE, seqlens=[384, 201], seed=55)
    O, L, Or, Lr = _run(p, bottom_right=True)
    compare(O, L, Or, Lr, "bottom-right causal, lengths")
    pc = W.dense(name="brc_len", B=2, Hq=2, Sq=384, D=128, mask=W.MASK_CAUSAL, seqlens=[384, 201], seed=55)
    Oc, Lc = A.attention_problem(pc)
    assert np.allclose(Or, Oc, equal_nan=True) and np.allclose(Lr, Lc, equal_nan=True)


def test_explicit_mask_shared_with_masked_rows():
    """A [Sq, Skv] mask shared by every batch and head (30 % of keys masked),
    two rows masked entirely, on a causal problem with a ragged tail."""
    p = W.dense(name="am", B=2, Hq=2, Sq=300, Skv=320, D=128, mask=W.MASK_CAUSAL, seed=56)
    m = _mask_bits((300, 320), 0.3, seed=561, full_rows=[(5,), (131,)])
    O, L, Or, Lr = _run(p, causal=True, mask=m)
    assert np.isinf(Lr[:, :, 5]).all() and np.isinf(Lr[:, :, 131]).all()
    compare(O, L, Or, Lr, "shared mask")


def test_explicit_mask_per_batch_and_head_gqa():
    """A [B, Hq, Sq, Skv] mask (a different pattern per head), GQA 4:1,
    fp16, per-batch lengths."""
    p = W.dense(name="am2", B=2, Hq=4, Hkv=1, Sq=256, D=64, dtype="fp16", mask=W.MASK_NONE,
                seqlens=[256, 150], seed=57)
    m = _mask_bits((2, 4, 256, 256), 0.5, seed=571)
    O, L, Or, Lr = _run(p, mask=m)
    compare(O, L, Or, Lr, "per-head mask")


@pytest.mark.parametrize("causal", [True, False])
def test_alibi(causal):
    """pse_type 2: -slope_h |i - j| with slope_h = 2^(-8 (h + 1) / Hq), 8 heads."""
    p = W.dense(name="alibi", B=1, Hq=8, Sq=512, D=128,
                mask=W.MASK_CAUSAL if causal else W.MASK_NONE, seed=58)
    O, L, Or, Lr = _run(p, causal=causal, alibi=True)
    compare(O, L, Or, Lr, f"alibi causal={causal}")


def test_window_mask_and_alibi_together():
    p = W.dense(name="all", B=1, Hq=4, Sq=640, D=128, mask=W.MASK_CAUSAL, seed=59)
    m = _mask_bits((640, 640), 0.2, seed=591)
    O, L, Or, Lr = _run(p, causal=True, window=(257, 0), mask=m, alibi=True)
    compare(O, L, Or, Lr, "window + mask + alibi")


@pytest.mark.parametrize("pse_type", [0, 1])
def test_pse_bias_shared(pse_type):
    """A [Sq, Skv] bf16 bias shared by every batch and head, causal."""
    p = W.dense(name="pse", B=2, Hq=2, Sq=384, D=128, mask=W.MASK_CAUSAL, seed=60)
    O, L, Or, Lr = _run(p, causal=True, pse=_bias((384, 384), "bf16", 601), pse_type=pse_type)
    compare(O, L, Or, Lr, f"pse shared type {pse_type}")


def test_pse_bias_per_head_fp16_with_window():
    """A [1, Hq, Sq, Skv] fp16 bias (one per head), D 64, GQA 4:2, with a
    two-sided window and a ragged key count (Skv 264)."""
    p = W.dense(name="pse2", B=1, Hq=4, Hkv=2, Sq=256, Skv=264, D=64, dtype="fp16",
                mask=W.MASK_NONE, seed=61)
    O, L, Or, Lr = _run(p, window=(100, 30), pse=_bias((1, 4, 256, 264), "fp16", 611), pse_type=0)
    compare(O, L, Or, Lr, "pse per head + window")


def test_dropout_causal():
    """keep_prob 0.9 on a causal problem: the Philox keep mask of every
    (batch, head, row, key), the kept P scaled by 1 / keep_prob, LSE the
    softmax's."""
    p = W.dense(name="drop", B=1, Hq=2, Sq=256, D=128, mask=W.MASK_CAUSAL, seed=62)
    O, L, Or, Lr = _run(p, causal=True, dropout=(0.9, 2024, 0))
    compare(O, L, Or, Lr, "dropout 0.9")


def test_dropout_offset_fp16_window_gqa():
    """keep_prob 0.75 from stream offset 4096 * 16, with a seed above 2^32,
    fp16 D 64, GQA 4:2, Sq 128 != Skv 384, and a key window."""
    p = W.dense(name="drop2", B=2, Hq=4, Hkv=2, Sq=128, Skv=384, D=64, dtype="fp16",
                mask=W.MASK_NONE, seed=63)
    O, L, Or, Lr = _run(p, window=(200, 150), dropout=(0.75, (7 << 32) + 12345, 4096 * 16))
    compare(O, L, Or, Lr, "dropout 0.75 + window")


@pytest.mark.parametrize("keep", [0.9, 0.6])
def test_dropout_mask_bit_exact(keep):
    """Every keep bit visible in the output: q = 0 makes P uniform (1/128)
    and v_j = e_j (one-hot), so O[i, j] = M_ij / (128 keep_prob): a single
    flipped bit would miss the bound by two orders of magnitude.  keep 0.6
    puts the byte bound next to an integer (float32 0.6 * 255 = 153.000006,
    so byte 153 is kept)."""
    import dataclasses
    p = W.dense(name="dropbits", B=1, Hq=2, Sq=128, D=128, dtype="fp16", mask=W.MASK_NONE, seed=64)
    q = np.zeros((1, 2, 128, 128), np.float32)
    v = np.broadcast_to(np.eye(128, dtype=np.float32), (1, 2, 128, 128)).copy()
    p = dataclasses.replace(p, q_bits=W.to_bits(q, "fp16"), v_bits=W.to_bits(v, "fp16"))
    O, L, Or, Lr = _run(p, dropout=(keep, 99, 16 * 1000))
    kept = Or * (128 * float(np.float32(keep)))
    assert np.allclose(kept, np.round(kept)) and 0.5 < kept.mean() / keep < 1.5
    compare(O, L, Or, Lr, f"dropout bits keep {keep}")


def test_alibi_sqrt_causal_gqa():
    """pse_type 3: -slope_h sqrt(|i - j|), 8 heads over 2 KV heads, causal."""
    p = W.dense(name="alibi3", B=1, Hq=8, Hkv=2, Sq=384, D=128, mask=W.MASK_CAUSAL, seed=65)
    O, L, Or, Lr = _run(p, causal=True, alibi=3)
    compare(O, L, Or, Lr, "alibi sqrt")

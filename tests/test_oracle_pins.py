"""Pins of the CPU oracle to things other than itself.

Each test ties oracle/attention.py (or online.py / metrics.py) to a closed
form, an invariant, brute force, a library routine, or a number printed on the
pages, so that a dropped term, a wrong sign, a wrong index or a transposed
operand in the oracle fails at least one of them.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from attention_forward_fa_gb300 import workloads as W
from oracle import attention as A
from oracle import metrics as M
from oracle import online as OL

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# ---------------------------------------------------------------- closed forms

def test_single_key_gives_v():
    """One key: P = 1, so O = V and LSE = the one scaled score (FlashAttention
    correctness verification, ai6s.net, 'Boundary condition tests', single token)."""
    q, k, v = rnd((1, 1, 1, 128), 1), rnd((1, 1, 1, 128), 2), rnd((1, 1, 1, 128), 3)
    O, L = A.attention_fwd(q, k, v, 1 / math.sqrt(128))
    assert np.array_equal(O, v)
    assert L[0, 0, 0] == pytest.approx(float(q[0, 0, 0] @ k[0, 0, 0]) / math.sqrt(128), rel=1e-14)


def test_causal_first_row_sees_one_key():
    q, k, v = rnd((2, 3, 9, 16), 4), rnd((2, 3, 9, 16), 5), rnd((2, 3, 9, 16), 6)
    O, L = A.attention_fwd(q, k, v, 0.3, mask=A.MASK_CAUSAL)
    assert np.allclose(O[:, :, 0], v[:, :, 0], rtol=0, atol=1e-15)
    assert np.allclose(L[:, :, 0], 0.3 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0]), atol=1e-13)


def test_equal_scores_give_mean_of_v():
    """q = 0: every score is 0, so O is the mean of V over the valid keys and
    LSE = ln |J|; under a causal mask row i averages keys 0..i."""
    B, H, S, D = 1, 2, 37, 8
    q = np.zeros((B, H, S, D))
    k, v = rnd((B, H, S, D), 7), rnd((B, H, S, D), 8)
    O, L = A.attention_fwd(q, k, v, 0.5, mask=A.MASK_CAUSAL)
    for i in range(S):
        assert np.allclose(O[:, :, i], v[:, :, : i + 1].mean(axis=2), atol=1e-14)
        assert np.allclose(L[:, :, i], math.log(i + 1), atol=1e-14)


def test_extreme_constant_inputs_are_finite_and_uniform():
    """All-equal huge scores (q = k = 1e3) and tiny ones (1e-10): no overflow,
    O = mean(V) (ai6s.net, 'Boundary condition tests', extreme values)."""
    for val in (1e3, 1e-10, 0.0):
        q = np.full((1, 1, 4, 128), val)
        k = np.full((1, 1, 4, 128), val)
        v = rnd((1, 1, 4, 128), 9)
        O, L = A.attention_fwd(q, k, v, 1 / math.sqrt(128))
        assert np.isfinite(O).all() and np.isfinite(L).all()
        assert np.allclose(O[0, 0], v[0, 0].mean(axis=0)[None], atol=1e-13)
        s = val * val * 128 / math.sqrt(128)
        assert L[0, 0, 0] == pytest.approx(s + math.log(4), rel=1e-12, abs=1e-12)
    q, k = rnd((1, 1, 4, 128), 10, 1e2), rnd((1, 1, 4, 128), 11, 1e2)
    O, L = A.attention_fwd(q, k, rnd((1, 1, 4, 128), 12), 1 / math.sqrt(128))
    assert np.isfinite(O).all() and np.isfinite(L).all()


def test_empty_rows_zero_output_infinite_lse():
    """Padded rows (i >= seqlens[b]) and rows with no valid key: O = 0, LSE = +inf."""
    q, k, v = rnd((2, 2, 10, 8), 13), rnd((2, 2, 10, 8), 14), rnd((2, 2, 10, 8), 15)
    O, L = A.attention_fwd(q, k, v, 0.4, mask=A.MASK_CAUSAL, seqlens=np.array([10, 0]))
    assert np.all(O[1] == 0) and np.all(np.isposinf(L[1]))
    assert np.isfinite(L[0]).all()
    idx = np.full((1, 2, 1, 3), -1, dtype=np.int32)  # only invalid slots
    O, L = A.attention_fwd(q[:1], k[:1], v[:1], 0.4, kv_block_idx=idx, block=16)
    assert np.all(O == 0) and np.all(np.isposinf(L))


# ---------------------------------------------------------------- invariants

def test_softmax_rows_nonnegative_sum_to_one():
    """Rows of P are >= 0, sum to 1 and their max exceeds their mean (ai6s.net,
    'Layered test framework', verify_softmax_properties)."""
    q, k, v = rnd((1, 2, 50, 16), 16), rnd((1, 2, 70, 16), 17), rnd((1, 2, 70, 16), 18)
    _, _, Ps = A.attention_fwd(q, k, v, 0.25, mask=A.MASK_CAUSAL, return_p=True)
    for p in Ps.values():
        assert (p >= 0).all()
        assert np.allclose(p.sum(axis=1), 1.0, atol=1e-12)
        assert (p.max(axis=1) > p.mean(axis=1)).all()


def test_masked_positions_do_not_leak():
    """Changing K/V where the mask hides them leaves O and LSE bit-identical:
    causal future keys, keys past seqlens, and blocks behind invalid slots."""
    B, H, S, D = 2, 2, 40, 8
    q, k, v = rnd((B, H, S, D), 19), rnd((B, H, S, D), 20), rnd((B, H, S, D), 21)
    sl = np.array([40, 23])
    O1, L1 = A.attention_fwd(q, k, v, 0.3, mask=A.MASK_CAUSAL, seqlens=sl)
    k2, v2 = k.copy(), v.copy()
    k2[1, :, 23:] = 1e4
    v2[1, :, 23:] = -7.0
    O2, L2 = A.attention_fwd(q, k2, v2, 0.3, mask=A.MASK_CAUSAL, seqlens=sl)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)
    # causal: row i must not depend on keys > i
    k3, v3 = k.copy(), v.copy()
    k3[:, :, 30:] += 5.0
    v3[:, :, 30:] += 5.0
    O3, L3 = A.attention_fwd(q, k3, v3, 0.3, mask=A.MASK_CAUSAL, seqlens=sl)
    assert np.array_equal(O1[:, :, :30], O3[:, :, :30])
    # block-sparse: blocks not listed are invisible
    idx = np.array([[[[0, -1], [1, 2], [2, 0]], [[2, -1], [0, 99], [1, 1]]]], dtype=np.int32)  # B=1,H=2,nqb=3
    qs, ks, vs = q[:1, :, :24], k[:1, :, :24], v[:1, :, :24]
    O4, L4 = A.attention_fwd(qs, ks, vs, 0.3, kv_block_idx=idx, block=8)
    ks2, vs2 = ks.copy(), vs.copy()
    ks2[0, 0, 8:16] = 50.0   # head 0, block 1 is listed only for q block 1
    vs2[0, 0, 8:16] = 50.0
    O5, L5 = A.attention_fwd(qs, ks2, vs2, 0.3, kv_block_idx=idx, block=8)
    assert np.array_equal(O4[0, 0, :8], O5[0, 0, :8])


def test_gqa_head_mapping_and_head_independence():
    """Query head h reads KV head h // (Hq/Hkv) ([B, Nkv, G, S, D] grouping of the
    FlashAttentionScoreGrad pytest framework page, section 5.1): running each
    KV group as its own MHA problem gives the same numbers."""
    B, Hq, Hkv, S, D = 2, 6, 2, 12, 8
    q, k, v = rnd((B, Hq, S, D), 22), rnd((B, Hkv, S, D), 23), rnd((B, Hkv, S, D), 24)
    O, L = A.attention_fwd(q, k, v, 0.35, mask=A.MASK_CAUSAL)
    for h in range(Hq):
        kh = h // 3
        O1, L1 = A.attention_fwd(q[:, h:h + 1], k[:, kh:kh + 1], v[:, kh:kh + 1], 0.35,
                                 mask=A.MASK_CAUSAL)
        assert np.array_equal(O[:, h:h + 1], O1) and np.array_equal(L[:, h:h + 1], L1)


# ---------------------------------------------------------------- brute force

def _brute_row(qi, K, V, scale, keys):
    """Exact rational-free brute force: exp without max subtraction, math.fsum."""
    e = [math.exp(scale * math.fsum(a * b for a, b in zip(qi, K[j]))) for j in keys]
    l = math.fsum(e)
    o = [math.fsum(e[t] * V[j][d] for t, j in enumerate(keys)) / l for d in range(len(V[0]))]
    return o, math.log(l)


@pytest.mark.parametrize("mask", [A.MASK_NONE, A.MASK_CAUSAL])
def test_brute_force_tiny(mask):
    rng = np.random.default_rng(25)
    for trial in range(6):
        Sq, Skv, D, Dv = rng.integers(1, 9), rng.integers(1, 9), rng.integers(1, 9), rng.integers(1, 9)
        q, k, v = rng.standard_normal((1, 1, Sq, D)), rng.standard_normal((1, 1, Skv, D)), rng.standard_normal((1, 1, Skv, Dv))
        O, L = A.attention_fwd(q, k, v, 0.7, mask=mask)
        Q, K, V = q[0, 0].tolist(), k[0, 0].tolist(), v[0, 0].tolist()
        for i in range(Sq):
            keys = [j for j in range(Skv) if mask == A.MASK_NONE or j <= i]
            if not keys:
                assert np.all(O[0, 0, i] == 0) and np.isposinf(L[0, 0, i])
                continue
            o, lse = _brute_row(Q[i], K, V, 0.7, keys)
            assert np.allclose(O[0, 0, i], o, rtol=1e-12, atol=1e-13)
            assert L[0, 0, i] == pytest.approx(lse, rel=1e-12, abs=1e-13)


def test_brute_force_exact_fractions_two_keys():
    """Two keys with scores 0 and ln 3: weights exactly 1/4 and 3/4."""
    q = np.array([[[[1.0]]]])
    k = np.array([[[[0.0], [math.log(3.0)]]]])
    v = np.array([[[[4.0, -8.0], [12.0, 0.0]]]])
    O, L = A.attention_fwd(q, k, v, 1.0)
    want = [float(Fraction(1, 4) * 4 + Fraction(3, 4) * 12), float(Fraction(1, 4) * -8)]
    assert np.allclose(O[0, 0, 0], want, rtol=1e-14)
    assert L[0, 0, 0] == pytest.approx(math.log(4.0), rel=1e-14)


# ---------------------------------------------------------------- library routines

@pytest.mark.parametrize("mask,G", [(A.MASK_NONE, 1), (A.MASK_CAUSAL, 1), (A.MASK_CAUSAL, 4)])
def test_matches_torch_sdpa_float64(mask, G):
    """Dense / causal / GQA reduce to torch's scaled_dot_product_attention (fp64 CPU)."""
    B, Hkv, Sq, Skv, D, Dv = 2, 2, 33, 33, 16, 12
    Hq = Hkv * G
    q, k, v = rnd((B, Hq, Sq, D), 26), rnd((B, Hkv, Skv, D), 27), rnd((B, Hkv, Skv, Dv), 28)
    O, L = A.attention_fwd(q, k, v, 0.21, mask=mask)
    tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
    tk = tk.repeat_interleave(G, dim=1)
    tv = tv.repeat_interleave(G, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, is_causal=(mask == A.MASK_CAUSAL), scale=0.21).numpy()
    assert np.allclose(O, ref, rtol=1e-12, atol=1e-13)
    s = 0.21 * torch.einsum("bhid,bhjd->bhij", tq, tk)
    if mask == A.MASK_CAUSAL:
        s = s.masked_fill(torch.ones(Sq, Skv, dtype=torch.bool).triu(1), float("-inf"))
    assert np.allclose(L, torch.logsumexp(s, dim=-1).numpy(), rtol=1e-13, atol=1e-13)


def test_block_sparse_matches_dense_mask_and_multiplicity():
    """A block list equals dense attention under the boolean mask the list
    spells out (Mask2Idx, BSA notes section 1); a block listed twice equals an
    additive ln 2 bias on its keys (slot semantics)."""
    bs, S, D = 8, 32, 8
    q, k, v = rnd((1, 2, S, D), 29), rnd((1, 2, S, D), 30), rnd((1, 2, S, D), 31)
    idx = np.array([[[[0, 2, -1], [1, -1, 3], [2, 0, 7], [3, 1, 0]],
                     [[1, 3, 2], [-1, -1, -1], [0, 2, 1], [3, 3, -1]]]], dtype=np.int32)
    for mask in (A.MASK_NONE, A.MASK_CAUSAL_DIAG_BLOCK, A.MASK_CAUSAL):
        O, L = A.attention_fwd(q, k, v, 0.3, mask=mask, kv_block_idx=idx, block=bs)
        for h in range(2):
            bias = np.full((S, S), -np.inf)
            for i in range(S):
                qb = i // bs
                for s_ in idx[0, h, qb]:
                    if s_ < 0 or s_ >= S // bs:
                        continue
                    for j in range(s_ * bs, (s_ + 1) * bs):
                        if mask == A.MASK_CAUSAL and j > i:
                            continue
                        if mask == A.MASK_CAUSAL_DIAG_BLOCK and s_ == qb and j > i:
                            continue
                        bias[i, j] = 0.0 if not np.isfinite(bias[i, j]) else bias[i, j] + math.log(2.0)
            tb = torch.from_numpy(bias)
            tq, tk, tv = (torch.from_numpy(x[0, h]) for x in (q, k, v))
            s = 0.3 * tq @ tk.T + tb
            lse = torch.logsumexp(s, dim=-1)
            p = torch.softmax(s, dim=-1).nan_to_num(0.0)
            o = p @ tv
            empty = torch.isinf(lse)
            o[empty] = 0.0
            assert np.allclose(O[0, h], o.numpy(), rtol=1e-12, atol=1e-13)
            got = L[0, h]
            assert np.array_equal(np.isposinf(got), empty.numpy())
            assert np.allclose(got[~empty.numpy()], lse.numpy()[~empty.numpy()], atol=1e-13)


def _parts_over_block_ranges(q, k, v, scale, mask, cuts, bs):
    """The oracle over each key-block range [cuts[i], cuts[i+1]) of every row,
    through its block-list path (a different code path from the dense one):
    normalised O_i and LSE_i, with -inf for a part that sees no key."""
    B, H, S, _ = q.shape
    nqb = S // bs
    os_, ls_ = [], []
    for a, b_ in zip(cuts[:-1], cuts[1:]):
        width = b_ - a
        idx = np.full((B, H, nqb, width), -1, np.int32)
        idx[..., :] = np.arange(a, b_, dtype=np.int32)
        O, L = A.attention_fwd(q, k, v, scale, mask=mask, kv_block_idx=idx, block=bs)
        os_.append(O)
        ls_.append(np.where(np.isposinf(L), -np.inf, L))
    return np.stack(os_), np.stack(ls_)


@pytest.mark.parametrize("mask", [A.MASK_NONE, A.MASK_CAUSAL])
@pytest.mark.parametrize("cuts", [(0, 3, 8), (0, 1, 2, 5, 8), (0, 8)])
def test_merge_of_key_ranges_equals_full_attention(mask, cuts):
    """Attention over disjoint key ranges, merged, equals attention over all
    keys (the pages' blockwise merge); with causal masking some parts of the
    early rows see no key and must weigh nothing."""
    bs, S, D = 8, 64, 16
    q, k, v = rnd((2, 3, S, D), 41, 2.0), rnd((2, 3, S, D), 42), rnd((2, 3, S, D), 43)
    full_o, full_l = A.attention_fwd(q, k, v, 0.25, mask=mask)
    o_p, l_p = _parts_over_block_ranges(q, k, v, 0.25, mask, list(cuts), bs)
    o, l = A.merge_partials(o_p, l_p)
    assert np.allclose(o, full_o, rtol=1e-12, atol=1e-13)
    assert np.allclose(l, full_l, rtol=0, atol=1e-12)


def test_merge_rows_without_keys():
    """A row with no key in any part: O = 0, LSE = +inf; a part without keys
    next to one with keys changes nothing."""
    o_p = np.stack([np.full((2, 4), 7.0), np.arange(8.0).reshape(2, 4)])
    l_p = np.array([[-np.inf, -np.inf], [-np.inf, 1.5]])
    o, l = A.merge_partials(o_p, l_p)
    assert np.array_equal(o[0], np.zeros(4)) and np.isposinf(l[0])
    assert np.array_equal(o[1], o_p[1, 1]) and l[1] == 1.5


def test_topk_matches_per_token_gather():
    """Top-k (MQA, shared indices): per token, softmax over the gathered keys
    only, with -1 and out-of-range slots ignored."""
    T, H, D, Dv, Wd = 20, 3, 12, 8, 6
    rng = np.random.default_rng(32)
    q, k = rnd((1, H, T, D), 33), rnd((1, 1, T, D), 34)
    v = k[..., :Dv]
    idx = np.full((1, T, Wd), -1, dtype=np.int32)
    for t in range(T):
        n = min(t + 1, Wd)
        idx[0, t, :n] = rng.choice(t + 1, size=n, replace=False)
    idx[0, 5, 3] = 999  # out of range: invalid
    O, L = A.attention_fwd(q, k, v, 0.29, topk_idx=idx)
    for t in range(T):
        sel = idx[0, t]
        sel = sel[(sel >= 0) & (sel < T)]
        tq = torch.from_numpy(q[0, :, t:t + 1])             # [H,1,D]
        tk = torch.from_numpy(k[0, 0, sel])[None].expand(H, -1, -1)
        tv = torch.from_numpy(v[0, 0, sel])[None].expand(H, -1, -1)
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=0.29)
        assert np.allclose(O[0, :, t], ref[:, 0].numpy(), rtol=1e-12, atol=1e-13)


def test_ragged_equals_cropped_problem():
    """Per-batch lengths: batch b equals the dense problem cropped to its length."""
    B, H, S, D = 3, 2, 30, 8
    q, k, v = rnd((B, H, S, D), 35), rnd((B, H, S, D), 36), rnd((B, H, S, D), 37)
    sl = np.array([30, 17, 1])
    O, L = A.attention_fwd(q, k, v, 0.3, mask=A.MASK_CAUSAL, seqlens=sl)
    for b in range(B):
        n = sl[b]
        O1, L1 = A.attention_fwd(q[b:b + 1, :, :n], k[b:b + 1, :, :n], v[b:b + 1, :, :n], 0.3,
                                 mask=A.MASK_CAUSAL)
        assert np.allclose(O[b:b + 1, :, :n], O1, rtol=0, atol=1e-15)
        assert np.all(O[b, :, n:] == 0) and np.all(np.isposinf(L[b, :, n:]))


def test_sampled_rows_match_full():
    q, k, v = rnd((1, 2, 300, 8), 38), rnd((1, 2, 300, 8), 39), rnd((1, 2, 300, 8), 40)
    O, L = A.attention_fwd(q, k, v, 0.3, mask=A.MASK_CAUSAL)
    rows = np.array([0, 7, 128, 299])
    Os, Ls = A.attention_fwd(q, k, v, 0.3, mask=A.MASK_CAUSAL, rows=rows, heads=np.array([1]))
    assert np.array_equal(Os[0, 1, rows], O[0, 1, rows])
    assert np.isnan(Os[0, 0]).all()


# ---------------------------------------------------------------- loop invariant

@pytest.mark.parametrize("threshold", [0.0, 8.0, 3.5, 40.0])
def test_blockwise_online_equals_definition(threshold):
    """Any split of the keys into blocks, in any order, with any stale-max
    threshold, reaches softmax(S) V exactly (ai6s.net, 'Formal verification
    outline': invariant, inductive step, termination)."""
    rng = np.random.default_rng(41)
    n, Skv, D, Dv = 17, 90, 16, 10
    q, k, v = rng.standard_normal((n, D)) * 2, rng.standard_normal((Skv, D)), rng.standard_normal((Skv, Dv))
    O, L = A.attention_fwd(q[None, None], k[None, None], v[None, None], 0.3)
    for trial in range(5):
        perm = rng.permutation(Skv)
        cuts = np.sort(rng.choice(np.arange(1, Skv), size=rng.integers(1, 12), replace=False))
        blocks = np.split(perm, cuts)
        O2, L2 = OL.online_attention(q, k, v, 0.3, blocks, threshold=threshold)
        assert np.allclose(O2, O[0, 0], rtol=1e-11, atol=1e-12)
        assert np.allclose(L2, L[0, 0], rtol=1e-12, atol=1e-12)


def test_blockwise_online_masked_rows():
    """Masking inside blocks and rows that stay empty for several blocks
    (-inf guard) end at the definition too."""
    rng = np.random.default_rng(42)
    S, D = 64, 8
    q, k, v = rng.standard_normal((S, D)), rng.standard_normal((S, D)), rng.standard_normal((S, D))
    rows = np.arange(S)
    valid = lambda keys: keys[None, :] <= rows[:, None]   # noqa: E731
    blocks = OL.split_blocks(np.arange(S)[::-1], 16)    # causal, walked backwards
    O2, L2 = OL.online_attention(q, k, v, 0.4, blocks, valid=valid, threshold=8.0)
    O, L = A.attention_fwd(q[None, None], k[None, None], v[None, None], 0.4, mask=A.MASK_CAUSAL)
    assert np.allclose(O2, O[0, 0], rtol=1e-11, atol=1e-12)
    assert np.allclose(L2, L[0, 0], atol=1e-12)


# ---------------------------------------------------------------- metrics vs printed numbers

def test_row_gain_closed_form():
    r = rnd((5, 64), 43)
    g = np.array([0.0, 1e-3, -2e-3, 0.5, -0.25])
    assert np.allclose(M.row_gain((1 + g)[:, None] * r, r), g, atol=1e-15)
    x = r + rnd((5, 64), 44) * 1e-3
    assert M.rel_l2(x, r) == pytest.approx(np.linalg.norm(x - r) / np.linalg.norm(r))


@pytest.fixture(scope="module")
def mla_emulation():
    """Emulate a bf16-P kernel on a token sample of the sparse-MLA measurement
    setup (T=S=4096, W=2048, H=128, D=576 = 512 latent + 64 rope, peaked)."""
    toks = np.sort(np.random.default_rng(0).choice(4096, 24, replace=False))
    q, k, idx, scale = W.sparse_mla_rows(toks)
    v = k[:, :512]
    out = {}
    for thr in (0.0, 8.0):
        for order in ("self_last", "self_first"):
            rows = []
            for r in range(toks.size):
                slots = idx[r] if order == "self_last" else idx[r][::-1]
                blocks = [b[b >= 0] for b in OL.split_blocks(slots, 64)[::-1]]
                o, _ = OL.online_attention(q[:, r], k, v, scale, blocks, threshold=thr,
                                           p_dtype="bf16", acc="fp32", out_dtype="bf16")
                rows.append(o)
            out[(thr, order)] = np.stack(rows)
    refs = []
    for r in range(toks.size):
        sel = idx[r][idx[r] >= 0]
        O, _ = A.attention_fwd(q[:, r][None, :, None], k[sel][None, None], v[sel][None, None], scale)
        refs.append(O[0, :, 0])
    return out, np.stack(refs)


def test_metrics_reproduce_printed_sparse_mla_numbers(mla_emulation):
    """The sparse-MLA page prints: bf16 floor 1.66e-3; exact-max row gain
    1.38e-4..1.46e-4 in both orders; lazy (threshold 8) with the dominant key
    last: rel-L2 2.07e-3, row gain 1.23e-3; order-difference coherent/floor
    1.05 (exact) and 6.4 (lazy)."""
    g = json.load(open(os.path.join(GOLDEN, "sparse_mla_measurements.json")))["printed"]
    out, ref = mla_emulation
    assert M.bf16_output_floor(ref) == pytest.approx(g["bf16_output_floor_rel_l2"], rel=0.03)
    for order in ("self_last", "self_first"):
        rg = M.rms(M.row_gain(out[(0.0, order)], ref))
        assert g["exact_row_gain_rms_min"] * 0.85 <= rg <= g["exact_row_gain_rms_max"] * 1.15
    assert M.rms(M.row_gain(out[(8.0, "self_last")], ref)) == pytest.approx(
        g["lazy_dominant_last_row_gain_rms"], rel=0.15)
    assert M.rms(M.row_gain(out[(8.0, "self_first")], ref)) == pytest.approx(
        g["lazy_dominant_first_row_gain_rms"], rel=0.15)
    assert M.rel_l2(out[(8.0, "self_last")], ref) == pytest.approx(g["lazy_dominant_last_rel_l2"], rel=0.1)
    c0, f0 = M.order_difference(out[(0.0, "self_last")], out[(0.0, "self_first")], ref)
    c8, f8 = M.order_difference(out[(8.0, "self_last")], out[(8.0, "self_first")], ref)
    assert c0 / f0 == pytest.approx(g["exact_order_difference_coherent_over_floor"], rel=0.25)
    assert c8 / f8 == pytest.approx(g["lazy_order_difference_coherent_over_floor"], rel=0.25)

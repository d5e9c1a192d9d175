"""GPU parity of the top-k sparse-MLA path through the C ABI against the fp64
oracle: one latent KV head shared by all query heads, K rows [latent | rope]
(D = 576), V = the latent part of K (Dv = 512), per-token gathered key lists
("Sparse-MLA training forward: exact running max vs lazy rescale", cf-1.com,
sections "Background: sparse MLA and top-k gathered KV" and "Measurement")."""
import dataclasses

import numpy as np
import pytest

from attention_forward_fa_gb300 import workloads as W
from oracle import attention as A
from oracle import metrics as M

from tests.parity import compare, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from attention_forward_fa_gb300 import build
    build.build()


def full_check(p, threshold=0.0):
    O, L = run_gpu(p, threshold)
    Or, Lr = A.attention_problem(p)
    return compare(O, L, Or, Lr, where=p.name), O, Or


# ------------------------------------------------------------ small, every output

@pytest.mark.parametrize("reverse", [False, True])
@pytest.mark.parametrize("threshold", [0.0, 8.0])
def test_small_all_tokens(threshold, reverse):
    # token t sees t + 1 keys: short rows (hi+lo P split), partial last tiles,
    # invalid slots after the keys (given order) or before them (reversed)
    p = W.sparse_mla(name="mla_T300_W384", T=300, W=384, seed=41, reverse=reverse)
    full_check(p, threshold)


def test_fp16_inputs():
    p = W.sparse_mla(name="mla_fp16", T=260, W=320, seed=42, dtype="fp16")
    full_check(p)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_rows_just_above_256_keys(dtype):
    """Peaked rows of 256-300 keys: with fp16 P alone the fp16 case exceeded the
    elementwise bound (1.16x at token 298), so every token below 512 keys takes
    the hi + lo split."""
    p = W.sparse_mla(name=f"mla_T300_{dtype}", T=300, W=320, seed=36, dtype=dtype)
    full_check(p)


@pytest.mark.parametrize("Hq", [64, 192])
def test_partial_head_groups(Hq):
    p = W.sparse_mla(name=f"mla_H{Hq}", T=150, Hq=Hq, W=160, seed=43)
    full_check(p)


def edited(p, idx, mask=None):
    return dataclasses.replace(p, topk_idx=np.ascontiguousarray(idx, dtype=np.int32),
                               mask=p.mask if mask is None else mask)


def test_invalid_duplicate_and_empty_slots():
    p = W.sparse_mla(name="mla_slots", T=180, W=200, seed=44)
    rng = np.random.Generator(np.random.PCG64(7))
    idx = p.topk_idx.copy()
    # invalid values anywhere in the list: negative, == Skv, far out of range
    hit = rng.random(idx.shape) < 0.15
    idx[hit] = rng.choice(np.array([-1, -7, p.Skv, p.Skv + 5, 1 << 30], dtype=np.int64),
                          size=int(hit.sum())).astype(np.int32)
    # duplicates: a key listed by several slots counts once per slot
    idx[0, 120, :50] = 3
    idx[0, 121, 10:20] = idx[0, 121, 0]
    # a token without any valid slot: O = 0, LSE = +inf
    idx[0, 17, :] = -1
    idx[0, 18, :] = p.Skv
    full_check(edited(p, idx))


def test_causal_flag_masks_future_keys():
    p = W.sparse_mla(name="mla_causal", T=200, W=256, seed=45)
    rng = np.random.Generator(np.random.PCG64(8))
    idx = p.topk_idx.copy()
    # replace a quarter of the slots by arbitrary keys, many of them > t
    hit = rng.random(idx.shape) < 0.25
    idx[hit] = rng.integers(0, p.Skv, size=int(hit.sum()), dtype=np.int32)
    full_check(edited(p, idx, mask=W.MASK_CAUSAL))


def test_slot_count_not_a_tile_multiple():
    p = W.sparse_mla(name="mla_W100", T=400, W=100, seed=46)
    full_check(p, 8.0)


def test_ragged_batches():
    a = W.sparse_mla(name="a", T=160, W=128, seed=47)
    b = W.sparse_mla(name="b", T=160, W=128, seed=48)
    p = dataclasses.replace(
        a, name="mla_ragged_B2", B=2,
        q_bits=np.concatenate([a.q_bits, b.q_bits]), k_bits=np.concatenate([a.k_bits, b.k_bits]),
        topk_idx=np.concatenate([a.topk_idx, b.topk_idx]),
        seqlens=np.array([160, 97], dtype=np.int32))
    full_check(p)


# ------------------------------------------------------------ full-size workload, sampled tokens

# 511 tokens: every token below 64 (few keys, hi + lo P split), a band of 128
# around 2048 (where the key lists stop being every earlier token), and 319
# more spread evenly over the sequence.
TOKENS = np.unique(np.r_[np.arange(64), np.arange(1984, 2112),
                         np.round(np.linspace(64, 4095, 330)).astype(int)])
_C5 = {}


def c5(reverse):
    if "p" not in _C5:
        _C5["p"] = W.config(5)
    p = _C5["p"]
    if reverse:
        p = dataclasses.replace(p, name=p.name + "_reversed",
                                topk_idx=np.ascontiguousarray(p.topk_idx[:, :, ::-1]))
    return p


def oracle_tokens(p, tokens):
    """The oracle on the sampled tokens only: rows are independent without a
    causal mask or lengths, so the sub-problem of those rows is exact.  The
    reversed problem lists the same slots per token, so both orders share one
    reference (computed once)."""
    assert p.mask == W.MASK_NONE and p.seqlens is None
    if "ref" not in _C5:
        base = c5(False)
        sub = dataclasses.replace(base, Sq=len(tokens), q_bits=base.q_bits[:, :, tokens],
                                  topk_idx=base.topk_idx[:, tokens])
        _C5["ref"] = A.attention_problem(sub)
    return _C5["ref"]


@pytest.mark.parametrize("reverse", [False, True])
@pytest.mark.parametrize("threshold", [0.0, 8.0])
def test_config5_full_size_sampled(threshold, reverse):
    """Sparse MLA (T4096 Hq128 D576 Dv512 W2048, peaked) on 511 tokens: the
    elementwise bound at both thresholds and orders, and with the exact
    running max the coherent row gain within twice the bf16 output floor, the
    acceptance of "Sparse-MLA training forward: exact running max vs lazy
    rescale" (cf-1.com), sections "Measurement" and "Tests: order-invariance
    verification"."""
    assert len(TOKENS) >= 500
    p = c5(reverse)
    O, L = run_gpu(p, threshold)
    Or, Lr = oracle_tokens(p, TOKENS)
    Og, Lg = O[:, :, TOKENS], L[:, :, TOKENS]
    compare(Og, Lg, Or, Lr, where=p.name + " (sampled)")
    gain = M.rms(M.row_gain(Og, Or))
    floor = M.bf16_row_gain_floor(Or)
    if threshold == 0.0:
        assert gain <= 2.0 * floor, (gain, floor)


def test_bf16_query_beyond_fp16_range_is_reported():
    """Q.K^T of the top-k path runs on fp16 copies: a bf16 query value above
    65504 is reported as FA_ERR_RANGE (once), like an out-of-range latent."""
    import torch
    import attention_forward_fa_gb300 as fa
    p = W.sparse_mla(name="mla_range", T=130, W=160, seed=49)
    d = to_device(p)
    d["q"][0, 3, 100, 17] = -80000.0
    assert fa.fa_check_status() == 0
    o, lse = fa.flash_attention_forward(d["q"], d["k"], None, scale=p.scale,
                                        topk_idx=d["topk_idx"])
    assert fa.fa_check_status() == -8
    d["k"][0, 0, 5, 3] = 66000.0
    fa.flash_attention_forward(d["q"][:, :, :1].contiguous(), d["k"], None, scale=p.scale,
                               topk_idx=d["topk_idx"][:, :1].contiguous())
    assert fa.fa_check_status() == -8
    assert fa.fa_check_status() == 0


def test_config5_order_difference_exact_max():
    """The same problem with its slots in the given and in the reversed order,
    exact running max: the coherent (whole-row) part of the difference of the
    two outputs stays under twice its noise floor, elem_rms * sqrt(3 / Dv)
    ("Sparse-MLA training forward: exact running max vs lazy rescale", cf-1.com,
    section "Measurement")."""
    import torch
    import attention_forward_fa_gb300 as fa
    outs = []
    for reverse in (False, True):
        p = c5(reverse)
        d = to_device(p)
        o, _ = fa.flash_attention_forward(d["q"], d["k"], None, scale=p.scale, mask_mode=p.mask,
                                          topk_idx=d["topk_idx"], rescale_threshold=0.0)
        assert fa.fa_check_status() == 0
        sel = torch.from_numpy(TOKENS).to(o.device)
        outs.append(o[:, :, sel].float().cpu().double().numpy())
        del o, d
    Or, _ = oracle_tokens(c5(False), TOKENS)
    coherent, floor = M.order_difference(outs[0], outs[1], Or)
    assert coherent < 2.0 * floor, (coherent, floor)

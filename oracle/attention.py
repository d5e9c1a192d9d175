"""fp64 CPU oracle for the FlashAttention forward (materialises S and P).

TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference arm may import or run anything in this package; the
product path (attention_forward_fa_gb300) never does, and nothing here imports
the product path.

What it computes is the plain definition of attention, written out:

  S[i, j] = scale * sum_d Q[i, d] K[j, d]
  P[i, j] = exp(S[i, j] - m_i) / sum_j' exp(S[i, j'] - m_i),  m_i = max_j S[i, j]
  O[i]    = sum_j P[i, j] V[j]
  LSE[i]  = m_i + ln sum_j exp(S[i, j] - m_i)

  * the three-line definition of standard attention and the numerically stable
    softmax of FlashAttention correctness verification (ai6s.net), sections
    "Standard Attention vs FlashAttention: mathematical equivalence" and
    "Layered test framework" (standard_attention);
  * scale and masking as in the FlashAttentionScore operator doc (gitcode
    ops-transformer), section "Function description", forward formula;
  * LSE as the natural log of the row sum over scaled scores, the quantity the
    backward re-uses as P = exp(scale*S - LSE) (BSA PyPTO implementation notes,
    section 3.2 "Core design strategies", recomputation strategy).

The valid key set J(i) of each query row is where the variants differ:
  * dense: every key j < kv_len;
  * causal (mask_mode 1): keys j > i are masked (top-left aligned);
  * per-batch lengths: keys j >= seqlens[b] are masked; query rows
    i >= seqlens[b] are padding (BSA notes, section 3.2, per-batch boundary mask);
  * block-sparse: the keys of the KV blocks listed for the row's 128-row Q block
    (Mask2Idx compact lists, BSA notes section 1); a slot < 0 or >= #blocks is
    invalid and contributes nothing; mask_mode 2 applies j > i only inside the
    diagonal block;
  * top-k (sparse MLA): the keys listed for the row's token, shared by all heads
    (sparse-MLA exact-max page, section "Background: sparse MLA and top-k
    gathered KV"); a slot < 0 or >= kv_len is invalid.
A key listed by two valid slots contributes twice (slot semantics).

Readings where the pages are silent: a row with no valid key, and a padded row
i >= seqlens[b], gets O = 0 and LSE = +inf (so that a backward's
exp(scale*S - LSE) is 0 there).  The lazy-rescale threshold does not change
this result: every threshold reaches the same exact value.

Everything is float64 from the exact bf16/fp16 input values; numpy's matmul is
the only library step.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np

BLOCK = 128
MASK_NONE, MASK_CAUSAL, MASK_CAUSAL_DIAG_BLOCK = 0, 1, 2


def _softmax_rows(s: np.ndarray, w: np.ndarray):
    """Masked softmax over the last axis.

    s: scaled scores (float64); w: non-negative integer multiplicity of each
    column (0 = masked).  Returns (P, LSE) with P rows of empty sets = 0 and
    LSE = +inf for them.
    """
    valid = w > 0
    neg = np.where(valid, s, -np.inf)
    m = neg.max(axis=-1, keepdims=True)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(np.where(valid, s - m_safe, -np.inf)) * w
    l = e.sum(axis=-1, keepdims=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(empty, 0.0, e / np.where(empty, 1.0, l))
        lse = np.where(empty, np.inf, m_safe + np.log(np.where(empty, 1.0, l)))
    return p, lse[..., 0]


def attention_fwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                  mask: int = MASK_NONE, seqlens: Optional[np.ndarray] = None,
                  kv_block_idx: Optional[np.ndarray] = None,
                  topk_idx: Optional[np.ndarray] = None,
                  block: int = BLOCK, rows: Optional[np.ndarray] = None,
                  heads: Optional[np.ndarray] = None, batches: Optional[np.ndarray] = None,
                  return_p: bool = False, extras: Optional["Extras"] = None):
    """Reference forward.

    q [B,Hq,Sq,D], k [B,Hkv,Skv,D], v [B,Hkv,Skv,Dv] (float64 values).
    kv_block_idx [B, Hq or 1, ceil(Sq/block), max_sel]; topk_idx [B, Sq, W].
    ``rows``/``heads``/``batches`` optionally restrict which outputs are
    computed (for sampling large problems); skipped outputs stay NaN.
    Returns O [B,Hq,Sq,Dv] and LSE [B,Hq,Sq] (float64); with return_p also a
    dict (b, h) -> (P over the full key axis with multiplicity folded in).
    ``extras`` adds the operator doc's mask, position-bias, window and dropout
    terms (class Extras); LSE stays the softmax's (dropout comes after it).
    """
    B, Hq, Sq, D = q.shape
    _, Hkv, Skv, _ = k.shape
    Dv = v.shape[-1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    O = np.full((B, Hq, Sq, Dv), np.nan)
    LSE = np.full((B, Hq, Sq), np.nan)
    Ps = {}
    row_set = np.arange(Sq) if rows is None else np.asarray(rows)
    head_set = np.arange(Hq) if heads is None else np.asarray(heads)
    batch_set = np.arange(B) if batches is None else np.asarray(batches)
    nkb = (Skv + block - 1) // block
    for b in batch_set:
        qlen = Sq if seqlens is None else int(seqlens[b])
        kvlen = Skv if seqlens is None else int(seqlens[b])
        for h in head_set:
            kh = h // G
            for r0 in range(0, row_set.size, 256):
                ri = row_set[r0:r0 + 256]
                w = _multiplicity(ri, b, h, qlen, kvlen, Skv, nkb, block, mask,
                                  kv_block_idx, topk_idx)
                if extras is None:
                    s = scale * (q[b, h, ri, :] @ k[b, kh].T)
                else:
                    s = extras.scores(q[b, h, ri, :] @ k[b, kh].T, scale, b, h, ri, Hq, Sq, Skv)
                    w = w * extras.visible(b, h, ri, Sq, Skv, qlen, kvlen)
                p, lse = _softmax_rows(s, w)
                if extras is not None:
                    p = p * extras.keep(b, h, ri, Skv)
                O[b, h, ri, :] = p @ v[b, kh]
                LSE[b, h, ri] = lse
                if return_p:
                    Ps[(int(b), int(h), int(r0))] = p
    if return_p:
        return O, LSE, Ps
    return O, LSE


def merge_partials(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Merge attention results computed over disjoint key subsets of each row.

    The pages' blockwise merge (FlashAttention correctness verification,
    ai6s.net, section "Standard Attention vs FlashAttention: mathematical
    equivalence", the final merge): block i with row max m_i and row sum l_i
    enters with weight exp(m_i - m) * l_i / L, L = sum_i exp(m_i - m) * l_i
    (the page prints "/ l_i" where the sum needs the factor l_i; reading taken:
    multiply).  With each part carried as its normalised output O_i and its
    LSE_i = m_i + ln l_i, that weight is exp(LSE_i - m) / L with
    m = max_i LSE_i and L = sum_i exp(LSE_i - m), and the merged LSE is
    m + ln L.

    o_parts [n, ..., Dv], lse_parts [n, ...] (float64).  A part with no key
    carries LSE_i = -inf and weight 0; a row with no key in any part gets
    O = 0 and LSE = +inf, as the forward does.
    """
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    o_parts = np.asarray(o_parts, dtype=np.float64)
    m = lse_parts.max(axis=0)
    empty = ~np.isfinite(m)
    m_safe = np.where(empty, 0.0, m)
    w = np.exp(lse_parts - m_safe[None])            # exp(-inf) = 0 for empty parts
    L = w.sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        wn = np.where(empty[None], 0.0, w / np.where(empty, 1.0, L)[None])
        lse = np.where(empty, np.inf, m_safe + np.log(np.where(empty, 1.0, L)))
    o = (wn[..., None] * o_parts).sum(axis=0)
    return o, lse


def _multiplicity(ri, b, h, qlen, kvlen, Skv, nkb, block, mask, kv_block_idx, topk_idx):
    """Integer weight of every (row, key) pair: how many valid slots list the
    key for the row (1 for dense), 0 where masked."""
    n = ri.size
    j = np.arange(Skv)
    w = np.zeros((n, Skv), dtype=np.float64)
    if topk_idx is not None:
        for t, i in enumerate(ri):
            sl = topk_idx[b, i]
            sl = sl[(sl >= 0) & (sl < kvlen)]
            np.add.at(w[t], sl, 1.0)
    elif kv_block_idx is not None:
        hl = h if kv_block_idx.shape[1] > 1 else 0
        for t, i in enumerate(ri):
            qb = i // block
            for s in kv_block_idx[b, hl, qb]:
                if s < 0 or s >= nkb:
                    continue
                lo, hi = s * block, min((s + 1) * block, Skv)
                if mask == MASK_CAUSAL_DIAG_BLOCK and s == qb:
                    hi = min(hi, i + 1)
                w[t, lo:hi] += 1.0
    else:
        w[:, :] = 1.0
    w[:, j >= kvlen] = 0.0
    if mask == MASK_CAUSAL:
        w[j[None, :] > ri[:, None]] = 0.0
    w[ri >= qlen, :] = 0.0
    return w


def attention_problem(p, **kw):
    """Run the oracle on a workloads.Problem-like object (duck-typed: needs
    q()/k()/v(), scale, mask, seqlens, kv_block_idx, topk_idx)."""
    return attention_fwd(p.q(), p.k(), p.v(), p.scale, mask=p.mask, seqlens=p.seqlens,
                         kv_block_idx=p.kv_block_idx, topk_idx=p.topk_idx, **kw)


@dataclass
class Extras:
    """The FlashAttentionScore operator doc's optional terms (gitcode
    ops-transformer, section "Function description", the forward formula and
    the parameter table), with the test-framework write-up of
    FlashAttentionScoreGrad (section 5, CPU golden) for how each is built:

      s = (Q K^T + pse) * scale         pse_type 1 (add, then multiply)
      s = Q K^T * scale + pse           pse_type 0, 2, 3 (multiply, then add)
      s masked where atten_mask is 1, outside the sparse_mode window
      P = softmax(s),  O = (P * drop_mask / keep_prob) V

    * atten_mask: 0/1 array broadcastable to [B, Hq, Sq, Skv] (1 = masked).
    * pse: array broadcastable to [B, Hq, Sq, Skv]; pse_type 2 / 3 build it
      instead as ALiBi, -slope_h * d and -slope_h * sqrt(d) with d = |i - j|
      and slope_h = 2^(-8 (h + 1) / Hq), the geometric series of ratio
      2^(-8/n) (Sq == Skv only, as the doc requires).
    * sparse_mode 0: key j visible from query i when
      i - pre_tokens <= j <= i + next_tokens; 2: j <= i (top-left causal);
      3: j <= i + kv_len - q_len (bottom-right causal: the last query of a
      sequence sees up to its last key, by the batch's actual lengths when
      they are given, else Skv - Sq); None: no window.
    * drop_mask: 0/1 array broadcastable to [B, Hq, Sq, Skv] (1 = kept), with
      keep_prob in (0, 1]; philox_dropout_mask draws one as the write-up does.
    Masked scores take no part in the softmax (the write-up's golden fills
    -40000; the oracle's reading is -inf, as for every other mask).
    """
    atten_mask: Optional[np.ndarray] = None
    pse: Optional[np.ndarray] = None
    pse_type: int = 1
    sparse_mode: Optional[int] = None
    pre_tokens: int = 2 ** 31 - 1
    next_tokens: int = 2 ** 31 - 1
    drop_mask: Optional[np.ndarray] = None
    keep_prob: float = 1.0

    def bias(self, b, h, ri, Hq, Sq, Skv):
        if self.pse_type in (2, 3):
            if Sq != Skv:
                raise ValueError("ALiBi position bias needs Sq == Skv")
            slope = 2.0 ** (-8.0 * (h + 1) / Hq)
            d = np.abs(ri[:, None] - np.arange(Skv)[None, :]).astype(np.float64)
            return -slope * (np.sqrt(d) if self.pse_type == 3 else d)
        if self.pse is None:
            return None
        return _pick(self.pse, b, h, ri, Skv)

    def scores(self, qk, scale, b, h, ri, Hq, Sq, Skv):
        bias = self.bias(b, h, ri, Hq, Sq, Skv)
        if bias is None:
            return scale * qk
        if self.pse_type == 1:
            return (qk + bias) * scale
        return qk * scale + bias

    def visible(self, b, h, ri, Sq, Skv, qlen=None, kvlen=None):
        """qlen / kvlen: the batch's actual lengths (default Sq, Skv); the
        bottom-right causal mask aligns the last query of the sequence with
        its last key, so it is offset by kvlen - qlen."""
        qlen = Sq if qlen is None else min(qlen, Sq)
        kvlen = Skv if kvlen is None else min(kvlen, Skv)
        i = ri[:, None]
        j = np.arange(Skv)[None, :]
        vis = np.ones((len(ri), Skv))
        if self.sparse_mode == 0:
            vis *= (j >= i - self.pre_tokens) & (j <= i + self.next_tokens)
        elif self.sparse_mode == 2:
            vis *= j <= i
        elif self.sparse_mode == 3:
            vis *= j <= i + (kvlen - qlen)
        elif self.sparse_mode is not None:
            raise ValueError("sparse_mode must be None, 0, 2 or 3")
        if self.atten_mask is not None:
            vis *= 1.0 - _pick(self.atten_mask, b, h, ri, Skv)
        return vis

    def keep(self, b, h, ri, Skv):
        if self.drop_mask is None:
            # dropout draws which elements it drops: a keep_prob below 1 with
            # no mask would only rescale P, which is not the formula
            if self.keep_prob != 1.0:
                raise ValueError("keep_prob < 1 needs a drop_mask "
                                 "(draw one with oracle.backward.philox_dropout_mask)")
            return 1.0
        return _pick(self.drop_mask, b, h, ri, Skv) / self.keep_prob


def _pick(x, b, h, ri, Skv):
    """Rows ri of (b, h) of an array broadcastable to [B, H, S, Skv]."""
    x = np.asarray(x, dtype=np.float64)
    while x.ndim < 4:
        x = x[None]
    xb = x[b if x.shape[0] > 1 else 0, h if x.shape[1] > 1 else 0]
    return np.broadcast_to(xb[ri] if xb.shape[0] > 1 else xb, (len(ri), Skv))

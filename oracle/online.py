"""Blockwise online-softmax attention on the CPU (fp64, or an emulation of
reduced-precision P).

TEST INFRASTRUCTURE, like the rest of this package (see oracle/attention.py).

This is the FlashAttention algorithm itself, taken in the order the pages give
it, for two uses:

1. In float64 it is a second, independent route to the exact result: the loop
   invariant of FlashAttention correctness verification (ai6s.net), section
   "Formal verification outline" (steps 1-4: invariant, base case m_0 = -inf,
   L_0 = 0; inductive step L_{i+1} = L_i * exp(m_i - m_{i+1}) + l_{i+1};
   termination) says that any split of the keys into blocks, processed in any
   order, ends at softmax(S) V.  Tests compare it with the materialised
   definition in oracle/attention.py.

2. With ``p_dtype`` set it emulates a kernel whose P operand of the P.V product
   is rounded to bf16 or fp16 while the row sum is accumulated from the
   unrounded fp32 p, with the stale-max ("lazy rescale") rule of the sparse-MLA
   exact-max page, section "Verifying the threshold branch from source": the
   running max is kept while the block max exceeds it by less than
   ``threshold`` (log2 units of scaled scores); threshold 0 is the exact running
   max.  The -inf guard (a row with no valid key so far uses 0 in place of its
   max) is the m_safe step of the ai6s.net blockwise code.

p = exp2(S*c - m*c) with c = scale*log2(e) (the folded scale of the sparse-MLA
page, section "Mechanism").
"""
from __future__ import annotations

import math
from typing import Callable, Iterable, Optional, Sequence

import numpy as np

LOG2E = 1.0 / math.log(2.0)


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float values to the nearest bf16 (ties to even), returned as float64."""
    f = np.ascontiguousarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def round_fp16(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float32).astype(np.float16).astype(np.float64)


def round_fp32(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, dtype=np.float32).astype(np.float64)


_ROUND = {None: lambda x: x, "fp64": lambda x: x, "bf16": round_bf16, "fp16": round_fp16,
          "fp32": round_fp32}


def online_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                     blocks: Sequence[np.ndarray],
                     valid: Optional[Callable[[np.ndarray], np.ndarray]] = None,
                     threshold: float = 0.0, p_dtype: Optional[str] = None,
                     acc: str = "fp64", out_dtype: Optional[str] = None):
    """Online softmax over key blocks.

    q [n, D] query rows; k [Skv, D]; v [Skv, Dv]; ``blocks`` is the processing
    order, a sequence of key-index arrays (one per step; an index may appear in
    several steps and then counts each time).  ``valid(keys) -> bool [n, len]``
    masks (row, key) pairs of a step.  ``acc`` = "fp64" for exact arithmetic or
    "fp32" to round the running state and scores to fp32 as a kernel would.
    Returns (O [n, Dv], LSE [n]) in float64; rows with no valid key give O = 0,
    LSE = +inf.
    """
    r_acc = _ROUND[acc]
    r_p = _ROUND[p_dtype]
    n = q.shape[0]
    c = scale * LOG2E
    m = np.full(n, -np.inf)
    l = np.zeros(n)
    o = np.zeros((n, v.shape[1]))
    for keys in blocks:
        keys = np.asarray(keys)
        if keys.size == 0:
            continue
        s = r_acc(q @ k[keys].T)                      # raw scores
        if valid is not None:
            s = np.where(valid(keys), s, -np.inf)
        m_blk = s.max(axis=1)
        m_new = np.maximum(m, m_blk)
        with np.errstate(invalid="ignore"):
            step = np.where(np.isfinite(m), (m - m_new) * c, -np.inf)   # <= 0, log2 units
        keep = np.isfinite(m) & (step >= -threshold)
        m_use = np.where(keep, m, m_new)
        alpha = np.where(keep, 1.0, np.where(np.isfinite(m), np.exp2(step), 0.0))
        m_safe = np.where(np.isfinite(m_use), m_use, 0.0)
        p = r_acc(np.exp2(r_acc(s * c - (m_safe * c)[:, None])))
        l = r_acc(alpha * l + r_acc(p.sum(axis=1)))
        o = r_acc(alpha[:, None] * o + r_acc(r_p(p) @ v[keys]))
        m = m_use
    empty = l == 0
    with np.errstate(divide="ignore", invalid="ignore"):
        O = np.where(empty[:, None], 0.0, o / np.where(empty, 1.0, l)[:, None])
        lse = np.where(empty, np.inf, np.where(np.isfinite(m), m, 0.0) * scale
                       + np.log(np.where(empty, 1.0, l)))
    if out_dtype is not None:
        O = _ROUND[out_dtype](O)
    return O, lse


def split_blocks(keys: np.ndarray, n: int) -> list:
    """Split a key-index list into consecutive steps of n keys."""
    keys = np.asarray(keys)
    return [keys[i:i + n] for i in range(0, keys.size, n)]

"""Seeded synthetic workloads for the FlashAttention forward.

This module only draws and rounds random inputs and builds index lists; it
holds none of the attention arithmetic.  The same host arrays feed the fp64
oracle and the CUDA path (one input set for both sides, the pattern of the
"FlashAttentionScoreGrad pytest framework" page, section 2, CalculusContext).

Workload shapes follow the problem statements on the pages:
  * BNSD layout, fp16/bf16 Q/K/V, fp32 LSE, GQA with Hq % Hkv == 0
    (BSA PyPTO implementation notes, section 1 "Overview").
  * per-batch actual sequence lengths (same page, section 3.2).
  * compact per-Q-block KV-block lists with an invalid pad slot (same page,
    section 1, Mask2Idx).
  * top-k gathered keys shared by all heads (MQA), self key in slot 0, peaked
    rows q_t += 0.25 k_t (sparse-MLA exact-max page, section "Measurement:
    experiment setup").

Draw order: one numpy PCG64 generator per workload, fp32 standard normals for
Q, then K, then V (V is not drawn when it is the latent part of K), rounded to
nearest-even into bf16 or fp16.  Index lists are drawn from the same generator
afterwards.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

# mask_mode flag word (mirrors include/fa_fwd.h)
MASK_NONE = 0
MASK_CAUSAL = 1
MASK_CAUSAL_DIAG_BLOCK = 2
DTYPE_FP16 = 0x100
V_FROM_K = 0x200

BLOCK = 128  # block-sparse granularity (rows and keys per block)


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (inputs are finite, so
    the 32-bit sum below cannot wrap); chunked to stay in cache."""
    src = np.ascontiguousarray(x, dtype=np.float32).reshape(-1).view(np.uint32)
    out = np.empty(src.size, dtype=np.uint16)
    step = 1 << 20
    for s in range(0, src.size, step):
        u = src[s:s + step]
        r = (u >> 16) & 1
        r += u
        r += 0x7FFF
        r >>= 16
        out[s:s + step] = r
    return out.reshape(np.shape(x))


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_to_fp16_bits(x: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def fp16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return b.view(np.float16).astype(np.float64)


def to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    return round_to_bf16_bits(x) if dtype == "bf16" else round_to_fp16_bits(x)


def bits_to_f64(b: np.ndarray, dtype: str) -> np.ndarray:
    return bf16_bits_to_f64(b) if dtype == "bf16" else fp16_bits_to_f64(b)


@dataclasses.dataclass
class Problem:
    """One forward problem: exact input values plus every call argument."""
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Skv: int
    D: int
    Dv: int
    dtype: str                     # "bf16" | "fp16"
    mask: int                      # MASK_* (low bits of mask_mode)
    scale: float
    q_bits: np.ndarray             # [B,Hq,Sq,D] uint16
    k_bits: np.ndarray             # [B,Hkv,Skv,D]
    v_bits: Optional[np.ndarray]   # [B,Hkv,Skv,Dv] or None when V is K[..., :Dv]
    seqlens: Optional[np.ndarray] = None        # [B] int32
    kv_block_idx: Optional[np.ndarray] = None   # [B,H*,nqb,max_sel] int32
    block_idx_per_head: bool = True
    topk_idx: Optional[np.ndarray] = None       # [B,Sq,W] int32
    v_from_k: bool = False
    seed: int = 0

    @property
    def mask_mode(self) -> int:
        m = self.mask
        if self.dtype == "fp16":
            m |= DTYPE_FP16
        if self.v_from_k:
            m |= V_FROM_K
        return m

    def q(self) -> np.ndarray:
        return bits_to_f64(self.q_bits, self.dtype)

    def k(self) -> np.ndarray:
        return bits_to_f64(self.k_bits, self.dtype)

    def v(self) -> np.ndarray:
        if self.v_from_k:
            return self.k()[..., : self.Dv]
        return bits_to_f64(self.v_bits, self.dtype)


def _draw(rng, shape):
    return rng.standard_normal(size=shape, dtype=np.float32)


def dense(name="dense", B=1, Hq=2, Hkv=None, Sq=128, Skv=None, D=64, Dv=None,
          dtype="bf16", mask=MASK_NONE, seqlens=None, seed=1001, scale=None) -> Problem:
    """Dense / causal / GQA / ragged problem with i.i.d. N(0,1) inputs."""
    Hkv = Hq if Hkv is None else Hkv
    Skv = Sq if Skv is None else Skv
    Dv = D if Dv is None else Dv
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _draw(rng, (B, Hq, Sq, D))
    k = _draw(rng, (B, Hkv, Skv, D))
    v = _draw(rng, (B, Hkv, Skv, Dv))
    return Problem(name=name, B=B, Hq=Hq, Hkv=Hkv, Sq=Sq, Skv=Skv, D=D, Dv=Dv,
                   dtype=dtype, mask=mask,
                   scale=float(1.0 / np.sqrt(D)) if scale is None else scale,
                   q_bits=to_bits(q, dtype), k_bits=to_bits(k, dtype), v_bits=to_bits(v, dtype),
                   seqlens=None if seqlens is None else np.asarray(seqlens, dtype=np.int32),
                   seed=seed)


def upstream_grad(shape, dtype="bf16", seed=2001) -> np.ndarray:
    """Seeded upstream gradient dO of a backward call: i.i.d. N(0,1) fp32
    draws rounded to the input type (the bits)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return to_bits(_draw(rng, tuple(shape)), dtype)


def block_sparse(name="block_sparse", B=1, H=16, S=16384, D=128, dtype="fp16",
                 n_random=15, pad_slots=1, mask=MASK_CAUSAL_DIAG_BLOCK, seed=1004,
                 per_head=True) -> Problem:
    """Block-sparse problem: each Q block attends to its diagonal KV block plus
    ``n_random`` distinct other KV blocks drawn uniformly, listed ascending,
    followed by ``pad_slots`` invalid (-1) slots."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _draw(rng, (B, H, S, D))
    k = _draw(rng, (B, H, S, D))
    v = _draw(rng, (B, H, S, D))
    nqb = (S + BLOCK - 1) // BLOCK
    nkb = nqb
    n_random = min(n_random, nkb - 1)
    max_sel = 1 + n_random + pad_slots
    Hl = H if per_head else 1
    idx = np.full((B, Hl, nqb, max_sel), -1, dtype=np.int32)
    for b in range(B):
        for h in range(Hl):
            for qb in range(nqb):
                others = np.delete(np.arange(nkb), qb)
                pick = rng.choice(others, size=n_random, replace=False)
                sel = np.sort(np.concatenate([[qb], pick]))
                idx[b, h, qb, : sel.size] = sel
    return Problem(name=name, B=B, Hq=H, Hkv=H, Sq=S, Skv=S, D=D, Dv=D, dtype=dtype,
                   mask=mask, scale=float(1.0 / np.sqrt(D)),
                   q_bits=to_bits(q, dtype), k_bits=to_bits(k, dtype), v_bits=to_bits(v, dtype),
                   kv_block_idx=idx, block_idx_per_head=per_head, seed=seed)


def sparse_mla(name="sparse_mla", T=4096, Hq=128, D=576, Dv=512, W=2048, peak=0.25,
               dtype="bf16", seed=1005, reverse=False, v_from_k=True, scale=None) -> Problem:
    """Sparse-MLA top-k problem (MQA: one latent KV head shared by all query heads).

    K rows are [latent(Dv) | rope(D-Dv)]; V is the latent part of K.  Peaked rows:
    q_t += peak * k_t for every head, added in fp32 before rounding.  Token t
    gathers W key slots: slot 0 is t itself; when t < W the other slots hold a
    permutation of [0, t) then -1; otherwise W-1 distinct keys drawn uniformly
    from [0, t).  ``reverse`` reverses every token's slot order (the self key
    then sits in the last slot, invalid slots first).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _draw(rng, (1, Hq, T, D))
    k = _draw(rng, (1, 1, T, D))
    q = q + np.float32(peak) * k  # broadcast over heads, fp32
    idx = np.full((1, T, W), -1, dtype=np.int32)
    for t in range(T):
        idx[0, t, 0] = t
        if t + 1 <= W:
            idx[0, t, 1 : t + 1] = rng.permutation(t)
        else:
            idx[0, t, 1:] = rng.choice(t, size=W - 1, replace=False)
    if reverse:
        idx = np.ascontiguousarray(idx[:, :, ::-1])
    kb = to_bits(k, dtype)
    return Problem(name=name, B=1, Hq=Hq, Hkv=1, Sq=T, Skv=T, D=D, Dv=Dv, dtype=dtype,
                   mask=MASK_NONE,
                   scale=float(1.0 / np.sqrt(D)) if scale is None else scale,
                   q_bits=to_bits(q, dtype), k_bits=kb,
                   v_bits=None if v_from_k else np.ascontiguousarray(kb[..., :Dv]),
                   topk_idx=idx, v_from_k=v_from_k, seed=seed)


def sparse_mla_rows(tokens, T=4096, Hq=128, D=576, Dv=512, W=2048, peak=0.25,
                    dtype="bf16", seed=2005):
    """Sampled sparse-MLA problem for statistics on the CPU: the same recipe as
    ``sparse_mla`` but queries and index rows are drawn only for ``tokens``
    (from a stream of their own, so values differ from the full workload).

    Returns (q [Hq, n, D] float64, k [T, D] float64, idx [n, W] int32, scale)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    k = _draw(rng, (T, D))
    tokens = np.asarray(tokens)
    q = _draw(rng, (Hq, tokens.size, D)) + np.float32(peak) * k[tokens][None]
    idx = np.full((tokens.size, W), -1, dtype=np.int32)
    for r, t in enumerate(tokens):
        idx[r, 0] = t
        if t + 1 <= W:
            idx[r, 1 : t + 1] = rng.permutation(t)
        else:
            idx[r, 1:] = rng.choice(t, size=W - 1, replace=False)
    qb = bits_to_f64(to_bits(q, dtype), dtype)
    kb = bits_to_f64(to_bits(k, dtype), dtype)
    return qb, kb, idx, float(1.0 / np.sqrt(D))


# The five workloads of the benchmark, at full size.
def config(n: int, **over) -> Problem:
    if n == 1:
        return dense(name="c1_dense_B1_H2_S128_D64", B=1, Hq=2, Sq=128, D=64,
                     mask=MASK_NONE, seed=1001, **over)
    if n == 2:
        return dense(name="c2_causal_B2_H16_S2048_D128", B=2, Hq=16, Sq=2048, D=128,
                     mask=MASK_CAUSAL, seed=1002, **over)
    if n == 3:
        return dense(name="c3_gqa_ragged_B4_Hq32_Hkv8_S4096_D128", B=4, Hq=32, Hkv=8,
                     Sq=4096, D=128, mask=MASK_CAUSAL,
                     seqlens=[4096, 3001, 517, 14], seed=1003, **over)
    if n == 4:
        return block_sparse(name="c4_block_sparse_H16_S16384_D128", B=1, H=16, S=16384,
                            D=128, dtype="fp16", seed=1004, **over)
    if n == 5:
        return sparse_mla(name="c5_sparse_mla_T4096_H128_D576_W2048", seed=1005, **over)
    raise ValueError(n)


def valid_pairs(p: Problem) -> int:
    """Number of unmasked valid (query, key) pairs summed over heads; the unit
    of algorithmic work (2*(D+Dv) flops each).  Slot semantics: a key listed
    by two valid slots counts twice."""
    B, Hq = p.B, p.Hq
    if p.topk_idx is not None:
        total = 0
        for b in range(B):
            kvlen = p.Skv if p.seqlens is None else int(p.seqlens[b])
            qlen = p.Sq if p.seqlens is None else int(p.seqlens[b])
            idx = p.topk_idx[b, :qlen]
            ok = (idx >= 0) & (idx < kvlen)
            if p.mask == MASK_CAUSAL:
                ok &= idx <= np.arange(qlen)[:, None]
            total += int(ok.sum())
        return total * Hq
    if p.kv_block_idx is not None:
        total = 0
        nkb = (p.Skv + BLOCK - 1) // BLOCK
        for b in range(B):
            kvlen = p.Skv if p.seqlens is None else int(p.seqlens[b])
            qlen = p.Sq if p.seqlens is None else int(p.seqlens[b])
            for h in range(Hq):
                hl = h if p.block_idx_per_head else 0
                for qb in range(p.kv_block_idx.shape[2]):
                    rows = np.arange(qb * BLOCK, min((qb + 1) * BLOCK, qlen))
                    if rows.size == 0:
                        continue
                    for s in p.kv_block_idx[b, hl, qb]:
                        if s < 0 or s >= nkb:
                            continue
                        keys = np.arange(s * BLOCK, min((s + 1) * BLOCK, kvlen))
                        if keys.size == 0:
                            continue
                        if p.mask == MASK_CAUSAL or (p.mask == MASK_CAUSAL_DIAG_BLOCK and s == qb):
                            total += int((keys[None, :] <= rows[:, None]).sum())
                        else:
                            total += rows.size * keys.size
        return total
    total = 0
    for b in range(B):
        kvlen = p.Skv if p.seqlens is None else int(p.seqlens[b])
        qlen = p.Sq if p.seqlens is None else int(p.seqlens[b])
        if p.mask == MASK_CAUSAL:
            i = np.arange(qlen)
            total += int(np.minimum(i + 1, kvlen).clip(min=0).sum())
        else:
            total += qlen * kvlen
    return total * Hq


def algorithmic_flops(p: Problem) -> float:
    return 2.0 * (p.D + p.Dv) * valid_pairs(p)

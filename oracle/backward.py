"""fp64 CPU oracle for the attention backward (dQ, dK, dV), materialising P.

TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and bench.py's
cpu_baseline / reference arm may import or run anything in this package; the
product path (attention_forward_fa_gb300) never does, and nothing here imports
the product path.

What it computes is the gradient of the forward's plain definition
(oracle.attention) for an upstream gradient dO, written out as the BSA PyPTO
implementation notes describe the backward:

  P[i, j]  = w[i, j] * exp(scale * S[i, j] - LSE[i])   recomputed from the saved
                                                      LSE, S and P not stored
                                                      (section 3.2 "Core design
                                                      strategies", recomputation)
  d_row[i] = sum_d dO[i, d] * O[i, d]                  (section 8.4, "D_row
                                                      precompute")
  dV       = P^T dO                                     (no scale on dV)
  dP       = dO V^T
  dS       = P * (dP - d_row)
  dQ       = scale * dS K,   dK = scale * dS^T Q        (scale on dQ and dK:
                                                      section 1, data types and
                                                      precision)

Here S[i, j] = sum_d Q[i, d] K[j, d] (unscaled) and w[i, j] is the number of
valid slots that list key j for row i (1 for dense, 0 where masked): the same
valid key sets as the forward, from the same multiplicity rule, so that a key
listed twice enters P twice, as it does the forward.

  * GQA: dK and dV of a KV head are the sums over the query heads of its group
    (BSA notes, section 1: GQA compatible).
  * Padded query rows (i >= seqlens[b]) and rows without a valid key carry
    LSE = +inf from the forward, so P = 0 there: they contribute nothing and
    get dQ = 0 (the notes' padded-row defence, section 3.2: such rows must not
    leak into dK / dV).  Keys j >= seqlens[b] get dK = dV = 0.
  * Sparse MLA (V is the latent part of K, one KV head): the key latent's
    gradient is dK plus dV on its first Dv columns; ``latent_grad`` forms it.

Everything is float64; numpy's matmul is the only library step.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

from .attention import BLOCK, MASK_NONE, _multiplicity


def attention_bwd(q: np.ndarray, k: np.ndarray, v: np.ndarray, o: np.ndarray, lse: np.ndarray,
                  do: np.ndarray, scale: float, mask: int = MASK_NONE,
                  seqlens: Optional[np.ndarray] = None,
                  kv_block_idx: Optional[np.ndarray] = None,
                  topk_idx: Optional[np.ndarray] = None, block: int = BLOCK, extras=None):
    """Reference backward.  ``extras`` (oracle.attention.Extras): masks and
    position bias change P only; dropout enters as the FlashAttentionScoreGrad
    write-up gives it (section 5.2): dV = (P * M / keep_prob)^T dO and
    dS = P * (dP * M / keep_prob - d_row).

    q [B,Hq,Sq,D], k [B,Hkv,Skv,D], v [B,Hkv,Skv,Dv], o / do [B,Hq,Sq,Dv] and
    lse [B,Hq,Sq] (the forward's outputs; +inf on rows without keys), all
    float64 values.  Mask arguments as oracle.attention.attention_fwd.
    Returns dQ [B,Hq,Sq,D], dK [B,Hkv,Skv,D], dV [B,Hkv,Skv,Dv] (float64).
    """
    B, Hq, Sq, D = q.shape
    _, Hkv, Skv, _ = k.shape
    Dv = v.shape[-1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    nkb = (Skv + block - 1) // block
    dq = np.zeros((B, Hq, Sq, D))
    dk = np.zeros((B, Hkv, Skv, D))
    dv = np.zeros((B, Hkv, Skv, Dv))
    rows = np.arange(Sq)
    for b in range(B):
        qlen = Sq if seqlens is None else int(seqlens[b])
        kvlen = Skv if seqlens is None else int(seqlens[b])
        for h in range(Hq):
            kh = h // G
            w = _multiplicity(rows, b, h, qlen, kvlen, Skv, nkb, block, mask, kv_block_idx,
                              topk_idx)
            s = q[b, h] @ k[b, kh].T
            keep = 1.0
            if extras is None:
                st = scale * s
            else:
                st = extras.scores(s, scale, b, h, rows, Hq, Sq, Skv)
                w = w * extras.visible(b, h, rows, Sq, Skv, qlen, kvlen)
                keep = extras.keep(b, h, rows, Skv)
            lse_h = lse[b, h][:, None]
            live = np.isfinite(lse_h) & (w > 0)
            with np.errstate(over="ignore", invalid="ignore"):
                p = np.where(live, w * np.exp(st - np.where(np.isfinite(lse_h), lse_h, 0.0)), 0.0)
            d_row = (do[b, h] * o[b, h]).sum(axis=-1)
            d_row = np.where(np.isfinite(lse[b, h]), d_row, 0.0)
            dv[b, kh] += (p * keep).T @ do[b, h]
            dp = (do[b, h] @ v[b, kh].T) * keep
            ds = p * (dp - d_row[:, None])
            dq[b, h] = scale * (ds @ k[b, kh])
            dk[b, kh] += scale * (ds.T @ q[b, h])
    return dq, dk, dv


def latent_grad(dk: np.ndarray, dv: np.ndarray) -> np.ndarray:
    """Gradient of a shared key latent whose first Dv columns also serve as V
    (sparse MLA): dK with dV added on those columns."""
    g = dk.copy()
    g[..., :dv.shape[-1]] += dv
    return g


def backward_emulation(q: np.ndarray, k: np.ndarray, v: np.ndarray, o_out: np.ndarray,
                       lse: np.ndarray, do: np.ndarray, scale: float, causal: bool,
                       o_lo: Optional[np.ndarray] = None, op_dtype: str = "fp16",
                       hilo_keys: int = 512, out_dtype: str = "bf16"):
    """Emulation of a tensor-core backward's roundings, for one (batch, head).

    q [Sq, D], k [Skv, D], v [Skv, Dv], do [Sq, Dv] hold the exact values of
    the low-precision inputs; o_out is the forward's rounded output and o_lo
    its rounding residual (or None); lse the forward's fp32 LSE.  The steps of
    attention_bwd, with these roundings:
      * d_row = rowsum(dO * (o_out [+ o_lo])) in fp32 (the backward sees only
        the forward's stored output, and the residual when given);
      * P (fp32) and dS = P * (dP - d_row) (fp32) enter the products
        dV = P^T dO, dQ = dS K and dK = dS^T Q as ``op_dtype`` operands; on
        query rows with fewer than ``hilo_keys`` valid keys as a pair
        fp16(x) + fp16(x - fp16(x)) (the forward's hi + lo split), when
        op_dtype is fp16;
      * products accumulate exactly (fp32 accumulation over these lengths is
        far below the operand roundings); outputs rounded to ``out_dtype``.
    Returns dQ, dK, dV (float64).
    """
    from .online import round_bf16, round_fp16, round_fp32
    rnd = {"bf16": round_bf16, "fp16": round_fp16, "fp32": round_fp32, None: lambda x: x}
    Sq, Skv = q.shape[0], k.shape[0]
    masked = (np.arange(Skv)[None, :] > np.arange(Sq)[:, None]) if causal else np.zeros((Sq, Skv), bool)
    p = round_fp32(np.where(masked, 0.0, np.exp(scale * (q @ k.T) - lse[:, None])))
    o_seen = o_out if o_lo is None else o_out + o_lo
    d_row = round_fp32((do * o_seen).sum(-1))
    ds = p * (round_fp32(do @ v.T) - d_row[:, None])
    short = ((~masked).sum(1) < hilo_keys)[:, None]

    def operand(x):
        hi = rnd[op_dtype](x)
        if op_dtype != "fp16":
            return hi
        return hi + np.where(short, round_fp16(x - hi), 0.0)

    p_op, ds_op = operand(p), operand(ds)
    out = rnd[out_dtype]
    return (out(scale * (ds_op @ k)), out(scale * (ds_op.T @ q)), out(p_op.T @ do))



# ------------------------------------------------------------------ dropout masks
_M0, _M1 = 0xD2511F53, 0xCD9E8D57      # Philox4x32 round multipliers
_W0, _W1 = 0x9E3779B9, 0xBB67AE85      # key schedule increments (Weyl)


def philox4x32(counter, key, rounds: int = 10):
    """Philox4x32-R (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
    easy as 1, 2, 3", SC 2011): 4 x 32-bit counter, 2 x 32-bit key.  Each
    round maps (c0, c1, c2, c3) to (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2),
    hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)); the key grows by the Weyl constants
    between rounds."""
    c = [int(x) & 0xFFFFFFFF for x in counter]
    k0, k1 = (int(x) & 0xFFFFFFFF for x in key)
    for r in range(rounds):
        p0 = _M0 * c[0]
        p1 = _M1 * c[2]
        c = [((p1 >> 32) ^ c[1] ^ k0) & 0xFFFFFFFF, p1 & 0xFFFFFFFF,
             ((p0 >> 32) ^ c[3] ^ k1) & 0xFFFFFFFF, p0 & 0xFFFFFFFF]
        if r + 1 < rounds:
            k0 = (k0 + _W0) & 0xFFFFFFFF
            k1 = (k1 + _W1) & 0xFFFFFFFF
    return c


def philox_dropout_mask(seed: int, offset: int, n: int, keep_prob: float) -> np.ndarray:
    """0/1 keep mask of n elements as the FlashAttentionScoreGrad write-up
    draws it (section 5.3): the seed's low and high 32 bits are the key, the
    counter starts at offset / 16, every Philox output gives 16 bytes (words
    in order, bytes of a word low first; the pages leave the order open), and
    an element is kept when its byte is below keep_prob * 255."""
    key = (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    ctr0 = offset // 16
    out = np.empty(((n + 15) // 16) * 16, dtype=np.uint8)
    for t in range(len(out) // 16):
        c = ctr0 + t
        words = philox4x32((c & 0xFFFFFFFF, (c >> 32) & 0xFFFFFFFF, 0, 0), key)
        out[16 * t:16 * t + 16] = np.array(words, dtype="<u4").view(np.uint8)
    return (out[:n] < keep_prob * 255).astype(np.uint8)

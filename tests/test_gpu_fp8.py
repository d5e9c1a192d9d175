"""GPU parity of the FP8-input forward (fa_fwd_fp8) against the fp64 oracle.

The operator doc's FP8 inputs with full-quantisation dequant scales
("FlashAttentionScore", gitcode ops-transformer, parameter table), formed
per 128-row block along S as the "FlashAttentionScoreGrad" write-up, section
5.1, gives them: the attention is the attention on x_q * d_scale
(oracle.fp8.dequant), compared under the forward's tolerances."""
import numpy as np
import pytest

from oracle import attention as A
from oracle import fp8 as F8
from tests.parity import compare

pytestmark = pytest.mark.gpu


def _inputs(B, Hq, Hkv, Sq, Skv, D, fmt, seed):
    """Seeded FP8 inputs: N(0,1) draws times a width that keeps them inside
    the format, cast to fp8 by torch, and random per-block scales."""
    import torch
    g = torch.Generator().manual_seed(seed)
    tdt = torch.float8_e4m3fn if fmt == "e4m3" else torch.float8_e5m2
    amp = 64.0 if fmt == "e4m3" else 4096.0
    xs, ds = [], []
    for (H, S) in ((Hq, Sq), (Hkv, Skv), (Hkv, Skv)):
        x8 = (torch.randn(B, H, S, D, generator=g) * amp).to(tdt)
        d = (torch.rand(B, H, (S + 127) // 128, generator=g) * 3.0 + 0.5) / amp
        xs.append(x8)
        ds.append(d.float())
    return xs, ds


def _run(B, Hq, Hkv, Sq, Skv, D, fmt, causal, seed, seqlens=None):
    import torch
    import attention_forward_fa_gb300 as fa
    (q8, k8, v8), (dq, dk, dv) = _inputs(B, Hq, Hkv, Sq, Skv, D, fmt, seed)
    dev = torch.device("cuda")
    sl = torch.tensor(seqlens, dtype=torch.int32, device=dev) if seqlens is not None else None
    o, lse = fa.flash_attention_forward_fp8(q8.to(dev), k8.to(dev), v8.to(dev), dq.to(dev),
                                            dk.to(dev), dv.to(dev), fp8_format=fmt, causal=causal,
                                            seqlens=sl)
    code = fa.fa_check_status()
    assert code == 0, fa.fa_strerror(code)
    torch.cuda.synchronize()
    q = F8.dequant(q8.double().numpy(), dq.double().numpy())
    k = F8.dequant(k8.double().numpy(), dk.double().numpy())
    v = F8.dequant(v8.double().numpy(), dv.double().numpy())
    Or, Lr = A.attention_fwd(q, k, v, D ** -0.5, mask=A.MASK_CAUSAL if causal else A.MASK_NONE,
                             seqlens=None if seqlens is None else np.asarray(seqlens))
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy(), Or, Lr


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_causal(fmt):
    O, L, Or, Lr = _run(1, 2, 2, 512, 512, 128, fmt, True, 71)
    compare(O, L, Or, Lr, f"fp8 {fmt} causal")


def test_fp8_gqa_lengths_d64():
    O, L, Or, Lr = _run(2, 4, 2, 384, 384, 64, "e4m3", True, 72, seqlens=[384, 200])
    compare(O, L, Or, Lr, "fp8 e4m3 GQA lengths D 64")


def test_fp8_no_mask_sq_ne_skv():
    O, L, Or, Lr = _run(1, 2, 1, 256, 640, 128, "e5m2", False, 73)
    compare(O, L, Or, Lr, "fp8 e5m2 256 x 640")

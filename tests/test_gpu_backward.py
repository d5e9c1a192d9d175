"""GPU parity of the backward (fa_bwd) against the fp64 backward oracle.

The forward runs on the GPU first (fa_fwd_o_lo: o, its rounding residual and
the LSE, which the backward takes as inputs, as a training step would), then
fa_bwd; dQ, dK and dV are compared element by element with
oracle.backward.attention_bwd evaluated on the exact forward (oracle O and
LSE) under the BSA PyPTO implementation notes' tolerances (section 6.1: atol
1e-4, rtol 7.8125e-3, the same bound as the forward's).  The recomputation
P = exp(scale S - LSE) and the precomputed d_row = rowsum(dO * (o + o_lo))
follow the notes' sections 3.2 and 8.4; fa_bwd materialises S, P, dP and dS
per batch of heads in fp32, with fp32 GEMMs for the products.
"""
import numpy as np
import pytest

from attention_forward_fa_gb300 import workloads as W
from oracle import attention as A
from oracle import backward as BW
from tests.parity import ATOL, RTOL

pytestmark = pytest.mark.gpu


def _run(p, heads=None, seed=2001):
    """Forward + backward on the GPU; returns (dq, dk, dv, oracle dq, dk, dv)
    as float64, restricted to `heads` (query heads; with Hq == Hkv the same
    KV heads) when given."""
    import torch
    import attention_forward_fa_gb300 as fa
    from tests.parity import to_device

    d = to_device(p)
    tdt = torch.bfloat16 if p.dtype == "bf16" else torch.float16
    do_bits = W.upstream_grad((p.B, p.Hq, p.Sq, p.Dv), p.dtype, seed=seed)
    dout = torch.from_numpy(do_bits.view(np.int16).copy()).cuda().view(tdt)
    causal = p.mask == W.MASK_CAUSAL
    o, lse, o_lo = fa.flash_attention_forward(d["q"], d["k"], d["v"], scale=p.scale, causal=causal,
                                              seqlens=d["seqlens"], o_lo=True)
    dq, dk, dv = fa.flash_attention_backward(d["q"], d["k"], d["v"], o, lse, dout, o_lo=o_lo,
                                             scale=p.scale, causal=causal, seqlens=d["seqlens"])
    code = fa.fa_check_status()
    assert code == 0, fa.fa_strerror(code)
    torch.cuda.synchronize()
    g = [x.float().cpu().double().numpy() for x in (dq, dk, dv)]
    q, k, v = p.q(), p.k(), p.v()
    do = W.bits_to_f64(do_bits, p.dtype)
    seq = p.seqlens
    if heads is not None:
        assert p.Hq == p.Hkv
        q, k, v, do = q[:, heads], k[:, heads], v[:, heads], do[:, heads]
        g = [x[:, heads] for x in g]
    O, L = A.attention_fwd(q, k, v, p.scale, mask=p.mask, seqlens=seq)
    ref = BW.attention_bwd(q, k, v, O, L, do, p.scale, mask=p.mask, seqlens=seq)
    return g, ref


def _check(g, ref, where):
    for name, x, r in zip(("dQ", "dK", "dV"), g, ref):
        assert np.isfinite(x).all(), f"{where} {name}: non-finite"
        ratio = float((np.abs(x - r) / (ATOL + RTOL * np.abs(r))).max())
        rel = float(np.linalg.norm(x - r) / max(np.linalg.norm(r), 1e-30))
        assert ratio <= 1.0, f"{where} {name}: max |d|/bound {ratio:.3f} (rel-L2 {rel:.2e})"


CASES = [
    # name, workloads.dense arguments
    ("causal_256", dict(B=1, Hq=2, Sq=256, D=128, mask=W.MASK_CAUSAL, seed=31)),
    ("full_384_fp16", dict(B=1, Hq=2, Sq=384, D=128, mask=W.MASK_NONE, dtype="fp16", seed=32)),
    ("causal_ragged_300", dict(B=1, Hq=2, Sq=300, D=128, mask=W.MASK_CAUSAL, seed=33)),
    ("gqa_lengths", dict(B=2, Hq=4, Hkv=2, Sq=640, D=128, mask=W.MASK_CAUSAL, seqlens=[640, 333], seed=34)),
    ("gqa8_full", dict(B=1, Hq=8, Hkv=1, Sq=256, D=128, mask=W.MASK_NONE, seed=35)),
    ("causal_1024", dict(B=1, Hq=1, Sq=1024, D=128, mask=W.MASK_CAUSAL, seed=36)),
    ("sq_ne_skv", dict(B=1, Hq=2, Sq=256, Skv=512, D=128, mask=W.MASK_NONE, seed=37)),
    ("d64_causal_ragged", dict(B=1, Hq=2, Sq=700, D=64, mask=W.MASK_CAUSAL, seed=39)),
    ("d64_gqa_fp16_lengths", dict(B=2, Hq=4, Hkv=2, Sq=600, D=64, mask=W.MASK_CAUSAL, dtype="fp16",
                                  seqlens=[600, 250], seed=40)),
]


@pytest.mark.parametrize("name,kw", CASES, ids=[c[0] for c in CASES])
def test_backward_matches_oracle(name, kw):
    p = W.dense(name=name, **kw)
    g, ref = _run(p)
    _check(g, ref, name)


def test_backward_benchmark_workload_sampled_heads():
    """The dense causal benchmark workload (B 2, H 16, S 2048, D 128, bf16):
    every element of dQ, dK and dV of three whole heads (heads are
    independent with Hq == Hkv, so the oracle runs on those alone)."""
    p = W.config(2)
    g, ref = _run(p, heads=[0, 7, 15])
    _check(g, ref, "c2 heads 0, 7, 15")


def test_backward_across_several_plane_batches():
    """16 heads at S 4096 hold 2 GiB of S and dP, so fa_bwd runs two batches
    of 8 planes (1 GiB each) and 8 causal row blocks per batch: every element
    of heads 0 and 7 (first batch) and 8 and 15 (second)."""
    p = W.dense(name="batches", B=1, Hq=16, Sq=4096, D=64, mask=W.MASK_CAUSAL, seed=41)
    g, ref = _run(p, heads=[0, 7, 8, 15])
    _check(g, ref, "S 4096, heads 0, 7, 8, 15")


def test_backward_empty_rows_have_zero_gradients():
    """A batch of length 0 and rows past a batch's length: zero dQ, dK, dV."""
    p = W.dense(name="empty", B=2, Hq=2, Sq=256, D=128, mask=W.MASK_CAUSAL, seqlens=[0, 77], seed=38)
    g, ref = _run(p)
    _check(g, ref, "lengths 0 / 77")
    for x in g:
        assert not np.any(x[0]), "batch of length 0"
        assert not np.any(x[1, :, 77:]), "rows past the length"

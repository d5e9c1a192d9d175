"""fa_fwd_noalloc: the entry point for callers that cannot let a library
allocate device memory (programs that hand out all device memory from their
own arena, latency-critical call sites where a driver allocation is not
acceptable).  fa_fwd takes stream-ordered scratch in two cases: the fp16 copy
of a bf16 top-k key latent, and the fp32 partial results of a dense problem
whose KV tiles are split into pieces because it has too few units to fill the
GPU.  fa_fwd_noalloc puts either into one fixed 32 MiB array inside the
library.  Both entry points run the same kernels with the same split on the
same inputs, so their results must be identical bit for bit, including on a
second call, which finds the previous call's data still in the shared array.
One of them is also compared with the fp64 oracle.

This file is collected last on purpose (a failure here then leaves every other
test already run)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

# The dense cases: B=2, Hq=4, Hkv=2 pairs the two heads of each GQA group in
# one unit, so there are B * Hq/2 * ceil(700/128) = 24 units.  The library
# splits a dense problem whose units * 2 <= SMs into
# min(max_split, ceil(SMs / units), KV tiles / 2) pieces: 3 here on any GPU
# with at least 48 SMs, with the cap pinned to 3.
DENSE_UNITS = 24
DENSE_SPLIT = 3


def _dense(seed, dtype="bf16"):
    from attention_forward_fa_gb300 import workloads as W
    return W.dense(name=f"noalloc{seed}", B=2, Hq=4, Hkv=2, Sq=700, D=128, dtype=dtype,
                   mask=W.MASK_CAUSAL, seqlens=[700, 333], seed=seed)


def _mla(seed, dtype="bf16"):
    from attention_forward_fa_gb300 import workloads as W
    return W.sparse_mla(name=f"noalloc_mla{seed}", T=300, W=320, seed=seed, dtype=dtype)


def _run(entry, p):
    import torch
    from tests.parity import to_device
    d = to_device(p)
    o = torch.empty((p.B, p.Hq, p.Sq, p.Dv), dtype=d["q"].dtype, device="cuda")
    lse = torch.empty((p.B, p.Hq, p.Sq), dtype=torch.float32, device="cuda")
    tk = None
    if d["topk_idx"] is not None:
        ti = d["topk_idx"]
        tk = (ti, ti.shape[-1], ti.shape[-2] * ti.shape[-1])
    code = entry(d["q"], d["k"], None if p.v_from_k else d["v"], o, lse, p.B, p.Hq, p.Hkv, p.Sq,
                 p.Skv, p.D, p.Dv, p.scale, p.mask_mode, d["seqlens"], None, tk, 0.0)
    assert code == 0
    import attention_forward_fa_gb300 as fa
    assert fa.fa_check_status() == 0
    torch.cuda.synchronize()
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy()


def test_noalloc_matches_fa_fwd_on_two_calls_in_a_row():
    import torch
    from attention_forward_fa_gb300 import build
    build.build()
    import attention_forward_fa_gb300 as fa
    from oracle import attention as A
    from tests.parity import compare
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert DENSE_UNITS * 2 <= sms, "the dense cases would not split on this GPU"
    assert fa.fa_set_max_kv_split(DENSE_SPLIT) == 0
    try:
        cases = [_dense(31), _dense(32), _dense(33, "fp16"), _mla(34), _mla(35), _mla(36, "fp16")]
        for p in cases:
            O_ref, L_ref = _run(fa.fa_fwd, p)
            O, L = _run(fa.fa_fwd_noalloc, p)
            assert np.array_equal(O, O_ref), f"{p.name}: O differs from fa_fwd's"
            assert np.array_equal(L, L_ref), f"{p.name}: LSE differs from fa_fwd's"
            Or, Lr = A.attention_problem(p)
            compare(O, L, Or, Lr, where=f"fa_fwd_noalloc vs the oracle, {p.name}")
    finally:
        fa.fa_set_max_kv_split(8)


def test_noalloc_rejects_a_latent_beyond_its_scratch():
    """A bf16 key latent whose fp16 copy exceeds 32 MiB is refused before
    anything runs (real buffers of the refused size)."""
    import torch
    import attention_forward_fa_gb300 as fa
    Skv = 29128   # 29128 * 576 * 2 bytes > 32 MiB
    q = torch.zeros((1, 128, 1, 576), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 1, Skv, 576), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros((1, 128, 1, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 128, 1), dtype=torch.float32, device="cuda")
    idx = torch.zeros((1, 1, 64), dtype=torch.int32, device="cuda")
    code = fa.fa_fwd_noalloc(q, k, None, o, lse, 1, 128, 1, 1, Skv, 576, 512, 0.1,
                             fa.FA_V_FROM_K, None, None, (idx, 64, 64), 0.0)
    assert code == -9
    assert "scratch" in fa.fa_strerror(code)
    torch.cuda.synchronize()
    assert fa.fa_check_status() == 0
    assert torch.count_nonzero(o) == 0   # nothing was launched

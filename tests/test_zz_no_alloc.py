"""fa_fwd_noalloc: the entry point for callers that cannot let a library
allocate device memory (programs that hand out all device memory from their
own arena, latency-critical call sites where a driver allocation is not
acceptable).  It uses a fixed 32 MiB array inside the library instead of
stream-ordered scratch; its results must equal fa_fwd's on the same inputs,
including on a second call, which finds the previous call's data still in the
shared array.

This file is collected last on purpose (a failure here then leaves every other
test already run)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu


def _problem(seed, dtype="bf16"):
    from attention_forward_fa_gb300 import workloads as W
    return W.dense(name=f"noalloc{seed}", B=2, Hq=4, Hkv=2, Sq=700, D=128, dtype=dtype,
                   mask=W.MASK_CAUSAL, seqlens=[700, 333], seed=seed)


def _run(entry, p):
    import torch
    from tests.parity import to_device
    d = to_device(p)
    o = torch.empty((p.B, p.Hq, p.Sq, p.Dv), dtype=d["q"].dtype, device="cuda")
    lse = torch.empty((p.B, p.Hq, p.Sq), dtype=torch.float32, device="cuda")
    code = entry(d["q"], d["k"], d["v"], o, lse, p.B, p.Hq, p.Hkv, p.Sq, p.Skv, p.D, p.Dv,
                 p.scale, p.mask_mode, d["seqlens"], None, None, 0.0)
    assert code == 0
    import attention_forward_fa_gb300 as fa
    assert fa.fa_check_status() == 0
    torch.cuda.synchronize()
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy()


def test_noalloc_matches_fa_fwd_on_two_calls_in_a_row():
    from attention_forward_fa_gb300 import build
    build.build()
    import attention_forward_fa_gb300 as fa
    from tests.parity import compare
    for seed, dtype in ((31, "bf16"), (32, "bf16"), (33, "fp16")):
        p = _problem(seed, dtype)
        O_ref, L_ref = _run(fa.fa_fwd, p)
        O, L = _run(fa.fa_fwd_noalloc, p)
        compare(O, L, O_ref, L_ref, where=f"noalloc vs fa_fwd, seed {seed}")


def test_noalloc_rejects_v_beyond_its_scratch():
    """bf16 V of more than 32 MiB (fp16 copy) is refused before anything runs."""
    import attention_forward_fa_gb300 as fa
    import torch
    P = 0x10000   # aligned stand-in addresses: validation fails before any use
    B, Hkv, Skv, Dv = 1, 8, 16384, 128   # 16M elements -> 32 MiB fp16 + 1 row more
    code = fa.fa_fwd_noalloc(P, P, P, P, P, B, Hkv, Hkv, 128, Skv + 1, 128, Dv, 0.1, 0,
                             None, None, None, 0.0, torch.cuda.current_stream())
    assert code == -9
    assert "scratch" in fa.fa_strerror(code)

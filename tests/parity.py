"""Shared helpers of the parity tests: run a workloads.Problem through the C
ABI on the GPU and compare with the fp64 oracle under the stated tolerances."""
from __future__ import annotations

import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TOL = json.load(open(os.path.join(GOLDEN, "tolerances.json")))
ATOL = TOL["elementwise_atol"]
RTOL = TOL["elementwise_rtol"]
RELL2 = TOL["o_rel_l2_max"]
LSE_ABS = TOL["lse_abs_max"]


def to_device(p):
    """Upload the problem's exact input bits; returns a dict of CUDA tensors."""
    import torch
    dt = torch.bfloat16 if p.dtype == "bf16" else torch.float16
    dev = torch.device("cuda")

    def up(bits):
        return torch.from_numpy(bits.view(np.int16).copy()).to(dev).view(dt)

    d = {"q": up(p.q_bits), "k": up(p.k_bits), "v": up(p.v_bits) if p.v_bits is not None else None}
    d["seqlens"] = torch.from_numpy(p.seqlens).to(dev) if p.seqlens is not None else None
    d["block_idx"] = torch.from_numpy(p.kv_block_idx).to(dev) if p.kv_block_idx is not None else None
    d["topk_idx"] = torch.from_numpy(p.topk_idx).to(dev) if p.topk_idx is not None else None
    return d


def run_gpu(p, threshold=0.0, dev_inputs=None):
    """Run the problem through fa_fwd; returns (O float64 [B,Hq,Sq,Dv], LSE float64)."""
    import torch
    import attention_forward_fa_gb300 as fa
    d = dev_inputs or to_device(p)
    o, lse = fa.flash_attention_forward(
        d["q"], d["k"], None if p.v_from_k else d["v"], scale=p.scale, mask_mode=p.mask,
        seqlens=d["seqlens"], block_idx=d["block_idx"], topk_idx=d["topk_idx"],
        rescale_threshold=threshold)
    code = fa.fa_check_status()
    assert code == 0, fa.fa_strerror(code)
    torch.cuda.synchronize()
    return o.float().cpu().double().numpy(), lse.cpu().double().numpy()


def compare(O, L, Or, Lr, where=""):
    """Assert the tolerances: elementwise |dO| <= atol + rtol |ref|, rel-L2 of O,
    |dLSE| for finite rows, +inf rows identical.  Returns a stats dict."""
    sel = ~np.isnan(Lr)
    assert sel.any()
    o, orf = O[sel], Or[sel]
    l, lr = L[sel], Lr[sel]
    assert np.isfinite(o).all(), f"{where}: non-finite O"
    err = np.abs(o - orf)
    bound = ATOL + RTOL * np.abs(orf)
    ratio = float((err / bound).max())
    nrm = np.linalg.norm(orf)
    rel = float(np.linalg.norm(o - orf) / nrm) if nrm > 0 else float(np.linalg.norm(o))
    inf_ref = np.isposinf(lr)
    assert np.array_equal(np.isposinf(l), inf_ref), f"{where}: +inf LSE rows differ"
    lse_err = float(np.abs(l[~inf_ref] - lr[~inf_ref]).max()) if (~inf_ref).any() else 0.0
    stats = {"max_err_over_bound": ratio, "rel_l2": rel, "lse_max_abs": lse_err,
             "n_out": int(o.size)}
    assert ratio <= 1.0, f"{where}: elementwise bound exceeded {stats}"
    assert rel <= RELL2 or nrm == 0, f"{where}: rel-L2 {stats}"
    assert lse_err <= LSE_ABS, f"{where}: LSE {stats}"
    return stats

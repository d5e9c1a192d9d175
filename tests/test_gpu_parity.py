"""GPU parity: the CUDA path through the C ABI against the fp64 oracle, element
by element, on the same seeded inputs (dense, causal, ragged, GQA,
block-sparse, both rescale thresholds, bf16 and fp16, D = 64 and 128), plus
sampled rows of the full-size workloads in the launch configuration the
benchmark times."""
import numpy as np
import pytest

from attention_forward_fa_gb300 import workloads as W
from oracle import attention as A

from tests.parity import compare, run_gpu, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    from attention_forward_fa_gb300 import build
    build.build()


def full_check(p, threshold=0.0):
    O, L = run_gpu(p, threshold)
    Or, Lr = A.attention_problem(p)
    return compare(O, L, Or, Lr, where=p.name)


# ------------------------------------------------------------ small, full outputs

def test_config1_dense_tiny():
    full_check(W.config(1))


@pytest.mark.parametrize("threshold", [0.0, 8.0])
@pytest.mark.parametrize("S", [640, 700, 129])
def test_causal_mha_ragged_tail(S, threshold):
    # odd head count -> consecutive query tiles share a CTA; S % 128 != 0 -> ragged tail
    full_check(W.dense(name=f"causal_S{S}", B=1, Hq=3, Sq=S, D=128, mask=W.MASK_CAUSAL,
                       seed=11 + S), threshold)


def test_noncausal_cross_lengths_fp16():
    full_check(W.dense(name="cross_fp16", B=2, Hq=2, Sq=200, Skv=333, D=128, dtype="fp16",
                       mask=W.MASK_NONE, seed=12))


def test_causal_cross_lengths():
    full_check(W.dense(name="causal_cross", B=1, Hq=2, Sq=300, Skv=520, D=128,
                       mask=W.MASK_CAUSAL, seed=13))


@pytest.mark.parametrize("threshold", [0.0, 8.0])
def test_gqa_ragged_even_group(threshold):
    # G = 4 -> head pairs share K/V tiles; lengths cover full, ragged, 1 and 0
    full_check(W.dense(name="gqa_ragged", B=4, Hq=8, Hkv=2, Sq=700, D=128, mask=W.MASK_CAUSAL,
                       seqlens=[700, 129, 1, 0], seed=14), threshold)


def test_gqa_odd_group():
    full_check(W.dense(name="gqa_odd", B=1, Hq=6, Hkv=2, Sq=384, D=128, mask=W.MASK_CAUSAL,
                       seed=15))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("mask", [W.MASK_NONE, W.MASK_CAUSAL])
def test_head_dim_64(dtype, mask):
    full_check(W.dense(name="d64", B=2, Hq=2, Sq=300, D=64, dtype=dtype, mask=mask, seed=16))


def test_single_key_and_single_row():
    full_check(W.dense(name="one", B=1, Hq=2, Sq=1, Skv=1, D=128, seed=17))


@pytest.mark.parametrize("mask", [W.MASK_CAUSAL_DIAG_BLOCK, W.MASK_NONE, W.MASK_CAUSAL])
@pytest.mark.parametrize("threshold", [0.0, 8.0])
def test_block_sparse_small(mask, threshold):
    full_check(W.block_sparse(name="bs_small", B=1, H=4, S=1024, D=128, dtype="fp16",
                              n_random=3, mask=mask, seed=18), threshold)


def test_block_sparse_shared_lists_gqa_bf16_ragged():
    p = W.block_sparse(name="bs_shared", B=2, H=4, S=640, D=128, dtype="bf16", n_random=2,
                       seed=19, per_head=False)
    p.Hkv = 2
    p.k_bits = np.ascontiguousarray(p.k_bits[:, :2])
    p.v_bits = np.ascontiguousarray(p.v_bits[:, :2])
    p.seqlens = np.array([640, 333], dtype=np.int32)
    full_check(p)


def test_block_sparse_invalid_and_duplicate_slots():
    p = W.block_sparse(name="bs_dup", B=1, H=2, S=512, D=64, dtype="fp16", n_random=1,
                       pad_slots=2, seed=20)
    idx = p.kv_block_idx
    idx[0, 0, 1] = [1, 1, -1, 7]          # duplicate slot counts twice; 7 is out of range
    idx[0, 1, 2] = [-1, -1, -1, -1]       # nothing valid: O = 0, LSE = +inf
    idx[0, 1, 3] = [-5, 3, 0, 2]
    full_check(p)


def test_extreme_values_are_finite():
    """All-equal large scores (q = k = const) must not overflow."""
    p = W.dense(name="const", B=1, Hq=2, Sq=256, D=128, mask=W.MASK_CAUSAL, seed=21)
    p.q_bits[:] = W.round_to_bf16_bits(np.full(p.q_bits.shape, 3.0, np.float32))
    p.k_bits[:] = W.round_to_bf16_bits(np.full(p.k_bits.shape, 3.0, np.float32))
    full_check(p)


def test_repeated_calls_are_deterministic():
    p = W.dense(name="det", B=1, Hq=4, Sq=512, D=128, mask=W.MASK_CAUSAL, seed=22)
    d = to_device(p)
    O1, L1 = run_gpu(p, 0.0, d)
    O2, L2 = run_gpu(p, 0.0, d)
    assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


SPLIT_CASES = {
    # (units of (batch, head or head pair, query-tile pair) well under half the SMs)
    "causal_mha": lambda: W.dense(name="split_causal", B=1, Hq=2, Sq=2048, D=128,
                                  mask=W.MASK_CAUSAL, seed=51),
    "fp16_d64_tail": lambda: W.dense(name="split_d64", B=1, Hq=1, Sq=1500, D=64, dtype="fp16",
                                     mask=W.MASK_NONE, seed=52),
    "gqa_pairs": lambda: W.dense(name="split_gqa", B=1, Hq=4, Hkv=2, Sq=1024, D=128,
                                 mask=W.MASK_CAUSAL, seed=53),
    "seqlens": lambda: W.dense(name="split_ragged", B=2, Hq=2, Sq=2048, D=128,
                               mask=W.MASK_CAUSAL, seqlens=[2048, 700], seed=54),
    "cross": lambda: W.dense(name="split_cross", B=1, Hq=2, Sq=300, Skv=3000, D=128,
                             mask=W.MASK_CAUSAL, seed=55),
}


@pytest.mark.parametrize("max_split", [8, 1])
@pytest.mark.parametrize("case", sorted(SPLIT_CASES))
def test_split_kv_small_grids(case, max_split):
    """Problems with too few units to fill the GPU split each unit's KV tiles
    into pieces that a second kernel merges (the pages' blockwise merge); with
    the split turned off (at most 1 piece) they run unsplit.  Both match the
    oracle."""
    import attention_forward_fa_gb300 as fa
    p = SPLIT_CASES[case]()
    assert fa.fa_set_max_kv_split(max_split) == 0
    try:
        full_check(p, threshold=8.0 if case == "gqa_pairs" else 0.0)
    finally:
        fa.fa_set_max_kv_split(8)


O_LO_CASES = {
    "dense_bf16": lambda: W.dense(name="olo_dense", B=2, Hq=4, Hkv=2, Sq=700, D=128,
                                  mask=W.MASK_CAUSAL, seqlens=[700, 333], seed=61),
    "split_fp16": lambda: W.dense(name="olo_split", B=1, Hq=2, Sq=2048, D=64, dtype="fp16",
                                  mask=W.MASK_CAUSAL, seed=62),
    "mla_bf16": lambda: W.sparse_mla(name="olo_mla", T=300, W=320, seed=63),
    # 64 heads: half of the kernel's 128-row head group is padding
    "mla_padded_heads": lambda: W.sparse_mla(name="olo_mla_h64", T=150, Hq=64, W=160, seed=64),
}


@pytest.mark.parametrize("case", sorted(O_LO_CASES))
def test_o_lo_residual(case):
    """fa_fwd_o_lo: o equals fa_fwd's bit for bit, o_lo is within half an ulp
    of o, and o + o_lo is closer to the fp64 oracle than o (the precise-dpsum
    forward check of the sparse-MLA page); the split-KV case gets its residual
    from the merge kernel, the top-k case from its own epilogue."""
    import torch
    import attention_forward_fa_gb300 as fa
    from tests.parity import to_device
    p = O_LO_CASES[case]()
    d = to_device(p)
    kw = dict(scale=p.scale, mask_mode=p.mask_mode, seqlens=d["seqlens"], topk_idx=d["topk_idx"])
    v = None if p.v_from_k else d["v"]
    o_ref, l_ref = fa.flash_attention_forward(d["q"], d["k"], v, **kw)
    o, lse, o_lo = fa.flash_attention_forward(d["q"], d["k"], v, o_lo=True, **kw)
    torch.cuda.synchronize()
    assert fa.fa_check_status() == 0
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    Or, _ = A.attention_problem(p)
    sel = ~np.isnan(Or)
    hi = o.float().cpu().double().numpy()
    lo = o_lo.float().cpu().double().numpy()
    ulp_half = 2.0 ** -8 if p.dtype == "bf16" else 2.0 ** -11
    tiny = 1e-30 if p.dtype == "bf16" else 2.0 ** -25
    assert (np.abs(lo) <= ulp_half * np.abs(hi) + tiny).all()
    e_hi = np.linalg.norm((hi - Or)[sel]) / np.linalg.norm(Or[sel])
    e_sum = np.linalg.norm((hi + lo - Or)[sel]) / np.linalg.norm(Or[sel])
    assert e_sum < (0.5 if p.dtype == "bf16" else 1.0) * e_hi, (e_sum, e_hi)


def test_chained_calls_wait_for_the_previous_call():
    """Two calls back to back on one stream, the second taking the first's
    output as its queries.  The second kernel may be scheduled while the first
    drains (programmatic dependent launch) and must still wait for it before
    its first read: its result equals that of the synchronised run, bit for bit."""
    import torch
    import attention_forward_fa_gb300 as fa
    p = W.dense(name="chain", B=2, Hq=16, Sq=2048, D=128, mask=W.MASK_CAUSAL, seed=23)
    d = to_device(p)
    kw = dict(scale=p.scale, mask_mode=p.mask)
    o1, _ = fa.flash_attention_forward(d["q"], d["k"], d["v"], **kw)
    torch.cuda.synchronize()
    o2_ref, l2_ref = fa.flash_attention_forward(o1.clone(), d["k"], d["v"], **kw)
    torch.cuda.synchronize()
    a = torch.empty_like(o1)
    b = torch.empty_like(o1)
    lb = torch.empty_like(l2_ref)
    for _ in range(4):
        a.fill_(0.5)   # stale values that the second call must not read
        fa.flash_attention_forward(d["q"], d["k"], d["v"], out=a, **kw)
        fa.flash_attention_forward(a, d["k"], d["v"], out=b, lse=lb, **kw)
        torch.cuda.synchronize()
        assert fa.fa_check_status() == 0
        assert torch.equal(b, o2_ref) and torch.equal(lb, l2_ref)


# ------------------------------------------------------------ full-size workloads, sampled rows

def sampled_check(p, rows, heads, batches, threshold=0.0):
    O, L = run_gpu(p, threshold)
    Or, Lr = A.attention_problem(p, rows=np.asarray(rows), heads=np.asarray(heads),
                                 batches=np.asarray(batches))
    return compare(O, L, Or, Lr, where=p.name + " (sampled)")


_ORACLE = {}


def oracle_cached(key, fn):
    """The oracle of a full-size workload, computed once per test session."""
    if key not in _ORACLE:
        _ORACLE[key] = fn()
    return _ORACLE[key]


def merged(a, b):
    """Two partial oracle results (NaN where not computed) as one."""
    (Oa, La), (Ob, Lb) = a, b
    O = np.where(np.isnan(Oa), Ob, Oa)
    L = np.where(np.isnan(La), Lb, La)
    return O, L


@pytest.mark.parametrize("threshold", [0.0, 8.0])
def test_config2_full_size_every_output(threshold):
    """The benchmark's workload (B2 H16 S2048 D128 causal, bf16), every output
    row against the oracle, at both thresholds."""
    p = W.config(2)
    O, L = run_gpu(p, threshold)
    Or, Lr = oracle_cached("c2", lambda: A.attention_problem(p))
    assert not np.isnan(Lr).any()
    compare(O, L, Or, Lr, where=p.name + " (every row)")


def test_config3_full_size_whole_heads_and_tile_edges():
    """GQA causal with ragged lengths (B4 Hq32 Hkv8 S4096, lengths 4096, 3001,
    517, 14): every row of two heads in every batch (one head of each of two
    KV groups), plus the first and last row of every 128-row query tile of
    every head."""
    p = W.config(3)
    O, L = run_gpu(p, 0.0)

    def ref():
        n_qt = (p.Sq + 127) // 128
        edges = np.sort(np.r_[np.arange(n_qt) * 128, np.minimum(np.arange(n_qt) * 128 + 127, p.Sq - 1)])
        R = A.attention_problem(p, rows=edges)
        for b in range(p.B):
            heads = [(5 * b) % p.Hq, (5 * b + 17) % p.Hq]
            R = merged(R, A.attention_problem(p, heads=np.asarray(heads), batches=np.asarray([b])))
        return R

    Or, Lr = oracle_cached("c3", ref)
    compare(O, L, Or, Lr, where=p.name + " (two heads per batch + tile edges)")


def test_config4_full_size_two_whole_heads():
    """Block-sparse H16 S16384 fp16 (diagonal + 15 random blocks + 1 invalid
    slot per query block, causal inside the diagonal block): every row of two
    heads, whose lists differ."""
    p = W.config(4)
    O, L = run_gpu(p, 0.0)
    Or, Lr = oracle_cached("c4", lambda: A.attention_problem(p, heads=np.asarray([3, 12])))
    compare(O, L, Or, Lr, where=p.name + " (heads 3, 12, every row)")


def test_preconverted_fp16_v_equals_in_call_conversion():
    """FA_V_FP16 with a V converted by fa_convert_v_fp16 gives the same bits as
    letting fa_fwd convert V itself."""
    import torch
    import attention_forward_fa_gb300 as fa
    p = W.dense(name="v16", B=2, Hq=4, Hkv=2, Sq=500, D=128, mask=W.MASK_CAUSAL, seed=23)
    d = to_device(p)
    O1, L1 = run_gpu(p, 0.0, d)
    v16 = torch.empty(d["v"].shape, dtype=torch.float16, device="cuda")
    assert fa.fa_convert_v_fp16(d["v"], v16, d["v"].numel()) == 0
    o = torch.empty((p.B, p.Hq, p.Sq, p.Dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((p.B, p.Hq, p.Sq), dtype=torch.float32, device="cuda")
    assert fa.fa_fwd(d["q"], d["k"], v16, o, lse, p.B, p.Hq, p.Hkv, p.Sq, p.Skv, p.D, p.Dv,
                     p.scale, p.mask | fa.FA_V_FP16) == 0
    assert fa.fa_check_status() == 0
    assert np.array_equal(o.float().cpu().double().numpy(), O1)
    assert np.array_equal(lse.cpu().double().numpy(), L1)


def test_bf16_v_beyond_fp16_range_is_reported():
    """A bf16 V value above 65504 cannot enter the fp16 P.V product: the call
    completes and fa_check_status reports FA_ERR_RANGE once, then clears."""
    import torch
    import attention_forward_fa_gb300 as fa
    p = W.dense(name="range", B=1, Hq=2, Sq=256, D=128, mask=W.MASK_CAUSAL, seed=27)
    d = to_device(p)
    d["v"][0, 1, 77, 5] = 70000.0
    o = torch.empty((p.B, p.Hq, p.Sq, p.Dv), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((p.B, p.Hq, p.Sq), dtype=torch.float32, device="cuda")
    assert fa.fa_check_status() == 0
    assert fa.fa_fwd(d["q"], d["k"], d["v"], o, lse, p.B, p.Hq, p.Hkv, p.Sq, p.Skv, p.D, p.Dv,
                     p.scale, p.mask) == 0
    assert fa.fa_check_status() == -8
    assert fa.fa_check_status() == 0

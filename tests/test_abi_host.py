"""Host-side checks of the C ABI that need no GPU: the library builds for
sm_103a, loads, exports every function include/fa_fwd.h declares, and rejects
bad arguments synchronously with the documented codes."""
import ctypes
import os
import re

import pytest

from attention_forward_fa_gb300 import _binding as B
from attention_forward_fa_gb300 import build as BUILD

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa_fwd.h")


@pytest.fixture(scope="module")
def lib():
    BUILD.build()
    return B.library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(fa_\w+)\s*\(", src, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("fa_fwd", "fa_check_status", "fa_strerror", "fa_set_wait_timeout_ns",
              "fa_set_max_kv_split",
              "fa_last_cuda_error", "fa_last_cuda_error_string"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_error_strings(lib):
    for code in range(-8, 1):
        assert B.fa_strerror(code)
    assert "unknown" in B.fa_strerror(-99)


P = 0x10000  # a 16-byte aligned stand-in address; validation fails before any use


def _device_visible() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(autouse=True)
def no_device_for_stand_in_addresses(request):
    """The calls below pass stand-in addresses and rely on the argument checks
    failing before any CUDA call.  They run only where no GPU is visible, so
    that a regression in the order of the checks can never launch a kernel on
    those addresses."""
    if request.node.name.startswith(("test_header", "test_library", "test_error_strings",
                                     "test_backward_wrapper")):
        return
    if _device_visible():
        pytest.skip("stand-in device addresses: host-only check, no GPU may be visible")


def call(lib, **kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, B=1, Hq=2, Hkv=2, Sq=128, Skv=128, D=128, Dv=128,
             scale=0.1, mask_mode=0, seqlens=None, kv_block_idx=None, topk_idx=None,
             rescale_threshold=0.0, stream=0)
    a.update(kw)
    return B.fa_fwd(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1), (dict(k=None), -1), (dict(o=None), -1), (dict(lse=None), -1),
    (dict(v=None), -1),
    (dict(B=0), -2), (dict(Hq=3, Hkv=2), -2), (dict(Sq=-1), -2), (dict(D=0), -2),
    (dict(mask_mode=3), -2), (dict(mask_mode=2), -2), (dict(mask_mode=0x800), -2),
    (dict(kv_block_idx=(P, 17, 64, 0, 0)), -2), (dict(kv_block_idx=(P, 0, 128, 0, 0)), -2),
    (dict(kv_block_idx=(P, 513, 128, 0, 0)), -2),
    (dict(kv_block_idx=(P, 4, 128, 0, 0), topk_idx=(P, 8, 0)), -2),
    (dict(rescale_threshold=-1.0), -5), (dict(rescale_threshold=16.0), -5),
    (dict(rescale_threshold=float("nan")), -5), (dict(scale=float("inf")), -2),
    (dict(D=96, Dv=96), -3), (dict(D=128, Dv=64), -3), (dict(D=256, Dv=256), -3),
    (dict(q=P + 8), -4), (dict(o=P + 2), -4), (dict(lse=P + 2), -4),
])
def test_argument_errors_are_synchronous(lib, kw, code):
    assert call(lib, **kw) == code


MLA = dict(Hq=128, Hkv=1, D=576, Dv=512, v=None, mask_mode=0x200, topk_idx=(P, 2048, 0))


@pytest.mark.parametrize("kw,code", [
    (dict(topk_idx=(P, 2049, 0)), -2), (dict(topk_idx=(P, 0, 0)), -2),
    (dict(topk_idx=(P, 64, -1)), -2), (dict(mask_mode=0x202), -2),
    (dict(Hq=4, Hkv=2), -3), (dict(mask_mode=0), -1), (dict(D=512), -3), (dict(Dv=576), -3),
    (dict(topk_idx=(P + 2, 64, 0)), -4), (dict(q=P + 8), -4),
])
def test_topk_argument_errors(lib, kw, code):
    a = dict(MLA)
    a.update(kw)
    assert call(lib, **a) == code


def test_topk_without_latent_is_unsupported(lib):
    assert call(lib, topk_idx=(P, 64, 0)) == -3   # D = Dv = 128 with a separate V


def test_timeout_setter(lib):
    B.fa_set_wait_timeout_ns(5_000_000)
    B.fa_set_wait_timeout_ns(0)   # back to the default


def test_o_lo_pointer_checks(lib):
    """fa_fwd_o_lo refuses a NULL or misaligned residual buffer before anything runs."""
    args = [P, P, P, P]
    tail = [P, 1, 2, 2, 128, 128, 128, 128, 0.1, 0, None, None, None, 0.0, None]
    assert lib.fa_fwd_o_lo(*args, None, *tail) == -1
    assert lib.fa_fwd_o_lo(*args, P + 2, *tail) == -4


@pytest.mark.parametrize("change, code", [
    (dict(q=None), -1), (dict(dout=None), -1), (dict(lse=None), -1),
    (dict(D=96, Dv=96), -3), (dict(Dv=64), -3),
    (dict(Hq=3, Hkv=2), -2), (dict(Sq=0), -2), (dict(mask_mode=2), -2), (dict(mask_mode=0x200), -2),
    (dict(dk=P + 8), -4), (dict(o_lo=P + 2), -4),
])
def test_bwd_argument_errors(lib, change, code):
    """fa_bwd checks its arguments before anything runs (no GPU needed)."""
    a = dict(q=P, k=P, v=P, o=P, o_lo=None, lse=P, dout=P, dq=P, dk=P, dv=P, B=1, Hq=2, Hkv=1,
             Sq=256, Skv=256, D=128, Dv=128, scale=0.1, mask_mode=1, seqlens=None, stream=0)
    a.update(change)
    assert B.fa_bwd(**a) == code


def test_kv_split_setter_range(lib):
    assert B.fa_set_max_kv_split(0) == -2
    assert B.fa_set_max_kv_split(9) == -2
    assert B.fa_set_max_kv_split(1) == 0
    assert B.fa_set_max_kv_split(8) == 0   # back to the default


@pytest.mark.parametrize("args,code", [
    ((None, P, 8), -1), ((P, None, 8), -1), ((P, P, 0), -2), ((P, P, 12), -2),
    ((P + 8, P, 8), -4), ((P, P + 2, 8), -4),
])
def test_convert_v_argument_errors(lib, args, code):
    assert B.fa_convert_v_fp16(*args, stream=0) == code


def test_backward_wrapper_rejects_host_or_mixed_tensors():
    torch = pytest.importorskip("torch")
    import attention_forward_fa_gb300 as fa
    q = torch.zeros(1, 2, 8, 128, dtype=torch.bfloat16)
    lse = torch.zeros(1, 2, 8)
    with pytest.raises(ValueError):
        fa.flash_attention_backward(q, q, q, q, lse, q)                  # host tensors
    with pytest.raises(ValueError):
        fa.flash_attention_backward(q, q.half(), q, q, lse, q)           # mixed types


def test_noalloc_rejects_a_latent_beyond_its_scratch_before_any_cuda_call(lib):
    """fa_fwd_noalloc refuses a bf16 key latent whose fp16 copy exceeds its
    32 MiB array with FA_ERR_SCRATCH, among the argument checks: no CUDA call
    is made (none could succeed here, without a GPU)."""
    Skv = 29128   # 29128 * 576 * 2 bytes > 32 MiB
    code = B.fa_fwd_noalloc(P, P, None, P, P, 1, 128, 1, 128, Skv, 576, 512, 0.1, B.FA_V_FROM_K,
                            None, None, (P, 2048, 0), 0.0, stream=0)
    assert code == -9
    assert "scratch" in B.fa_strerror(code)
    # an fp16 latent of the same size needs no scratch: it passes that check
    # (and then fails for want of a device, or of anything behind P)
    code16 = B.fa_fwd_noalloc(P, P, None, P, P, 1, 128, 1, 128, Skv, 576, 512, 0.1,
                              B.FA_V_FROM_K | B.FA_DTYPE_FP16, None, None, (P, 2048, 0), 0.0,
                              stream=0)
    assert code16 != -9



def call_ext(lib, ex, **kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, B=1, Hq=2, Hkv=2, Sq=128, Skv=128, D=128, Dv=128,
             scale=0.1, mask_mode=0, seqlens=None, rescale_threshold=0.0, stream=0)
    a.update(kw)
    return B.fa_fwd_ext(extras=ex, **a)


def _ex(**kw):
    e = B.fa_extras_t()
    for k, v in kw.items():
        setattr(e, k, v)
    return e


@pytest.mark.parametrize("ex,kw,code", [
    (None, {}, -1),
    (_ex(window=3), {}, -2), (_ex(window=-1), {}, -2), (_ex(alibi=3), {}, -2),
    (_ex(), dict(mask_mode=2), -2), (_ex(), dict(mask_mode=0x200, v=None), -3),
    (_ex(), dict(Skv=128 * 513), -2),
    (_ex(atten_mask=P, mask_stride_q=-16), {}, -2),
    (_ex(atten_mask=P + 8, mask_stride_q=128), {}, -4),
    (_ex(atten_mask=P, mask_stride_q=120), {}, -4),
    (_ex(atten_mask=P, mask_stride_q=128, mask_stride_h=8), {}, -4),
    (_ex(atten_mask=P, mask_stride_q=120), dict(Skv=120), -4),
    (_ex(), dict(D=576, Dv=512), -3), (_ex(), dict(q=P + 8), -4), (_ex(), dict(B=0), -2),
    (_ex(pse=P, alibi=1), {}, -2), (_ex(pse=P, pse_type=2), {}, -2),
    (_ex(pse=P, pse_stride_q=-8), {}, -2), (_ex(pse=P + 8, pse_stride_q=128), {}, -4),
    (_ex(pse=P, pse_stride_q=124), {}, -4), (_ex(pse=P, pse_stride_q=128), dict(Skv=124), -4),
    (_ex(keep_prob=-0.5), {}, -2), (_ex(keep_prob=1.5), {}, -2), (_ex(keep_prob=float("nan")), {}, -2),
    (_ex(keep_prob=0.9, offset=8), {}, -2), (_ex(keep_prob=0.9), dict(Skv=136), -2),
])
def test_ext_argument_errors(lib, ex, kw, code):
    assert call_ext(lib, ex, **kw) == code


def call_fp8(lib, **kw):
    a = dict(q8=P, k8=P, v8=P, d_scale_q=P, d_scale_k=P, d_scale_v=P, fp8_format=0, o=P, lse=P,
             B=1, Hq=2, Hkv=2, Sq=128, Skv=128, D=128, Dv=128, scale=0.1, mask_mode=0,
             seqlens=None, extras=None, rescale_threshold=0.0, stream=0)
    a.update(kw)
    return B.fa_fwd_fp8(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(d_scale_q=None), -1), (dict(d_scale_v=None), -1), (dict(q8=None), -1),
    (dict(fp8_format=2), -2), (dict(mask_mode=0x100), -2), (dict(mask_mode=2), -2),
    (dict(D=96, Dv=96), -3), (dict(q8=P + 8), -4), (dict(d_scale_k=P + 2), -4),
    (dict(extras=_ex(window=5)), -2), (dict(B=0), -2), (dict(Skv=128 * 513), -2),
])
def test_fp8_argument_errors(lib, kw, code):
    assert call_fp8(lib, **kw) == code


def test_binding_constants_match_the_header():
    """Every FA_* integer #define of include/fa_fwd.h has the same value in the
    Python binding."""
    import re
    from pathlib import Path
    import attention_forward_fa_gb300._binding as B

    text = (Path(__file__).resolve().parents[1] / "include" / "fa_fwd.h").read_text()
    found = re.findall(r"^#define\s+(FA_[A-Z0-9_]+)\s+(-?(?:0x[0-9A-Fa-f]+|\d+))\b", text, re.M)
    assert len(found) >= 10
    for name, val in found:
        if hasattr(B, name):
            assert getattr(B, name) == int(val, 0), name
    for name in ("FA_OK", "FA_ERR_RANGE", "FA_ERR_DEVICE_TIMEOUT", "FA_MASK_CAUSAL", "FA_DTYPE_FP16"):
        assert name in dict(found), name

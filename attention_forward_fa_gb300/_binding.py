"""ctypes binding of libfa_fwd.so (see include/fa_fwd.h for the contract)."""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(PKG, "libfa_fwd.so")

FA_MASK_NONE = 0
FA_MASK_CAUSAL = 1
FA_MASK_CAUSAL_DIAG_BLOCK = 2
FA_DTYPE_FP16 = 0x100
FA_V_FROM_K = 0x200
FA_V_FP16 = 0x400
FA_FP8_E4M3 = 0
FA_FP8_E5M2 = 1

FA_OK = 0
FA_ERR_NULL = -1
FA_ERR_SHAPE = -2
FA_ERR_UNSUPPORTED = -3
FA_ERR_ALIGN = -4
FA_ERR_THRESHOLD = -5
FA_ERR_CUDA = -6
FA_ERR_DEVICE_TIMEOUT = -7
FA_ERR_RANGE = -8
FA_ERR_SCRATCH = -9


class FaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"fa_fwd error {code}: {msg}")
        self.code = code


class fa_block_sparse_t(ctypes.Structure):
    _fields_ = [("idx", ctypes.c_void_p), ("max_sel", ctypes.c_int32), ("block", ctypes.c_int32),
                ("stride_b", ctypes.c_int64), ("stride_h", ctypes.c_int64)]


class fa_topk_t(ctypes.Structure):
    _fields_ = [("idx", ctypes.c_void_p), ("topk", ctypes.c_int32), ("stride_b", ctypes.c_int64)]


class fa_extras_t(ctypes.Structure):
    _fields_ = [("window", ctypes.c_int32), ("pre_tokens", ctypes.c_int32),
                ("next_tokens", ctypes.c_int32), ("alibi", ctypes.c_int32),
                ("atten_mask", ctypes.c_void_p), ("mask_stride_b", ctypes.c_int64),
                ("mask_stride_h", ctypes.c_int64), ("mask_stride_q", ctypes.c_int64),
                ("pse", ctypes.c_void_p), ("pse_stride_b", ctypes.c_int64),
                ("pse_stride_h", ctypes.c_int64), ("pse_stride_q", ctypes.c_int64),
                ("pse_type", ctypes.c_int32), ("keep_prob", ctypes.c_float),
                ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint64)]


_lib = None


def library_path() -> str:
    return _LIB_PATH


def library() -> ctypes.CDLL:
    """Load libfa_fwd.so (raises OSError if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise OSError(f"{_LIB_PATH} is missing: build it with "
                          "`python -m attention_forward_fa_gb300.build`")
        lib = ctypes.CDLL(_LIB_PATH)
        lib.fa_fwd.restype = ctypes.c_int
        lib.fa_fwd.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_void_p] + [ctypes.c_int] * 7 + [
            ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(fa_block_sparse_t),
            ctypes.POINTER(fa_topk_t), ctypes.c_float, ctypes.c_void_p]
        lib.fa_fwd_noalloc.restype = ctypes.c_int
        lib.fa_fwd_noalloc.argtypes = lib.fa_fwd.argtypes
        lib.fa_fwd_fp8.restype = ctypes.c_int
        lib.fa_fwd_fp8.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_int, ctypes.c_void_p,
                                                           ctypes.c_void_p] + [ctypes.c_int] * 7 + [
            ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(fa_extras_t),
            ctypes.c_float, ctypes.c_void_p]
        lib.fa_fwd_ext.restype = ctypes.c_int
        lib.fa_fwd_ext.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_void_p] + [ctypes.c_int] * 7 + [
            ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.POINTER(fa_extras_t),
            ctypes.c_float, ctypes.c_void_p]
        lib.fa_fwd_o_lo.restype = ctypes.c_int
        lib.fa_fwd_o_lo.argtypes = lib.fa_fwd.argtypes[:4] + [ctypes.c_void_p] + lib.fa_fwd.argtypes[4:]
        lib.fa_bwd.restype = ctypes.c_int
        lib.fa_bwd.argtypes = [ctypes.c_void_p] * 10 + [ctypes.c_int] * 7 + [
            ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p]
        lib.fa_convert_v_fp16.restype = ctypes.c_int
        lib.fa_convert_v_fp16.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64,
                                          ctypes.c_void_p]
        lib.fa_check_status.restype = ctypes.c_int
        lib.fa_check_status.argtypes = [ctypes.c_void_p]
        lib.fa_set_wait_timeout_ns.restype = None
        lib.fa_set_wait_timeout_ns.argtypes = [ctypes.c_int64]
        lib.fa_set_max_kv_split.restype = ctypes.c_int
        lib.fa_set_max_kv_split.argtypes = [ctypes.c_int]
        lib.fa_wait_probe.restype = ctypes.c_int
        lib.fa_wait_probe.argtypes = [ctypes.c_void_p]
        lib.fa_strerror.restype = ctypes.c_char_p
        lib.fa_strerror.argtypes = [ctypes.c_int]
        lib.fa_last_cuda_error.restype = ctypes.c_int
        lib.fa_last_cuda_error_string.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def _ptr(x) -> Optional[int]:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def fa_strerror(code: int) -> str:
    return library().fa_strerror(code).decode()


def fa_fwd(q, k, v, o, lse, B: int, Hq: int, Hkv: int, Sq: int, Skv: int, D: int, Dv: int,
           scale: float, mask_mode: int, seqlens=None, kv_block_idx=None, topk_idx=None,
           rescale_threshold: float = 0.0, stream=None) -> int:
    """Direct call of the C entry point.  Tensors (or raw device pointers) for
    q, k, v, o, lse, seqlens; kv_block_idx = (idx, max_sel, block, stride_b,
    stride_h) and topk_idx = (idx, topk, stride_b) with device index arrays.
    Returns the FA_* code."""
    lib = library()
    bs = None
    if kv_block_idx is not None:
        idx, max_sel, block, sb, sh = kv_block_idx
        bs = ctypes.pointer(fa_block_sparse_t(_ptr(idx), max_sel, block, sb, sh))
    tk = None
    if topk_idx is not None:
        idx, topk, sb = topk_idx
        tk = ctypes.pointer(fa_topk_t(_ptr(idx), topk, sb))
    return lib.fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Skv, D, Dv,
                      float(scale), int(mask_mode), _ptr(seqlens), bs, tk,
                      float(rescale_threshold), _stream(stream))


def fa_fwd_o_lo(q, k, v, o, o_lo, lse, B: int, Hq: int, Hkv: int, Sq: int, Skv: int, D: int,
                Dv: int, scale: float, mask_mode: int, seqlens=None, kv_block_idx=None,
                topk_idx=None, rescale_threshold: float = 0.0, stream=None) -> int:
    """fa_fwd that also writes o_lo = fp32(O) - O rounded to o's type (same
    type and layout as o).  Same arguments as fa_fwd plus o_lo after o."""
    lib = library()
    bs = None
    if kv_block_idx is not None:
        idx, max_sel, block, sb, sh = kv_block_idx
        bs = ctypes.pointer(fa_block_sparse_t(_ptr(idx), max_sel, block, sb, sh))
    tk = None
    if topk_idx is not None:
        idx, topk, sb = topk_idx
        tk = ctypes.pointer(fa_topk_t(_ptr(idx), topk, sb))
    return lib.fa_fwd_o_lo(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(o_lo), _ptr(lse), B, Hq, Hkv,
                           Sq, Skv, D, Dv, float(scale), int(mask_mode), _ptr(seqlens), bs, tk,
                           float(rescale_threshold), _stream(stream))


def fa_bwd(q, k, v, o, o_lo, lse, dout, dq, dk, dv, B: int, Hq: int, Hkv: int, Sq: int, Skv: int,
           D: int, Dv: int, scale: float, mask_mode: int, seqlens=None, stream=None) -> int:
    """Direct call of the backward entry point (see include/fa_fwd.h); o_lo
    may be None.  Returns the FA_* code."""
    return library().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(o_lo), _ptr(lse), _ptr(dout),
                            _ptr(dq), _ptr(dk), _ptr(dv), B, Hq, Hkv, Sq, Skv, D, Dv, float(scale),
                            int(mask_mode), _ptr(seqlens), _stream(stream))


def fa_fwd_ext(q, k, v, o, lse, B: int, Hq: int, Hkv: int, Sq: int, Skv: int, D: int, Dv: int,
               scale: float, mask_mode: int, seqlens, extras, rescale_threshold: float = 0.0,
               stream=None) -> int:
    """Direct call of fa_fwd_ext (see include/fa_fwd.h).  extras: an
    fa_extras_t (or None, which the library rejects).  Returns the FA_* code."""
    return library().fa_fwd_ext(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Skv,
                                D, Dv, float(scale), int(mask_mode), _ptr(seqlens),
                                ctypes.byref(extras) if extras is not None else None,
                                float(rescale_threshold), _stream(stream))


def fa_fwd_fp8(q8, k8, v8, d_scale_q, d_scale_k, d_scale_v, fp8_format: int, o, lse, B: int,
               Hq: int, Hkv: int, Sq: int, Skv: int, D: int, Dv: int, scale: float,
               mask_mode: int, seqlens=None, extras=None, rescale_threshold: float = 0.0,
               stream=None) -> int:
    """Direct call of fa_fwd_fp8 (see include/fa_fwd.h).  Returns the FA_* code."""
    return library().fa_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v8), _ptr(d_scale_q), _ptr(d_scale_k),
                                _ptr(d_scale_v), int(fp8_format), _ptr(o), _ptr(lse), B, Hq, Hkv,
                                Sq, Skv, D, Dv, float(scale), int(mask_mode), _ptr(seqlens),
                                ctypes.byref(extras) if extras is not None else None,
                                float(rescale_threshold), _stream(stream))


def flash_attention_forward_fp8(q8, k8, v8, d_scale_q, d_scale_k, d_scale_v, *, fp8_format="e4m3",
                                scale: Optional[float] = None, causal: bool = False, seqlens=None,
                                rescale_threshold: float = 0.0, stream=None):
    """Allocating wrapper over fa_fwd_fp8: q8 / k8 / v8 CUDA tensors of fp8 bytes
    (torch float8_e4m3fn / float8_e5m2 or uint8) [B, H, S, D], d_scale_* fp32
    [B, H, ceil(S / 128)].  Returns (o fp16, lse)."""
    import torch
    B, Hq, Sq, D = q8.shape
    _, Hkv, Skv, _ = k8.shape
    Dv = v8.shape[-1]
    for t in (q8, k8, v8, d_scale_q, d_scale_k, d_scale_v):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("FP8 inputs and scales must be contiguous CUDA tensors")
    fmt = {"e4m3": FA_FP8_E4M3, "e5m2": FA_FP8_E5M2}[fp8_format]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    out = torch.empty((B, Hq, Sq, Dv), dtype=torch.float16, device=q8.device)
    lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q8.device)
    _raise(fa_fwd_fp8(q8, k8, v8, d_scale_q, d_scale_k, d_scale_v, fmt, out, lse, B, Hq, Hkv, Sq,
                      Skv, D, Dv, scale, FA_MASK_CAUSAL if causal else FA_MASK_NONE, seqlens, None,
                      rescale_threshold, stream))
    return out, lse


def fa_fwd_noalloc(q, k, v, o, lse, B: int, Hq: int, Hkv: int, Sq: int, Skv: int, D: int,
                   Dv: int, scale: float, mask_mode: int, seqlens=None, kv_block_idx=None,
                   topk_idx=None, rescale_threshold: float = 0.0, stream=None) -> int:
    """fa_fwd without any memory allocation (fixed 32 MiB scratch inside the
    library; bf16 V larger than that is rejected with FA_ERR_SCRATCH).  Same
    arguments as fa_fwd.  Calls that overlap on the GPU race on the scratch."""
    lib = library()
    bs = None
    if kv_block_idx is not None:
        idx, max_sel, block, sb, sh = kv_block_idx
        bs = ctypes.pointer(fa_block_sparse_t(_ptr(idx), max_sel, block, sb, sh))
    tk = None
    if topk_idx is not None:
        idx, topk, sb = topk_idx
        tk = ctypes.pointer(fa_topk_t(_ptr(idx), topk, sb))
    return lib.fa_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Sq, Skv,
                              D, Dv, float(scale), int(mask_mode), _ptr(seqlens), bs, tk,
                              float(rescale_threshold), _stream(stream))


def fa_convert_v_fp16(v_bf16, v_fp16, n_elems: int, stream=None) -> int:
    """fp16 copy of a bf16 V (see include/fa_fwd.h); returns the FA_* code."""
    return library().fa_convert_v_fp16(_ptr(v_bf16), _ptr(v_fp16), int(n_elems), _stream(stream))


def fa_check_status(stream=None) -> int:
    return library().fa_check_status(_stream(stream))


def fa_set_wait_timeout_ns(ns: int) -> None:
    library().fa_set_wait_timeout_ns(int(ns))


def fa_set_max_kv_split(n: int) -> int:
    """Most KV pieces per unit for under-filled dense problems (1 = never split)."""
    return library().fa_set_max_kv_split(int(n))


def fa_wait_probe(stream=None) -> int:
    return library().fa_wait_probe(_stream(stream))


def _raise(code: int):
    if code != FA_OK:
        lib = library()
        msg = lib.fa_strerror(code).decode()
        if code == -6:
            msg += f" ({lib.fa_last_cuda_error_string().decode()})"
        raise FaError(code, msg)


def flash_attention_forward(q, k, v=None, *, scale: Optional[float] = None, causal: bool = False,
                            mask_mode: Optional[int] = None, seqlens=None, block_idx=None,
                            topk_idx=None, rescale_threshold: float = 0.0, out=None, lse=None,
                            o_lo=None, window=None, bottom_right_causal: bool = False,
                            atten_mask=None, alibi: bool = False, pse=None, pse_type: int = 0,
                            dropout=None, stream=None):
    """Allocating convenience wrapper over fa_fwd.

    q [B,Hq,Sq,D], k [B,Hkv,Skv,D], v [B,Hkv,Skv,Dv] (or None with top-k and a
    shared latent), bf16 or fp16 CUDA tensors.  block_idx: int32 tensor
    [B, Hq or 1, ceil(Sq/128), max_sel]; topk_idx: int32 [B, Sq, W].
    o_lo: True (allocate) or a tensor like out to also receive the output's
    rounding residual (fa_fwd_o_lo).  Returns (o, lse), or (o, lse, o_lo).

    The operator's optional terms go through fa_fwd_ext: window=(pre_tokens,
    next_tokens) (sparse_mode 0), bottom_right_causal (sparse_mode 3),
    atten_mask (bool or uint8 CUDA tensor [..., Sq, Skv] broadcastable to
    [B, Hq, Sq, Skv], True / nonzero = masked; its last dimension contiguous),
    alibi (True or 2: pse_type 2, -slope |i - j|; 3: pse_type 3, -slope
    sqrt|i - j|), pse (a bias tensor of q's type [..., Sq, Skv]
    broadcastable like atten_mask, last dim contiguous) with pse_type 0
    (added after the scale) or 1 (before), dropout=(keep_prob, seed, offset)
    (the Philox mask of include/fa_fwd.h)."""
    import torch
    if q.dtype not in (torch.bfloat16, torch.float16):
        raise TypeError("q, k, v must be bf16 or fp16")
    for t in (q, k, v):
        if t is not None and (not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype):
            raise ValueError("q, k, v must be contiguous CUDA tensors of one dtype")
    B, Hq, Sq, D = q.shape
    _, Hkv, Skv, _ = k.shape
    v_from_k = v is None
    Dv = v.shape[-1] if v is not None else 512
    if mask_mode is None:
        mask_mode = FA_MASK_CAUSAL if causal else FA_MASK_NONE
    if q.dtype == torch.float16:
        mask_mode |= FA_DTYPE_FP16
    if v_from_k:
        mask_mode |= FA_V_FROM_K
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty((B, Hq, Sq, Dv), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, Hq, Sq), dtype=torch.float32, device=q.device)
    bs = None
    if block_idx is not None:
        assert block_idx.dtype == torch.int32 and block_idx.is_contiguous()
        nb, hh, nqb, ms = block_idx.shape
        bs = (block_idx, ms, 128, hh * nqb * ms, nqb * ms if hh > 1 else 0)
    tk = None
    if topk_idx is not None:
        assert topk_idx.dtype == torch.int32 and topk_idx.is_contiguous()
        tk = (topk_idx, topk_idx.shape[-1], topk_idx.shape[-2] * topk_idx.shape[-1])
    if seqlens is not None:
        assert seqlens.dtype == torch.int32 and seqlens.is_cuda
    if (window is not None or bottom_right_causal or atten_mask is not None or alibi
            or pse is not None or dropout is not None):
        if o_lo not in (None, False) or bs is not None or tk is not None:
            raise ValueError("the optional terms apply to dense problems without o_lo")
        ex = fa_extras_t()
        ex.window = 1 if window is not None else (2 if bottom_right_causal else 0)
        if window is not None and bottom_right_causal:
            raise ValueError("window and bottom_right_causal are exclusive")
        ex.pre_tokens, ex.next_tokens = (int(window[0]), int(window[1])) if window is not None else (0, 0)
        ex.alibi = {False: 0, True: 1, 2: 1, 3: 2}[alibi]   # True = pse_type 2
        if dropout is not None:
            ex.keep_prob, ex.seed, ex.offset = float(dropout[0]), int(dropout[1]), int(dropout[2])
        keep = None
        if atten_mask is not None:
            m = atten_mask
            if m.dtype == torch.bool:
                m = m.view(torch.uint8)
            if m.dtype != torch.uint8 or not m.is_cuda or m.stride(-1) != 1:
                raise ValueError("atten_mask must be a bool / uint8 CUDA tensor with a contiguous last dim")
            while m.dim() < 4:
                m = m.unsqueeze(0)
            def st(d):
                return 0 if m.shape[d] == 1 else m.stride(d)
            ex.atten_mask = m.data_ptr()
            ex.mask_stride_b, ex.mask_stride_h, ex.mask_stride_q = st(0), st(1), st(2)
            keep = m
        keep_pse = None
        if pse is not None:
            b_ = pse
            if b_.dtype != q.dtype or not b_.is_cuda or b_.stride(-1) != 1:
                raise ValueError("pse must be a CUDA tensor of q's dtype with a contiguous last dim")
            while b_.dim() < 4:
                b_ = b_.unsqueeze(0)
            def stp(d):
                return 0 if b_.shape[d] == 1 else b_.stride(d)
            ex.pse = b_.data_ptr()
            ex.pse_stride_b, ex.pse_stride_h, ex.pse_stride_q = stp(0), stp(1), stp(2)
            ex.pse_type = int(pse_type)
            keep_pse = b_
        code = fa_fwd_ext(q, k, v, out, lse, B, Hq, Hkv, Sq, Skv, D, Dv, scale, mask_mode, seqlens,
                          ex, rescale_threshold, stream)
        del keep, keep_pse
        _raise(code)
        return out, lse
    if o_lo is None or o_lo is False:
        code = fa_fwd(q, k, v, out, lse, B, Hq, Hkv, Sq, Skv, D, Dv, scale, mask_mode, seqlens, bs,
                      tk, rescale_threshold, stream)
        _raise(code)
        return out, lse
    if o_lo is True:
        o_lo = torch.empty_like(out)
    code = fa_fwd_o_lo(q, k, v, out, o_lo, lse, B, Hq, Hkv, Sq, Skv, D, Dv, scale, mask_mode,
                       seqlens, bs, tk, rescale_threshold, stream)
    _raise(code)
    return out, lse, o_lo


def flash_attention_backward(q, k, v, o, lse, dout, *, o_lo=None, scale: Optional[float] = None,
                             causal: bool = False, seqlens=None, dq=None, dk=None, dv=None,
                             stream=None):
    """Allocating wrapper over fa_bwd: q, o, dout [B,Hq,Sq,D], k, v
    [B,Hkv,Skv,D] (D = 64 or 128; bf16 or fp16 CUDA tensors, contiguous), lse [B,Hq,Sq]
    fp32 from the forward, o_lo its residual (recommended).  Returns
    (dq, dk, dv) in the inputs' type."""
    import torch
    for t in (q, k, v, o, dout) + ((o_lo,) if o_lo is not None else ()):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype:
            raise ValueError("q, k, v, o, dout (and o_lo) must be contiguous CUDA tensors of one dtype")
    B, Hq, Sq, D = q.shape
    _, Hkv, Skv, _ = k.shape
    Dv = v.shape[-1]
    mask_mode = FA_MASK_CAUSAL if causal else FA_MASK_NONE
    if q.dtype == torch.float16:
        mask_mode |= FA_DTYPE_FP16
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _raise(fa_bwd(q, k, v, o, o_lo, lse, dout, dq, dk, dv, B, Hq, Hkv, Sq, Skv, D, Dv, scale,
                  mask_mode, seqlens, stream))
    return dq, dk, dv

"""ctypes binding of the C ABI in ``include/attn.h`` (argument marshalling only).

Every function here forwards torch tensors' device pointers to the library;
all arithmetic runs in the library's CUDA kernels.  There is no CPU or PyTorch
fallback: if ``libattn.so`` is missing or fails to load, :func:`lib` raises.
"""
from __future__ import annotations

import ctypes
import math
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libattn.so")

ATTN_OK = 0
STATUS = {
    0: "ATTN_OK", -1: "ATTN_ERR_NULL", -2: "ATTN_ERR_DIM", -3: "ATTN_ERR_GQA",
    -4: "ATTN_ERR_HEAD_DIM", -5: "ATTN_ERR_ALIGN", -6: "ATTN_ERR_SCALE", -7: "ATTN_ERR_CUDA",
    -8: "ATTN_ERR_TIMEOUT", -9: "ATTN_ERR_DEVICE", -10: "ATTN_ERR_SEQLEN",
    -11: "ATTN_ERR_CHUNK", -12: "ATTN_ERR_CAPACITY", -13: "ATTN_ERR_PAGE",
}

_c_int, _c_float, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_void_p
SIGNATURES = {
    "attn_fwd": (_c_int, [_vp, _vp, _vp, _vp, _vp] + [_c_int] * 6 + [_c_float, _c_int, _c_int, _vp]),
    "attn_fwd_fp32": (_c_int, [_vp, _vp, _vp, _vp, _vp] + [_c_int] * 6 + [_c_float, _c_int, _c_int, _vp]),
    "attn_fwd_fp16": (_c_int, [_vp, _vp, _vp, _vp, _vp] + [_c_int] * 6 + [_c_float, _c_int, _c_int, _vp]),
    "attn_fwd_varlen": (_c_int, [_vp] * 7 + [_c_int] * 7 + [_c_float, _c_int, _c_int, _vp]),
    "attn_fwd_softcap_sink": (_c_int, [_vp] * 5 + [_c_int] * 6 + [_c_float, _c_int, _c_int, _c_float, _vp, _vp]),
    "attn_decode_workspace_size": (ctypes.c_size_t, [_c_int] * 5),
    "attn_decode_splitkv": (_c_int, [_vp] * 5 + [_c_int] * 5 + [_c_float, _c_int, _vp]),
    "attn_decode_combine": (_c_int, [_vp] * 4 + [_c_int] * 5 + [_vp]),
    "attn_decode_splitkv_paged": (_c_int, [_vp] * 6 + [_c_int] * 7 + [_c_float, _c_int, _vp]),
    "attn_decode_noalloc": (_c_int, [_vp] * 6 + [_c_int] * 5 + [_c_float, _c_int, _vp]),
    "attn_decode_splitkv_fp8": (_c_int, [_vp] * 3 + [_c_float] * 2 + [_vp] * 2 + [_c_int] * 5
                                + [_c_float, _c_int, _vp]),
    "attn_decode_splitkv_paged_fp8": (_c_int, [_vp] * 3 + [_c_float] * 2 + [_vp] * 3 + [_c_int] * 7
                                      + [_c_float, _c_int, _vp]),
    "attn_fwd_fp8_workspace_size": (ctypes.c_size_t, [_c_int] * 4),
    "attn_fwd_fp8": (_c_int, [_vp] * 3 + [_c_float] * 3 + [_vp] * 3 + [_c_int] * 6
                     + [_c_float, _c_int, _c_int, _vp]),
    "attn_bwd_workspace_size": (ctypes.c_size_t, [_c_int] * 3),
    "attn_bwd": (_c_int, [_vp] * 10 + [_c_int] * 6 + [_c_float, _c_int, _c_int, _vp]),
    "attn_get_device_error": (_c_int, [_vp]),
    "attn_strerror": (ctypes.c_char_p, [_c_int]),
}

_LIB = None


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS.get(code, code)} ({strerror(code)})")


def lib(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load ``libattn.so`` (once) and declare its signatures."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run softmax_attention_attn_gb300.build.build() first")
        handle = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype, fn.argtypes = res, args
        _LIB = handle
    return _LIB


def strerror(code: int) -> str:
    return lib().attn_strerror(int(code)).decode()


def _check(code: int, where: str) -> None:
    if code != ATTN_OK:
        raise AttnError(code, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _require(t, dtype, name):
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _fwd(name, dtype, q, k, v, o, lse, scale, causal, window, stream):
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _require(t, dtype, n)
    B, Hq, Nq, D = q.shape
    _, Hkv, Nk, _ = k.shape
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, Hq, Nq, device=q.device, dtype=torch.float32)
    _require(o, dtype, "o")
    _require(lse, torch.float32, "lse")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    code = getattr(lib(), name)(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk, D,
                                scale, int(bool(causal)), int(window), _stream(stream))
    _check(code, name)
    return o, lse


def attn_fwd(q, k, v, o=None, lse=None, scale=None, causal=False, window=0, stream=None):
    """bf16 forward: q ``[B,Hq,Nq,D]``, k/v ``[B,Hkv,Nk,D]`` -> (o, lse)."""
    import torch
    return _fwd("attn_fwd", torch.bfloat16, q, k, v, o, lse, scale, causal, window, stream)


def attn_fwd_softcap_sink(q, k, v, o=None, lse=None, scale=None, causal=False, window=0, softcap=0.0,
                          sinks=None, stream=None):
    """bf16 forward with a softcap on the scaled scores (``softcap > 0``) and one
    sink logit per query head (``sinks``: float32 CUDA tensor ``[Hq]``, or None)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _require(t, torch.bfloat16, n)
    B, Hq, Nq, D = q.shape
    _, Hkv, Nk, _ = k.shape
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, Hq, Nq, device=q.device, dtype=torch.float32)
    _require(o, torch.bfloat16, "o")
    _require(lse, torch.float32, "lse")
    if sinks is not None:
        _require(sinks, torch.float32, "sinks")
        if sinks.numel() != Hq:
            raise ValueError(f"sinks must hold Hq = {Hq} values")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    code = lib().attn_fwd_softcap_sink(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, Nq, Nk, D,
                                       scale, int(bool(causal)), int(window), float(softcap),
                                       _ptr(sinks) if sinks is not None else None, _stream(stream))
    _check(code, "attn_fwd_softcap_sink")
    return o, lse


def attn_bwd(q, k, v, o, do, lse, dq=None, dk=None, dv=None, workspace=None, scale=None, causal=False,
             window=0, stream=None):
    """bf16 backward: (dq fp32 ``[B,Hq,Nq,D]``, dk, dv bf16 ``[B,Hkv,Nk,D]``) for the
    upstream gradient ``do``, from the forward's ``o`` and ``lse``."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (do, "do")):
        _require(t, torch.bfloat16, n)
    _require(lse, torch.float32, "lse")
    B, Hq, Nq, D = q.shape
    _, Hkv, Nk, _ = k.shape
    if dq is None:
        dq = torch.empty(B, Hq, Nq, D, device=q.device, dtype=torch.float32)
    if dk is None:
        dk = torch.empty_like(k)
    if dv is None:
        dv = torch.empty_like(v)
    need = int(lib().attn_bwd_workspace_size(B, Hq, Nq))
    if workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    if workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace holds fewer than {need} bytes")
    _require(dq, torch.float32, "dq")
    _require(dk, torch.bfloat16, "dk")
    _require(dv, torch.bfloat16, "dv")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    code = lib().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                          _ptr(workspace), B, Hq, Hkv, Nq, Nk, D, scale, int(bool(causal)), int(window),
                          _stream(stream))
    _check(code, "attn_bwd")
    return dq, dk, dv


def attn_fwd_fp16(q, k, v, o=None, lse=None, scale=None, causal=False, window=0, stream=None):
    """fp16 forward: same layouts as :func:`attn_fwd`."""
    import torch
    return _fwd("attn_fwd_fp16", torch.float16, q, k, v, o, lse, scale, causal, window, stream)


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, o=None, lse=None, scale=None,
                    causal=False, window=0, stream=None):
    """Ragged bf16 forward: q ``[total_q,Hq,D]``, k/v ``[total_k,Hkv,D]`` -> (o, lse ``[Hq,total_q]``)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _require(t, torch.bfloat16, n)
    _require(cu_seqlens_q, torch.int32, "cu_seqlens_q")
    _require(cu_seqlens_k, torch.int32, "cu_seqlens_k")
    total_q, Hq, D = q.shape
    total_k, Hkv, _ = k.shape
    B = cu_seqlens_q.numel() - 1
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(Hq, total_q, device=q.device, dtype=torch.float32)
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    code = lib().attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens_q),
                                 _ptr(cu_seqlens_k), B, Hq, Hkv, int(max_seqlen_q), total_q, total_k, D,
                                 scale, int(bool(causal)), int(window), _stream(stream))
    _check(code, "attn_fwd_varlen")
    return o, lse


def attn_fwd_fp32(q, k, v, o=None, lse=None, scale=None, causal=False, window=0, stream=None):
    """fp32 forward: same layouts as :func:`attn_fwd`."""
    import torch
    return _fwd("attn_fwd_fp32", torch.float32, q, k, v, o, lse, scale, causal, window, stream)


def attn_decode_workspace_size(B, Hq, D, Nk_max, chunk=512) -> int:
    return int(lib().attn_decode_workspace_size(B, Hq, D, Nk_max, chunk))


def attn_decode_splitkv(q, k_cache, v_cache, seqlens, workspace, scale=None, chunk=512, stream=None):
    """Partial step: fills ``workspace`` (uint8 CUDA tensor) with per-chunk O and LSE."""
    import torch
    _require(q, torch.bfloat16, "q")
    _require(k_cache, torch.bfloat16, "k_cache")
    _require(v_cache, torch.bfloat16, "v_cache")
    _require(seqlens, torch.int32, "seqlens")
    B, Hq, D = q.shape
    _, Nk_max, Hkv, _ = k_cache.shape
    need = attn_decode_workspace_size(B, Hq, D, Nk_max, chunk)
    if workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace holds fewer than {need} bytes")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    code = lib().attn_decode_splitkv(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), _ptr(workspace),
                                     B, Hq, Hkv, Nk_max, D, scale, int(chunk), _stream(stream))
    _check(code, "attn_decode_splitkv")
    return workspace


def attn_decode_combine(workspace, seqlens, B, Hq, Nk_max, D, o=None, lse=None, chunk=512,
                        device=None, stream=None):
    """Combine step: merges the chunk results into ``o [B,Hq,D]`` bf16 and ``lse [B,Hq]``."""
    import torch
    device = workspace.device if device is None else device
    if o is None:
        o = torch.empty(B, Hq, D, device=device, dtype=torch.bfloat16)
    if lse is None:
        lse = torch.empty(B, Hq, device=device, dtype=torch.float32)
    _require(o, torch.bfloat16, "o")
    _require(lse, torch.float32, "lse")
    _require(seqlens, torch.int32, "seqlens")
    code = lib().attn_decode_combine(_ptr(workspace), _ptr(seqlens), _ptr(o), _ptr(lse),
                                     B, Hq, Nk_max, D, int(chunk), _stream(stream))
    _check(code, "attn_decode_combine")
    return o, lse


def attn_decode(q, k_cache, v_cache, seqlens, workspace=None, o=None, lse=None, scale=None,
                chunk=512, stream=None):
    """Split-KV decode: partial step then combine step on the same stream."""
    import torch
    B, Hq, D = q.shape
    Nk_max = k_cache.shape[1]
    if workspace is None:
        workspace = torch.empty(attn_decode_workspace_size(B, Hq, D, Nk_max, chunk),
                                device=q.device, dtype=torch.uint8)
    attn_decode_splitkv(q, k_cache, v_cache, seqlens, workspace, scale, chunk, stream)
    return attn_decode_combine(workspace, seqlens, B, Hq, Nk_max, D, o, lse, chunk, q.device, stream)


def attn_decode_paged(q, k_pages, v_pages, block_table, seqlens, workspace=None, o=None, lse=None,
                      scale=None, chunk=512, stream=None):
    """Split-KV decode on a paged cache: partial step, then combine step."""
    import torch
    _require(q, torch.bfloat16, "q")
    _require(k_pages, torch.bfloat16, "k_pages")
    _require(v_pages, torch.bfloat16, "v_pages")
    _require(block_table, torch.int32, "block_table")
    _require(seqlens, torch.int32, "seqlens")
    B, Hq, D = q.shape
    num_pages, page_size, Hkv, _ = k_pages.shape
    max_pages = block_table.shape[1]
    nk_max = max_pages * page_size
    need = attn_decode_workspace_size(B, Hq, D, nk_max, chunk)
    if workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    if workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace holds fewer than {need} bytes")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    code = lib().attn_decode_splitkv_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                           _ptr(seqlens), _ptr(workspace), B, Hq, Hkv, num_pages,
                                           page_size, max_pages, D, scale, int(chunk), _stream(stream))
    _check(code, "attn_decode_splitkv_paged")
    return attn_decode_combine(workspace, seqlens, B, Hq, nk_max, D, o, lse, chunk, q.device, stream)


def _require_fp8(t, name):
    """fp8 E4M3 cache tensor: uint8 codes or torch.float8_e4m3fn, CUDA, contiguous."""
    import torch
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in (torch.uint8, torch.float8_e4m3fn):
        raise TypeError(f"{name} must hold E4M3 codes (uint8 or float8_e4m3fn), got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def attn_fwd_fp8_workspace_size(B, Hkv, Nk, D) -> int:
    return int(lib().attn_fwd_fp8_workspace_size(int(B), int(Hkv), int(Nk), int(D)))


def attn_fwd_fp8(q, k, v, q_scale=1.0, k_scale=1.0, v_scale=1.0, o=None, lse=None, workspace=None,
                 scale=None, causal=False, window=0, stream=None):
    """Forward on fp8 E4M3 q ``[B,Hq,Nq,D]`` and k/v ``[B,Hkv,Nk,D]`` (values = code *
    per-tensor scale) -> (o bf16, lse fp32).  ``workspace`` (uint8, at least
    :func:`attn_fwd_fp8_workspace_size` bytes) is allocated when None."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _require_fp8(t, n)
    B, Hq, Nq, D = q.shape
    _, Hkv, Nk, _ = k.shape
    need = attn_fwd_fp8_workspace_size(B, Hkv, Nk, D)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    if workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace holds fewer than {need} bytes")
    if o is None:
        o = torch.empty(B, Hq, Nq, D, device=q.device, dtype=torch.bfloat16)
    if lse is None:
        lse = torch.empty(B, Hq, Nq, device=q.device, dtype=torch.float32)
    _require(o, torch.bfloat16, "o")
    _require(lse, torch.float32, "lse")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    code = lib().attn_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), float(q_scale), float(k_scale), float(v_scale),
                              _ptr(o), _ptr(lse), _ptr(workspace), B, Hq, Hkv, Nq, Nk, D, scale,
                              int(bool(causal)), int(window), _stream(stream))
    _check(code, "attn_fwd_fp8")
    return o, lse


def attn_decode_fp8(q, k_cache, v_cache, seqlens, k_scale=1.0, v_scale=1.0, workspace=None, o=None,
                    lse=None, scale=None, chunk=512, stream=None):
    """Split-KV decode on an fp8 E4M3 cache ``[B,Nk_max,Hkv,D]`` (values = code * scale):
    partial step, then combine step."""
    import torch
    _require(q, torch.bfloat16, "q")
    _require_fp8(k_cache, "k_cache")
    _require_fp8(v_cache, "v_cache")
    _require(seqlens, torch.int32, "seqlens")
    B, Hq, D = q.shape
    _, Nk_max, Hkv, _ = k_cache.shape
    need = attn_decode_workspace_size(B, Hq, D, Nk_max, chunk)
    if workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    if workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace holds fewer than {need} bytes")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    code = lib().attn_decode_splitkv_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), float(k_scale),
                                         float(v_scale), _ptr(seqlens), _ptr(workspace), B, Hq, Hkv,
                                         Nk_max, D, scale, int(chunk), _stream(stream))
    _check(code, "attn_decode_splitkv_fp8")
    return attn_decode_combine(workspace, seqlens, B, Hq, Nk_max, D, o, lse, chunk, q.device, stream)


def attn_decode_paged_fp8(q, k_pages, v_pages, block_table, seqlens, k_scale=1.0, v_scale=1.0,
                          workspace=None, o=None, lse=None, scale=None, chunk=512, stream=None):
    """Split-KV decode on a paged fp8 E4M3 cache ``[num_pages,page_size,Hkv,D]``."""
    import torch
    _require(q, torch.bfloat16, "q")
    _require_fp8(k_pages, "k_pages")
    _require_fp8(v_pages, "v_pages")
    _require(block_table, torch.int32, "block_table")
    _require(seqlens, torch.int32, "seqlens")
    B, Hq, D = q.shape
    num_pages, page_size, Hkv, _ = k_pages.shape
    max_pages = block_table.shape[1]
    nk_max = max_pages * page_size
    need = attn_decode_workspace_size(B, Hq, D, nk_max, chunk)
    if workspace is None:
        workspace = torch.empty(need, device=q.device, dtype=torch.uint8)
    if workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace holds fewer than {need} bytes")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    code = lib().attn_decode_splitkv_paged_fp8(_ptr(q), _ptr(k_pages), _ptr(v_pages), float(k_scale),
                                               float(v_scale), _ptr(block_table), _ptr(seqlens),
                                               _ptr(workspace), B, Hq, Hkv, num_pages, page_size,
                                               max_pages, D, scale, int(chunk), _stream(stream))
    _check(code, "attn_decode_splitkv_paged_fp8")
    return attn_decode_combine(workspace, seqlens, B, Hq, nk_max, D, o, lse, chunk, q.device, stream)


def attn_decode_noalloc(q, k_cache, v_cache, seqlens, o=None, lse=None, scale=None, chunk=512,
                        stream=None):
    """Split-KV decode without a caller workspace (scratch inside the library)."""
    import torch
    _require(q, torch.bfloat16, "q")
    _require(k_cache, torch.bfloat16, "k_cache")
    _require(v_cache, torch.bfloat16, "v_cache")
    _require(seqlens, torch.int32, "seqlens")
    B, Hq, D = q.shape
    _, Nk_max, Hkv, _ = k_cache.shape
    if o is None:
        o = torch.empty(B, Hq, D, device=q.device, dtype=torch.bfloat16)
    if lse is None:
        lse = torch.empty(B, Hq, device=q.device, dtype=torch.float32)
    _require(o, torch.bfloat16, "o")
    _require(lse, torch.float32, "lse")
    scale = 1.0 / math.sqrt(D) if scale is None else float(scale)
    code = lib().attn_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seqlens), _ptr(o), _ptr(lse),
                                     B, Hq, Hkv, Nk_max, D, scale, int(chunk), _stream(stream))
    _check(code, "attn_decode_noalloc")
    return o, lse


def get_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device error word."""
    return int(lib().attn_get_device_error(_stream(stream)))

"""Python binding of libfa.so: argument marshalling only (ctypes).

Every step of the attention path runs in the library's CUDA kernels; PyTorch supplies device
memory and the current stream.  There is no fallback: when libfa.so is missing or the device
is not an sm_103 GPU, the calls raise.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional, Tuple

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa.so")

FA_FP16, FA_BF16 = 0, 1
FA_OK, FA_ERR_INVALID, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = 0, -1, -2, -3, -4
FA_ERR_INTERNAL = -5
FA_NOALLOC_MAX_ROWS = 1 << 20  # B*H*N limit of fa_bwd_noalloc

# exported names and their signatures, in the order include/fa.h declares them
_vp, _i, _f, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
_u64 = ctypes.c_ulonglong
SIGNATURES = {
    "fa_fwd": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp]),
    "fa_fwd_blocksparse": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _vp]),
    "fa_fwd_gqa": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _vp]),
    "fa_fwd_fp8_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "fa_fwd_fp8": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _f, _f, _f, _i, _vp,
                        _vp, _sz, _vp]),
    "fa_bwd_workspace_bytes": (_sz, [_i, _i, _i, _i]),
    "fa_bwd": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i, _i,
                    _f, _i, _vp, _vp]),
    "fa_bwd_gqa_workspace_bytes": (_sz, [_i, _i, _i, _i, _i]),
    "fa_bwd_gqa": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i,
                        _i, _i, _f, _i, _vp, _vp]),
    "fa_fwd_dropout": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _f,
                            _u64, _u64, _vp]),
    "fa_bwd_dropout": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _i, _i, _i, _i,
                            _i, _i, _f, _i, _vp, _f, _u64, _u64, _vp]),
    "fa_bwd_preprocess": (_i, [_vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "fa_bwd_dkdv": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i,
                         _vp, _vp]),
    "fa_bwd_dq": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _vp]),
    "fa_bwd_noalloc": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i,
                            _f, _i, _vp, _vp]),
    "fa_decode_workspace_bytes": (_sz, [_i, _i, _i, _i, _i, _i]),
    "fa_decode": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp,
                       _sz, _vp]),
    "fa_sync_status": (_i, [_vp]),
    "fa_status_string": (ctypes.c_char_p, [_i]),
    "fa_debug_set_visit_log": (_i, [_vp, _sz]),
    "fa_debug_set_wait_limit_ns": (_i, [ctypes.c_ulonglong]),
    "fa_debug_set_fault": (_i, [_i]),
    "fa_debug_set_dkdv_splits": (_i, [_i]),
}

_lib = None
_lock = threading.Lock()


class FAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


def load(path: str = LIB_PATH):
    """Load libfa.so (built by ``exact_attention_staged_gb300.build``); raise if absent."""
    global _lib
    lib = _lib
    if lib is not None:  # loaded: no lock on the per-call path
        return lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it with "
                                   "`python -m exact_attention_staged_gb300.build`")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    return load().fa_status_string(int(code)).decode()


def _check(code: int, where: str):
    if code != FA_OK:
        raise FAError(code, where)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return FA_BF16
    if t.dtype == torch.float16:
        return FA_FP16
    raise TypeError(f"unsupported dtype {t.dtype}: use torch.bfloat16 or torch.float16")


def _dev(t: Optional[torch.Tensor], name: str, like: Optional[torch.Tensor] = None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if like is not None and (t.shape != like.shape or t.dtype != like.dtype):
        raise ValueError(f"{name} must match q in shape and dtype")
    return t.data_ptr()  # ctypes passes the int as the c_void_p argument


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream: Optional[torch.cuda.Stream], like: Optional[torch.Tensor] = None) -> int:
    """The CUDA stream handle to launch on: `stream`, else the current stream of the tensor's
    device (read as a raw handle: no Stream object is built on the per-call path)."""
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None and like is not None:
        return _raw_stream(like.device.index)
    return torch.cuda.current_stream().cuda_stream


def _shape(q: torch.Tensor):
    if q.dim() != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    return tuple(int(x) for x in q.shape)


def fwd(q, k, v, scale: Optional[float] = None, causal: bool = False, block_mask=None,
        out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
        stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """O, LSE = attention forward (fa_fwd, or fa_fwd_blocksparse when block_mask is given)."""
    lib = load()
    B, H, N, d = _shape(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be fp32 [B, H, N]")
    args = [_dev(q, "q"), _dev(k, "k", q), _dev(v, "v", q), _dev(out, "out", q), _dev(lse, "lse"),
            B, H, N, d, _dtype_code(q), float(scale), int(bool(causal))]
    if block_mask is None:
        _check(lib.fa_fwd(*args, _stream(stream, q)), "fa_fwd")
    else:
        if block_mask.dtype != torch.uint8:
            raise TypeError("block_mask must be uint8")
        _check(lib.fa_fwd_blocksparse(*args, _dev(block_mask, "block_mask"), _stream(stream, q)),
               "fa_fwd_blocksparse")
    return out, lse


def workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load().fa_bwd_workspace_bytes(B, H, N, d))


def bwd(q, k, v, o, lse, dout, scale: Optional[float] = None, causal: bool = False,
        block_mask=None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """dQ, dK, dV = attention backward (fa_bwd)."""
    lib = load()
    B, H, N, d = _shape(q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    nbytes = workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError("workspace too small")
    mask_ptr = None if block_mask is None else _dev(block_mask, "block_mask")
    _check(lib.fa_bwd(_dev(q, "q"), _dev(k, "k", q), _dev(v, "v", q), _dev(o, "o", q),
                      _dev(dout, "dout", q), _dev(lse, "lse"), _dev(dq, "dq", q),
                      _dev(dk, "dk", q), _dev(dv, "dv", q), _dev(workspace, "workspace"),
                      nbytes, B, H, N, d, _dtype_code(q), float(scale), int(bool(causal)),
                      mask_ptr, _stream(stream, q)), "fa_bwd")
    return dq, dk, dv


def bwd_preprocess(o, dout, delta, stream=None):
    B, H, N, d = _shape(o)
    _check(load().fa_bwd_preprocess(_dev(o, "o"), _dev(dout, "dout", o), _dev(delta, "delta"),
                                    B, H, N, d, _dtype_code(o), _stream(stream, o)),
           "fa_bwd_preprocess")
    return delta


def bwd_dkdv(q, k, v, dout, lse, delta, dk, dv, scale=None, causal=False, block_mask=None,
             stream=None):
    B, H, N, d = _shape(q)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    mask_ptr = None if block_mask is None else _dev(block_mask, "block_mask")
    _check(load().fa_bwd_dkdv(_dev(q, "q"), _dev(k, "k", q), _dev(v, "v", q),
                              _dev(dout, "dout", q), _dev(lse, "lse"), _dev(delta, "delta"),
                              _dev(dk, "dk", q), _dev(dv, "dv", q), B, H, N, d, _dtype_code(q),
                              float(scale), int(bool(causal)), mask_ptr, _stream(stream, q)),
           "fa_bwd_dkdv")
    return dk, dv


def bwd_dq(q, k, v, dout, lse, delta, dq, scale=None, causal=False, block_mask=None,
           stream=None):
    B, H, N, d = _shape(q)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    mask_ptr = None if block_mask is None else _dev(block_mask, "block_mask")
    _check(load().fa_bwd_dq(_dev(q, "q"), _dev(k, "k", q), _dev(v, "v", q),
                            _dev(dout, "dout", q), _dev(lse, "lse"), _dev(delta, "delta"),
                            _dev(dq, "dq", q), B, H, N, d, _dtype_code(q), float(scale),
                            int(bool(causal)), mask_ptr, _stream(stream, q)), "fa_bwd_dq")
    return dq


def _kv_check(q, k, v):
    """K, V of grouped-query attention: [B, H_kv, N, d] with H_kv dividing H; returns H_kv."""
    B, H, N, d = _shape(q)
    for name, t in (("k", k), ("v", v)):
        if t.dim() != 4 or t.dtype != q.dtype or t.shape[0] != B or t.shape[2:] != q.shape[2:]:
            raise ValueError(f"{name} must be [B, H_kv, N, d] with the dtype of q")
    if k.shape != v.shape:
        raise ValueError("k and v must have the same shape")
    return int(k.shape[1])


def fwd_gqa(q, k, v, scale: Optional[float] = None, causal: bool = False, block_mask=None,
            out: Optional[torch.Tensor] = None, lse: Optional[torch.Tensor] = None,
            stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """O, LSE = grouped-query attention forward (fa_fwd_gqa): k, v are [B, H_kv, N, d]."""
    lib = load()
    B, H, N, d = _shape(q)
    Hkv = _kv_check(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be fp32 [B, H, N]")
    mask_ptr = None if block_mask is None else _dev(block_mask, "block_mask")
    _check(lib.fa_fwd_gqa(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(out, "out", q),
                          _dev(lse, "lse"), B, H, Hkv, N, d, _dtype_code(q), float(scale),
                          int(bool(causal)), mask_ptr, _stream(stream, q)), "fa_fwd_gqa")
    return out, lse


def fp8_workspace_bytes(B: int, H_kv: int, N: int, d: int) -> int:
    return int(load().fa_fwd_fp8_workspace_bytes(B, H_kv, N, d))


def fwd_fp8(q, k, v, descale_q: float, descale_k: float, descale_v: float,
            scale: Optional[float] = None, causal: bool = False, block_mask=None, out=None,
            lse=None, workspace=None, stream=None):
    """O (bf16), LSE of attention on e4m3 codes (uint8 tensors) with per-tensor scales
    (fa_fwd_fp8): q [B, H, N, d], k, v [B, H_kv, N, d]."""
    lib = load()
    B, H, N, d = _shape(q)
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.uint8:
            raise TypeError(f"{name} must hold e4m3 codes as torch.uint8")
    if k.dim() != 4 or k.shape != v.shape or k.shape[0] != B or k.shape[2:] != q.shape[2:]:
        raise ValueError("k and v must be [B, H_kv, N, d]")
    Hkv = int(k.shape[1])
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = torch.empty((B, H, N, d), dtype=torch.bfloat16, device=q.device) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    nbytes = fp8_workspace_bytes(B, Hkv, N, d)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    mask_ptr = None if block_mask is None else _dev(block_mask, "block_mask")
    _check(lib.fa_fwd_fp8(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(out, "out"),
                          _dev(lse, "lse"), B, H, Hkv, N, d, float(scale), float(descale_q),
                          float(descale_k), float(descale_v), int(bool(causal)), mask_ptr,
                          _dev(workspace, "workspace"),
                          workspace.numel() * workspace.element_size(), _stream(stream, q)),
           "fa_fwd_fp8")
    return out, lse


def gqa_workspace_bytes(B: int, H: int, H_kv: int, N: int, d: int) -> int:
    return int(load().fa_bwd_gqa_workspace_bytes(B, H, H_kv, N, d))


def bwd_gqa(q, k, v, o, lse, dout, scale: Optional[float] = None, causal: bool = False,
            block_mask=None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """dQ, dK, dV = grouped-query attention backward (fa_bwd_gqa); dk, dv are [B, H_kv, N, d]."""
    lib = load()
    B, H, N, d = _shape(q)
    Hkv = _kv_check(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    nbytes = gqa_workspace_bytes(B, H, Hkv, N, d)
    if nbytes == 0:
        raise ValueError("invalid grouped-query sizes")
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError("workspace too small")
    mask_ptr = None if block_mask is None else _dev(block_mask, "block_mask")
    _check(lib.fa_bwd_gqa(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(o, "o", q),
                          _dev(dout, "dout", q), _dev(lse, "lse"), _dev(dq, "dq", q),
                          _dev(dk, "dk", k), _dev(dv, "dv", k), _dev(workspace, "workspace"),
                          nbytes, B, H, Hkv, N, d, _dtype_code(q), float(scale),
                          int(bool(causal)), mask_ptr, _stream(stream, q)), "fa_bwd_gqa")
    return dq, dk, dv


def decode_workspace_bytes(B: int, H: int, H_kv: int, Nq: int, Nk: int, d: int) -> int:
    return int(load().fa_decode_workspace_bytes(B, H, H_kv, Nq, Nk, d))


def decode(q, k, v, scale: Optional[float] = None, causal: bool = False, kv_len=None,
           out=None, lse=None, workspace=None, stream=None):
    """O, LSE of Nq new rows q [B, H, Nq, d] against the cache k, v [B, H_kv, Nk, d] (fa_decode).

    kv_len: int32 CUDA tensor [B] of valid cache lengths, or None for Nk.
    """
    lib = load()
    B, H, Nq, d = _shape(q)
    if k.dim() != 4 or k.shape != v.shape or k.shape[0] != B or k.shape[3] != d \
            or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k and v must be [B, H_kv, Nk, d] with the dtype of q")
    Hkv, Nk = int(k.shape[1]), int(k.shape[2])
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Nq):
        raise ValueError("lse must be fp32 [B, H, Nq]")
    if kv_len is not None and (kv_len.dtype != torch.int32 or tuple(kv_len.shape) != (B,)):
        raise ValueError("kv_len must be int32 [B]")
    nbytes = decode_workspace_bytes(B, H, Hkv, Nq, Nk, d)
    if workspace is None and nbytes > 0:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    ws = None if workspace is None else _dev(workspace, "workspace")
    _check(lib.fa_decode(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(out, "out", q),
                         _dev(lse, "lse"), None if kv_len is None else _dev(kv_len, "kv_len"),
                         B, H, Hkv, Nq, Nk, d, _dtype_code(q), float(scale), int(bool(causal)),
                         ws, nbytes, _stream(stream, q)), "fa_decode")
    return out, lse


def fwd_dropout(q, k, v, p_drop: float, seed: int, offset: int = 0,
                scale: Optional[float] = None, causal: bool = False, block_mask=None, out=None,
                lse=None, stream=None):
    """O, LSE with dropout on the probabilities (fa_fwd_dropout); k, v may have H_kv heads."""
    lib = load()
    B, H, N, d = _shape(q)
    Hkv = _kv_check(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    mask_ptr = None if block_mask is None else _dev(block_mask, "block_mask")
    _check(lib.fa_fwd_dropout(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(out, "out", q),
                              _dev(lse, "lse"), B, H, Hkv, N, d, _dtype_code(q), float(scale),
                              int(bool(causal)), mask_ptr, float(p_drop), int(seed), int(offset),
                              _stream(stream, q)), "fa_fwd_dropout")
    return out, lse


def bwd_dropout(q, k, v, o, lse, dout, p_drop: float, seed: int, offset: int = 0,
                scale: Optional[float] = None, causal: bool = False, block_mask=None, dq=None,
                dk=None, dv=None, workspace=None, stream=None):
    """dQ, dK, dV of the forward with dropout (fa_bwd_dropout), same dropout arguments."""
    lib = load()
    B, H, N, d = _shape(q)
    Hkv = _kv_check(q, k, v)
    scale = 1.0 / math.sqrt(d) if scale is None else scale
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    nbytes = gqa_workspace_bytes(B, H, Hkv, N, d)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    if workspace.numel() * workspace.element_size() < nbytes:
        raise ValueError("workspace too small")
    mask_ptr = None if block_mask is None else _dev(block_mask, "block_mask")
    _check(lib.fa_bwd_dropout(_dev(q, "q"), _dev(k, "k"), _dev(v, "v"), _dev(o, "o", q),
                              _dev(dout, "dout", q), _dev(lse, "lse"), _dev(dq, "dq", q),
                              _dev(dk, "dk", k), _dev(dv, "dv", k), _dev(workspace, "workspace"),
                              nbytes, B, H, Hkv, N, d, _dtype_code(q), float(scale),
                              int(bool(causal)), mask_ptr, float(p_drop), int(seed), int(offset),
                              _stream(stream, q)), "fa_bwd_dropout")
    return dq, dk, dv


def sync_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(load().fa_sync_status(_stream(stream)))


def debug_set_visit_log(buf: Optional[torch.Tensor]):
    if buf is None:
        _check(load().fa_debug_set_visit_log(None, 0), "fa_debug_set_visit_log")
    else:
        if buf.dtype != torch.uint8:
            raise TypeError("visit log must be uint8")
        _check(load().fa_debug_set_visit_log(_dev(buf, "visit_log"), buf.numel()),
               "fa_debug_set_visit_log")


def debug_set_wait_limit_ns(ns: int):
    _check(load().fa_debug_set_wait_limit_ns(int(ns)), "fa_debug_set_wait_limit_ns")


def debug_set_fault(mode: int):
    _check(load().fa_debug_set_fault(int(mode)), "fa_debug_set_fault")


def debug_set_dkdv_splits(splits: int):
    _check(load().fa_debug_set_dkdv_splits(int(splits)), "fa_debug_set_dkdv_splits")

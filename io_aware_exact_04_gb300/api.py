"""PyTorch-facing wrappers of the C ABI: argument checks and marshalling only.

PyTorch provides device memory and the current CUDA stream; every step of the
attention computation runs in the library's kernels.
"""

from __future__ import annotations

import ctypes
import math
from typing import Optional, Tuple

import torch

from . import _lib


def _lib_fa():
    return _lib.load("libfa.so")


def _p(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _check_bhnd(name: str, t: torch.Tensor, shape=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise ValueError(f"{name} must be bfloat16")
    if t.dim() != 4 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous [B, H, N, d] tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _kv(kv_len: Optional[torch.Tensor], B: int, device) -> Optional[torch.Tensor]:
    if kv_len is None:
        return None
    if kv_len.dtype != torch.int32 or kv_len.shape != (B,) or not kv_len.is_contiguous():
        raise ValueError("kv_len must be a contiguous int32 tensor of shape [B]")
    if kv_len.device != device:
        raise ValueError("kv_len must live on the same device as q")
    return kv_len


def _kv_shape(q, k):
    """[B, H, N_k, d] of k: q's batch, heads and head dim with its own length."""
    _check_bhnd("k", k)
    if k.shape[0] != q.shape[0] or k.shape[1] != q.shape[1] or k.shape[3] != q.shape[3]:
        raise ValueError(f"k has shape {tuple(k.shape)}; q is {tuple(q.shape)} (only N may differ)")
    return tuple(k.shape)


def forward(q, k, v, causal: bool = False, scale: Optional[float] = None, kv_len=None, out=None,
            lse=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """O, LSE of exact softmax attention (include/fa.h: fa_forward_qk). q is [B, H, N_q, d];
    k and v are [B, H, N_k, d] (N_k may differ; causal aligns the queries with the last keys)."""
    _check_bhnd("q", q)
    B, H, N, d = q.shape
    kshape = _kv_shape(q, k)
    _check_bhnd("v", v, kshape)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q) if out is None else out
    _check_bhnd("out", o, q.shape)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    kv = _kv(kv_len, B, q.device)
    with torch.cuda.device(q.device):
        rc = _lib_fa().fa_forward_qk(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, N, kshape[2], d, scale,
                                     int(bool(causal)), _p(kv), _stream(q.device))
    _lib.check(rc, "fa_forward_qk")
    return o, lse


def _check_hTd(name: str, t: torch.Tensor, shape=None):
    if not t.is_cuda or t.dtype != torch.bfloat16 or t.dim() != 3 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bfloat16 CUDA tensor [H, T, d]")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _cu(cu_seqlens: torch.Tensor, device) -> torch.Tensor:
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens must be a contiguous int32 tensor [B + 1]")
    if cu_seqlens.device != device:
        raise ValueError("cu_seqlens must live on the same device as q")
    return cu_seqlens


def forward_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = False, scale: Optional[float] = None):
    """O, LSE over packed sequences (include/fa.h: fa_forward_varlen): q, k, v [H, T, d], sequence
    b at rows cu_seqlens[b] .. cu_seqlens[b + 1]; lse [H, T]."""
    _check_hTd("q", q)
    H, T, d = q.shape
    _check_hTd("k", k, q.shape)
    _check_hTd("v", v, q.shape)
    cu = _cu(cu_seqlens, q.device)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    o = torch.empty_like(q)
    lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    with torch.cuda.device(q.device):
        rc = _lib_fa().fa_forward_varlen(_p(q), _p(k), _p(v), _p(o), _p(lse), _p(cu), cu.numel() - 1, H, T,
                                         int(max_seqlen), d, scale, int(bool(causal)), _stream(q.device))
    _lib.check(rc, "fa_forward_varlen")
    return o, lse


def backward_varlen(q, k, v, o, do, lse, cu_seqlens, max_seqlen: int, causal: bool = False,
                    scale: Optional[float] = None):
    """dQ, dK, dV over packed sequences (include/fa.h: fa_backward_varlen); shapes as forward_varlen."""
    _check_hTd("q", q)
    H, T, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("do", do)):
        _check_hTd(name, t, q.shape)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (H, T) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [H, T] tensor")
    cu = _cu(cu_seqlens, q.device)
    B = cu.numel() - 1
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    lib = _lib_fa()
    need = int(lib.fa_backward_varlen_workspace_size(B, H, T, d))
    work = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    with torch.cuda.device(q.device):
        rc = lib.fa_backward_varlen(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv), _p(cu), B, H,
                                    T, int(max_seqlen), d, scale, int(bool(causal)), _p(work), work.numel(),
                                    _stream(q.device))
    _lib.check(rc, "fa_backward_varlen")
    return dq, dk, dv


def forward_split(q, k, v, causal: bool = False, scale: Optional[float] = None, kv_len=None,
                  n_split: Optional[int] = None, with_lse: bool = False, out=None, workspace=None):
    """Inference forward with split keys (include/fa.h: fa_forward_split): O, and LSE when
    with_lse (else None). n_split defaults to the library's choice for the shape."""
    _check_bhnd("q", q)
    B, H, N, d = q.shape
    kshape = _kv_shape(q, k)
    _check_bhnd("v", v, kshape)
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    lib = _lib_fa()
    if n_split is None:
        with torch.cuda.device(q.device):
            n_split = int(lib.fa_forward_split_count(B, H, N, kshape[2], d))
    o = torch.empty_like(q) if out is None else out
    _check_bhnd("out", o, q.shape)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if with_lse else None
    need = int(lib.fa_forward_split_workspace_size(B, H, N, d, n_split))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    kv = _kv(kv_len, B, q.device)
    with torch.cuda.device(q.device):
        rc = lib.fa_forward_split(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, N, kshape[2], d, scale,
                                  int(bool(causal)), _p(kv), int(n_split), _p(workspace), workspace.numel(),
                                  _stream(q.device))
    _lib.check(rc, "fa_forward_split")
    return o, lse


def workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(_lib_fa().fa_backward_workspace_size(B, H, N, d))


def backward(q, k, v, o, do, lse, causal: bool = False, scale: Optional[float] = None, kv_len=None,
             dq=None, dk=None, dv=None, workspace=None):
    """dQ, dK, dV by recomputation from Q, K, V, O, dO and LSE (fa_backward_qk); shapes as
    for forward."""
    _check_bhnd("q", q)
    B, H, N, d = q.shape
    kshape = _kv_shape(q, k)
    for name, t, shp in (("v", v, kshape), ("o", o, q.shape), ("do", do, q.shape)):
        _check_bhnd(name, t, shp)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous float32 [B, H, N] tensor")
    scale = 1.0 / math.sqrt(d) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(k) if dv is None else dv
    need = workspace_bytes(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    kv = _kv(kv_len, B, q.device)
    with torch.cuda.device(q.device):
        rc = _lib_fa().fa_backward_qk(_p(q), _p(k), _p(v), _p(o), _p(do), _p(lse), _p(dq), _p(dk), _p(dv),
                                      B, H, N, kshape[2], d, scale, int(bool(causal)), _p(kv), _p(workspace),
                                      workspace.numel(), _stream(q.device))
    _lib.check(rc, "fa_backward_qk")
    return dq, dk, dv


def device_status(device=None):
    """(code, [code, site, blockIdx.x, blockIdx.y]) of the device status word; clears it."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    detail = (ctypes.c_int * 4)()
    with torch.cuda.device(dev):
        rc = _lib_fa().fa_get_last_device_status_detail(_stream(dev), detail)
    return rc, list(detail)


class _Attention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal, scale, kv_len):
        o, lse = forward(q, k, v, causal=causal, scale=scale, kv_len=kv_len)
        ctx.save_for_backward(q, k, v, o, lse, kv_len if kv_len is not None else torch.empty(0))
        ctx.causal, ctx.scale, ctx.has_kv = causal, scale, kv_len is not None
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse, kv = ctx.saved_tensors
        dq, dk, dv = backward(q, k, v, o, do.contiguous(), lse, causal=ctx.causal, scale=ctx.scale,
                              kv_len=kv if ctx.has_kv else None)
        return dq, dk, dv, None, None, None


def attention(q, k, v, causal: bool = False, scale: Optional[float] = None, kv_len=None) -> torch.Tensor:
    """Differentiable exact attention: O only; only the LSE is kept for backward."""
    return _Attention.apply(q, k, v, causal, scale, kv_len)

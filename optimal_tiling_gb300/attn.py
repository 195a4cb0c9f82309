"""Thin Python binding of the C ABI in ``include/attn.h``.

Argument marshalling only: every step of the computation runs in the CUDA
library.  PyTorch provides device memory and the current stream.  The library
is loaded on first use; if it has not been built, calls raise -- there is no
fallback of any kind.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import threading

import torch

from . import build as _build

ATTN_OK = 0
ATTN_ERR_INVALID_ARG = 1
ATTN_ERR_UNSUPPORTED = 2
ATTN_ERR_CUDA = 3
ATTN_ERR_TIMEOUT = 4
ATTN_ERR_WORKSPACE = 5

ATTN_DTYPE_F32 = 0
ATTN_DTYPE_BF16 = 1

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t


class BlockMask(ctypes.Structure):
    """attn_block_mask: device mask pointer, block side (64 or 128), bytes between heads' masks."""
    _fields_ = [("blocks", _vp), ("block", _i), ("head_stride", ctypes.c_longlong)]


class AttnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


def library_path() -> str:
    return _build.LIB_PATH


def load():
    """Load the built library (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_PATH
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library {path} is not built; run optimal_tiling_gb300.build.build()")
            lib = ctypes.CDLL(path)
            lib.attn_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp, _vp]
            lib.attn_fwd.restype = _i
            lib.attn_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i,
                                     _vp, _vp, _sz, _vp]
            lib.attn_bwd.restype = _i
            _bm = ctypes.POINTER(BlockMask)
            lib.attn_fwd_masked.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _bm, _vp]
            lib.attn_fwd_masked.restype = _i
            lib.attn_bwd_masked.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i,
                                            _bm, _vp, _sz, _vp]
            lib.attn_bwd_masked.restype = _i
            lib.attn_bwd_workspace_size.argtypes = [_i, _i, _i, _i, _i]
            lib.attn_bwd_workspace_size.restype = _sz
            lib.attn_fwd_materialized.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f, _i, _vp,
                                                  _vp, _sz, _vp]
            lib.attn_fwd_materialized.restype = _i
            lib.attn_fwd_materialized_workspace_size.argtypes = [_i, _i, _i, _i, _i]
            lib.attn_fwd_materialized_workspace_size.restype = _sz
            lib.attn_bwd_static_workspace.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i,
                                                      _i, _f, _i, _vp, _vp]
            lib.attn_bwd_static_workspace.restype = _i
            lib.attn_bwd_materialized.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _f,
                                                  _i, _vp, _vp, _sz, _vp]
            lib.attn_bwd_materialized.restype = _i
            lib.attn_bwd_materialized_workspace_size.argtypes = [_i, _i, _i, _i, _i]
            lib.attn_bwd_materialized_workspace_size.restype = _sz
            lib.attn_decode.argtypes = [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _sz, _vp]
            lib.attn_decode.restype = _i
            lib.attn_decode_workspace_size.argtypes = [_i, _i, _i, _i, _i, _i]
            lib.attn_decode_workspace_size.restype = _sz
            lib.attn_selftest_timeout.argtypes = [ctypes.c_uint, _vp]
            lib.attn_selftest_timeout.restype = _i
            lib.attn_device_status.argtypes = [_vp]
            lib.attn_device_status.restype = _i
            lib.attn_status_string.argtypes = [_i]
            lib.attn_status_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().attn_status_string(int(status)).decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return ATTN_DTYPE_F32
    if t.dtype == torch.bfloat16:
        return ATTN_DTYPE_BF16
    raise TypeError(f"unsupported dtype {t.dtype}: use float32 or bfloat16")


def _shape(q: torch.Tensor):
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, d] tensors")
    return tuple(int(x) for x in q.shape)


def _check(*ts):
    dev = ts[0].device
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda or t.device != dev:
            raise ValueError("all tensors must be CUDA tensors on one device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _on(stream):
    """Context for the tensors a wrapper allocates (outputs, LSE, workspace): they belong to
    the stream the library launches on, so that the caching allocator does not hand their
    memory to another stream's allocation while the kernels still use it."""
    return torch.cuda.stream(stream) if stream is not None else contextlib.nullcontext()


def _raise(status, where):
    if status != ATTN_OK:
        raise AttnError(status, where)


def attn_bwd_workspace_size(B, H, N, d, dtype_code) -> int:
    return int(load().attn_bwd_workspace_size(B, H, N, d, dtype_code))


def attn_fwd_materialized_workspace_size(B, H, N, d, dtype_code) -> int:
    return int(load().attn_fwd_materialized_workspace_size(B, H, N, d, dtype_code))


def attn_fwd(q, k, v, scale: float, block_mask=None, out=None, lse=None, stream=None):
    """O, LSE = softmax(scale q k^T) v, logsumexp; tensors [B, H, N, d]."""
    lib = load()
    B, H, N, d = _shape(q)
    with _on(stream):
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    _check(q, k, v, out, lse, block_mask)
    st = lib.attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d, float(scale),
                      _dtype_code(q), _ptr(block_mask), _stream(stream))
    _raise(st, "attn_fwd")
    return out, lse


def _block_mask(mask, block: int, B: int, H: int, N: int):
    """attn_block_mask for a uint8 mask tensor: [nb, nb] shared by every head, or
    [B*H, nb, nb] / [B, H, nb, nb] one per head (nb = ceil(N / block))."""
    if mask is None:
        return BlockMask(None, int(block), 0)
    nb = (N + block - 1) // block
    if mask.dtype != torch.uint8 or not mask.is_contiguous():
        raise ValueError("block mask must be a contiguous uint8 tensor")
    if tuple(mask.shape[-2:]) != (nb, nb):
        raise ValueError(f"block mask must end in [{nb}, {nb}] for N={N}, block={block}")
    if mask.dim() == 2:
        stride = 0
    elif mask.numel() == B * H * nb * nb and mask.dim() in (3, 4):
        stride = nb * nb
    else:
        raise ValueError("block mask must be [nb, nb], [B*H, nb, nb] or [B, H, nb, nb]")
    return BlockMask(ctypes.c_void_p(mask.data_ptr()), int(block), stride)


def attn_fwd_masked(q, k, v, scale: float, mask=None, block: int = 128, out=None, lse=None, stream=None):
    """attn_fwd with a general block mask: 64- or 128-blocks, shared or one per head."""
    lib = load()
    B, H, N, d = _shape(q)
    with _on(stream):
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    _check(q, k, v, out, lse, mask)
    bm = _block_mask(mask, block, B, H, N)
    st = lib.attn_fwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d, float(scale),
                             _dtype_code(q), ctypes.byref(bm), _stream(stream))
    _raise(st, "attn_fwd_masked")
    return out, lse


def attn_bwd_masked(q, k, v, o, do, lse, scale: float, mask=None, block: int = 128, dq=None, dk=None, dv=None,
                    workspace=None, stream=None):
    """attn_bwd with a general block mask (the one the forward used)."""
    lib = load()
    B, H, N, d = _shape(q)
    code = _dtype_code(q)
    need = attn_bwd_workspace_size(B, H, N, d, code)
    with _on(stream):
        dq = torch.empty_like(q) if dq is None else dq
        dk = torch.empty_like(q) if dk is None else dk
        dv = torch.empty_like(q) if dv is None else dv
        if workspace is None:
            workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    _check(q, k, v, o, do, lse, dq, dk, dv, workspace, mask)
    bm = _block_mask(mask, block, B, H, N)
    st = lib.attn_bwd_masked(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                             B, H, N, d, float(scale), code, ctypes.byref(bm), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream))
    _raise(st, "attn_bwd_masked")
    return dq, dk, dv


def attn_bwd(q, k, v, o, do, lse, scale: float, block_mask=None, dq=None, dk=None, dv=None,
             workspace=None, stream=None):
    """dQ, dK, dV of attn_fwd for upstream gradient ``do``."""
    lib = load()
    B, H, N, d = _shape(q)
    code = _dtype_code(q)
    need = attn_bwd_workspace_size(B, H, N, d, code)
    with _on(stream):
        dq = torch.empty_like(q) if dq is None else dq
        dk = torch.empty_like(q) if dk is None else dk
        dv = torch.empty_like(q) if dv is None else dv
        if workspace is None:
            workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    _check(q, k, v, o, do, lse, dq, dk, dv, workspace, block_mask)
    st = lib.attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                      B, H, N, d, float(scale), code, _ptr(block_mask), _ptr(workspace),
                      workspace.numel() * workspace.element_size(), _stream(stream))
    _raise(st, "attn_bwd")
    return dq, dk, dv


def attn_bwd_static_workspace(q, k, v, o, do, lse, scale: float, block_mask=None, dq=None, dk=None, dv=None,
                              stream=None):
    """attn_bwd without a workspace argument: the scratch is the library's fixed
    64 MiB device array (for callers that cannot allocate device memory)."""
    lib = load()
    B, H, N, d = _shape(q)
    with _on(stream):
        dq = torch.empty_like(q) if dq is None else dq
        dk = torch.empty_like(q) if dk is None else dk
        dv = torch.empty_like(q) if dv is None else dv
    _check(q, k, v, o, do, lse, dq, dk, dv, block_mask)
    st = lib.attn_bwd_static_workspace(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                                       _ptr(dk), _ptr(dv), B, H, N, d, float(scale), _dtype_code(q),
                                       _ptr(block_mask), _stream(stream))
    _raise(st, "attn_bwd_static_workspace")
    return dq, dk, dv


def attn_fwd_materialized(q, k, v, scale: float, block_mask=None, out=None, lse=None, workspace=None,
                          stream=None):
    """Same result as attn_fwd through the materialising two-GEMM schedule (bf16)."""
    lib = load()
    B, H, N, d = _shape(q)
    code = _dtype_code(q)
    need = attn_fwd_materialized_workspace_size(B, H, N, d, code)
    with _on(stream):
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
        if workspace is None:
            workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    _check(q, k, v, out, lse, workspace, block_mask)
    st = lib.attn_fwd_materialized(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, d, float(scale),
                                   code, _ptr(block_mask), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream))
    _raise(st, "attn_fwd_materialized")
    return out, lse


def attn_bwd_materialized_workspace_size(B, H, N, d, dtype_code) -> int:
    return int(load().attn_bwd_materialized_workspace_size(B, H, N, d, dtype_code))


def attn_bwd_materialized(q, k, v, o, do, lse, scale: float, block_mask=None, dq=None, dk=None, dv=None,
                          workspace=None, stream=None):
    """dQ, dK, dV through the materialising schedule (P and dS stored in HBM), bf16."""
    lib = load()
    B, H, N, d = _shape(q)
    code = _dtype_code(q)
    need = attn_bwd_materialized_workspace_size(B, H, N, d, code)
    with _on(stream):
        dq = torch.empty_like(q) if dq is None else dq
        dk = torch.empty_like(q) if dk is None else dk
        dv = torch.empty_like(q) if dv is None else dv
        if workspace is None:
            workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    _check(q, k, v, o, do, lse, dq, dk, dv, workspace, block_mask)
    st = lib.attn_bwd_materialized(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk),
                                   _ptr(dv), B, H, N, d, float(scale), code, _ptr(block_mask), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _stream(stream))
    _raise(st, "attn_bwd_materialized")
    return dq, dk, dv


def attn_decode_workspace_size(B, H, Nq, Nk, d, dtype_code) -> int:
    return int(load().attn_decode_workspace_size(B, H, Nq, Nk, d, dtype_code))


def attn_decode(q, k, v, scale: float, out=None, lse=None, workspace=None, stream=None):
    """Decode-shaped attention: q [B, H, Nq, d] against k, v [B, H, Nk, d] (bf16)."""
    lib = load()
    B, H, Nq, d = _shape(q)
    Nk = int(k.shape[2])
    if tuple(k.shape) != (B, H, Nk, d) or tuple(v.shape) != tuple(k.shape):
        raise ValueError("k and v must be [B, H, Nk, d] with q's B, H and d")
    code = _dtype_code(q)
    need = attn_decode_workspace_size(B, H, Nq, Nk, d, code)
    with _on(stream):
        if out is None:
            out = torch.empty_like(q)
        if lse is None:
            lse = torch.empty((B, H, Nq), device=q.device, dtype=torch.float32)
        if workspace is None:
            workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    _check(q, k, v, out, lse, workspace)
    st = lib.attn_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, Nq, Nk, d, float(scale), code,
                         _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    _raise(st, "attn_decode")
    return out, lse


def attn_selftest_timeout(limit_us: int, stream=None) -> None:
    """Enqueue the bounded-wait self-test (a wait that nothing completes)."""
    _raise(load().attn_selftest_timeout(int(limit_us), _stream(stream)), "attn_selftest_timeout")


def attn_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(load().attn_device_status(_stream(stream)))

"""Python binding of libsdm.so, the GB300 (sm_103a) sparse-routed gated
delta-rule memory scan.

Argument marshalling only: every function here checks shapes and dtypes of
CUDA tensors, passes their device pointers and the current CUDA stream to the
C ABI declared in ``include/sdm.h`` (same function names), and raises
``SdmError`` with the library's message on a non-zero status.  All compute
runs in the library's kernels.  There is no CPU fallback: importing works
without a GPU, but every call needs the built library and a CUDA device.

Build the library with ``python -m delta_rule_memory_gb300.build``.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

__all__ = [
    "SdmError", "lib", "library_path", "sdm_version", "sdm_check", "sdm_address", "sdm_scan", "sdm_scan_workspace_size",
    "sdm_scan_noalloc", "sdm_forward_host", "sdm_forward_host_workspace_size", "sdm_scan_train",
    "sdm_scan_backward", "sdm_scan_backward_workspace_size", "sdm_address_backward", "sdm_scan_chunked",
    "sdm_scan_chunked_workspace_size",
    "gdn_scan", "gdn_scan_workspace_size", "gdn2_scan", "gdn2_scan_workspace_size", "sse_scan", "sse_scan_workspace_size", "SDM_RESID_SHARED", "SDM_RESID_PERSLOT", "SSE_WRITE_ADDITIVE", "SSE_WRITE_DELTA",
    "SDM_RESID_ADDITIVE", "SDM_DEVERR_INDEX_RANGE", "SDM_DEVERR_INDEX_REPEAT", "SDM_DEVERR_NONFINITE",
    "SDM_DEVERR_TIMEOUT", "SDM_ERR_DEVICE",
]

SDM_OK, SDM_ERR_INVALID_ARG, SDM_ERR_SHAPE, SDM_ERR_ALIGN, SDM_ERR_UNSUPPORTED, SDM_ERR_CUDA, SDM_ERR_DEVICE = range(7)
SDM_DEVERR_INDEX_RANGE, SDM_DEVERR_INDEX_REPEAT, SDM_DEVERR_NONFINITE, SDM_DEVERR_TIMEOUT = 1, 2, 4, 8
SDM_DTYPE_F32, SDM_DTYPE_BF16 = 0, 1
SDM_RESID_SHARED, SDM_RESID_PERSLOT, SDM_RESID_ADDITIVE = 0, 1, 2
SSE_WRITE_ADDITIVE, SSE_WRITE_DELTA = 0, 1

_HERE = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_HERE, "libsdm.so")
_lock = threading.Lock()
_lib = None

_P, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
_SIGNATURES = {
    "sdm_version": (_I, []),
    "sdm_last_error": (ctypes.c_char_p, []),
    "sdm_check": (_I, [_P, _P]),
    "sdm_address": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    "sdm_scan_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "sdm_scan": (_I, [_P, _P, _I, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P, _P]),
    "sdm_scan_noalloc": (_I, [_P, _P, _I, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P]),
    "sdm_scan_train": (_I, [_P, _P, _I, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _SZ, _P,
                            _P]),
    "sdm_scan_backward_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "sdm_address_backward": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P]),
    "sdm_scan_chunked_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "sdm_scan_chunked": (_I, [_P, _P, _I, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _SZ, _P,
                              _P]),
    "sdm_scan_backward": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P,
                               _P, _P, _P, _P, _P, _SZ, _P, _P]),
    "sdm_forward_host_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I, _I, _I]),
    "sdm_forward_host": (_I, [_P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _P, _I, _P,
                              _SZ, _P, _P]),
    "gdn_scan_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "gdn_scan": (_I, [_P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _P, _P, _SZ, _P, _P]),
    "gdn2_scan_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "gdn2_scan": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _SZ, _P, _P]),
    "sse_scan_workspace_size": (_SZ, [_I, _I, _I, _I, _I, _I, _I, _I]),
    "sse_scan": (_I, [_P, _P, _I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P, _P, _SZ, _P, _P]),
}


class SdmError(RuntimeError):
    """A libsdm call returned a non-zero status."""

    def __init__(self, fn: str, code: int, msg: str):
        super().__init__(f"{fn} failed with status {code}: {msg}")
        self.code = code


def lib() -> ctypes.CDLL:
    """The loaded libsdm.so.  Raises if it was not built: there is no fallback."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(library_path):
                raise RuntimeError(f"libsdm.so is not built ({library_path}); run "
                                   "`python -m delta_rule_memory_gb300.build`")
            h = ctypes.CDLL(library_path)
            for name, (res, args) in _SIGNATURES.items():
                fn = getattr(h, name, None)
                if fn is None:
                    continue
                fn.restype = res
                fn.argtypes = args
            _lib = h
    return _lib


def _check(fn: str, rc: int):
    if rc != SDM_OK:
        raise SdmError(fn, rc, lib().sdm_last_error().decode(errors="replace"))


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _req(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def sdm_version() -> int:
    return lib().sdm_version()


def sdm_check(dev_err=None, stream=None) -> None:
    """Synchronise the stream and raise SdmError (status SDM_ERR_DEVICE) if
    the error word `dev_err` or the library's own timeout record holds a bit.
    The timeout record is cleared by the check; `dev_err` is not."""
    if dev_err is not None:
        _req(dev_err, "dev_err", torch.int32)
    _check("sdm_check", lib().sdm_check(_ptr(dev_err), _stream(stream)))


def sdm_address(s1: torch.Tensor, s2: torch.Tensor, k: int, W: int, idx_out=None, w_out=None, dev_err=None,
                stream=None):
    """Product-key addressing of fp32 score halves [B,T,H,sqrtN].
    Returns (idx int32 [B,T,H,W] in rank order, w fp32 [B,T,H,W])."""
    _req(s1, "s1", torch.float32)
    if s1.dim() != 4:
        raise ValueError("s1 must be [B,T,H,sqrtN]")
    _req(s2, "s2", torch.float32, s1.shape)
    B, T, H, sq = s1.shape
    if idx_out is None:
        idx_out = torch.empty((B, T, H, W), dtype=torch.int32, device=s1.device)
    if w_out is None:
        w_out = torch.empty((B, T, H, W), dtype=torch.float32, device=s1.device)
    _req(idx_out, "idx_out", torch.int32, (B, T, H, W))
    _req(w_out, "w_out", torch.float32, (B, T, H, W))
    if dev_err is not None:
        _req(dev_err, "dev_err", torch.int32)
    rc = lib().sdm_address(s1.data_ptr(), s2.data_ptr(), B, T, H, sq, int(k), int(W), idx_out.data_ptr(),
                           w_out.data_ptr(), _ptr(dev_err), _stream(stream))
    _check("sdm_address", rc)
    return idx_out, w_out


def sdm_scan_workspace_size(B: int, T: int, H: int, W: int, R: int) -> int:
    return int(lib().sdm_scan_workspace_size(B, T, H, W, R))


def _scan_shapes(state, v, alpha, beta, idx_w, w_w, idx_r, w_r):
    _req(state, "state", torch.float32)
    if state.dim() != 4:
        raise ValueError("state must be [B,H,N,d_v]")
    B, H, N, dv = state.shape
    if v.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("v must be float32 or bfloat16")
    _req(v, "v", v.dtype)
    if v.dim() != 4 or v.shape[0] != B or v.shape[2] != H or v.shape[3] != dv:
        raise ValueError(f"v must be [B,T,H,d_v] = [{B},T,{H},{dv}]")
    T = v.shape[1]
    _req(alpha, "alpha", torch.float32, (B, T, H))
    _req(beta, "beta", torch.float32, (B, T, H))
    _req(idx_w, "idx_w", torch.int32)
    W = idx_w.shape[-1]
    _req(idx_w, "idx_w", torch.int32, (B, T, H, W))
    _req(w_w, "w_w", torch.float32, (B, T, H, W))
    _req(idx_r, "idx_r", torch.int32)
    R = idx_r.shape[-1]
    _req(idx_r, "idx_r", torch.int32, (B, T, H, R))
    _req(w_r, "w_r", torch.float32, (B, T, H, R))
    return B, T, H, N, dv, W, R


def sdm_scan_chunked(state, v, alpha, beta, idx_w, w_w, idx_r, w_r, resid_mode=SDM_RESID_SHARED, y=None,
                     workspace=None, dev_err=None, stream=None):
    """The sparse scan in chunked form (64-token chunks, the work inside a
    chunk in parallel); same arguments and result as sdm_scan, shared or
    additive write, W, R <= 16."""
    B, T, H, N, dv, W, R = _scan_shapes(state, v, alpha, beta, idx_w, w_w, idx_r, w_r)
    if y is None:
        y = torch.empty((B, T, H, dv), dtype=torch.float32, device=state.device)
    _req(y, "y", torch.float32, (B, T, H, dv))
    need = int(lib().sdm_scan_chunked_workspace_size(B, T, H, W, R))
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=state.device)
    _req(workspace, "workspace", torch.uint8)
    if dev_err is not None:
        _req(dev_err, "dev_err", torch.int32)
    vdt = SDM_DTYPE_BF16 if v.dtype == torch.bfloat16 else SDM_DTYPE_F32
    rc = lib().sdm_scan_chunked(state.data_ptr(), v.data_ptr(), vdt, alpha.data_ptr(), beta.data_ptr(),
                                idx_w.data_ptr(), w_w.data_ptr(), W, idx_r.data_ptr(), w_r.data_ptr(), R, B, T, H, N,
                                dv, int(resid_mode), y.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                _ptr(dev_err), _stream(stream))
    _check("sdm_scan_chunked", rc)
    return y


def sdm_scan_chunked_workspace_size(B: int, T: int, H: int, W: int, R: int) -> int:
    return int(lib().sdm_scan_chunked_workspace_size(B, T, H, W, R))


def sdm_scan_train(state, v, alpha, beta, idx_w, w_w, idx_r, w_r, resid_mode=SDM_RESID_SHARED, y=None, undo=None,
                   workspace=None, dev_err=None, stream=None):
    """sdm_scan that also returns the undo log fp32 [B,T,H,W,d_v] (the
    written rows before each token's decay) for sdm_scan_backward.
    Returns (y, undo)."""
    B, T, H, N, dv, W, R = _scan_shapes(state, v, alpha, beta, idx_w, w_w, idx_r, w_r)
    if y is None:
        y = torch.empty((B, T, H, dv), dtype=torch.float32, device=state.device)
    _req(y, "y", torch.float32, (B, T, H, dv))
    if undo is None:
        undo = torch.empty((B, T, H, W, dv), dtype=torch.float32, device=state.device)
    _req(undo, "undo", torch.float32, (B, T, H, W, dv))
    need = sdm_scan_workspace_size(B, T, H, W, R)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=state.device)
    _req(workspace, "workspace", torch.uint8)
    if dev_err is not None:
        _req(dev_err, "dev_err", torch.int32)
    vdt = SDM_DTYPE_BF16 if v.dtype == torch.bfloat16 else SDM_DTYPE_F32
    rc = lib().sdm_scan_train(state.data_ptr(), v.data_ptr(), vdt, alpha.data_ptr(), beta.data_ptr(),
                              idx_w.data_ptr(), w_w.data_ptr(), W, idx_r.data_ptr(), w_r.data_ptr(), R, B, T, H, N, dv,
                              int(resid_mode), y.data_ptr(), undo.data_ptr(), workspace.data_ptr(), workspace.numel(),
                              _ptr(dev_err), _stream(stream))
    _check("sdm_scan_train", rc)
    return y, undo


def sdm_address_backward(idx, w, dw, sqrtN: int, dev_err=None, stream=None):
    """Gradient of sdm_address's weights w.r.t. the score halves: idx int32,
    w and dw fp32 [B,T,H,W] -> (ds1, ds2) fp32 [B,T,H,sqrtN]."""
    _req(idx, "idx", torch.int32)
    B, T, H, W = idx.shape
    _req(w, "w", torch.float32, (B, T, H, W))
    _req(dw, "dw", torch.float32, (B, T, H, W))
    ds1 = torch.empty((B, T, H, sqrtN), dtype=torch.float32, device=idx.device)
    ds2 = torch.empty((B, T, H, sqrtN), dtype=torch.float32, device=idx.device)
    if dev_err is not None:
        _req(dev_err, "dev_err", torch.int32)
    rc = lib().sdm_address_backward(idx.data_ptr(), w.data_ptr(), dw.data_ptr(), B, T, H, int(sqrtN), W,
                                    ds1.data_ptr(), ds2.data_ptr(), _ptr(dev_err), _stream(stream))
    _check("sdm_address_backward", rc)
    return ds1, ds2


def sdm_scan_backward_workspace_size(B: int, T: int, H: int, W: int, R: int, d_v: int) -> int:
    return int(lib().sdm_scan_backward_workspace_size(B, T, H, W, R, d_v))


def sdm_scan_backward(state, dstate, v, alpha, beta, idx_w, w_w, idx_r, w_r, undo, dy, resid_mode=SDM_RESID_SHARED,
                      workspace=None, dev_err=None, stream=None):
    """Gradients of sdm_scan_train.  `state` holds M_T and becomes M_0;
    `dstate` holds dL/dM_T and becomes dL/dM_0 (both in place).  Returns
    (dv, dalpha, dbeta, dw_w, dw_r), fp32."""
    B, T, H, N, dv_, W, R = _scan_shapes(state, v, alpha, beta, idx_w, w_w, idx_r, w_r)
    _req(dstate, "dstate", torch.float32, (B, H, N, dv_))
    _req(undo, "undo", torch.float32, (B, T, H, W, dv_))
    _req(dy, "dy", torch.float32, (B, T, H, dv_))
    dev = state.device
    dv = torch.empty((B, T, H, dv_), dtype=torch.float32, device=dev)
    dalpha = torch.empty((B, T, H), dtype=torch.float32, device=dev)
    dbeta = torch.empty((B, T, H), dtype=torch.float32, device=dev)
    dw_w = torch.empty((B, T, H, W), dtype=torch.float32, device=dev)
    dw_r = torch.empty((B, T, H, R), dtype=torch.float32, device=dev)
    need = sdm_scan_backward_workspace_size(B, T, H, W, R, dv_)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
    _req(workspace, "workspace", torch.uint8)
    if dev_err is not None:
        _req(dev_err, "dev_err", torch.int32)
    vdt = SDM_DTYPE_BF16 if v.dtype == torch.bfloat16 else SDM_DTYPE_F32
    rc = lib().sdm_scan_backward(state.data_ptr(), dstate.data_ptr(), v.data_ptr(), vdt, alpha.data_ptr(),
                                 beta.data_ptr(), idx_w.data_ptr(), w_w.data_ptr(), W, idx_r.data_ptr(), w_r.data_ptr(),
                                 R, B, T, H, N, dv_, int(resid_mode), undo.data_ptr(), dy.data_ptr(), dv.data_ptr(),
                                 dalpha.data_ptr(), dbeta.data_ptr(), dw_w.data_ptr(), dw_r.data_ptr(),
                                 workspace.data_ptr(), workspace.numel(), _ptr(dev_err), _stream(stream))
    _check("sdm_scan_backward", rc)
    return dv, dalpha, dbeta, dw_w, dw_r


def sdm_scan(state, v, alpha, beta, idx_w, w_w, idx_r, w_r, resid_mode=SDM_RESID_SHARED, y=None, workspace=None,
             dev_err=None, stream=None):
    """Sparse delta-rule scan; updates `state` [B,H,N,d_v] in place and
    returns y fp32 [B,T,H,d_v].  v is fp32 or bf16 [B,T,H,d_v]."""
    _req(state, "state", torch.float32)
    if state.dim() != 4:
        raise ValueError("state must be [B,H,N,d_v]")
    B, H, N, dv = state.shape
    if v.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("v must be float32 or bfloat16")
    _req(v, "v", v.dtype)
    if v.dim() != 4 or v.shape[0] != B or v.shape[2] != H or v.shape[3] != dv:
        raise ValueError(f"v must be [B,T,H,d_v] = [{B},T,{H},{dv}]")
    T = v.shape[1]
    _req(alpha, "alpha", torch.float32, (B, T, H))
    _req(beta, "beta", torch.float32, (B, T, H))
    _req(idx_w, "idx_w", torch.int32)
    W = idx_w.shape[-1]
    _req(idx_w, "idx_w", torch.int32, (B, T, H, W))
    _req(w_w, "w_w", torch.float32, (B, T, H, W))
    _req(idx_r, "idx_r", torch.int32)
    R = idx_r.shape[-1]
    _req(idx_r, "idx_r", torch.int32, (B, T, H, R))
    _req(w_r, "w_r", torch.float32, (B, T, H, R))
    if y is None:
        y = torch.empty((B, T, H, dv), dtype=torch.float32, device=state.device)
    _req(y, "y", torch.float32, (B, T, H, dv))
    need = sdm_scan_workspace_size(B, T, H, W, R)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=state.device)
    _req(workspace, "workspace", torch.uint8)
    if dev_err is not None:
        _req(dev_err, "dev_err", torch.int32)
    vdt = SDM_DTYPE_BF16 if v.dtype == torch.bfloat16 else SDM_DTYPE_F32
    rc = lib().sdm_scan(state.data_ptr(), v.data_ptr(), vdt, alpha.data_ptr(), beta.data_ptr(), idx_w.data_ptr(),
                        w_w.data_ptr(), W, idx_r.data_ptr(), w_r.data_ptr(), R, B, T, H, N, dv, int(resid_mode),
                        y.data_ptr(), workspace.data_ptr(), workspace.numel(), _ptr(dev_err), _stream(stream))
    _check("sdm_scan", rc)
    return y


def sdm_forward_host_workspace_size(B, T, H, sqrtN, d_v, W, R, v_bf16: bool, chunk_T: int) -> int:
    return int(lib().sdm_forward_host_workspace_size(B, T, H, sqrtN, d_v, W, R,
                                                     SDM_DTYPE_BF16 if v_bf16 else SDM_DTYPE_F32, chunk_T))


def _req_host(t: torch.Tensor, name: str, dtype, shape=None):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise TypeError(f"{name} must be a CPU (preferably pinned) tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def sdm_forward_host(s1w, s2w, s1r, s2r, v, alpha, beta, k: int, W: int, R: int, state, y=None,
                     resid_mode=SDM_RESID_SHARED, chunk_T: int = 512, workspace=None, dev_err=None, stream=None):
    """Whole sparse step from host tensors (pinned for overlap): addressing of
    both score-half pairs and the scan, pipelined over chunks of chunk_T
    tokens.  `state` is the CUDA table [B,H,N,d_v]; returns the host y
    [B,T,H,d_v], valid once `stream` is synchronised."""
    _req_host(s1w, "s1w", torch.float32)
    if s1w.dim() != 4:
        raise ValueError("s1w must be [B,T,H,sqrtN]")
    B, T, H, sq = s1w.shape
    for n_, t_ in (("s2w", s2w), ("s1r", s1r), ("s2r", s2r)):
        _req_host(t_, n_, torch.float32, (B, T, H, sq))
    _req(state, "state", torch.float32, (B, H, sq * sq, state.shape[-1]))
    dv = state.shape[-1]
    if v.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("v must be float32 or bfloat16")
    _req_host(v, "v", v.dtype, (B, T, H, dv))
    _req_host(alpha, "alpha", torch.float32, (B, T, H))
    _req_host(beta, "beta", torch.float32, (B, T, H))
    if y is None:
        y = torch.empty((B, T, H, dv), dtype=torch.float32).pin_memory()
    _req_host(y, "y", torch.float32, (B, T, H, dv))
    bf = v.dtype == torch.bfloat16
    need = sdm_forward_host_workspace_size(B, T, H, sq, dv, W, R, bf, chunk_T)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=state.device)
    _req(workspace, "workspace", torch.uint8)
    if dev_err is not None:
        _req(dev_err, "dev_err", torch.int32)
    rc = lib().sdm_forward_host(s1w.data_ptr(), s2w.data_ptr(), s1r.data_ptr(), s2r.data_ptr(), v.data_ptr(),
                                SDM_DTYPE_BF16 if bf else SDM_DTYPE_F32, alpha.data_ptr(), beta.data_ptr(), B, T, H,
                                sq, int(k), int(W), int(R), dv, int(resid_mode), state.data_ptr(), y.data_ptr(),
                                int(chunk_T), workspace.data_ptr(), workspace.numel(), _ptr(dev_err), _stream(stream))
    _check("sdm_forward_host", rc)
    return y


def sdm_scan_noalloc(state, v, alpha, beta, idx_w, w_w, idx_r, w_r, resid_mode=SDM_RESID_SHARED, y=None,
                     dev_err=None, stream=None):
    """sdm_scan without a workspace argument, for callers that cannot
    allocate device memory while running.  The library keeps the scratch in
    one fixed 32 MiB device array per GPU, shared by all calls: B*T*H may be
    at most 99,864 when W, R <= 16 and 25,890 otherwise (larger calls raise,
    SDM_ERR_SHAPE); calls that overlap on the GPU race on the array."""
    _req(state, "state", torch.float32)
    if state.dim() != 4:
        raise ValueError("state must be [B,H,N,d_v]")
    B, H, N, dv = state.shape
    if v.dtype not in (torch.float32, torch.bfloat16):
        raise TypeError("v must be float32 or bfloat16")
    _req(v, "v", v.dtype)
    T = v.shape[1]
    _req(v, "v", v.dtype, (B, T, H, dv))
    _req(alpha, "alpha", torch.float32, (B, T, H))
    _req(beta, "beta", torch.float32, (B, T, H))
    W, R = idx_w.shape[-1], idx_r.shape[-1]
    _req(idx_w, "idx_w", torch.int32, (B, T, H, W))
    _req(w_w, "w_w", torch.float32, (B, T, H, W))
    _req(idx_r, "idx_r", torch.int32, (B, T, H, R))
    _req(w_r, "w_r", torch.float32, (B, T, H, R))
    if y is None:
        y = torch.empty((B, T, H, dv), dtype=torch.float32, device=state.device)
    _req(y, "y", torch.float32, (B, T, H, dv))
    if dev_err is not None:
        _req(dev_err, "dev_err", torch.int32)
    vdt = SDM_DTYPE_BF16 if v.dtype == torch.bfloat16 else SDM_DTYPE_F32
    rc = lib().sdm_scan_noalloc(state.data_ptr(), v.data_ptr(), vdt, alpha.data_ptr(), beta.data_ptr(),
                                idx_w.data_ptr(), w_w.data_ptr(), W, idx_r.data_ptr(), w_r.data_ptr(), R, B, T, H, N,
                                dv, int(resid_mode), y.data_ptr(), _ptr(dev_err), _stream(stream))
    _check("sdm_scan_noalloc", rc)
    return y


def gdn_scan_workspace_size(B: int, T: int, H: int, dk: int, dv: int, per_channel: bool) -> int:
    return int(lib().gdn_scan_workspace_size(B, T, H, dk, dv, int(bool(per_channel))))


def gdn_scan(state, q, k, v, alpha, beta, per_channel: bool, y=None, workspace=None, dev_err=None, stream=None):
    """Dense GDN / KDA scan; updates `state` [B,H,dk,dv] in place and returns
    y fp32 [B,T,H,dv].  q, k bf16 [B,T,H,dk]; v bf16 [B,T,H,dv]; alpha fp32
    [B,T,H] (GDN) or [B,T,H,dk] (KDA); beta fp32 [B,T,H]."""
    _req(state, "state", torch.float32)
    if state.dim() != 4:
        raise ValueError("state must be [B,H,dk,dv]")
    B, H, dk, dv = state.shape
    _req(q, "q", torch.bfloat16)
    T = q.shape[1]
    _req(q, "q", torch.bfloat16, (B, T, H, dk))
    _req(k, "k", torch.bfloat16, (B, T, H, dk))
    _req(v, "v", torch.bfloat16, (B, T, H, dv))
    _req(alpha, "alpha", torch.float32, (B, T, H, dk) if per_channel else (B, T, H))
    _req(beta, "beta", torch.float32, (B, T, H))
    if y is None:
        y = torch.empty((B, T, H, dv), dtype=torch.float32, device=state.device)
    _req(y, "y", torch.float32, (B, T, H, dv))
    need = gdn_scan_workspace_size(B, T, H, dk, dv, per_channel)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=state.device)
    if workspace is not None:
        _req(workspace, "workspace", torch.uint8)
    if dev_err is not None:
        _req(dev_err, "dev_err", torch.int32)
    rc = lib().gdn_scan(state.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), alpha.data_ptr(),
                        int(bool(per_channel)), beta.data_ptr(), B, T, H, dk, dv, y.data_ptr(), _ptr(workspace),
                        0 if workspace is None else workspace.numel(), _ptr(dev_err), _stream(stream))
    _check("gdn_scan", rc)
    return y


def gdn2_scan_workspace_size(B: int, T: int, H: int, dk: int, dv: int) -> int:
    return int(lib().gdn2_scan_workspace_size(B, T, H, dk, dv))


def gdn2_scan(state, q, k, v, alpha, b_erase, w_write, y=None, workspace=None, dev_err=None, stream=None):
    """GDN2 scan; updates `state` [B,H,dk,dv] in place and returns y fp32
    [B,T,H,dv].  q, k bf16 [B,T,H,dk]; v bf16 [B,T,H,dv]; alpha and b_erase
    fp32 [B,T,H,dk]; w_write fp32 [B,T,H,dv]."""
    _req(state, "state", torch.float32)
    if state.dim() != 4:
        raise ValueError("state must be [B,H,dk,dv]")
    B, H, dk, dv = state.shape
    _req(q, "q", torch.bfloat16)
    T = q.shape[1]
    _req(q, "q", torch.bfloat16, (B, T, H, dk))
    _req(k, "k", torch.bfloat16, (B, T, H, dk))
    _req(v, "v", torch.bfloat16, (B, T, H, dv))
    _req(alpha, "alpha", torch.float32, (B, T, H, dk))
    _req(b_erase, "b_erase", torch.float32, (B, T, H, dk))
    _req(w_write, "w_write", torch.float32, (B, T, H, dv))
    if y is None:
        y = torch.empty((B, T, H, dv), dtype=torch.float32, device=state.device)
    _req(y, "y", torch.float32, (B, T, H, dv))
    need = gdn2_scan_workspace_size(B, T, H, dk, dv)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=state.device)
    if workspace is not None:
        _req(workspace, "workspace", torch.uint8)
    if dev_err is not None:
        _req(dev_err, "dev_err", torch.int32)
    rc = lib().gdn2_scan(state.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), alpha.data_ptr(),
                         b_erase.data_ptr(), w_write.data_ptr(), B, T, H, dk, dv, y.data_ptr(), _ptr(workspace),
                         0 if workspace is None else workspace.numel(), _ptr(dev_err), _stream(stream))
    _check("gdn2_scan", rc)
    return y


def sse_scan_workspace_size(B: int, T: int, H: int, N: int, topk: int, c: int = 128, d: int = 128,
                            write_mode: int = 0) -> int:
    return int(lib().sse_scan_workspace_size(B, T, H, N, topk, c, d, write_mode))


def sse_scan(state, route_logits, topk: int, k_logits, q, v, alpha, y=None, sel_out=None, workspace=None,
             dev_err=None, stream=None, write_mode: int = 0):
    """Sparse State Expansion scan; updates `state` [B,H,N+1,c,d] in place and
    returns y fp32 [B,T,H,d] (and fills sel_out int32 [B,T,H,topk] if given).
    write_mode: SSE_WRITE_ADDITIVE (0) or SSE_WRITE_DELTA (1)."""
    _req(state, "state", torch.float32)
    if state.dim() != 5:
        raise ValueError("state must be [B,H,N+1,c,d]")
    B, H, Np1, c, d = state.shape
    N = Np1 - 1
    _req(route_logits, "route_logits", torch.float32)
    T = route_logits.shape[1]
    _req(route_logits, "route_logits", torch.float32, (B, T, H, N))
    _req(k_logits, "k_logits", torch.float32, (B, T, H, c))
    _req(q, "q", torch.bfloat16, (B, T, H, c))
    _req(v, "v", torch.bfloat16, (B, T, H, d))
    _req(alpha, "alpha", torch.float32, (B, T, H, c))
    if y is None:
        y = torch.empty((B, T, H, d), dtype=torch.float32, device=state.device)
    _req(y, "y", torch.float32, (B, T, H, d))
    if sel_out is not None:
        _req(sel_out, "sel_out", torch.int32, (B, T, H, topk))
    if dev_err is not None:
        _req(dev_err, "dev_err", torch.int32)
    if workspace is None:
        workspace = torch.empty(max(sse_scan_workspace_size(B, T, H, N, topk, c, d, write_mode), 1), dtype=torch.uint8,
                                device=state.device)
    _req(workspace, "workspace", torch.uint8)
    rc = lib().sse_scan(state.data_ptr(), route_logits.data_ptr(), int(topk), k_logits.data_ptr(), q.data_ptr(),
                        v.data_ptr(), alpha.data_ptr(), int(write_mode), B, T, H, N, c, d, y.data_ptr(), _ptr(sel_out),
                        workspace.data_ptr(), workspace.numel(), _ptr(dev_err), _stream(stream))
    _check("sse_scan", rc)
    return y

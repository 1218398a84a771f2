"""fp64 CPU oracle for the delta-rule memory scans (numpy front end).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg (and its ``--impl reference`` arm) may import
this package.  The product library (``delta_rule_memory_gb300``) never imports
it and shares no code with it; the only module both sides use is ``synth``,
which draws the seeded inputs.

The arithmetic lives in ``oracle.c`` (plain C, fp64, built with gcc without
fast-math or FMA contraction).  This file only compiles it, widens inputs to
fp64 and marshals numpy arrays through ctypes.

Pins: every function here is checked by ``tests/test_oracle_pins.py`` against
worked examples printed on the pages (``tests/golden/``), closed forms,
special-case reductions and brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

RESID_SHARED, RESID_PERSLOT, RESID_ADDITIVE = 0, 1, 2
SSE_WRITE_ADDITIVE, SSE_WRITE_DELTA = 0, 1


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -O2, no fast-math,
    no FP contraction).  Returns the library path."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_address.argtypes = [P, P, I, I, I, I, I, I, P, P]
            lib.oracle_address_backward.argtypes = [P, P, P, ctypes.c_long, I, I, P, P]
            lib.oracle_sdm_scan.argtypes = [P, P, P, P, P, P, I, P, P, I, I, I, I, I, I, I, P, P]
            lib.oracle_sdm_scan_backward.argtypes = [P, P, P, P, P, P, P, I, P, P, I, I, I, I, I, I, I, P, P, P, P, P,
                                                     P, P]
            lib.oracle_gdn_scan.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, P]
            lib.oracle_gdn2_scan.argtypes = [P, P, P, P, P, P, P, I, I, I, I, I, P]
            lib.oracle_sse_scan.argtypes = [P, P, I, P, P, P, P, I, I, I, I, I, I, P, P, I]
            lib.oracle_widen_bf16.argtypes = [P, P, ctypes.c_long]
            for f in (lib.oracle_address, lib.oracle_address_backward, lib.oracle_sdm_scan, lib.oracle_sdm_scan_backward, lib.oracle_gdn_scan,
                      lib.oracle_gdn2_scan, lib.oracle_sse_scan):
                f.restype = I
            _lib = lib
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def widen(x: np.ndarray, is_bf16: bool | None = None) -> np.ndarray:
    """Exact fp64 copy of an fp32 array or of a uint16 array of bf16 bits."""
    if is_bf16 or (is_bf16 is None and x.dtype == np.uint16):
        src = _c(x, np.uint16)
        out = np.empty(src.shape, np.float64)
        _load().oracle_widen_bf16(_p(src), _p(out), src.size)
        return out
    return np.asarray(x, dtype=np.float64)


def address(s1: np.ndarray, s2: np.ndarray, k: int, W: int):
    """Product-key addressing.  s1, s2: fp32 [B,T,H,sqrtN].
    Returns (idx int32 [B,T,H,W] in rank order, w fp64 [B,T,H,W])."""
    s1 = _c(s1, np.float32)
    s2 = _c(s2, np.float32)
    assert s1.shape == s2.shape and s1.ndim == 4
    B, T, H, sq = s1.shape
    idx = np.empty((B, T, H, W), np.int32)
    w = np.empty((B, T, H, W), np.float64)
    rc = _load().oracle_address(_p(s1), _p(s2), B, T, H, sq, k, W, _p(idx), _p(w))
    if rc != 0:
        raise ValueError(f"oracle_address: bad sizes (rc={rc})")
    return idx, w


def address_backward(idx, w, dw, sqrtN: int):
    """Gradient of the addressing weights w.r.t. the score halves: idx int32,
    w and dw [..., W] -> (ds1, ds2) fp64 [..., sqrtN]."""
    ix = _c(idx, np.int32)
    ww, dd = _c(w, np.float64), _c(dw, np.float64)
    W = ix.shape[-1]
    rows = ix.size // W
    lead = ix.shape[:-1]
    ds1 = np.zeros(lead + (sqrtN,))
    ds2 = np.zeros(lead + (sqrtN,))
    rc = _load().oracle_address_backward(_p(ix), _p(ww), _p(dd), rows, sqrtN, W, _p(ds1), _p(ds2))
    if rc != 0:
        raise ValueError(f"oracle_address_backward failed (rc={rc})")
    return ds1, ds2


def sdm_scan(state, v, alpha, beta, idx_w, w_w, idx_r, w_r, mode=RESID_SHARED, keep_undo=False):
    """Sparse delta-rule scan.  state [B,H,N,dv] (copied, fp64); v [B,T,H,dv]
    (fp32, fp64 or bf16 bits); alpha, beta [B,T,H]; idx_*/w_* [B,T,H,W|R].
    Returns (final state fp64, y fp64 [B,T,H,dv]), plus the undo log
    [B,T,H,W,dv] (rows of I^w before each token's decay) if keep_undo."""
    M = np.array(state, dtype=np.float64, copy=True, order="C")
    B, H, N, dv = M.shape
    vv = _c(widen(v), np.float64)
    T = vv.shape[1]
    iw = _c(idx_w, np.int32)
    ir = _c(idx_r, np.int32)
    W, R = iw.shape[-1], ir.shape[-1]
    ww = _c(w_w, np.float64)
    wr = _c(w_r, np.float64)
    a = _c(alpha, np.float64)
    b = _c(beta, np.float64)
    assert vv.shape == (B, T, H, dv) and iw.shape == (B, T, H, W) and ir.shape == (B, T, H, R)
    assert a.shape == (B, T, H) and b.shape == (B, T, H)
    y = np.zeros((B, T, H, dv), np.float64)
    undo = np.zeros((B, T, H, W, dv), np.float64) if keep_undo else None
    rc = _load().oracle_sdm_scan(_p(M), _p(vv), _p(a), _p(b), _p(iw), _p(ww), W, _p(ir), _p(wr), R,
                                 B, T, H, N, dv, int(mode), _p(y), _p(undo) if keep_undo else None)
    if rc != 0:
        raise ValueError(f"oracle_sdm_scan failed (rc={rc})")
    return (M, y, undo) if keep_undo else (M, y)


def sdm_scan_backward(state_T, dstate_T, v, alpha, beta, idx_w, w_w, idx_r, w_r, mode, undo, dy):
    """Gradients of sdm_scan by undoing its writes.  state_T: the forward's
    final table; dstate_T: dL/dM_T; undo: the forward's log; dy: dL/dy.
    Returns (M_0, dL/dM_0, dv, dalpha, dbeta, dw_w, dw_r), all fp64."""
    M = np.array(state_T, dtype=np.float64, copy=True, order="C")
    dM = np.array(dstate_T, dtype=np.float64, copy=True, order="C")
    B, H, N, dv = M.shape
    vv = _c(widen(v), np.float64)
    T = vv.shape[1]
    iw, ir = _c(idx_w, np.int32), _c(idx_r, np.int32)
    W, R = iw.shape[-1], ir.shape[-1]
    ww, wr, a, b = (_c(x, np.float64) for x in (w_w, w_r, alpha, beta))
    un, g = _c(undo, np.float64), _c(dy, np.float64)
    assert dM.shape == M.shape and un.shape == (B, T, H, W, dv) and g.shape == (B, T, H, dv)
    dvo = np.zeros((B, T, H, dv))
    da, db = np.zeros((B, T, H)), np.zeros((B, T, H))
    dww, dwr = np.zeros((B, T, H, W)), np.zeros((B, T, H, R))
    rc = _load().oracle_sdm_scan_backward(_p(M), _p(dM), _p(vv), _p(a), _p(b), _p(iw), _p(ww), W, _p(ir), _p(wr), R,
                                          B, T, H, N, dv, int(mode), _p(un), _p(g), _p(dvo), _p(da), _p(db),
                                          _p(dww), _p(dwr))
    if rc != 0:
        raise ValueError(f"oracle_sdm_scan_backward failed (rc={rc})")
    return M, dM, dvo, da, db, dww, dwr


def gdn_scan(state, q, k, v, alpha, beta, per_channel: bool):
    """Dense GDN (per_channel False, alpha [B,T,H]) or KDA (alpha [B,T,H,dk]).
    state [B,H,dk,dv]; q, k [B,T,H,dk]; v [B,T,H,dv] (fp32/fp64/bf16 bits).
    Returns (final state, y [B,T,H,dv]) in fp64."""
    S = np.array(state, dtype=np.float64, copy=True, order="C")
    B, H, dk, dv = S.shape
    qq, kk, vv = (_c(widen(x), np.float64) for x in (q, k, v))
    T = qq.shape[1]
    a = _c(alpha, np.float64)
    b = _c(beta, np.float64)
    assert qq.shape == (B, T, H, dk) and kk.shape == (B, T, H, dk) and vv.shape == (B, T, H, dv)
    assert a.shape == ((B, T, H, dk) if per_channel else (B, T, H)) and b.shape == (B, T, H)
    y = np.zeros((B, T, H, dv), np.float64)
    rc = _load().oracle_gdn_scan(_p(S), _p(qq), _p(kk), _p(vv), _p(a), int(bool(per_channel)), _p(b),
                                 B, T, H, dk, dv, _p(y))
    if rc != 0:
        raise ValueError(f"oracle_gdn_scan failed (rc={rc})")
    return S, y


def gdn2_scan(state, q, k, v, alpha, b_erase, w_write):
    """GDN2: per-key-channel decay alpha [B,T,H,dk], erase gate b_erase
    [B,T,H,dk] and write gate w_write [B,T,H,dv].  state [B,H,dk,dv];
    q, k [B,T,H,dk]; v [B,T,H,dv].  Returns (final state, y) in fp64."""
    S = np.array(state, dtype=np.float64, copy=True, order="C")
    B, H, dk, dv = S.shape
    qq, kk, vv = (_c(widen(x), np.float64) for x in (q, k, v))
    T = qq.shape[1]
    a, be, wr = (_c(x, np.float64) for x in (alpha, b_erase, w_write))
    assert qq.shape == (B, T, H, dk) and kk.shape == (B, T, H, dk) and vv.shape == (B, T, H, dv)
    assert a.shape == (B, T, H, dk) and be.shape == (B, T, H, dk) and wr.shape == (B, T, H, dv)
    y = np.zeros((B, T, H, dv), np.float64)
    rc = _load().oracle_gdn2_scan(_p(S), _p(qq), _p(kk), _p(vv), _p(a), _p(be), _p(wr), B, T, H, dk, dv, _p(y))
    if rc != 0:
        raise ValueError(f"oracle_gdn2_scan failed (rc={rc})")
    return S, y


def sse_scan(state, route, topk, klog, q, v, alpha, mode=0):
    """SSE scan.  state [B,H,N+1,c,d]; route fp32 [B,T,H,N]; klog fp32
    [B,T,H,c]; q [B,T,H,c]; v [B,T,H,d]; alpha [B,T,H,c]; mode
    SSE_WRITE_ADDITIVE (0) or SSE_WRITE_DELTA (1).
    Returns (final state, y [B,T,H,d], sel int32 [B,T,H,topk])."""
    S = np.array(state, dtype=np.float64, copy=True, order="C")
    B, H, Np1, c, d = S.shape
    N = Np1 - 1
    rt = _c(route, np.float32)
    kl = _c(klog, np.float32)
    qq, vv = (_c(widen(x), np.float64) for x in (q, v))
    T = rt.shape[1]
    a = _c(alpha, np.float64)
    assert rt.shape == (B, T, H, N) and kl.shape == (B, T, H, c) and qq.shape == (B, T, H, c)
    assert vv.shape == (B, T, H, d) and a.shape == (B, T, H, c)
    y = np.zeros((B, T, H, d), np.float64)
    sel = np.zeros((B, T, H, topk), np.int32)
    rc = _load().oracle_sse_scan(_p(S), _p(rt), int(topk), _p(kl), _p(qq), _p(vv), _p(a), B, T, H, N, c, d,
                                 _p(y), _p(sel), int(mode))
    if rc != 0:
        raise ValueError(f"oracle_sse_scan failed (rc={rc})")
    return S, y, sel


def sdm_forward(inp: dict, k: int, W: int, R: int, state=None, mode=RESID_SHARED):
    """Full SDM path on synth inputs: write addressing, read addressing, scan.
    Returns dict with idx_w, w_w, idx_r, w_r, state, y."""
    idx_w, w_w = address(inp["s1w"], inp["s2w"], k, W)
    idx_r, w_r = address(inp["s1r"], inp["s2r"], k, R)
    B, T, H, _ = inp["s1w"].shape
    dv = inp["v"].shape[-1]
    N = inp["s1w"].shape[-1] ** 2
    if state is None:
        state = np.zeros((B, H, N, dv), np.float64)
    M, y = sdm_scan(state, inp["v"], inp["alpha"], inp["beta"], idx_w, w_w, idx_r, w_r, mode)
    return {"idx_w": idx_w, "w_w": w_w, "idx_r": idx_r, "w_r": w_r, "state": M, "y": y}

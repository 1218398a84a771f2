"""sdm_scan_noalloc: the scan for callers that cannot allocate device memory
(for example a host that serves every device buffer from its own pool and
forbids raw cudaMalloc while running).  It keeps its scratch in a fixed
device array inside the library instead of a caller workspace.

Checked through the C ABI against sdm_scan (the entry point that takes a
workspace) on the same inputs, for two calls in a row that continue the same
table, within the parity tolerance the other tests use.  This file is
collected last on purpose; it must pass on its own in a fresh process and
after every other test."""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from helpers import assert_state_close, assert_y_close, dev, host, need_gpu

pytestmark = pytest.mark.gpu


def _call(sdm, fn, state, v, inp_d, iw, ww, ir, wr, y, err, ws=None):
    import torch
    L = sdm.lib()
    B, H, N, dv = state.shape
    T = v.shape[1]
    W, R = iw.shape[-1], ir.shape[-1]
    common = (state.data_ptr(), v.data_ptr(), 1, inp_d["alpha"].data_ptr(), inp_d["beta"].data_ptr(), iw.data_ptr(),
              ww.data_ptr(), W, ir.data_ptr(), wr.data_ptr(), R, B, T, H, N, dv, 0, y.data_ptr())
    stream = torch.cuda.current_stream().cuda_stream
    if fn == "sdm_scan":
        rc = L.sdm_scan(*common, ws.data_ptr(), ws.numel(), err.data_ptr(), stream)
    else:
        rc = L.sdm_scan_noalloc(*common, err.data_ptr(), stream)
    assert rc == 0, L.sdm_last_error()


def test_noalloc_matches_workspace_scan_on_two_calls_in_a_row():
    sdm = need_gpu()
    import torch
    sh = synth.SDM_14B_LAYER.with_(B=2, T=192)
    inp = synth.sdm_inputs(sh, seed=31)
    iw, ww = oracle.address(inp["s1w"], inp["s2w"], sh.k, sh.W)
    ir, wr = oracle.address(inp["s1r"], inp["s2r"], sh.k, sh.R)
    iw, ww, ir, wr = dev(iw), dev(ww.astype(np.float32)), dev(ir), dev(wr.astype(np.float32))
    inp_d = {"alpha": dev(inp["alpha"]), "beta": dev(inp["beta"])}
    v = dev(inp["v"])
    M0 = synth.random_state((sh.B, sh.H, sh.N, sh.d_v), seed=32, scale=0.1)
    st_ref, st_new = dev(M0), dev(M0)
    y_ref = torch.empty((sh.B, sh.T, sh.H, sh.d_v), device="cuda")
    y_new = torch.empty_like(y_ref)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(sdm.sdm_scan_workspace_size(sh.B, sh.T, sh.H, sh.W, sh.R), dtype=torch.uint8, device="cuda")
    for _ in range(2):   # the second call continues both tables
        y_new.fill_(float("nan"))
        _call(sdm, "sdm_scan", st_ref, v, inp_d, iw, ww, ir, wr, y_ref, err, ws)
        _call(sdm, "sdm_scan_noalloc", st_new, v, inp_d, iw, ww, ir, wr, y_new, err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert_y_close(host(y_new), host(y_ref))
        assert_state_close(host(st_new), host(st_ref))


def test_noalloc_rejects_sizes_beyond_its_array():
    sdm = need_gpu()
    L = sdm.lib()
    # 64*8192*2 token-head records of 336 bytes exceed the 32 MiB array: refused before any launch
    rc = L.sdm_scan_noalloc(1 << 20, 1 << 20, 1, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 16, 1 << 20, 1 << 20, 16,
                            64, 8192, 2, 57600, 960, 0, 1 << 20, None, None)
    assert rc == sdm.SDM_ERR_SHAPE
    assert b"static" in L.sdm_last_error()

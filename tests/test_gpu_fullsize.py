"""GPU parity at the configured sizes of the state-scaling sweep and of the
training path, in the launch configuration the benchmark times, against the
fp64 oracle on sampled (batch, head) sequences.

* Sweep (Sparse Delta Memory deck, "Head count controls a cubic state
  expansion", Eq. 6): d = 1920, H in {2, 4, 8} (N = 57,600 / 14,400 / 3,600,
  d_v = 960 / 480 / 240), B = 8, T = 8192, W = R = 16, in both the shared
  (Fig. 2) and the per-slot (printed Eq. 4) residual modes.  The GPU runs the
  whole workload; the oracle runs two sequences on 48 value columns (value
  columns evolve independently because the addresses do not depend on the
  table).
* Training path (same deck, "Backup: undoing writes avoids repeated
  full-table snapshots", App. A.3): the 1.4B layer (B = 8, T = 4096, H = 2,
  N = 57,600, d_v = 960) through sdm_scan_train, sdm_scan_backward and both
  sdm_address_backward calls.  The oracle runs two whole sequences (every
  column, since the gate and weight gradients sum over columns); their
  initial table and dL/dM_T are random, every other sequence's are zero (the
  sequences are independent).
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_state_close, assert_y_close, dev, host, need_gpu

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

MODES = [(0, oracle.RESID_SHARED), (1, oracle.RESID_PERSLOT)]


@pytest.mark.parametrize("H", [2, 4, 8])
@pytest.mark.parametrize("gmode,omode", MODES, ids=["shared", "perslot"])
def test_sweep_full_size_sampled(H, gmode, omode):
    sdm = need_gpu()
    import torch
    sh = synth.sdm_sweep_shape(H)
    assert (sh.B, sh.T, sh.N, sh.d_v) == (8, 8192, (1920 // (4 * H)) ** 2, 1920 // H)
    inp = synth.sdm_inputs(sh, seed=100 + H)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = {k_: dev(inp[k_]) for k_ in ("s1w", "s2w", "s1r", "s2r")}
    iw, ww = sdm.sdm_address(s["s1w"], s["s2w"], sh.k, sh.W, dev_err=err)
    ir, wr = sdm.sdm_address(s["s1r"], s["s2r"], sh.k, sh.R, dev_err=err)
    del s
    state = torch.zeros((sh.B, sh.H, sh.N, sh.d_v), dtype=torch.float32, device="cuda")
    y = sdm.sdm_scan(state, dev(inp["v"]), dev(inp["alpha"]), dev(inp["beta"]), iw, ww, ir, wr, resid_mode=gmode,
                     dev_err=err)
    torch.cuda.synchronize()
    assert int(host(err)[0]) == 0
    cols = np.r_[0:16, sh.d_v // 2 - 8:sh.d_v // 2 + 8, sh.d_v - 16:sh.d_v]
    for (b, h) in [(0, 0), (sh.B - 1, H - 1)]:
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        ridx_w, rw_w = oracle.address(inp["s1w"][sl], inp["s2w"][sl], sh.k, sh.W)
        ridx_r, rw_r = oracle.address(inp["s1r"][sl], inp["s2r"][sl], sh.k, sh.R)
        np.testing.assert_array_equal(host(iw[sl]), ridx_w)
        np.testing.assert_array_equal(host(ir[sl]), ridx_r)
        M0 = np.zeros((1, 1, sh.N, len(cols)))
        Mr, yr = oracle.sdm_scan(M0, inp["v"][sl][..., cols], inp["alpha"][sl], inp["beta"][sl], ridx_w, rw_w,
                                 ridx_r, rw_r, omode)
        assert_y_close(host(y[sl])[..., cols], yr, what=f"y[b={b},h={h}]")
        assert_state_close(host(state[b:b + 1, h:h + 1])[..., cols], Mr, what=f"state[b={b},h={h}]")


@pytest.mark.parametrize("mode", [oracle.RESID_SHARED, oracle.RESID_PERSLOT, oracle.RESID_ADDITIVE],
                         ids=["shared", "perslot", "additive"])
def test_train_14b_layer_full_size_sampled(mode):
    sdm = need_gpu()
    import torch
    sh = synth.SDM_14B_LAYER
    inp = synth.sdm_inputs(sh, seed=110)
    sampled = [(0, 0), (sh.B - 1, sh.H - 1)]
    # nonzero initial table and final-table gradient on the sampled sequences only
    M0 = torch.zeros((sh.B, sh.H, sh.N, sh.d_v), dtype=torch.float32, device="cuda")
    dMT = torch.zeros_like(M0)
    M0_s, dMT_s = {}, {}
    for i, (b, h) in enumerate(sampled):
        M0_s[b, h] = synth.random_state((1, 1, sh.N, sh.d_v), seed=111 + i, scale=0.3)
        dMT_s[b, h] = synth.random_state((1, 1, sh.N, sh.d_v), seed=113 + i, scale=0.5)
        M0[b, h] = dev(M0_s[b, h][0, 0])
        dMT[b, h] = dev(dMT_s[b, h][0, 0])
    dy = synth.random_state((sh.B, sh.T, sh.H, sh.d_v), seed=115)

    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = {k_: dev(inp[k_]) for k_ in ("s1w", "s2w", "s1r", "s2r")}
    iw, ww = sdm.sdm_address(s["s1w"], s["s2w"], sh.k, sh.W, dev_err=err)
    ir, wr = sdm.sdm_address(s["s1r"], s["s2r"], sh.k, sh.R, dev_err=err)
    del s
    args = (dev(inp["v"]), dev(inp["alpha"]), dev(inp["beta"]), iw, ww, ir, wr)
    y, undo = sdm.sdm_scan_train(M0, *args, resid_mode=mode, dev_err=err)
    y_h = {bh: host(y[bh[0]:bh[0] + 1, :, bh[1]:bh[1] + 1]) for bh in sampled}
    MT_h = {bh: host(M0[bh[0]:bh[0] + 1, bh[1]:bh[1] + 1]) for bh in sampled}
    del y
    dv, da, db, dww, dwr = sdm.sdm_scan_backward(M0, dMT, *args, undo, dev(dy), resid_mode=mode, dev_err=err)
    del undo
    ds1w, ds2w = sdm.sdm_address_backward(iw, ww, dww, sh.sqrtN, dev_err=err)
    ds1r, ds2r = sdm.sdm_address_backward(ir, wr, dwr, sh.sqrtN, dev_err=err)
    torch.cuda.synchronize()
    assert int(host(err)[0]) == 0

    for (b, h) in sampled:
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        ridx_w, rw_w = oracle.address(inp["s1w"][sl], inp["s2w"][sl], sh.k, sh.W)
        ridx_r, rw_r = oracle.address(inp["s1r"][sl], inp["s2r"][sl], sh.k, sh.R)
        np.testing.assert_array_equal(host(iw[sl]), ridx_w)
        np.testing.assert_array_equal(host(ir[sl]), ridx_r)
        sel = (ridx_w, rw_w, ridx_r, rw_r)
        what = f"[b={b},h={h}]"
        MT, yr, undo_r = oracle.sdm_scan(M0_s[b, h], inp["v"][sl], inp["alpha"][sl], inp["beta"][sl], *sel, mode,
                                         keep_undo=True)
        assert_y_close(y_h[b, h], yr, what="y" + what)
        assert_state_close(MT_h[b, h], MT, what="M_T" + what)
        M0r, dM0r, dvr, dar, dbr, dwwr, dwrr = oracle.sdm_scan_backward(
            MT, dMT_s[b, h], inp["v"][sl], inp["alpha"][sl], inp["beta"][sl], *sel, mode, undo_r, dy[sl])
        del MT, undo_r
        # every write undone: the table is the initial one again, bit for bit
        np.testing.assert_array_equal(host(M0[b, h]), M0_s[b, h][0, 0])
        assert_state_close(host(dMT[b:b + 1, h:h + 1]), dM0r, what="dL/dM_0" + what)
        assert_y_close(host(dv[sl]), dvr, what="dL/dv" + what)
        assert_y_close(host(da[sl]), dar, what="dL/dalpha" + what)
        assert_y_close(host(db[sl]), dbr, what="dL/dbeta" + what)
        assert_y_close(host(dww[sl]), dwwr, what="dL/dw_w" + what)
        assert_y_close(host(dwr[sl]), dwrr, what="dL/dw_r" + what)
        # the score gradients of both addressing calls, end to end: the oracle
        # chain (its own weights and weight gradients) against the GPU chain
        r1, r2 = oracle.address_backward(ridx_w, rw_w, dwwr, sh.sqrtN)
        assert_y_close(host(ds1w[sl]), r1, what="ds1w" + what)
        assert_y_close(host(ds2w[sl]), r2, what="ds2w" + what)
        r1, r2 = oracle.address_backward(ridx_r, rw_r, dwrr, sh.sqrtN)
        assert_y_close(host(ds1r[sl]), r1, what="ds1r" + what)
        assert_y_close(host(ds2r[sl]), r2, what="ds2r" + what)

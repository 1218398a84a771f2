"""GPU parity of the sparse scan's training path through the C ABI:
sdm_scan_train (the forward plus its undo log) and sdm_scan_backward (the
gradients by undoing the writes, Sparse Delta Memory deck, App. A.3) against
the fp64 oracle."""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_state_close, assert_y_close, dev, host, need_gpu

pytestmark = pytest.mark.gpu

MODES = [oracle.RESID_SHARED, oracle.RESID_PERSLOT, oracle.RESID_ADDITIVE]
# tiny config (fp32 v), and a reduced 1.4B-layer-like shape (bf16 v, W = R = 16)
# whose d_v = 100 leaves a ragged last column tile
SHAPES = [synth.SDM_TINY, synth.SDM_14B_LAYER.with_(B=2, T=160, H=2, sqrtN=32, d_v=100)]


def _setup(shape, seed):
    inp = synth.sdm_inputs(shape, seed)
    iw, ww = oracle.address(inp["s1w"], inp["s2w"], shape.k, shape.W)
    ir, wr = oracle.address(inp["s1r"], inp["s2r"], shape.k, shape.R)
    M0 = synth.random_state((shape.B, shape.H, shape.N, shape.d_v), seed=seed + 1, scale=0.3)
    dy = synth.random_state((shape.B, shape.T, shape.H, shape.d_v), seed=seed + 2)
    dMT = synth.random_state((shape.B, shape.H, shape.N, shape.d_v), seed=seed + 3, scale=0.5)
    return inp, (iw, ww.astype(np.float32), ir, wr.astype(np.float32)), M0, dy, dMT


def _gpu_args(inp, sel):
    iw, ww, ir, wr = sel
    return (dev(inp["v"], bf16=inp["v_bf16"]), dev(inp["alpha"]), dev(inp["beta"]), dev(iw), dev(ww), dev(ir),
            dev(wr))


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_train_forward_is_the_scan_and_logs_the_written_rows(shape, mode):
    sdm = need_gpu()
    inp, sel, M0, _, _ = _setup(shape, seed=50 + mode)
    args = _gpu_args(inp, sel)
    s1 = dev(M0)
    y1 = sdm.sdm_scan(s1, *args, resid_mode=mode)
    s2 = dev(M0)
    y2, undo = sdm.sdm_scan_train(s2, *args, resid_mode=mode)
    np.testing.assert_array_equal(host(y2), host(y1))
    np.testing.assert_array_equal(host(s2), host(s1))
    _, _, undo_ref = oracle.sdm_scan(M0, inp["v"], inp["alpha"], inp["beta"], *sel, mode, keep_undo=True)
    assert_state_close(host(undo), undo_ref, what="undo log")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_backward_matches_the_oracle_and_restores_the_table(shape, mode):
    sdm = need_gpu()
    import torch
    inp, sel, M0, dy, dMT = _setup(shape, seed=60 + mode)
    args = _gpu_args(inp, sel)
    state = dev(M0)
    _, undo = sdm.sdm_scan_train(state, *args, resid_mode=mode)
    dstate = dev(dMT)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    dv, da, db, dww, dwr = sdm.sdm_scan_backward(state, dstate, *args, undo, dev(dy), resid_mode=mode, dev_err=err)
    assert int(host(err)[0]) == 0
    np.testing.assert_array_equal(host(state), M0)          # every write undone, bit for bit
    MT, _, undo_ref = oracle.sdm_scan(M0, inp["v"], inp["alpha"], inp["beta"], *sel, mode, keep_undo=True)
    _, dM0r, dvr, dar, dbr, dwwr, dwrr = oracle.sdm_scan_backward(MT, dMT, inp["v"], inp["alpha"], inp["beta"], *sel,
                                                                  mode, undo_ref, dy)
    assert_state_close(host(dstate), dM0r, what="dL/dM_0")
    assert_y_close(host(dv), dvr, what="dL/dv")
    assert_y_close(host(da), dar, what="dL/dalpha")
    assert_y_close(host(db), dbr, what="dL/dbeta")
    assert_y_close(host(dww), dwwr, what="dL/dw_w")
    assert_y_close(host(dwr), dwrr, what="dL/dw_r")


def test_address_backward_matches_the_oracle():
    """The 1.4B layer's halves (sqrtN = 240, k = 16, W = 16) on a reduced
    batch: the score gradients equal the oracle's (fp32 vs fp64)."""
    sdm = need_gpu()
    sh = synth.SDM_14B_LAYER.with_(B=2, T=64)
    inp = synth.sdm_inputs(sh, seed=70)
    idx, w = oracle.address(inp["s1w"], inp["s2w"], sh.k, sh.W)
    dw = synth.random_state(idx.shape, seed=71)
    ds1, ds2 = sdm.sdm_address_backward(dev(idx), dev(w.astype(np.float32)), dev(dw), sh.sqrtN)
    r1, r2 = oracle.address_backward(idx, w.astype(np.float32), dw, sh.sqrtN)
    assert_y_close(host(ds1), r1, what="ds1")
    assert_y_close(host(ds2), r2, what="ds2")
    assert np.all(host(ds1)[r1 == 0] == 0) and np.all(host(ds2)[r2 == 0] == 0)

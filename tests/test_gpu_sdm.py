"""GPU parity of the sparse path (sdm_address + sdm_scan) against the fp64 CPU
oracle, through the C ABI.  Indices bit-exact; y within 2e-3 * RMS(y_ref);
state within 1e-3 relative (Frobenius)."""
import os

import numpy as np
import pytest

import oracle
import synth
from helpers import assert_state_close, assert_y_close, dev, host, need_gpu

pytestmark = pytest.mark.gpu

MODES = [(0, oracle.RESID_SHARED), (1, oracle.RESID_PERSLOT), (2, oracle.RESID_ADDITIVE)]


def _gpu_address(sdm, s1, s2, k, W):
    import torch
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    idx, w = sdm.sdm_address(dev(s1), dev(s2), k, W, dev_err=err)
    return host(idx), host(w), int(host(err)[0])


def _check_address(sdm, s1, s2, k, W):
    idx, w, err = _gpu_address(sdm, s1, s2, k, W)
    ridx, rw = oracle.address(s1, s2, k, W)
    assert err == 0
    np.testing.assert_array_equal(idx, ridx)
    np.testing.assert_allclose(w, rw, rtol=2e-6, atol=1e-7)


# ----------------------------------------------------------------- addressing
def test_address_tiny_bitexact():
    sdm = need_gpu()
    sh = synth.SDM_TINY
    inp = synth.sdm_inputs(sh, seed=0)
    _check_address(sdm, inp["s1w"], inp["s2w"], sh.k, sh.W)
    _check_address(sdm, inp["s1r"], inp["s2r"], sh.k, sh.R)


def test_address_14b_layer_full_size_bitexact():
    """Every row of the 1.4B-layer workload (B=8, T=4096, H=2, sqrtN=240)."""
    sdm = need_gpu()
    sh = synth.SDM_14B_LAYER
    inp = synth.sdm_inputs(sh, seed=0)
    _check_address(sdm, inp["s1w"], inp["s2w"], sh.k, sh.W)
    _check_address(sdm, inp["s1r"], inp["s2r"], sh.k, sh.R)


@pytest.mark.parametrize("H", [4, 8])
def test_address_sweep_shapes_bitexact(H):
    sdm = need_gpu()
    sh = synth.sdm_sweep_shape(H, B=2, T=512)
    inp = synth.sdm_inputs(sh, seed=H)
    _check_address(sdm, inp["s1w"], inp["s2w"], sh.k, sh.W)


@pytest.mark.parametrize("sq,k,W", [(8, 4, 4), (16, 6, 5), (64, 32, 64), (512, 32, 64), (1, 1, 1), (33, 7, 49),
                                    (240, 16, 1)])
def test_address_shapes_and_limits(sq, k, W):
    sdm = need_gpu()
    s1 = synth.dyadic_scores((1, 37, 3, sq), sq)
    s2 = synth.dyadic_scores((1, 37, 3, sq), sq + 1)
    _check_address(sdm, s1, s2, k, W)
    g = np.random.default_rng(sq)
    _check_address(sdm, g.standard_normal((1, 37, 3, sq)).astype(np.float32),
                   g.standard_normal((1, 37, 3, sq)).astype(np.float32), k, W)


def test_address_exact_ties():
    sdm = need_gpu()
    g = np.random.default_rng(7)
    s1 = g.integers(-2, 3, (2, 64, 2, 16)).astype(np.float32)
    s2 = g.integers(-2, 3, (2, 64, 2, 16)).astype(np.float32)
    _check_address(sdm, s1, s2, 8, 16)
    z = np.zeros((1, 8, 1, 32), np.float32)          # everything ties
    _check_address(sdm, z, z, 5, 20)


def test_address_flags_nonfinite():
    sdm = need_gpu()
    s1 = np.zeros((1, 4, 1, 8), np.float32)
    s1[0, 2, 0, 3] = np.nan
    _, _, err = _gpu_address(sdm, s1, np.zeros_like(s1), 4, 4)
    assert err & sdm.SDM_DEVERR_NONFINITE


# ----------------------------------------------------------------------- scan
def _run_gpu_scan(sdm, M0, inp, idx_w, w_w, idx_r, w_r, mode, v_bf16=None):
    import torch
    state = dev(M0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    v = dev(inp["v"], bf16=inp["v"].dtype == np.uint16 if v_bf16 is None else v_bf16)
    y = sdm.sdm_scan(state, v, dev(inp["alpha"]), dev(inp["beta"]), dev(idx_w), dev(w_w), dev(idx_r), dev(w_r),
                     resid_mode=mode, dev_err=err)
    return host(state), host(y), int(host(err)[0])


@pytest.mark.parametrize("gmode,omode", MODES)
def test_scan_tiny_full_pipeline(gmode, omode):
    """The tiny workload end to end: GPU addressing + GPU scan vs the oracle's
    addressing + scan (zero initial state)."""
    sdm = need_gpu()
    sh = synth.SDM_TINY
    inp = synth.sdm_inputs(sh, seed=0)
    iw, ww, e1 = _gpu_address(sdm, inp["s1w"], inp["s2w"], sh.k, sh.W)
    ir, wr, e2 = _gpu_address(sdm, inp["s1r"], inp["s2r"], sh.k, sh.R)
    ref = oracle.sdm_forward(inp, sh.k, sh.W, sh.R, mode=omode)
    np.testing.assert_array_equal(iw, ref["idx_w"])
    np.testing.assert_array_equal(ir, ref["idx_r"])
    M0 = np.zeros((sh.B, sh.H, sh.N, sh.d_v), np.float32)
    M, y, err = _run_gpu_scan(sdm, M0, inp, iw, ww, ir, wr, gmode)
    assert err == e1 == e2 == 0
    assert_y_close(y, ref["y"])
    assert_state_close(M, ref["state"])


@pytest.mark.parametrize("d_v", [36, 68, 132])
@pytest.mark.parametrize("window", [4, 6, 8])
@pytest.mark.parametrize("tile", [16, 32])
@pytest.mark.parametrize("gmode,omode", MODES)
def test_scan_hazard_stress(monkeypatch, d_v, window, tile, gmode, omode):
    """Tiny tables with W = R = 16: rows are rewritten by almost every token,
    so nearly every slot is forwarded from the history ring.  Ragged d_v (a
    partial last column tile), random nonzero initial state, every compiled
    prefetch window and both column-tile widths."""
    sdm = need_gpu()
    monkeypatch.setenv("SDM_SCAN_WINDOW", str(window))
    monkeypatch.setenv("SDM_SCAN_TILE", str(tile))
    for sq, k, seed in ((4, 4, 1), (8, 8, 2)):
        sh = synth.SdmShape("stress", B=2, T=97, H=3, sqrtN=sq, d_v=d_v, k=k, W=16, R=16, v_bf16=False)
        inp = synth.sdm_inputs(sh, seed=seed)
        iw, ww = oracle.address(inp["s1w"], inp["s2w"], k, 16)
        ir, wr = oracle.address(inp["s1r"], inp["s2r"], k, 16)
        M0 = synth.random_state((sh.B, sh.H, sh.N, sh.d_v), seed=seed + 10)
        Mr, yr = oracle.sdm_scan(M0, inp["v"], inp["alpha"], inp["beta"], iw, ww, ir, wr, omode)
        M, y, err = _run_gpu_scan(sdm, M0, inp, iw, ww.astype(np.float32), ir, wr.astype(np.float32), gmode)
        assert err == 0
        assert_y_close(y, yr)
        assert_state_close(M, Mr)


@pytest.mark.parametrize("W,R", [(1, 1), (4, 12), (33, 64), (64, 20)])
def test_scan_list_sizes(W, R):
    sdm = need_gpu()
    sh = synth.SdmShape("sizes", B=1, T=40, H=2, sqrtN=16, d_v=64, k=16, W=W, R=R, v_bf16=True)
    inp = synth.sdm_inputs(sh, seed=W + R)
    iw, ww = oracle.address(inp["s1w"], inp["s2w"], 16, W)
    ir, wr = oracle.address(inp["s1r"], inp["s2r"], 16, R)
    M0 = synth.random_state((1, 2, sh.N, 64), seed=3)
    Mr, yr = oracle.sdm_scan(M0, inp["v"], inp["alpha"], inp["beta"], iw, ww, ir, wr, oracle.RESID_SHARED)
    M, y, err = _run_gpu_scan(sdm, M0, inp, iw, ww.astype(np.float32), ir, wr.astype(np.float32), 0)
    assert err == 0
    assert_y_close(y, yr)
    assert_state_close(M, Mr)


def _layer_case(sh, seed, cols, bh_list, mode):
    """GPU: addressing + scan of the whole workload.  Oracle: the same inputs
    restricted to the sampled (b, h) sequences and value columns (columns are
    independent: the addresses do not depend on the table)."""
    sdm = need_gpu()
    import torch
    inp = synth.sdm_inputs(sh, seed=seed)
    s = {k_: dev(inp[k_]) for k_ in ("s1w", "s2w", "s1r", "s2r")}
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    iw, ww = sdm.sdm_address(s["s1w"], s["s2w"], sh.k, sh.W, dev_err=err)
    ir, wr = sdm.sdm_address(s["s1r"], s["s2r"], sh.k, sh.R, dev_err=err)
    state = torch.zeros((sh.B, sh.H, sh.N, sh.d_v), dtype=torch.float32, device="cuda")
    y = sdm.sdm_scan(state, dev(inp["v"]), dev(inp["alpha"]), dev(inp["beta"]), iw, ww, ir, wr, resid_mode=mode,
                     dev_err=err)
    torch.cuda.synchronize()
    assert int(host(err)[0]) == 0
    iw, ww, ir, wr = host(iw), host(ww), host(ir), host(wr)
    cols = np.asarray(cols)
    for (b, h) in bh_list:
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        ridx_w, rw_w = oracle.address(inp["s1w"][sl], inp["s2w"][sl], sh.k, sh.W)
        ridx_r, rw_r = oracle.address(inp["s1r"][sl], inp["s2r"][sl], sh.k, sh.R)
        np.testing.assert_array_equal(iw[sl], ridx_w)
        np.testing.assert_array_equal(ir[sl], ridx_r)
        v = inp["v"][sl][..., cols]
        M0 = np.zeros((1, 1, sh.N, len(cols)))
        Mr, yr = oracle.sdm_scan(M0, v, inp["alpha"][sl], inp["beta"][sl], ridx_w, rw_w, ridx_r, rw_r, mode)
        assert_y_close(host(y[b:b + 1, :, h:h + 1][..., cols]), yr, what=f"y[b={b},h={h}]")
        assert_state_close(host(state[b:b + 1, h:h + 1][..., cols]), Mr, what=f"state[b={b},h={h}]")


def test_scan_14b_layer_reduced_T():
    sh = synth.SDM_14B_LAYER.with_(B=2, T=256)
    cols = list(range(0, 40)) + list(range(500, 530)) + list(range(930, 960))
    _layer_case(sh, 1, cols, [(0, 0), (1, 1)], 0)


@pytest.mark.slow
def test_scan_14b_layer_full_size_sampled():
    """The full 1.4B-layer workload (B=8, T=4096) in the launch configuration
    the benchmark times; oracle on two sequences and 96 sampled columns."""
    sh = synth.SDM_14B_LAYER
    cols = list(range(0, 32)) + list(range(416, 448)) + list(range(928, 960))
    _layer_case(sh, 0, cols, [(0, 0), (7, 1)], 0)


@pytest.mark.parametrize("H", [2, 4, 8])
@pytest.mark.parametrize("gmode,omode", MODES[:2])
def test_scan_sweep_shapes_reduced(H, gmode, omode):
    sh = synth.sdm_sweep_shape(H, B=2, T=128)
    cols = list(range(0, 24)) + list(range(sh.d_v - 24, sh.d_v))
    _layer_case(sh, H, cols, [(1, H - 1)], gmode)


# ------------------------------------------------------------------ invariants
def test_scan_untouched_rows_bit_unchanged():
    sdm = need_gpu()
    sh = synth.SDM_14B_LAYER.with_(B=1, T=64, H=2, sqrtN=64, d_v=128)
    inp = synth.sdm_inputs(sh, seed=5)
    iw, ww = oracle.address(inp["s1w"], inp["s2w"], sh.k, sh.W)
    ir, wr = oracle.address(inp["s1r"], inp["s2r"], sh.k, sh.R)
    M0 = synth.random_state((1, 2, sh.N, 128), seed=6)
    M, _, err = _run_gpu_scan(sdm, M0, inp, iw, ww.astype(np.float32), ir, wr.astype(np.float32), 0)
    for h in range(2):
        untouched = np.setdiff1d(np.arange(sh.N), np.unique(iw[0, :, h]))
        assert untouched.size > 1000
        assert np.array_equal(M[0, h, untouched].view(np.uint32), M0[0, h, untouched].view(np.uint32))


def test_scan_split_in_time_is_bit_identical():
    sdm = need_gpu()
    import torch
    sh = synth.SdmShape("split", B=2, T=150, H=2, sqrtN=8, d_v=64, k=8, W=16, R=16, v_bf16=True)
    inp = synth.sdm_inputs(sh, seed=9)
    iw, ww = oracle.address(inp["s1w"], inp["s2w"], sh.k, sh.W)
    ir, wr = oracle.address(inp["s1r"], inp["s2r"], sh.k, sh.R)
    M0 = synth.random_state((2, 2, sh.N, 64), seed=1)
    full_M, full_y, _ = _run_gpu_scan(sdm, M0, inp, iw, ww.astype(np.float32), ir, wr.astype(np.float32), 0)
    state = dev(M0)
    ys = []
    for lo, hi in ((0, 61), (61, 150)):
        sl = (slice(None), slice(lo, hi))
        ys.append(host(sdm.sdm_scan(state, dev(inp["v"][sl]), dev(inp["alpha"][sl]), dev(inp["beta"][sl]),
                                    dev(iw[sl]), dev(ww[sl].astype(np.float32)), dev(ir[sl]),
                                    dev(wr[sl].astype(np.float32)))))
    torch.cuda.synchronize()
    assert np.array_equal(np.concatenate(ys, axis=1), full_y)
    assert np.array_equal(host(state), full_M)


def test_scan_columns_are_independent_bit_identical():
    sdm = need_gpu()
    sh = synth.SdmShape("cols", B=1, T=80, H=2, sqrtN=16, d_v=96, k=8, W=16, R=16, v_bf16=False)
    inp = synth.sdm_inputs(sh, seed=11)
    iw, ww = oracle.address(inp["s1w"], inp["s2w"], sh.k, sh.W)
    ir, wr = oracle.address(inp["s1r"], inp["s2r"], sh.k, sh.R)
    M0 = synth.random_state((1, 2, sh.N, 96), seed=2)
    M, y, _ = _run_gpu_scan(sdm, M0, inp, iw, ww.astype(np.float32), ir, wr.astype(np.float32), 0)
    sub = dict(inp)
    sub["v"] = np.ascontiguousarray(inp["v"][..., 36:56])
    Ms, ys, _ = _run_gpu_scan(sdm, np.ascontiguousarray(M0[..., 36:56]), sub, iw, ww.astype(np.float32), ir,
                              wr.astype(np.float32), 0)
    assert np.array_equal(ys, y[..., 36:56])
    assert np.array_equal(Ms, M[..., 36:56])


def test_scan_out_of_range_index_is_flagged_and_skipped():
    sdm = need_gpu()
    sh = synth.SdmShape("bad", B=1, T=20, H=1, sqrtN=8, d_v=32, k=4, W=4, R=4, v_bf16=False)
    inp = synth.sdm_inputs(sh, seed=4)
    iw, ww = oracle.address(inp["s1w"], inp["s2w"], sh.k, sh.W)
    ir, wr = oracle.address(inp["s1r"], inp["s2r"], sh.k, sh.R)
    iw[0, 5, 0, 2] = sh.N + 7
    ir[0, 9, 0, 1] = -3
    M0 = synth.random_state((1, 1, sh.N, 32), seed=8)
    M, y, err = _run_gpu_scan(sdm, M0, inp, iw, ww.astype(np.float32), ir, wr.astype(np.float32), 0)
    assert err & sdm.SDM_DEVERR_INDEX_RANGE
    assert np.all(np.isfinite(y)) and np.all(np.isfinite(M))


def test_scan_repeated_write_slot_is_flagged():
    sdm = need_gpu()
    sh = synth.SdmShape("rep", B=1, T=6, H=1, sqrtN=8, d_v=16, k=4, W=4, R=4, v_bf16=False)
    inp = synth.sdm_inputs(sh, seed=4)
    iw, ww = oracle.address(inp["s1w"], inp["s2w"], sh.k, sh.W)
    ir, wr = oracle.address(inp["s1r"], inp["s2r"], sh.k, sh.R)
    iw[0, 3, 0, 1] = iw[0, 3, 0, 0]
    _, _, err = _run_gpu_scan(sdm, np.zeros((1, 1, sh.N, 16), np.float32), inp, iw, ww.astype(np.float32), ir,
                              wr.astype(np.float32), 0)
    assert err & sdm.SDM_DEVERR_INDEX_REPEAT


def test_deltanet_teaching_example_on_gpu(golden):
    """One unit-weight slot, prediction 2, target 5, beta 0.5 -> 3.5 (Linear
    Attention Architectures deck, Eq. 14 teaching example)."""
    sdm = need_gpu()
    g = golden("deltanet_teaching.txt")
    N, dv = 9, 4
    M0 = np.zeros((1, 1, N, dv), np.float32)
    M0[0, 0, 5] = g["prediction"][0]
    inp = {"v": np.full((1, 1, 1, dv), g["target"][0], np.float32), "alpha": np.ones((1, 1, 1), np.float32),
           "beta": np.full((1, 1, 1), g["beta"][0], np.float32)}
    idx = np.array([5], np.int32).reshape(1, 1, 1, 1)
    one = np.ones((1, 1, 1, 1), np.float32)
    for mode in (0, 1):
        M, y, _ = _run_gpu_scan(sdm, M0, inp, idx, one, idx, one, mode)
        np.testing.assert_allclose(y.ravel(), g["new_prediction"][0], rtol=0, atol=1e-6)


def test_two_slot_worked_example_on_gpu(golden):
    sdm = need_gpu()
    g = golden("two_slot_update.txt")
    M0 = np.array(g["m_prev"], np.float32).reshape(1, 1, 2, 1) * np.ones((1, 1, 2, 4), np.float32)
    inp = {"v": np.full((1, 1, 1, 4), g["v"][0], np.float32), "alpha": np.full((1, 1, 1), g["alpha"][0], np.float32),
           "beta": np.full((1, 1, 1), g["beta"][0], np.float32)}
    idx = np.array([0, 1], np.int32).reshape(1, 1, 1, 2)
    w = np.array(g["k"], np.float32).reshape(1, 1, 1, 2)
    for mode, key in ((1, "per_slot"), (0, "shared")):
        M, _, _ = _run_gpu_scan(sdm, M0, inp, idx, w, idx, w, mode)
        np.testing.assert_allclose(M[0, 0, :, 0], g[key], atol=1e-6)


# ------------------------------------------------------------- host path
@pytest.mark.parametrize("chunk", [3, 100, 4096])
def test_forward_host_matches_device_path_bitexact(chunk):
    """sdm_forward_host (host inputs and y, chunked copy/compute pipeline) gives
    the same bits as sdm_address x2 + sdm_scan on device inputs: one chunk
    (4096), quarter-size first and last chunks around even middle chunks
    (100: 25, 95, 94, 94, 25 tokens), one-token edges (3)."""
    sdm = need_gpu()
    import torch
    sh = synth.SDM_14B_LAYER.with_(B=2, T=333, H=2, sqrtN=64, d_v=96)
    inp = synth.sdm_inputs(sh, seed=17)
    M0 = synth.random_state((sh.B, sh.H, sh.N, sh.d_v), seed=18, scale=0.1)
    iw, ww = sdm.sdm_address(dev(inp["s1w"]), dev(inp["s2w"]), sh.k, sh.W)
    ir, wr = sdm.sdm_address(dev(inp["s1r"]), dev(inp["s2r"]), sh.k, sh.R)
    st_dev = dev(M0)
    y_dev = sdm.sdm_scan(st_dev, dev(inp["v"]), dev(inp["alpha"]), dev(inp["beta"]), iw, ww, ir, wr)
    hostt = lambda a: torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
    v_h = torch.from_numpy(inp["v"].view(np.int16).copy()).view(torch.bfloat16).pin_memory()
    st_host = dev(M0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y_h = sdm.sdm_forward_host(hostt(inp["s1w"]), hostt(inp["s2w"]), hostt(inp["s1r"]), hostt(inp["s2r"]), v_h,
                               hostt(inp["alpha"]), hostt(inp["beta"]), sh.k, sh.W, sh.R, st_host, chunk_T=chunk,
                               dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert np.array_equal(y_h.numpy(), host(y_dev))
    assert np.array_equal(host(st_host), host(st_dev))

"""GPU parity of the chunked form of the sparse scan (sdm_scan_chunked,
Sparse Delta Memory deck, App. A.1-A.2) against the fp64 sequential oracle,
through the C ABI."""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_state_close, assert_y_close, dev, host, need_gpu

pytestmark = pytest.mark.gpu

MODES = [oracle.RESID_SHARED, oracle.RESID_ADDITIVE]
SHAPES = [
    synth.SDM_TINY,                                                                    # 2 chunks, rows repeat
    synth.SdmShape("stress", B=2, T=150, H=2, sqrtN=8, d_v=64, k=8, W=16, R=16, v_bf16=True),  # N = 64: nearly every slot repeats
    synth.SDM_14B_LAYER.with_(B=2, T=300, H=2, sqrtN=32, d_v=100),                    # ragged chunk and column tile
]


def _case(shape, seed):
    inp = synth.sdm_inputs(shape, seed)
    iw, ww = oracle.address(inp["s1w"], inp["s2w"], shape.k, shape.W)
    ir, wr = oracle.address(inp["s1r"], inp["s2r"], shape.k, shape.R)
    M0 = synth.random_state((shape.B, shape.H, shape.N, shape.d_v), seed=seed + 1, scale=0.3)
    return inp, iw, ww.astype(np.float32), ir, wr.astype(np.float32), M0


def _gpu(sdm, inp, iw, ww, ir, wr, M0, mode):
    import torch
    state = dev(M0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = sdm.sdm_scan_chunked(state, dev(inp["v"], bf16=inp["v_bf16"]), dev(inp["alpha"]), dev(inp["beta"]),
                             dev(iw), dev(ww), dev(ir), dev(wr), resid_mode=mode, dev_err=err)
    return host(state), host(y), int(host(err)[0])


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: s.name)
def test_chunked_matches_the_oracle(shape, mode):
    sdm = need_gpu()
    inp, iw, ww, ir, wr, M0 = _case(shape, seed=80 + mode)
    M, y, err = _gpu(sdm, inp, iw, ww, ir, wr, M0, mode)
    assert err == 0
    Mr, yr = oracle.sdm_scan(M0, inp["v"], inp["alpha"], inp["beta"], iw, ww, ir, wr, mode)
    assert_y_close(y, yr)
    assert_state_close(M, Mr)
    for b in range(shape.B):
        for h in range(shape.H):
            untouched = np.setdiff1d(np.arange(shape.N), np.unique(iw[b, :, h]))
            assert np.array_equal(M[b, h, untouched].view(np.uint32), M0[b, h, untouched].view(np.uint32))


@pytest.mark.slow
def test_chunked_14b_layer_full_size_sampled():
    """The full 1.4B-layer workload; oracle on two sequences and 96 columns
    (columns are independent: the addresses do not depend on the table)."""
    sdm = need_gpu()
    import torch
    sh = synth.SDM_14B_LAYER
    inp = synth.sdm_inputs(sh, seed=0)
    s = {k_: dev(inp[k_]) for k_ in ("s1w", "s2w", "s1r", "s2r")}
    iw, ww = sdm.sdm_address(s["s1w"], s["s2w"], sh.k, sh.W)
    ir, wr = sdm.sdm_address(s["s1r"], s["s2r"], sh.k, sh.R)
    state = torch.zeros((sh.B, sh.H, sh.N, sh.d_v), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = sdm.sdm_scan_chunked(state, dev(inp["v"]), dev(inp["alpha"]), dev(inp["beta"]), iw, ww, ir, wr,
                             dev_err=err)
    torch.cuda.synchronize()
    assert int(host(err)[0]) == 0
    iw, ww, ir, wr = host(iw), host(ww), host(ir), host(wr)
    cols = np.asarray(list(range(0, 32)) + list(range(416, 448)) + list(range(928, 960)))
    for (b, h) in ((0, 1), (6, 0)):
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        Mr, yr = oracle.sdm_scan(np.zeros((1, 1, sh.N, len(cols))), inp["v"][sl][..., cols], inp["alpha"][sl],
                                 inp["beta"][sl], iw[sl], ww[sl], ir[sl], wr[sl], oracle.RESID_SHARED)
        assert_y_close(host(y[b:b + 1, :, h:h + 1][..., cols]), yr, what=f"y[b={b},h={h}]")
        assert_state_close(host(state[b:b + 1, h:h + 1][..., cols]), Mr, what=f"state[b={b},h={h}]")


def test_chunked_refuses_the_per_slot_residual():
    sdm = need_gpu()
    inp, iw, ww, ir, wr, M0 = _case(synth.SDM_TINY, seed=90)
    with pytest.raises(sdm.SdmError):
        _gpu(sdm, inp, iw, ww, ir, wr, M0, oracle.RESID_PERSLOT)

"""GPU parity of the dense (gdn_scan: GDN / KDA) and Sparse State Expansion
(sse_scan) paths against the fp64 CPU oracle, through the C ABI."""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_state_close, assert_y_close, dev, host, need_gpu

pytestmark = pytest.mark.gpu


# ---------------------------------------------------------------- dense GDN/KDA
def _gdn_gpu(sdm, S0, inp, per_channel):
    state = dev(S0)
    a = inp["alpha_kda"] if per_channel else inp["alpha_gdn"]
    y = sdm.gdn_scan(state, dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(a), dev(inp["beta"]), per_channel)
    return host(state), host(y)


@pytest.mark.parametrize("per_channel", [False, True])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 96), (16, 32)])
def test_gdn_reduced_parity(per_channel, dk, dv):
    sdm = need_gpu()
    sh = synth.GDN_DENSE.with_(B=2, T=200, H=3, dk=dk, dv=dv)
    inp = synth.gdn_inputs(sh, seed=dk + dv)
    S0 = synth.random_state((2, 3, dk, dv), seed=1, scale=0.3)
    a = inp["alpha_kda"] if per_channel else inp["alpha_gdn"]
    Sr, yr = oracle.gdn_scan(S0, inp["q"], inp["k"], inp["v"], a, inp["beta"], per_channel)
    S, y = _gdn_gpu(sdm, S0, inp, per_channel)
    assert_y_close(y, yr)
    assert_state_close(S, Sr)


@pytest.mark.slow
@pytest.mark.parametrize("per_channel", [False, True])
def test_gdn_full_size_sampled(per_channel):
    """The full dense workload (B=4, T=4096, H=16, dk=dv=128, zero state) on the
    GPU; the oracle recomputes three whole (b, h) sequences."""
    sdm = need_gpu()
    sh = synth.GDN_DENSE
    inp = synth.gdn_inputs(sh, seed=0)
    S0 = np.zeros((sh.B, sh.H, sh.dk, sh.dv), np.float32)
    S, y = _gdn_gpu(sdm, S0, inp, per_channel)
    a = inp["alpha_kda"] if per_channel else inp["alpha_gdn"]
    for b, h in ((0, 0), (2, 7), (3, 15)):
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        Sr, yr = oracle.gdn_scan(np.zeros((1, 1, sh.dk, sh.dv)), inp["q"][sl], inp["k"][sl], inp["v"][sl], a[sl],
                                 inp["beta"][sl], per_channel)
        assert_y_close(y[sl], yr, what=f"y[{b},{h}]")
        assert_state_close(S[b:b + 1, h:h + 1], Sr, what=f"state[{b},{h}]")


@pytest.mark.parametrize("chain", ["pair", "single"])
@pytest.mark.parametrize("per_channel", [False, True], ids=["gdn", "kda"])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200, 512, 700])
def test_gdn_chunked_path_lengths(T, per_channel, chain, monkeypatch):
    """Dense GDN and KDA at d_k = d_v = 128 run chunkwise (64 tokens) on the
    tensor cores: lengths below, at and across a chunk boundary, nonzero
    state, and longer sequences of 8 and 11 chunks; the chain on a CTA pair
    per (b, h) (value columns split) and on one CTA per (b, h)."""
    sdm = need_gpu()
    monkeypatch.setenv("SDM_GDN_PATH", "chunk")
    monkeypatch.setenv("SDM_GDN_CHAIN", chain)
    import torch
    sh = synth.GDN_DENSE.with_(B=2, T=T, H=2)
    inp = synth.gdn_inputs(sh, seed=40 + T)
    S0 = synth.random_state((2, 2, 128, 128), seed=41, scale=0.3)
    a = inp["alpha_kda"] if per_channel else inp["alpha_gdn"]
    Sr, yr = oracle.gdn_scan(S0, inp["q"], inp["k"], inp["v"], a, inp["beta"], per_channel)
    state = dev(S0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = sdm.gdn_scan(state, dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(a), dev(inp["beta"]),
                     per_channel, dev_err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    assert_y_close(host(y), yr)
    assert_state_close(host(state), Sr)


@pytest.mark.parametrize("per_channel", [False, True], ids=["gdn", "kda"])
def test_gdn_chunked_many_heads_default_chain_form(per_channel, monkeypatch):
    """B*H = 96 chains: more CTA pairs than a GB300 holds at once, so the
    default form there is one CTA per (b, h); whichever form the device
    size selects must match the oracle."""
    sdm = need_gpu()
    monkeypatch.setenv("SDM_GDN_PATH", "chunk")
    monkeypatch.delenv("SDM_GDN_CHAIN", raising=False)
    sh = synth.GDN_DENSE.with_(B=6, T=130, H=16)
    inp = synth.gdn_inputs(sh, seed=52)
    S0 = synth.random_state((6, 16, 128, 128), seed=53, scale=0.3)
    a = inp["alpha_kda"] if per_channel else inp["alpha_gdn"]
    Sr, yr = oracle.gdn_scan(S0, inp["q"], inp["k"], inp["v"], a, inp["beta"], per_channel)
    S, y = _gdn_gpu(sdm, S0, inp, per_channel)
    assert_y_close(y, yr)
    assert_state_close(S, Sr)


@pytest.mark.parametrize("chain", ["pair", "single"])
@pytest.mark.parametrize("scale", [1.0, 3.0, 6.0])
def test_kda_chunked_strong_per_channel_decay(scale, chain, monkeypatch):
    """KDA decays alpha = exp(-scale * softplus(N(0,1))) per key channel: at
    scale 6 the per-channel log decay over a 64-token chunk spans hundreds of
    units, so any factor formed as an inverse decay would overflow; every
    factor here is a decay ratio of at most 1."""
    sdm = need_gpu()
    monkeypatch.setenv("SDM_GDN_PATH", "chunk")
    monkeypatch.setenv("SDM_GDN_CHAIN", chain)
    sh = synth.GDN_DENSE.with_(B=1, T=300, H=2)
    inp = synth.gdn_inputs(sh, seed=48)
    a = np.exp(np.log(inp["alpha_kda"].astype(np.float64)) * scale).astype(np.float32)
    a = np.maximum(a, np.float32(1e-30))
    inp = dict(inp, alpha_kda=a)
    S0 = synth.random_state((1, 2, 128, 128), seed=49, scale=0.3)
    Sr, yr = oracle.gdn_scan(S0, inp["q"], inp["k"], inp["v"], a, inp["beta"], True)
    S, y = _gdn_gpu(sdm, S0, inp, True)
    assert_y_close(y, yr)
    assert_state_close(S, Sr)


@pytest.mark.parametrize("chain", ["pair", "single"])
@pytest.mark.parametrize("per_channel", [False, True], ids=["gdn", "kda"])
def test_gdn_chunked_is_deterministic_and_continues_the_state(per_channel, chain, monkeypatch):
    """The chunked path (T = 900: 15 chunks) gives the same bits on every
    call, and a sequence cut at a chunk boundary into two calls equals one
    call (the second call continues from the state the first left)."""
    sdm = need_gpu()
    monkeypatch.setenv("SDM_GDN_PATH", "chunk")
    monkeypatch.setenv("SDM_GDN_CHAIN", chain)
    sh = synth.GDN_DENSE.with_(B=2, T=900, H=2)
    inp = synth.gdn_inputs(sh, seed=46)
    S0 = synth.random_state((2, 2, 128, 128), seed=47, scale=0.3)
    S1, y1 = _gdn_gpu(sdm, S0, inp, per_channel)
    S2, y2 = _gdn_gpu(sdm, S0, inp, per_channel)
    np.testing.assert_array_equal(y1, y2)
    np.testing.assert_array_equal(S1, S2)
    cut = 576
    first = {k: v[:, :cut] for k, v in inp.items() if isinstance(v, np.ndarray) and v.ndim >= 3}
    second = {k: v[:, cut:] for k, v in inp.items() if isinstance(v, np.ndarray) and v.ndim >= 3}
    Sa, ya = _gdn_gpu(sdm, S0, first, per_channel)
    Sb, yb = _gdn_gpu(sdm, Sa, second, per_channel)
    assert_y_close(np.concatenate([ya, yb], axis=1), y1.astype(np.float64))
    assert_state_close(Sb, S1.astype(np.float64))


@pytest.mark.parametrize("per_channel", [False, True], ids=["gdn", "kda"])
def test_gdn_chunked_matches_token_recurrent(per_channel, monkeypatch):
    sdm = need_gpu()
    sh = synth.GDN_DENSE.with_(B=1, T=300, H=3)
    inp = synth.gdn_inputs(sh, seed=44)
    S0 = synth.random_state((1, 3, 128, 128), seed=45, scale=0.3)
    monkeypatch.setenv("SDM_GDN_PATH", "chunk")
    Sc, yc = _gdn_gpu(sdm, S0, inp, per_channel)
    monkeypatch.setenv("SDM_GDN_PATH", "recurrent")
    Sr, yr = _gdn_gpu(sdm, S0, inp, per_channel)
    assert_y_close(yc, yr)
    assert_state_close(Sc, Sr)


def test_kda_with_constant_channel_decay_is_gdn(monkeypatch):
    """KDA with alpha = alpha_t * 1 is GDN (Linear Attention Architectures
    deck, Eqs. 18-20): within tolerance between the two tensor-core paths, and
    bit-exact on the same token-by-token kernel."""
    sdm = need_gpu()
    sh = synth.GDN_DENSE.with_(B=1, T=200, H=2)
    inp = synth.gdn_inputs(sh, seed=3)
    inp2 = dict(inp)
    inp2["alpha_kda"] = np.repeat(inp["alpha_gdn"][..., None], sh.dk, axis=-1).copy()
    S0 = synth.random_state((1, 2, sh.dk, sh.dv), seed=4, scale=0.2)
    monkeypatch.setenv("SDM_GDN_PATH", "chunk")
    Sk, yk = _gdn_gpu(sdm, S0, inp2, True)          # chunked KDA
    Sc, yc = _gdn_gpu(sdm, S0, inp, False)          # chunked GDN
    assert_y_close(yc, yk)
    assert_state_close(Sc, Sk)
    monkeypatch.setenv("SDM_GDN_PATH", "recurrent")
    Skr, ykr = _gdn_gpu(sdm, S0, inp2, True)
    Sg, yg = _gdn_gpu(sdm, S0, inp, False)
    assert np.array_equal(yg, ykr) and np.array_equal(Sg, Skr)


def test_sparse_scan_with_every_row_selected_matches_dense():
    """sdm_scan with N = dk, all rows selected, weights k_t / q_t and the shared
    residual is gdn_scan (the dense limit of the sparse write)."""
    sdm = need_gpu()
    import torch
    sh = synth.GDN_DENSE.with_(B=1, T=96, H=2, dk=32, dv=64)
    inp = synth.gdn_inputs(sh, seed=8)
    S0 = synth.random_state((1, 2, 32, 64), seed=2, scale=0.5)
    Sg, yg = _gdn_gpu(sdm, S0, inp, False)
    kk = oracle.widen(inp["k"]).astype(np.float32)
    qq = oracle.widen(inp["q"]).astype(np.float32)
    idx = np.broadcast_to(np.arange(32, dtype=np.int32), (1, 96, 2, 32)).copy()
    state = dev(S0)
    y = sdm.sdm_scan(state, dev(inp["v"]), dev(inp["alpha_gdn"]), dev(inp["beta"]), dev(idx), dev(kk), dev(idx),
                     dev(qq))
    torch.cuda.synchronize()
    assert_y_close(host(y), yg)
    assert_state_close(host(state), Sg)


def test_gdn_teaching_example_on_gpu(golden):
    sdm = need_gpu()
    g = golden("deltanet_teaching.txt")
    dk, dv = 16, 32
    S0 = np.zeros((1, 1, dk, dv), np.float32)
    S0[0, 0, 3] = g["prediction"][0]
    e = np.zeros((1, 1, 1, dk), np.float32)
    e[..., 3] = 1.0
    inp = {"q": synth.to_bf16_bits(__import__("torch").from_numpy(e)), "k": None,
           "v": synth.to_bf16_bits(__import__("torch").full((1, 1, 1, dv), g["target"][0])),
           "alpha_gdn": np.ones((1, 1, 1), np.float32), "beta": np.full((1, 1, 1), g["beta"][0], np.float32)}
    inp["k"] = inp["q"]
    _, y = _gdn_gpu(sdm, S0, inp, False)
    np.testing.assert_allclose(y.ravel(), g["new_prediction"][0], atol=1e-6)


# ------------------------------------------------------------------------ GDN2
def _gdn2_gpu(sdm, S0, inp):
    state = dev(S0)
    y = sdm.gdn2_scan(state, dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(inp["alpha_kda"]),
                      dev(inp["b_erase"]), dev(inp["w_write"]))
    return host(state), host(y)


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 96), (16, 32)])
def test_gdn2_reduced_parity(dk, dv):
    sdm = need_gpu()
    sh = synth.GDN_DENSE.with_(B=2, T=200, H=3, dk=dk, dv=dv)
    inp = synth.gdn_inputs(sh, seed=3 * dk + dv)
    S0 = synth.random_state((2, 3, dk, dv), seed=4, scale=0.3)
    Sr, yr = oracle.gdn2_scan(S0, inp["q"], inp["k"], inp["v"], inp["alpha_kda"], inp["b_erase"], inp["w_write"])
    S, y = _gdn2_gpu(sdm, S0, inp)
    assert_y_close(y, yr)
    assert_state_close(S, Sr)


@pytest.mark.slow
def test_gdn2_full_size_sampled():
    """The dense workload's shape (B=4, T=4096, H=16, dk=dv=128) through GDN2;
    the oracle recomputes three whole (b, h) sequences."""
    sdm = need_gpu()
    sh = synth.GDN_DENSE
    inp = synth.gdn_inputs(sh, seed=0)
    S, y = _gdn2_gpu(sdm, np.zeros((sh.B, sh.H, sh.dk, sh.dv), np.float32), inp)
    for b, h in ((0, 0), (1, 9), (3, 15)):
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        Sr, yr = oracle.gdn2_scan(np.zeros((1, 1, sh.dk, sh.dv)), inp["q"][sl], inp["k"][sl], inp["v"][sl],
                                  inp["alpha_kda"][sl], inp["b_erase"][sl], inp["w_write"][sl])
        assert_y_close(y[sl], yr, what=f"y[{b},{h}]")
        assert_state_close(S[b:b + 1, h:h + 1], Sr, what=f"state[{b},{h}]")


@pytest.mark.parametrize("chain", ["pair", "single"])
@pytest.mark.parametrize("T", [1, 63, 64, 65, 200, 700])
def test_gdn2_chunked_path_lengths(T, chain, monkeypatch):
    """GDN2 at d_k = d_v = 128 runs in chunk form on the tensor cores (the KDA
    chunk form with erase rows e = b (.) k and Ut = (I + A)^-1 (w (.) v)):
    lengths around chunk edges from a nonzero state, on both chain forms."""
    sdm = need_gpu()
    monkeypatch.setenv("SDM_GDN_PATH", "chunk")
    monkeypatch.setenv("SDM_GDN_CHAIN", chain)
    sh = synth.GDN_DENSE.with_(B=2, T=T, H=2)
    inp = synth.gdn_inputs(sh, seed=70 + T)
    S0 = synth.random_state((2, 2, 128, 128), seed=71, scale=0.3)
    Sr, yr = oracle.gdn2_scan(S0, inp["q"], inp["k"], inp["v"], inp["alpha_kda"], inp["b_erase"], inp["w_write"])
    S, y = _gdn2_gpu(sdm, S0, inp)
    assert_y_close(y, yr)
    assert_state_close(S, Sr)


def test_gdn2_chunked_matches_token_recurrent(monkeypatch):
    sdm = need_gpu()
    sh = synth.GDN_DENSE.with_(B=1, T=300, H=3)
    inp = synth.gdn_inputs(sh, seed=72)
    S0 = synth.random_state((1, 3, 128, 128), seed=73, scale=0.3)
    monkeypatch.setenv("SDM_GDN_PATH", "chunk")
    Sc, yc = _gdn2_gpu(sdm, S0, inp)
    monkeypatch.setenv("SDM_GDN_PATH", "recurrent")
    Sr, yr = _gdn2_gpu(sdm, S0, inp)
    assert_y_close(yc, yr.astype(np.float64))
    assert_state_close(Sc, Sr.astype(np.float64))


def test_gdn2_chunked_gates_equal_to_beta_match_kda(monkeypatch):
    """b = w = beta 1 makes GDN2 KDA: the two chunked tensor-core paths agree
    within tolerance (they differ in where beta enters the products)."""
    sdm = need_gpu()
    monkeypatch.setenv("SDM_GDN_PATH", "chunk")
    sh = synth.GDN_DENSE.with_(B=1, T=200, H=2)
    inp = dict(synth.gdn_inputs(sh, seed=74))
    inp["b_erase"] = np.repeat(inp["beta"][..., None], 128, axis=-1).astype(np.float32)
    inp["w_write"] = np.repeat(inp["beta"][..., None], 128, axis=-1).astype(np.float32)
    S0 = synth.random_state((1, 2, 128, 128), seed=75, scale=0.3)
    S2, y2 = _gdn2_gpu(sdm, S0, inp)
    Sk, yk = _gdn_gpu(sdm, S0, inp, True)
    assert_y_close(y2, yk.astype(np.float64))
    assert_state_close(S2, Sk.astype(np.float64))


def test_gdn2_gates_equal_to_beta_match_the_kda_kernel():
    """b = w = beta 1 on the GPU gives the KDA kernel's result (within fp32
    rounding of the differently ordered products)."""
    sdm = need_gpu()
    sh = synth.GDN_DENSE.with_(B=1, T=150, H=2, dk=64, dv=64)
    inp = synth.gdn_inputs(sh, seed=31)
    S0 = synth.random_state((1, 2, 64, 64), seed=32, scale=0.3)
    inp = dict(inp)
    inp["b_erase"] = np.repeat(inp["beta"][..., None], 64, axis=-1).astype(np.float32)
    inp["w_write"] = np.repeat(inp["beta"][..., None], 64, axis=-1).astype(np.float32)
    S2, y2 = _gdn2_gpu(sdm, S0, inp)
    Sk, yk = _gdn_gpu(sdm, S0, inp, True)
    assert_y_close(y2, yk.astype(np.float64))
    assert_state_close(S2, Sk.astype(np.float64))


# ------------------------------------------------------------------------- SSE
def _sse_gpu(sdm, S0, inp, topk, mode=0):
    import torch
    B, T, H, N = inp["route"].shape
    state = dev(S0)
    sel = torch.zeros((B, T, H, topk), dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = sdm.sse_scan(state, dev(inp["route"]), topk, dev(inp["klog"]), dev(inp["q"]), dev(inp["v"]),
                     dev(inp["alpha"]), sel_out=sel, dev_err=err, write_mode=mode)
    return host(state), host(y), host(sel), int(host(err)[0])


@pytest.mark.parametrize("N,topk,c,d", [(8, 2, 128, 128), (4, 1, 64, 32), (16, 3, 32, 48), (1, 1, 16, 16)])
def test_sse_reduced_parity(N, topk, c, d):
    sdm = need_gpu()
    sh = synth.SSE_PART.with_(B=2, T=150, H=3, N=N, topk=topk, c=c, d=d)
    inp = synth.sse_inputs(sh, seed=N + c)
    S0 = synth.random_state((2, 3, N + 1, c, d), seed=5)
    Sr, yr, selr = oracle.sse_scan(S0, inp["route"], topk, inp["klog"], inp["q"], inp["v"], inp["alpha"])
    S, y, sel, err = _sse_gpu(sdm, S0, inp, topk)
    assert err == 0
    np.testing.assert_array_equal(sel, selr)
    assert_y_close(y, yr)
    assert_state_close(S, Sr)


@pytest.mark.slow
def test_sse_full_size_sampled():
    """The full SSE workload (B=4, T=4096, H=8, 8+1 partitions of 128x128,
    top-2) on the GPU; the oracle recomputes two whole (b, h) sequences."""
    sdm = need_gpu()
    sh = synth.SSE_PART
    inp = synth.sse_inputs(sh, seed=0)
    S0 = np.zeros((sh.B, sh.H, sh.N + 1, sh.c, sh.d), np.float32)
    S, y, sel, err = _sse_gpu(sdm, S0, inp, sh.topk)
    assert err == 0
    for b, h in ((0, 0), (3, 7)):
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        Sr, yr, selr = oracle.sse_scan(np.zeros((1, 1, sh.N + 1, sh.c, sh.d)), inp["route"][sl], sh.topk,
                                       inp["klog"][sl], inp["q"][sl], inp["v"][sl], inp["alpha"][sl])
        np.testing.assert_array_equal(sel[sl], selr)
        assert_y_close(y[sl], yr, what=f"y[{b},{h}]")
        assert_state_close(S[b:b + 1, h:h + 1], Sr, what=f"state[{b},{h}]")


@pytest.mark.parametrize("N,topk,c,d", [(8, 2, 128, 128), (4, 1, 64, 32), (16, 3, 32, 48), (1, 1, 16, 16)])
def test_sse_delta_reduced_parity(N, topk, c, d):
    """The delta write (shared residual per visited partition); partitions no
    token visits keep their bits."""
    sdm = need_gpu()
    sh = synth.SSE_PART.with_(B=2, T=150, H=3, N=N, topk=topk, c=c, d=d)
    inp = synth.sse_inputs(sh, seed=2 * N + c + 1)
    S0 = synth.random_state((2, 3, N + 1, c, d), seed=6, scale=0.5)
    Sr, yr, selr = oracle.sse_scan(S0, inp["route"], topk, inp["klog"], inp["q"], inp["v"], inp["alpha"],
                                   oracle.SSE_WRITE_DELTA)
    S, y, sel, err = _sse_gpu(sdm, S0, inp, topk, oracle.SSE_WRITE_DELTA)
    assert err == 0
    np.testing.assert_array_equal(sel, selr)
    assert_y_close(y, yr)
    assert_state_close(S, Sr)
    for b in range(2):
        for h in range(3):
            for p in set(range(N)) - set(sel[b, :, h].ravel().tolist()):
                np.testing.assert_array_equal(S[b, h, p], S0[b, h, p])


@pytest.mark.slow
def test_sse_delta_full_size_sampled():
    sdm = need_gpu()
    sh = synth.SSE_PART
    inp = synth.sse_inputs(sh, seed=1)
    S0 = np.zeros((sh.B, sh.H, sh.N + 1, sh.c, sh.d), np.float32)
    S, y, sel, err = _sse_gpu(sdm, S0, inp, sh.topk, oracle.SSE_WRITE_DELTA)
    assert err == 0
    for b, h in ((1, 2), (2, 6)):
        sl = (slice(b, b + 1), slice(None), slice(h, h + 1))
        Sr, yr, selr = oracle.sse_scan(np.zeros((1, 1, sh.N + 1, sh.c, sh.d)), inp["route"][sl], sh.topk,
                                       inp["klog"][sl], inp["q"][sl], inp["v"][sl], inp["alpha"][sl],
                                       oracle.SSE_WRITE_DELTA)
        np.testing.assert_array_equal(sel[sl], selr)
        assert_y_close(y[sl], yr, what=f"y[{b},{h}]")
        assert_state_close(S[b:b + 1, h:h + 1], Sr, what=f"state[{b},{h}]")


def test_sse_local_clock_on_gpu(golden):
    sdm = need_gpu()
    g = golden("sse_local_clock.txt")
    a, T, visits = g["decay"][0], int(g["tokens"][0]), int(g["visits"][0])
    N, c, d = 4, 16, 16
    route = np.full((1, T, 1, N), -5.0, np.float32)
    route[0, :, 0, 1] = 3.0
    route[0, np.linspace(0, T - 1, visits).astype(int), 0, 0] = 4.0
    S0 = synth.random_state((1, 1, N + 1, c, d), seed=21) + 2.0
    zeros_bf = np.zeros((1, T, 1, c), np.uint16)
    inp = {"route": route, "klog": np.zeros((1, T, 1, c), np.float32), "q": zeros_bf,
           "v": np.zeros((1, T, 1, d), np.uint16), "alpha": np.full((1, T, 1, c), a, np.float32)}
    S, _, sel, _ = _sse_gpu(sdm, S0, inp, 1)
    assert np.sum(sel == 0) == visits
    np.testing.assert_allclose(S[0, 0, 0] / S0[0, 0, 0], a ** visits, rtol=2e-6)
    np.testing.assert_allclose(S[0, 0, 0] / S0[0, 0, 0], g["sparse_retained"][0], atol=5e-4)
    np.testing.assert_allclose(S[0, 0, N] / S0[0, 0, N], g["dense_retained"][0], atol=5e-4)
    for p in (2, 3):
        assert np.array_equal(S[0, 0, p].view(np.uint32), S0[0, 0, p].view(np.uint32))

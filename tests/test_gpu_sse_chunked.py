"""GPU parity of the SSE scan's chunked prefill path (SSE deck, "Varlen
groups tokens while preserving causal order"; "One gate controls both writes
and reads", Eqs. 9-14) through the C ABI, against the fp64 oracle.

sse_scan takes this path for both writes with c = d = 128 once T reaches
one chunk of 64 visits: the additive write (Eq. 11) through its own prep and
chain kernels, the delta write (Eq. 12) through the per-channel-decay delta
chunk form of the dense KDA scan, run per partition on its visit
subsequence.  SDM_SSE_PATH=chunk forces the path for any T and
SDM_SSE_PATH=recurrent forces the token-by-token kernel."""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_state_close, assert_y_close, dev, host, need_gpu

pytestmark = pytest.mark.gpu

WRITES = pytest.mark.parametrize("mode", [oracle.SSE_WRITE_ADDITIVE, oracle.SSE_WRITE_DELTA],
                                 ids=["additive", "delta"])


def _run(sdm, S0, inp, topk, ws_extra=0, mode=0):
    import torch
    B, T, H, N = inp["route"].shape
    state = dev(S0)
    sel = torch.zeros((B, T, H, topk), dtype=torch.int32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    c, d = S0.shape[3], S0.shape[4]
    ws = torch.empty(sdm.sse_scan_workspace_size(B, T, H, N, topk, c, d, mode) + ws_extra, dtype=torch.uint8,
                     device="cuda")
    y = sdm.sse_scan(state, dev(inp["route"]), topk, dev(inp["klog"]), dev(inp["q"]), dev(inp["v"]),
                     dev(inp["alpha"]), sel_out=sel, workspace=ws, dev_err=err, write_mode=mode)
    return host(state), host(y), host(sel), int(host(err)[0])


def _check(sdm, S0, inp, topk, mode=0):
    Sr, yr, selr = oracle.sse_scan(S0, inp["route"], topk, inp["klog"], inp["q"], inp["v"], inp["alpha"], mode)
    S, y, sel, err = _run(sdm, S0, inp, topk, mode=mode)
    assert err == 0
    np.testing.assert_array_equal(sel, selr)
    assert_y_close(y, yr)
    assert_state_close(S, Sr)
    B, H, N = S0.shape[0], S0.shape[1], S0.shape[2] - 1
    for b in range(B):
        for h in range(H):
            for p in set(range(N)) - set(sel[b, :, h].ravel().tolist()):
                np.testing.assert_array_equal(S[b, h, p], S0[b, h, p])
    return S, y


@pytest.mark.parametrize("B,T,H,N,topk", [
    (2, 200, 2, 8, 2),     # several units per partition, ragged tails
    (1, 130, 3, 1, 1),     # one routed partition that every token visits
    (1, 64, 2, 5, 3),      # exactly one shared chunk
    (2, 300, 1, 16, 1),    # partitions with few visits (some with none)
    (1, 160, 1, 64, 8),    # the largest N and top-k
])
@WRITES
def test_chunked_sse_matches_the_oracle(B, T, H, N, topk, mode, monkeypatch):
    monkeypatch.setenv("SDM_SSE_PATH", "chunk")
    sdm = need_gpu()
    sh = synth.SSE_PART.with_(B=B, T=T, H=H, N=N, topk=topk)
    inp = synth.sse_inputs(sh, seed=T + N)
    S0 = synth.random_state((B, H, N + 1, 128, 128), seed=N, scale=0.5)
    _check(sdm, S0, inp, topk, mode)


@pytest.mark.parametrize("chain", ["pair", "single"])
@pytest.mark.parametrize("B,T,H,N,topk", [(2, 200, 2, 8, 2), (1, 64, 2, 5, 3), (1, 160, 1, 64, 8)])
def test_chunked_sse_delta_on_both_chain_forms(B, T, H, N, topk, chain, monkeypatch):
    """The delta write's chains: the shared partitions on CTA pairs (value
    columns split) beside the routed partitions on one CTA each, in one
    launch, and every chain on one CTA."""
    monkeypatch.setenv("SDM_SSE_PATH", "chunk")
    monkeypatch.setenv("SDM_GDN_CHAIN", chain)
    sdm = need_gpu()
    sh = synth.SSE_PART.with_(B=B, T=T, H=H, N=N, topk=topk)
    inp = synth.sse_inputs(sh, seed=3 * T + N)
    S0 = synth.random_state((B, H, N + 1, 128, 128), seed=N + 1, scale=0.5)
    _check(sdm, S0, inp, topk, oracle.SSE_WRITE_DELTA)


def test_chunked_sse_delta_many_heads_default_chain_form(monkeypatch):
    """B*H = 96: more shared-partition CTA pairs than a GB300 holds at once,
    so the default there puts every chain on one CTA; the result must match
    the oracle whichever form the device size selects."""
    monkeypatch.setenv("SDM_SSE_PATH", "chunk")
    monkeypatch.delenv("SDM_GDN_CHAIN", raising=False)
    sdm = need_gpu()
    sh = synth.SSE_PART.with_(B=6, T=100, H=16, N=4, topk=2)
    inp = synth.sse_inputs(sh, seed=77)
    S0 = synth.random_state((6, 16, 5, 128, 128), seed=78, scale=0.5)
    _check(sdm, S0, inp, 2, oracle.SSE_WRITE_DELTA)


@pytest.mark.parametrize("T", [1, 5, 63, 65])
@WRITES
def test_chunked_sse_short_sequences(T, mode, monkeypatch):
    """One ragged chunk (or one full chunk and a one-visit tail)."""
    monkeypatch.setenv("SDM_SSE_PATH", "chunk")
    sdm = need_gpu()
    sh = synth.SSE_PART.with_(B=2, T=T, H=2)
    inp = synth.sse_inputs(sh, seed=3 * T)
    S0 = synth.random_state((2, 2, sh.N + 1, 128, 128), seed=T, scale=0.5)
    _check(sdm, S0, inp, sh.topk, mode)


@WRITES
def test_chunked_sse_strong_decay_stays_accurate(mode, monkeypatch):
    """alpha down to 0.01: products over a whole chunk underflow, which a
    quotient form would turn into 0/0; the block-referenced factors keep every
    pair exact."""
    monkeypatch.setenv("SDM_SSE_PATH", "chunk")
    sdm = need_gpu()
    sh = synth.SSE_PART.with_(B=1, T=256, H=2)
    inp = dict(synth.sse_inputs(sh, seed=11))
    rng = np.random.default_rng(5)
    inp["alpha"] = rng.uniform(0.01, 1.0, inp["alpha"].shape).astype(np.float32)
    S0 = synth.random_state((1, 2, sh.N + 1, 128, 128), seed=12, scale=0.5)
    _check(sdm, S0, inp, sh.topk, mode)


@WRITES
def test_chunked_and_recurrent_paths_agree_and_are_deterministic(mode, monkeypatch):
    sdm = need_gpu()
    sh = synth.SSE_PART.with_(B=2, T=256, H=2)
    inp = synth.sse_inputs(sh, seed=21)
    S0 = synth.random_state((2, 2, sh.N + 1, 128, 128), seed=22, scale=0.5)
    monkeypatch.setenv("SDM_SSE_PATH", "chunk")
    Sc, yc, selc, e1 = _run(sdm, S0, inp, sh.topk, mode=mode)
    Sc2, yc2, _, e2 = _run(sdm, S0, inp, sh.topk, mode=mode)
    monkeypatch.setenv("SDM_SSE_PATH", "recurrent")
    Sr, yr, selr, e3 = _run(sdm, S0, inp, sh.topk, mode=mode)
    assert e1 == e2 == e3 == 0
    np.testing.assert_array_equal(selc, selr)
    np.testing.assert_array_equal(yc, yc2)      # fixed summation order: bit-reproducible
    np.testing.assert_array_equal(Sc, Sc2)
    assert_y_close(yc, yr.astype(np.float64))
    assert_state_close(Sc, Sr.astype(np.float64))


def test_chunked_sse_is_the_default_for_the_prefill_shape(monkeypatch):
    """Without SDM_SSE_PATH, c = d = 128 and T >= 64 takes the chunked path
    for either write (its workspace holds the units), other shapes do not."""
    monkeypatch.delenv("SDM_SSE_PATH", raising=False)
    sdm = need_gpu()
    rec_only = sdm.sse_scan_workspace_size(4, 4096, 8, 8, 2, 64, 128, 0)
    assert sdm.sse_scan_workspace_size(4, 4096, 8, 8, 2, 128, 128, 0) > rec_only + 4096 * 32 * 99072 // 64
    assert sdm.sse_scan_workspace_size(4, 4096, 8, 8, 2, 128, 128, 1) > rec_only + 4096 * 32 * 148224 // 64
    assert sdm.sse_scan_workspace_size(4, 4096, 8, 8, 2, 64, 128, 1) == rec_only
    assert sdm.sse_scan_workspace_size(4, 32, 8, 8, 2, 128, 128, 0) == sdm.sse_scan_workspace_size(
        4, 32, 8, 8, 2, 64, 128, 0)


@WRITES
def test_chunked_sse_rejects_a_short_workspace(mode, monkeypatch):
    monkeypatch.setenv("SDM_SSE_PATH", "chunk")
    sdm = need_gpu()
    sh = synth.SSE_PART.with_(B=1, T=70, H=1)
    inp = synth.sse_inputs(sh, seed=2)
    S0 = np.zeros((1, 1, sh.N + 1, 128, 128), np.float32)
    with pytest.raises(RuntimeError):
        _run(sdm, S0, inp, sh.topk, ws_extra=-256, mode=mode)


def test_chunked_sse_local_clock(golden, monkeypatch):
    """The deck's local-clock example on the chunked path: partition 0
    visited 10 times in 100 tokens with v = 0 keeps alpha^10 of its content;
    the shared partition decays every token; unvisited partitions keep their
    bits."""
    monkeypatch.setenv("SDM_SSE_PATH", "chunk")
    sdm = need_gpu()
    g = golden("sse_local_clock.txt")
    a, T, visits = g["decay"][0], int(g["tokens"][0]), int(g["visits"][0])
    N, c, d = 4, 128, 128
    route = np.full((1, T, 1, N), -5.0, np.float32)
    route[0, :, 0, 1] = 3.0
    route[0, np.linspace(0, T - 1, visits).astype(int), 0, 0] = 4.0
    S0 = synth.random_state((1, 1, N + 1, c, d), seed=21) + 2.0
    inp = {"route": route, "klog": np.zeros((1, T, 1, c), np.float32), "q": np.zeros((1, T, 1, c), np.uint16),
           "v": np.zeros((1, T, 1, d), np.uint16), "alpha": np.full((1, T, 1, c), a, np.float32)}
    S, _, sel, err = _run(sdm, S0, inp, 1)
    assert err == 0 and np.sum(sel == 0) == visits
    np.testing.assert_allclose(S[0, 0, 0] / S0[0, 0, 0], a ** visits, rtol=2e-6)
    np.testing.assert_allclose(S[0, 0, 0] / S0[0, 0, 0], g["sparse_retained"][0], atol=5e-4)
    np.testing.assert_allclose(S[0, 0, N] / S0[0, 0, N], g["dense_retained"][0], atol=5e-4)
    for p in (2, 3):
        assert np.array_equal(S[0, 0, p].view(np.uint32), S0[0, 0, p].view(np.uint32))


@pytest.mark.parametrize("N,topk,path", [(12, 6, "chunk"), (16, 3, "chunk"), (40, 5, "chunk"), (12, 6, "recurrent")])
@WRITES
def test_routing_ties_go_to_the_lower_partition(N, topk, path, mode, monkeypatch):
    """Router logits on a coarse integer grid, so most tokens have exact ties:
    the selected partitions must be the oracle's (lower partition first among
    equal logits) through the per-thread routing of the chunked path (N <= 16),
    the per-warp routing (N = 40) and the token-by-token path."""
    monkeypatch.setenv("SDM_SSE_PATH", path)
    sdm = need_gpu()
    sh = synth.SSE_PART.with_(B=1, T=96, H=2, N=N, topk=topk)
    inp = dict(synth.sse_inputs(sh, seed=40 + N))
    rng = np.random.default_rng(N + topk)
    inp["route"] = rng.integers(-2, 3, inp["route"].shape).astype(np.float32)
    S0 = synth.random_state((1, 2, N + 1, 128, 128), seed=41, scale=0.5)
    _check(sdm, S0, inp, topk, mode)

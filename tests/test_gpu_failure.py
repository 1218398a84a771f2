"""Failure detection on the GPU without a fault: the tensor-core chain kernels
bound every mbarrier wait, and when one runs out they drain their MMAs and
copies, free tensor memory, return normally and report SDM_DEVERR_TIMEOUT in
the caller's error word.  SDM_TEST_DROP_SIGNAL=1 makes the chain skip one
signal (a flag that nothing then sets), so a wait runs out on purpose; the
next call on the same context must still be exact."""
import numpy as np
import pytest

import oracle
import synth
from helpers import assert_state_close, assert_y_close, dev, host, need_gpu

pytestmark = pytest.mark.gpu

SDM_DEVERR_TIMEOUT = 8


def _gdn(sdm, S0, inp, per_channel=False):
    import torch
    state = dev(S0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = inp["alpha_kda"] if per_channel else inp["alpha_gdn"]
    y = sdm.gdn_scan(state, dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(a), dev(inp["beta"]),
                     per_channel, dev_err=err)
    torch.cuda.synchronize()
    return host(state), host(y), int(host(err)[0])


def _sse(sdm, S0, inp, topk, mode):
    import torch
    state = dev(S0)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = sdm.sse_scan(state, dev(inp["route"]), topk, dev(inp["klog"]), dev(inp["q"]), dev(inp["v"]),
                     dev(inp["alpha"]), dev_err=err, write_mode=mode)
    torch.cuda.synchronize()
    return host(state), host(y), int(host(err)[0])


@pytest.mark.parametrize("chain", ["pair", "single"])
@pytest.mark.parametrize("per_channel", [False, True], ids=["gdn", "kda"])
def test_gdn_chain_wait_runs_out_and_the_context_stays_usable(per_channel, chain, monkeypatch):
    sdm = need_gpu()
    monkeypatch.setenv("SDM_GDN_PATH", "chunk")
    monkeypatch.setenv("SDM_GDN_CHAIN", chain)
    sh = synth.GDN_DENSE.with_(B=1, T=200, H=2)
    inp = synth.gdn_inputs(sh, seed=90)
    S0 = synth.random_state((1, 2, 128, 128), seed=91, scale=0.3)
    monkeypatch.setenv("SDM_TEST_DROP_SIGNAL", "1")
    _, _, err = _gdn(sdm, S0, inp, per_channel)
    assert err & SDM_DEVERR_TIMEOUT
    monkeypatch.delenv("SDM_TEST_DROP_SIGNAL")
    S, y, err = _gdn(sdm, S0, inp, per_channel)
    assert err == 0
    a = inp["alpha_kda"] if per_channel else inp["alpha_gdn"]
    Sr, yr = oracle.gdn_scan(S0, inp["q"], inp["k"], inp["v"], a, inp["beta"], per_channel)
    assert_y_close(y, yr)
    assert_state_close(S, Sr)


@pytest.mark.parametrize("mode,chain", [(oracle.SSE_WRITE_ADDITIVE, "pair"), (oracle.SSE_WRITE_DELTA, "pair"),
                                        (oracle.SSE_WRITE_DELTA, "single")], ids=["additive", "delta", "delta-single"])
def test_sse_chain_wait_runs_out_and_the_context_stays_usable(mode, chain, monkeypatch):
    sdm = need_gpu()
    monkeypatch.setenv("SDM_SSE_PATH", "chunk")
    monkeypatch.setenv("SDM_GDN_CHAIN", chain)
    sh = synth.SSE_PART.with_(B=1, T=200, H=2)
    inp = synth.sse_inputs(sh, seed=92)
    S0 = synth.random_state((1, 2, sh.N + 1, 128, 128), seed=93, scale=0.5)
    monkeypatch.setenv("SDM_TEST_DROP_SIGNAL", "1")
    _, _, err = _sse(sdm, S0, inp, sh.topk, mode)
    assert err & SDM_DEVERR_TIMEOUT
    monkeypatch.delenv("SDM_TEST_DROP_SIGNAL")
    S, y, err = _sse(sdm, S0, inp, sh.topk, mode)
    assert err == 0
    Sr, yr, _ = oracle.sse_scan(S0, inp["route"], sh.topk, inp["klog"], inp["q"], inp["v"], inp["alpha"], mode)
    assert_y_close(y, yr)
    assert_state_close(S, Sr)
    assert np.all(np.isfinite(S))


def test_timeout_without_error_word_is_reported_by_sdm_check(monkeypatch):
    """A call made without dev_err still cannot lose a timeout: the library
    records it in its own device word and sdm_check reports it (then clears
    it, so the next check after a clean call passes)."""
    import torch
    sdm = need_gpu()
    try:  # start from a clean record (the tests above leave timeouts in it)
        sdm.sdm_check()
    except sdm.SdmError:
        pass
    sdm.sdm_check()
    monkeypatch.setenv("SDM_GDN_PATH", "chunk")
    sh = synth.GDN_DENSE.with_(B=1, T=200, H=2)
    inp = synth.gdn_inputs(sh, seed=94)
    S0 = synth.random_state((1, 2, 128, 128), seed=95, scale=0.3)
    monkeypatch.setenv("SDM_TEST_DROP_SIGNAL", "1")
    sdm.gdn_scan(dev(S0), dev(inp["q"]), dev(inp["k"]), dev(inp["v"]), dev(inp["alpha_gdn"]), dev(inp["beta"]),
                 False)
    with pytest.raises(sdm.SdmError) as e:
        sdm.sdm_check()
    assert e.value.code == sdm.SDM_ERR_DEVICE
    assert "wait gave up" in str(e.value)
    monkeypatch.delenv("SDM_TEST_DROP_SIGNAL")
    S, y, err = _gdn(sdm, S0, inp)
    assert err == 0
    sdm.sdm_check()
    # the caller's own word is reported too (and left as it is)
    word = torch.full((1,), SDM_DEVERR_TIMEOUT, dtype=torch.int32, device="cuda")
    with pytest.raises(sdm.SdmError):
        sdm.sdm_check(word)
    assert int(host(word)[0]) == SDM_DEVERR_TIMEOUT

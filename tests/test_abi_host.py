"""Host-side checks of the C ABI (no GPU): the library builds, loads, exports
every function that include/sdm.h declares, and rejects bad arguments with
the documented status codes before touching the device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "sdm.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^(?:SDM_API\s+)?(?:const\s+)?(?:int|size_t|char|void)\s*\*?\s*(\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def sdm():
    from delta_rule_memory_gb300 import build as b
    b.build()
    import delta_rule_memory_gb300 as m
    return m


def test_header_declares_the_boundary():
    names = _declared_functions()
    for fn in ("sdm_address", "sdm_scan", "gdn_scan", "gdn2_scan", "sse_scan", "sdm_version", "sdm_last_error",
               "sdm_check", "sdm_scan_workspace_size", "gdn_scan_workspace_size", "sse_scan_workspace_size"):
        assert fn in names


def test_library_exports_every_declared_symbol(sdm):
    lib = ctypes.CDLL(sdm.library_path)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, f"declared in sdm.h but not exported: {missing}"


def test_version_and_workspace(sdm):
    assert sdm.sdm_version() >= 10000
    # one packed record per token-head: 336 bytes for W, R <= 16, else 1296
    assert sdm.sdm_scan_workspace_size(8, 4096, 2, 16, 16) == 8 * 4096 * 2 * 336
    assert sdm.sdm_scan_workspace_size(1, 3, 1, 3, 4) == 1024
    assert sdm.sdm_scan_workspace_size(1, 1, 1, 17, 4) == 1536
    assert sdm.sdm_scan_workspace_size(0, 3, 1, 3, 4) == 0


def test_sse_workspace_sizes(sdm, monkeypatch):
    """Routing records only on the token-by-token path; on the chunked
    prefill path also the group tables (200 header words + topk*T entries per
    (batch, head)), ceil(T/64) + floor((topk*T + 63*N)/64) units per (batch,
    head) of 99,072 bytes (additive write) or 148,224 bytes (delta write), and
    (topk+1) staging rows of d fp32 per token."""
    monkeypatch.delenv("SDM_SSE_PATH", raising=False)
    B, T, H, N, k = 4, 4096, 8, 8, 2
    rec = B * T * H * 8 * 4                       # 2k + 2 words, rounded up to 4
    assert sdm.sse_scan_workspace_size(B, T, H, N, k, 64, 128, 0) == rec
    r256 = lambda n: (n + 255) // 256 * 256
    units = (T + 63) // 64 + (k * T + 63 * N) // 64
    chunk = lambda unit: (r256(B * H * (200 + k * T) * 4) + B * H * units * unit +
                          r256(B * T * H * (k + 1) * 128 * 4))
    assert sdm.sse_scan_workspace_size(B, T, H, N, k, 128, 128, 0) == rec + chunk(99072)
    assert sdm.sse_scan_workspace_size(B, T, H, N, k, 128, 128, 1) == rec + chunk(148224)
    assert sdm.sse_scan_workspace_size(B, T, H, N, k, 64, 128, 1) == rec     # c != 128: token by token
    assert sdm.sse_scan_workspace_size(1, 63, 1, N, k, 128, 128, 0) == r256(63 * 8 * 4)   # below one chunk
    monkeypatch.setenv("SDM_SSE_PATH", "chunk")
    assert sdm.sse_scan_workspace_size(1, 63, 1, N, k, 128, 128, 0) > r256(63 * 8 * 4)
    monkeypatch.setenv("SDM_SSE_PATH", "recurrent")
    assert sdm.sse_scan_workspace_size(B, T, H, N, k, 128, 128, 0) == rec


# Fake, 256-byte aligned "device" addresses: every call below must return an
# error during host validation, before any CUDA call.
A = 1 << 20
B_ = 2 << 20


def test_address_rejects_bad_arguments(sdm):
    L = sdm.lib()
    assert L.sdm_address(None, A, 1, 1, 1, 8, 4, 4, A, A, None, None) == sdm.SDM_ERR_INVALID_ARG
    assert L.sdm_address(A, A, -1, 1, 1, 8, 4, 4, A, A, None, None) == sdm.SDM_ERR_INVALID_ARG
    assert L.sdm_address(A, A, 1, 1, 1, 8, 9, 4, A, A, None, None) == sdm.SDM_ERR_SHAPE      # k > sqrtN
    assert L.sdm_address(A, A, 1, 1, 1, 8, 4, 17, A, A, None, None) == sdm.SDM_ERR_SHAPE     # W > k^2
    assert L.sdm_address(A, A, 1, 1, 1, 600, 4, 4, A, A, None, None) == sdm.SDM_ERR_SHAPE    # sqrtN > 512
    assert L.sdm_address(A, A, 1, 1, 1, 64, 33, 4, A, A, None, None) == sdm.SDM_ERR_SHAPE    # k > 32
    assert L.sdm_address(A + 2, A, 1, 1, 1, 8, 4, 4, A, A, None, None) == sdm.SDM_ERR_ALIGN
    assert b"sdm_address" in L.sdm_last_error()


def test_scan_rejects_bad_arguments(sdm):
    L = sdm.lib()

    def call(**kw):
        a = dict(state=A, v=A, vdt=1, alpha=A, beta=A, iw=A, ww=A, W=16, ir=A, wr=A, R=16, B=1, T=4, H=1,
                 N=64, dv=16, mode=0, y=A, ws=B_, wsb=1 << 20, err=None)
        a.update(kw)
        return L.sdm_scan(a["state"], a["v"], a["vdt"], a["alpha"], a["beta"], a["iw"], a["ww"], a["W"], a["ir"],
                          a["wr"], a["R"], a["B"], a["T"], a["H"], a["N"], a["dv"], a["mode"], a["y"], a["ws"],
                          a["wsb"], a["err"], None)

    assert call(state=None) == sdm.SDM_ERR_INVALID_ARG
    assert call(W=0) == sdm.SDM_ERR_SHAPE
    assert call(R=65) == sdm.SDM_ERR_SHAPE
    assert call(dv=18) == sdm.SDM_ERR_SHAPE
    assert call(vdt=7) == sdm.SDM_ERR_UNSUPPORTED
    assert call(mode=3) == sdm.SDM_ERR_UNSUPPORTED
    assert call(state=A + 4) == sdm.SDM_ERR_ALIGN
    assert call(v=A + 4) == sdm.SDM_ERR_ALIGN                 # bf16 v needs 8-byte alignment
    assert call(wsb=16) == sdm.SDM_ERR_INVALID_ARG            # workspace too small
    assert call(ws=None) == sdm.SDM_ERR_INVALID_ARG
    assert call(ws=B_ + 8) == sdm.SDM_ERR_ALIGN
    assert b"workspace" in L.sdm_last_error()


def test_binding_fails_loudly_without_cuda_tensors(sdm):
    import torch
    with pytest.raises(TypeError):
        sdm.sdm_address(torch.zeros(1, 1, 1, 8), torch.zeros(1, 1, 1, 8), 4, 4)

"""Shared helpers for the GPU parity tests: device transfer of the seeded
inputs and the tolerance checks.

Tolerances (floating point): max |y - y_ref| <= 2e-3 * RMS(y_ref) over the
whole output, and ||state - state_ref||_F / ||state_ref||_F <= 1e-3.  Index
outputs are compared bit for bit."""
import numpy as np
import pytest
import torch

Y_REL = 2e-3
STATE_REL = 1e-3


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import delta_rule_memory_gb300 as sdm
    sdm.lib()          # raises if libsdm.so is missing: no fallback
    return sdm


def dev(x, bf16: bool = False) -> torch.Tensor:
    """numpy -> CUDA tensor; uint16 arrays (or bf16=True) become bfloat16 bits."""
    x = np.ascontiguousarray(x)
    if bf16 or x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).cuda()
    if x.dtype == np.float64:
        x = x.astype(np.float32)
    return torch.from_numpy(x.copy()).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def assert_y_close(y, y_ref, rel=Y_REL, what="y"):
    y = np.asarray(y, np.float64)
    y_ref = np.asarray(y_ref, np.float64)
    assert y.shape == y_ref.shape
    assert np.all(np.isfinite(y)), f"{what}: non-finite values"
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    err = float(np.max(np.abs(y - y_ref))) if y.size else 0.0
    assert err <= rel * rms + 1e-30, f"{what}: max abs err {err:.3e} > {rel} * RMS {rms:.3e}"
    return err / max(rms, 1e-30)


def assert_state_close(s, s_ref, rel=STATE_REL, what="state"):
    s = np.asarray(s, np.float64)
    s_ref = np.asarray(s_ref, np.float64)
    assert s.shape == s_ref.shape
    assert np.all(np.isfinite(s)), f"{what}: non-finite values"
    ref = float(np.linalg.norm(s_ref))
    diff = float(np.linalg.norm(s - s_ref))
    assert diff <= rel * ref + 1e-30, f"{what}: relative Frobenius error {diff / max(ref, 1e-30):.3e} > {rel}"
    return diff / max(ref, 1e-30)

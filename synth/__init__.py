"""Seeded synthetic inputs for the delta-rule memory scans.

This module is shared by the CPU oracle tests and the CUDA path's tests and
benchmark.  It only draws random numbers and shapes them into the workload
recipes (distributions, dtypes, sizes); it holds none of the scan's own
arithmetic.  Every draw comes from a ``torch.Generator`` seeded explicitly, in
fp32, in a fixed tensor order; casts to bf16 happen after the draw.

bf16 tensors are returned as ``numpy.uint16`` arrays holding the raw bit
patterns (round-to-nearest-even from fp32), so both the oracle and the CUDA
path read exactly the same bits.

Workloads (sizes from the Sparse Delta Memory deck, "Head count controls a
cubic state expansion", Eq. 6, and the scan configurations built on it):

* ``sdm``  - product-key score halves, values, forget/input gates.
* ``gdn``  - dense Gated DeltaNet / KDA inputs (q, k L2-normalised).
* ``sse``  - Sparse State Expansion router logits, key logits, q, v, decay.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

__all__ = [
    "SdmShape", "GdnShape", "SseShape",
    "SDM_TINY", "SDM_14B_LAYER", "sdm_sweep_shape", "GDN_DENSE", "SSE_PART",
    "sdm_inputs", "gdn_inputs", "sse_inputs", "to_bf16_bits", "bf16_bits_to_f32",
    "sdm_layer_sizes",
]


def to_bf16_bits(x: torch.Tensor) -> np.ndarray:
    """fp32 tensor -> uint16 array of bf16 bits (round to nearest even)."""
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> exact float32 values."""
    return (b.astype(np.uint32) << 16).view(np.float32)


def sdm_layer_sizes(d: int, H: int) -> dict:
    """Slot count, value width and per-layer table size for model width d and
    H heads: N = (d/4H)^2, d_v = d/H, H*N*d_v = d^3/(16 H^2) (SDM deck, Eq. 6)."""
    assert d % (4 * H) == 0
    sqrt_n = d // (4 * H)
    n = sqrt_n * sqrt_n
    d_v = d // H
    return {"sqrtN": sqrt_n, "N": n, "d_v": d_v, "elements": H * n * d_v}


@dataclasses.dataclass(frozen=True)
class SdmShape:
    name: str
    B: int
    T: int
    H: int
    sqrtN: int
    d_v: int
    k: int
    W: int
    R: int
    v_bf16: bool

    @property
    def N(self) -> int:
        return self.sqrtN * self.sqrtN

    def with_(self, **kw) -> "SdmShape":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class GdnShape:
    name: str
    B: int
    T: int
    H: int
    dk: int
    dv: int

    def with_(self, **kw) -> "GdnShape":
        return dataclasses.replace(self, **kw)


@dataclasses.dataclass(frozen=True)
class SseShape:
    name: str
    B: int
    T: int
    H: int
    N: int       # routed partitions (one more, shared, is always active)
    topk: int
    c: int       # rows per partition
    d: int       # value width

    def with_(self, **kw) -> "SseShape":
        return dataclasses.replace(self, **kw)


# Tiny SDM scan: N = 64 slots, d_v = 16, fp32 values.
SDM_TINY = SdmShape("sdm_tiny", B=1, T=128, H=1, sqrtN=8, d_v=16, k=4, W=4, R=4, v_bf16=False)
# SDM 1.4B-layer shape: d = 1920, H = 2 -> N = 57600, d_v = 960.
SDM_14B_LAYER = SdmShape("sdm_1.4b_layer", B=8, T=4096, H=2, sqrtN=240, d_v=960, k=16, W=16, R=16,
                         v_bf16=True)


def sdm_sweep_shape(H: int, d: int = 1920, B: int = 8, T: int = 8192) -> SdmShape:
    """State-scaling sweep at model width d: N = (d/4H)^2, d_v = d/H."""
    s = sdm_layer_sizes(d, H)
    return SdmShape(f"sdm_sweep_H{H}", B=B, T=T, H=H, sqrtN=s["sqrtN"], d_v=s["d_v"], k=16, W=16, R=16,
                    v_bf16=True)


GDN_DENSE = GdnShape("gdn_dense", B=4, T=4096, H=16, dk=128, dv=128)
SSE_PART = SseShape("sse_partitions", B=4, T=4096, H=8, N=8, topk=2, c=128, d=128)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(seed)
    return g


def sdm_inputs(shape: SdmShape, seed: int = 0) -> dict:
    """Draw, in this order: write halves s1w, s2w, read halves s1r, s2r
    (N(0,1), [B,T,H,sqrtN]); v (N(0,1), [B,T,H,d_v], bf16 bits if v_bf16);
    alpha = sigmoid(N(3,1)) and beta = sigmoid(N(0,1)), both [B,T,H]."""
    g = _gen(seed)
    B, T, H, s, dv = shape.B, shape.T, shape.H, shape.sqrtN, shape.d_v
    out = {}
    for name in ("s1w", "s2w", "s1r", "s2r"):
        out[name] = torch.randn((B, T, H, s), generator=g, dtype=torch.float32).numpy()
    v = torch.randn((B, T, H, dv), generator=g, dtype=torch.float32)
    out["v"] = to_bf16_bits(v) if shape.v_bf16 else v.numpy()
    out["v_bf16"] = shape.v_bf16
    out["alpha"] = torch.sigmoid(torch.randn((B, T, H), generator=g) + 3.0).numpy()
    out["beta"] = torch.sigmoid(torch.randn((B, T, H), generator=g)).numpy()
    return out


def gdn_inputs(shape: GdnShape, seed: int = 0) -> dict:
    """Draw q, k, v (N(0,1), [B,T,H,d]); q and k L2-normalised per head in
    fp32, then all three cast to bf16 bits.  alpha_gdn = exp(-softplus(N(0,1)))
    [B,T,H]; alpha_kda the same recipe per key channel [B,T,H,dk];
    beta = sigmoid(N(0,1)) [B,T,H]; then the GDN2 gates b_erase =
    sigmoid(N(0,1)) [B,T,H,dk] and w_write = sigmoid(N(0,1)) [B,T,H,dv] (both
    in (0,1), drawn after everything else so the earlier tensors keep their
    values)."""
    g = _gen(seed)
    B, T, H, dk, dv = shape.B, shape.T, shape.H, shape.dk, shape.dv
    q = torch.randn((B, T, H, dk), generator=g)
    k = torch.randn((B, T, H, dk), generator=g)
    v = torch.randn((B, T, H, dv), generator=g)
    q = q / q.norm(dim=-1, keepdim=True)
    k = k / k.norm(dim=-1, keepdim=True)
    a_gdn = torch.exp(-torch.nn.functional.softplus(torch.randn((B, T, H), generator=g)))
    a_kda = torch.exp(-torch.nn.functional.softplus(torch.randn((B, T, H, dk), generator=g)))
    beta = torch.sigmoid(torch.randn((B, T, H), generator=g))
    b_erase = torch.sigmoid(torch.randn((B, T, H, dk), generator=g))
    w_write = torch.sigmoid(torch.randn((B, T, H, dv), generator=g))
    return {"q": to_bf16_bits(q), "k": to_bf16_bits(k), "v": to_bf16_bits(v),
            "alpha_gdn": a_gdn.numpy(), "alpha_kda": a_kda.numpy(), "beta": beta.numpy(),
            "b_erase": b_erase.numpy(), "w_write": w_write.numpy()}


def sse_inputs(shape: SseShape, seed: int = 0) -> dict:
    """Draw router logits (N(0,1), [B,T,H,N]), key logits (N(0,1), [B,T,H,c]),
    q ([B,T,H,c]) and v ([B,T,H,d]) as N(0,1) cast to bf16 bits, and the
    per-row decay alpha = sigmoid(N(3,1)) [B,T,H,c]."""
    g = _gen(seed)
    B, T, H, N, c, d = shape.B, shape.T, shape.H, shape.N, shape.c, shape.d
    route = torch.randn((B, T, H, N), generator=g)
    klog = torch.randn((B, T, H, c), generator=g)
    q = torch.randn((B, T, H, c), generator=g)
    v = torch.randn((B, T, H, d), generator=g)
    alpha = torch.sigmoid(torch.randn((B, T, H, c), generator=g) + 3.0)
    return {"route": route.numpy(), "klog": klog.numpy(), "q": to_bf16_bits(q), "v": to_bf16_bits(v),
            "alpha": alpha.numpy()}


def random_state(shape_tuple, seed: int, scale: float = 1.0) -> np.ndarray:
    """A nonzero fp32 initial state ~ scale * N(0,1) (for invariant tests)."""
    g = _gen(seed)
    return (torch.randn(shape_tuple, generator=g) * scale).numpy()


def dyadic_scores(shape_tuple, seed: int) -> np.ndarray:
    """fp32 scores that are multiples of 2^-10 in [-8, 8]: any sum of two is
    exact in fp32, so no rounding ties can occur."""
    g = _gen(seed)
    ints = torch.randint(-8 * 1024, 8 * 1024 + 1, shape_tuple, generator=g)
    return (ints.to(torch.float64) / 1024.0).to(torch.float32).numpy()


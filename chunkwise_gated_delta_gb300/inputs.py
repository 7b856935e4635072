"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module holds no arithmetic of the method: it only draws random tensors
with the shapes and distributions of the workloads and casts them to the
storage dtype.  Both the CUDA path and the CPU oracle receive the same cast
values (the oracle upcasts them to float64).

Draws come from a CPU ``torch.Generator`` seeded with ``seed`` in a fixed
order -- q, k, v, beta logits, g logits, h0, then (backward workloads only) the
output gradient dO and the final-state gradient dht, then (DPLR only) a, the
noise for a', the cosines and the eta logits -- all in float64 before the cast.

Distributions (one per workload family):

* q, k ~ N(0, 1), then L2-normalised per token and head;
* v ~ N(0, 1);
* beta = sigmoid(N(0, 1)) per token and head;
* g = -softplus(N(0, 1)) * 0.1 per channel (KDA, GLA, DPLR) or one value per
  token and head (GDN); absent for DeltaNet;
* h0 ~ 0.1 N(0, 1) in float32 when requested;
* backward: dO ~ N(0, 1) in the storage dtype, dht ~ N(0, 1) in float32;
* DPLR: a unit; a' unit with cos(a, a') ~ U[0.9, 1]; b = eta a' with
  eta = 2 sigmoid(N(0, 1)).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import torch

VARIANTS = ("kda", "gdn", "deltanet", "gla", "dplr")


@dataclass(frozen=True)
class Workload:
    name: str
    variant: str
    B: int
    T: int
    H: int
    dk: int
    dv: int
    dtype: torch.dtype
    h0: bool
    chunk: int = 64
    grads: bool = False        # backward workload: also draw dO and dht

    @property
    def tokens(self) -> int:
        return self.B * self.T

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The workloads: a small fp32 KDA case, the KDA throughput case, the
# special-case sweep, the general DPLR case and the KDA backward case.
WORKLOADS = {
    "kda_fp32_b1t256h1d64": Workload("kda_fp32_b1t256h1d64", "kda", 1, 256, 1, 64, 64, torch.float32, False),
    "kda_bf16_b4t4096h16d128": Workload("kda_bf16_b4t4096h16d128", "kda", 4, 4096, 16, 128, 128, torch.bfloat16, True),
    "gdn_bf16_b8t2048h32d128": Workload("gdn_bf16_b8t2048h32d128", "gdn", 8, 2048, 32, 128, 128, torch.bfloat16, False),
    "deltanet_bf16_b8t2048h32d128": Workload("deltanet_bf16_b8t2048h32d128", "deltanet", 8, 2048, 32, 128, 128, torch.bfloat16, False),
    "gla_bf16_b8t2048h32d128": Workload("gla_bf16_b8t2048h32d128", "gla", 8, 2048, 32, 128, 128, torch.bfloat16, False),
    "dplr_bf16_b2t8192h16d128": Workload("dplr_bf16_b2t8192h16d128", "dplr", 2, 8192, 16, 128, 128, torch.bfloat16, False),
    "kda_bwd_bf16_b4t4096h16d128": Workload("kda_bwd_bf16_b4t4096h16d128", "kda", 4, 4096, 16, 128, 128,
                                            torch.bfloat16, True, grads=True),
    "dplr_bwd_bf16_b2t8192h16d128": Workload("dplr_bwd_bf16_b2t8192h16d128", "dplr", 2, 8192, 16, 128, 128,
                                             torch.bfloat16, False, grads=True),
}


def _l2n(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True)


def make_inputs(w: Workload, seed: int = 0) -> dict:
    """Draw the inputs of workload ``w`` on the CPU.

    Returns a dict of CPU tensors in the storage dtype: q, k, v and, depending
    on the variant, g, beta, a, b and h0 (float32).  ``scale_v`` tells whether
    beta scales v (KDA, GDN, DeltaNet) or not (GLA, DPLR).
    """
    if w.variant not in VARIANTS:
        raise ValueError(f"unknown variant {w.variant}")
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    f64 = dict(generator=gen, dtype=torch.float64)
    B, T, H, dk, dv = w.B, w.T, w.H, w.dk, w.dv

    q = _l2n(torch.randn(B, T, H, dk, **f64))
    k = _l2n(torch.randn(B, T, H, dk, **f64))
    v = torch.randn(B, T, H, dv, **f64)
    beta_logits = torch.randn(B, T, H, **f64)
    gshape = (B, T, H) if w.variant == "gdn" else (B, T, H, dk)
    g_logits = torch.randn(*gshape, **f64)
    h0 = (0.1 * torch.randn(B, H, dv, dk, **f64)) if w.h0 else None
    if w.grads:
        do = torch.randn(B, T, H, dv, **f64)
        dht = torch.randn(B, H, dv, dk, **f64)

    out = {"q": q, "k": k, "v": v}
    if w.variant in ("kda", "gdn", "deltanet"):
        out["beta"] = torch.sigmoid(beta_logits)
        out["scale_v"] = True
    else:
        out["scale_v"] = False
    if w.variant != "deltanet":
        out["g"] = -torch.nn.functional.softplus(g_logits) * 0.1
    if w.variant == "dplr":
        a = _l2n(torch.randn(B, T, H, dk, **f64))
        noise = torch.randn(B, T, H, dk, **f64)
        cos = 0.9 + 0.1 * torch.rand(B, T, H, 1, **f64)
        eta = 2.0 * torch.sigmoid(torch.randn(B, T, H, 1, **f64))
        ortho = _l2n(noise - (noise * a).sum(-1, keepdim=True) * a)
        a_prime = cos * a + torch.sqrt(1.0 - cos * cos) * ortho
        out["a"] = a
        out["b"] = eta * a_prime
        out["eta"] = eta[..., 0]
        out["a_prime"] = a_prime

    if w.grads:
        out["do"] = do
        out["dht"] = dht.to(torch.float32)
    for key in ("q", "k", "v", "g", "beta", "a", "b", "do"):
        if key in out:
            out[key] = out[key].to(w.dtype)
    if h0 is not None:
        out["h0"] = h0.to(torch.float32)
    return out


def custom(variant: str, B: int, T: int, H: int, dk: int, dv: int,
           dtype=torch.bfloat16, h0: bool = False, grads: bool = False) -> Workload:
    """A workload of arbitrary shape with the distributions above (tests)."""
    return Workload(f"{variant}_custom", variant, B, T, H, dk, dv, dtype, h0, grads=grads)

"""DPLR backward and the eq. (7) gate clip, CUDA (through the C ABI) vs the float64 oracle.

The oracle differentiates the token recurrence (``oracle.dplr_bwd``), with the
clip of page "How to make GDN2 more stable", eq. (7), applied before it when
asked (``clip=True``).  Tolerances (relative Frobenius norm per tensor): 1e-5
for float32 inputs, 5e-3 for bfloat16 inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from chunkwise_gated_delta_gb300 import dplr_chunk_bwd, dplr_chunk_fwd, dplr_factor_norms
from chunkwise_gated_delta_gb300.inputs import WORKLOADS, custom, make_inputs

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 5e-3}
DEV = "cuda:0"


def rel(x, ref):
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


def f64(t):
    return None if t is None else t.double().numpy()


def _inputs(dtype, B, T, H, dk, dv, seed=0, gate="channel", eta_scale=1.0, h0=True):
    x = make_inputs(custom("dplr", B, T, H, dk, dv, dtype=dtype, h0=h0, grads=True), seed=seed)
    if eta_scale != 1.0:
        x["b"] = (x["b"].double() * eta_scale).to(dtype)
    if gate == "none":
        x.pop("g")
    elif gate == "scalar":
        x["g"] = x["g"][..., 0].contiguous()
    return x


def _oracle_gate(x):
    g = f64(x.get("g"))
    if g is None:
        return np.zeros(x["q"].shape)
    return np.repeat(g[..., None], x["q"].shape[-1], axis=-1) if g.ndim == 3 else g


def run_bwd(x, gate, clip):
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    out = dplr_chunk_bwd(d["q"], d["k"], d["v"], d["a"], d["b"], d.get("g"), d.get("h0"), d["do"], d["dht"],
                         gate=gate, clip=clip)
    torch.cuda.synchronize()
    return {k: v.double().cpu().numpy() for k, v in out.items()}


def oracle_bwd(x, clip, heads=None):
    ref = oracle.dplr_bwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["a"]), f64(x["b"]), _oracle_gate(x),
                          f64(x["do"]), h0=f64(x.get("h0")), dht=f64(x["dht"]), clip=clip, heads=heads)
    g = x.get("g")
    if g is None:
        ref.pop("dg")
    elif g.dim() == 3:
        ref["dg"] = ref["dg"].sum(-1)
    return ref


def compare(got, ref, tol, heads=None):
    errs = {}
    for key, r in ref.items():
        g = got[key]
        if heads is not None:
            if key == "dh0":
                g, r = np.stack([g[b, h] for b, h in heads]), np.stack([r[b, h] for b, h in heads])
            else:
                g, r = np.stack([g[b, :, h] for b, h in heads]), np.stack([r[b, :, h] for b, h in heads])
        errs[key] = rel(g, r)
    bad = {k: f"{e:.2e}" for k, e in errs.items() if not e <= tol}
    assert not bad, f"over {tol}: {bad} (all: { {k: f'{e:.1e}' for k, e in errs.items()} })"
    return errs


def check(dtype, B, T, H, dk, dv, seed=0, gate="channel", clip=False, eta_scale=1.0, h0=True):
    x = _inputs(dtype, B, T, H, dk, dv, seed, gate, eta_scale, h0)
    compare(run_bwd(x, gate, clip), oracle_bwd(x, clip), TOL[dtype])


# ---------------------------------------------------------------- the clip in the forward
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_clipped_forward(dtype):
    x = _inputs(dtype, 2, 150, 2, 128, 128, seed=3, eta_scale=1.5)
    d = {k: v.to(DEV) for k, v in x.items() if isinstance(v, torch.Tensor)}
    o, ht = dplr_chunk_fwd(d["q"], d["k"], d["v"], d["a"], d["b"], d["g"], d["h0"], clip=True)
    torch.cuda.synchronize()
    ro, rh = oracle.dplr_fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["a"]), f64(x["b"]), f64(x["g"]),
                             f64(x["h0"]), clip=True)
    assert rel(o.double().cpu().numpy(), ro) <= TOL[dtype] and rel(ht.double().cpu().numpy(), rh) <= TOL[dtype]
    # the clip changed the result
    r_unclipped, _ = oracle.dplr_fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["a"]), f64(x["b"]),
                                     f64(x["g"]), f64(x["h0"]))
    assert rel(r_unclipped, ro) > 1e-3


def test_clipped_factor_norms_at_most_one():
    """With the clip every step's exact factor norm is at most 1 (eq. (7) bounds it by rho / rho)."""
    x = make_inputs(WORKLOADS["dplr_bf16_b2t8192h16d128"], seed=0)
    d = {k: v.to(DEV) for k, v in x.items() if isinstance(v, torch.Tensor)}
    _, nrm0, mx0 = dplr_factor_norms(d["a"], d["b"], d["g"])
    _, nrm, mx = dplr_factor_norms(d["a"], d["b"], d["g"], clip=True)
    torch.cuda.synchronize()
    assert float(mx0[1]) > 1.0
    assert float(mx[1]) <= 1.0 + 2e-5
    assert bool((nrm <= nrm0 + 1e-6).all())


# ---------------------------------------------------------------- backward, float32
@pytest.mark.parametrize("T", [1, 15, 16, 17, 70])
def test_fp32_lengths(T):
    check(torch.float32, 1, T, 2, 64, 64)


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64)])
def test_fp32_dims(dk, dv):
    check(torch.float32, 2, 50, 2, dk, dv)


@pytest.mark.parametrize("gate", ["scalar", "none"])
def test_fp32_gate_kinds(gate):
    check(torch.float32, 1, 60, 2, 64, 64, gate=gate)


@pytest.mark.parametrize("gate", ["channel", "scalar", "none"])
def test_fp32_clip(gate):
    check(torch.float32, 1, 90, 2, 64, 64, gate=gate, clip=True, eta_scale=1.5, seed=2)


def test_fp32_no_h0():
    check(torch.float32, 1, 40, 2, 64, 64, h0=False)


# ---------------------------------------------------------------- backward, bfloat16
@pytest.mark.parametrize("clip", [False, True])
def test_bf16(clip):
    check(torch.bfloat16, 2, 200, 2, 128, 128, clip=clip, seed=4)


def test_full_dplr_bwd_b2t8192h16d128_every_head():
    w = WORKLOADS["dplr_bwd_bf16_b2t8192h16d128"]
    x = make_inputs(w, seed=0)
    got = run_bwd(x, "channel", False)
    for v in got.values():
        assert np.isfinite(v).all()
    ref = oracle_bwd(x, False)
    worst = {}
    for b in range(w.B):
        for h in range(w.H):
            errs = compare(got, ref, 5e-3, heads=[(b, h)])
            for k, e in errs.items():
                worst[k] = max(worst.get(k, 0.0), e)
    print("parity: dplr_bwd_bf16_b2t8192h16d128 worst head per gradient:",
          {k: f"{e:.3e}" for k, e in worst.items()})


# ---------------------------------------------------------------- packed variable-length batches
@pytest.mark.parametrize("dtype,clip", [(torch.float32, False), (torch.float32, True), (torch.bfloat16, False)])
def test_packed_sequences(dtype, clip):
    """cu_seqlens: ragged lengths below, at and above a 16-token chunk, an empty sequence and a
    one-token one, against the oracle's backward of each sequence alone (an empty sequence's dh0
    is its dht)."""
    lens, H, dk, dv = [40, 16, 0, 1, 70, 17], 2, 128, 64
    parts = [_inputs(dtype, 1, max(n, 1), H, dk, dv, seed=40 + i, eta_scale=1.5 if clip else 1.0)
             for i, n in enumerate(lens)]
    rows = ("q", "k", "v", "a", "b", "g", "do")
    x = {name: torch.cat([p_[name][:, :n] for p_, n in zip(parts, lens)], 1).contiguous() for name in rows}
    for name in ("h0", "dht"):
        x[name] = torch.cat([p_[name] for p_ in parts], 0).contiguous()
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=DEV)
    d = {k: v.to(DEV) for k, v in x.items()}
    out = dplr_chunk_bwd(d["q"], d["k"], d["v"], d["a"], d["b"], d["g"], d["h0"], d["do"], d["dht"],
                         gate="channel", clip=clip, cu_seqlens=cu)
    torch.cuda.synchronize()
    got = {k: v.double().cpu().numpy() for k, v in out.items()}
    starts = np.concatenate([[0], np.cumsum(lens)])
    for i, (p_, n) in enumerate(zip(parts, lens)):
        if n == 0:
            assert rel(got["dh0"][i], f64(p_["dht"])[0]) <= 1e-6, i
            continue
        sub = {name: (p_[name][:, :n] if name in rows else p_[name]) for name in p_}
        mine = {k: (v[i:i + 1] if k == "dh0" else v[:, starts[i]:starts[i + 1]]) for k, v in got.items()}
        compare(mine, oracle_bwd(sub, clip), TOL[dtype])

"""Backward of the chunkwise gated delta rule, CUDA (through the C ABI) vs the float64 oracle.

The oracle is the reverse mode of the token recurrence (``oracle.recurrence_bwd``),
for L = <dO, o> + <dht, ht>.  Every gradient (dq, dk, dv, dg, dbeta, dh0) is
compared by relative Frobenius norm: 1e-5 for float32 inputs; 5e-3 for
bfloat16 inputs (float32 arithmetic, gradients rounded to bf16 on store).
"""
import numpy as np
import pytest
import torch

import oracle
from chunkwise_gated_delta_gb300 import kda_chunk_bwd
from chunkwise_gated_delta_gb300.inputs import WORKLOADS, custom, make_inputs

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 5e-3}
DEV = "cuda:0"
GATE = {"kda": "channel", "gla": "channel", "gdn": "scalar", "deltanet": "none"}


def rel(x, ref):
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


def f64(t):
    return None if t is None else t.double().numpy()


def run_gpu(x, variant, with_dht=True):
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    out = kda_chunk_bwd(d["q"], d["k"], d["v"], d.get("g"), d.get("beta"), d.get("h0"), d["do"],
                        d["dht"] if with_dht else None, gate=GATE[variant], scale_v=x["scale_v"])
    torch.cuda.synchronize()
    return {k: v.double().cpu().numpy() for k, v in out.items()}


def run_oracle(x, variant, with_dht=True, heads=None):
    kw = dict(h0=f64(x.get("h0")), dht=f64(x["dht"]) if with_dht else None, heads=heads)
    q, k, v, do = f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["do"])
    if variant == "kda":
        return oracle.kda_bwd(q, k, v, f64(x["g"]), f64(x["beta"]), do, **kw)
    if variant == "gdn":
        return oracle.gdn_bwd(q, k, v, f64(x["g"]), f64(x["beta"]), do, **kw)
    if variant == "deltanet":
        return oracle.deltanet_bwd(q, k, v, f64(x["beta"]), do, **kw)
    return oracle.gla_bwd(q, k, v, f64(x["g"]), do, **kw)


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


def check(variant, dtype, B, T, H, dk, dv, h0=True, seed=0, with_dht=True):
    x = make_inputs(custom(variant, B, T, H, dk, dv, dtype=dtype, h0=h0, grads=True), seed=seed)
    got = run_gpu(x, variant, with_dht)
    ref = run_oracle(x, variant, with_dht)
    return compare(got, ref, TOL[dtype])


# ---------------------------------------------------------------- float32
@pytest.mark.parametrize("T", [1, 31, 32, 33, 100, 256])
def test_fp32_kda_lengths(T):
    check("kda", torch.float32, 1, T, 2, 64, 64)


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_fp32_kda_dims(dk, dv):
    check("kda", torch.float32, 2, 90, 2, dk, dv)


@pytest.mark.parametrize("variant", ["gdn", "deltanet", "gla"])
def test_fp32_special_cases(variant):
    check(variant, torch.float32, 1, 130, 2, 64, 64)


def test_fp32_no_h0_no_dht():
    check("kda", torch.float32, 1, 97, 2, 64, 64, h0=False, with_dht=False)


# ---------------------------------------------------------------- bfloat16
@pytest.mark.parametrize("T", [1, 64, 65, 300])
def test_bf16_kda_lengths(T):
    check("kda", torch.bfloat16, 1, T, 2, 128, 128)


@pytest.mark.parametrize("variant", ["gdn", "deltanet", "gla"])
def test_bf16_special_cases(variant):
    check(variant, torch.bfloat16, 2, 200, 2, 128, 128)


def test_bf16_deterministic():
    x = make_inputs(custom("kda", 2, 150, 2, 128, 128, dtype=torch.bfloat16, h0=True, grads=True), seed=5)
    a, b = run_gpu(x, "kda"), run_gpu(x, "kda")
    for key in a:
        assert np.array_equal(a[key], b[key]), key


def test_full_kda_bwd_b4t4096h16d128_every_head():
    """The backward workload B4 T4096 H16 d128 bf16: every gradient of every (batch, head) pair."""
    w = WORKLOADS["kda_bwd_bf16_b4t4096h16d128"]
    x = make_inputs(w, seed=0)
    got = run_gpu(x, "kda")
    for v in got.values():
        assert np.isfinite(v).all()
    ref = run_oracle(x, "kda")
    worst = {}
    for b in range(w.B):
        for h in range(w.H):
            errs = compare(got, ref, 5e-3, heads=[(b, h)])
            for k, e in errs.items():
                worst[k] = max(worst.get(k, 0.0), e)
    print("parity: kda_bwd_bf16_b4t4096h16d128 worst head per gradient:",
          {k: f"{e:.3e}" for k, e in worst.items()})


# ---------------------------------------------------------------- packed variable-length batches
def _packed_bwd(variant, dtype, lens, dk, dv, seed=20):
    """Sequences of the given lengths packed into one [1, T, H, d] batch: the packed backward
    against the oracle's backward of each sequence on its own (an empty sequence's dh0 is its dht)."""
    H = 2
    parts = [make_inputs(custom(variant, 1, max(n, 1), H, dk, dv, dtype=dtype, h0=True, grads=True),
                         seed=seed + i) for i, n in enumerate(lens)]
    rows = ("q", "k", "v", "g", "beta", "do")
    x = {name: torch.cat([p_[name][:, :n] for p_, n in zip(parts, lens)], 1).contiguous()
         for name in rows if name in parts[0]}
    for name in ("h0", "dht"):
        x[name] = torch.cat([p_[name] for p_ in parts], 0).contiguous()
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=DEV)
    d = {k_: v_.to(DEV) for k_, v_ in x.items()}
    out = kda_chunk_bwd(d["q"], d["k"], d["v"], d.get("g"), d.get("beta"), d["h0"], d["do"], d["dht"],
                        gate=GATE[variant], scale_v=parts[0]["scale_v"], cu_seqlens=cu)
    torch.cuda.synchronize()
    got = {k_: v_.double().cpu().numpy() for k_, v_ in out.items()}
    starts = np.concatenate([[0], np.cumsum(lens)])
    worst = {}
    for i, (p_, n) in enumerate(zip(parts, lens)):
        if n == 0:
            assert rel(got["dh0"][i], f64(p_["dht"])[0]) <= 1e-6, i
            continue
        sub = {name: (p_[name][:, :n] if name in rows else p_[name]) for name in p_ if name != "scale_v"}
        sub["scale_v"] = p_["scale_v"]
        ref = run_oracle(sub, variant)
        mine = {k_: (v_[i:i + 1] if k_ == "dh0" else v_[:, starts[i]:starts[i + 1]]) for k_, v_ in got.items()}
        for k_, e in compare(mine, ref, TOL[dtype]).items():
            worst[k_] = max(worst.get(k_, 0.0), e)
    return worst


@pytest.mark.parametrize("dtype,dk,dv", [(torch.float32, 64, 64), (torch.bfloat16, 128, 128),
                                         (torch.bfloat16, 128, 64)])
def test_packed_kda_bwd(dtype, dk, dv):
    """cu_seqlens: ragged lengths below, at and above a 32-token chunk, an empty sequence and a
    one-token one; no gradient crosses a boundary."""
    _packed_bwd("kda", dtype, [100, 32, 0, 1, 193, 37], dk, dv)


@pytest.mark.parametrize("variant", ["gdn", "deltanet", "gla"])
def test_packed_special_cases_bwd(variant):
    _packed_bwd(variant, torch.bfloat16, [70, 0, 130, 33], 128, 128)


def test_packed_bwd_equals_dense_on_equal_lengths():
    """Equal lengths packed with cu_seqlens give the same gradients as the dense [B, T] batch
    (bit for bit: the same chunks, products and sums in the same order)."""
    x = make_inputs(custom("kda", 3, 96, 2, 128, 128, dtype=torch.bfloat16, h0=True, grads=True), seed=23)
    d = {k_: (v_.to(DEV) if isinstance(v_, torch.Tensor) else v_) for k_, v_ in x.items()}
    dense = kda_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], d["do"], d["dht"], gate="channel")
    flat = {k_: d[k_].reshape(1, -1, *d[k_].shape[2:]).contiguous() for k_ in ("q", "k", "v", "g", "beta", "do")}
    cu = torch.tensor([0, 96, 192, 288], dtype=torch.int32, device=DEV)
    packed = kda_chunk_bwd(flat["q"], flat["k"], flat["v"], flat["g"], flat["beta"], d["h0"], flat["do"],
                           d["dht"], gate="channel", cu_seqlens=cu)
    torch.cuda.synchronize()
    for key, t in dense.items():
        assert torch.equal(packed[key].reshape(t.shape), t), key

"""General gated DPLR forward and the transition-norm report, CUDA vs the float64 oracle.

The forward follows page "Diagonal Plus Low Rank", section 2 (token recurrence
S_t = S_{t-1} Diag(alpha_t)(I - b_t a_t^T) + v_t k_t^T, o_t = S_t q_t); the
norms follow page "How to make GDN2 more stable", eqs. (4) and (12).

Tolerances (relative Frobenius norm on o and on the final state): 1e-5 for
float32 inputs, 5e-3 for bfloat16 inputs (float32 arithmetic, o rounded to
bf16).  rho is a closed form evaluated in float32: 1e-5 relative per token.
The factor norm comes from float32 bisection on eigenvalue counts of the
factor's Gram matrix: within 2e-5 relative of numpy's SVD of the same factor.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import spectral
from chunkwise_gated_delta_gb300 import dplr_chunk_fwd, dplr_factor_norms
from chunkwise_gated_delta_gb300.inputs import WORKLOADS, custom, make_inputs

pytestmark = pytest.mark.gpu

TOL = {torch.float32: 1e-5, torch.bfloat16: 5e-3}
DEV = "cuda:0"


def rel(x, ref):
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-300))


def f64(t):
    return None if t is None else t.double().numpy()


def run_gpu(x, gate="channel"):
    d = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in x.items()}
    o, ht = dplr_chunk_fwd(d["q"], d["k"], d["v"], d["a"], d["b"], d.get("g"), d.get("h0"), gate=gate)
    torch.cuda.synchronize()
    return o.double().cpu().numpy(), ht.double().cpu().numpy()


def run_oracle(x, heads=None):
    g = f64(x.get("g"))
    if g is not None and g.ndim == 3:            # scalar gate: broadcast over the key channels
        g = np.repeat(g[..., None], x["q"].shape[-1], axis=-1)
    if g is None:
        g = np.zeros(x["q"].shape)
    return oracle.dplr_fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["a"]), f64(x["b"]), g,
                           h0=f64(x.get("h0")), heads=heads)


def check(dtype, B, T, H, dk, dv, h0, seed=0, gate="channel"):
    x = make_inputs(custom("dplr", B, T, H, dk, dv, dtype=dtype, h0=h0), seed=seed)
    if gate == "none":
        x.pop("g")
    elif gate == "scalar":
        x["g"] = x["g"][..., 0].contiguous()
    o, ht = run_gpu(x, gate)
    ro, rh = run_oracle(x)
    eo, eh = rel(o, ro), rel(ht, rh)
    assert eo <= TOL[dtype] and eh <= TOL[dtype], f"o {eo:.3e} ht {eh:.3e}"


# ---------------------------------------------------------------- forward, float32
@pytest.mark.parametrize("T", [1, 31, 32, 33, 100, 256])
def test_fp32_lengths(T):
    check(torch.float32, 1, T, 2, 64, 64, h0=True)


@pytest.mark.parametrize("dk,dv", [(64, 64), (128, 128), (64, 128), (128, 64), (128, 32), (64, 256)])
def test_fp32_dims(dk, dv):
    check(torch.float32, 2, 90, 2, dk, dv, h0=True)


@pytest.mark.parametrize("gate", ["scalar", "none"])
def test_fp32_gate_kinds(gate):
    check(torch.float32, 1, 130, 2, 64, 64, h0=True, gate=gate)


def test_fp32_kda_mapping():
    """a = k, b = beta k and v scaled by beta: the DPLR call computes KDA."""
    x = make_inputs(custom("kda", 1, 200, 2, 64, 64, dtype=torch.float32, h0=True), seed=6)
    beta = x["beta"].double()[..., None]
    y = dict(q=x["q"], k=x["k"], v=(x["v"].double() * beta).float(), a=x["k"],
             b=(x["k"].double() * beta).float(), g=x["g"], h0=x["h0"])
    o, ht = run_gpu(y)
    ro, rh = oracle.kda_fwd(f64(x["q"]), f64(x["k"]), f64(x["v"]), f64(x["g"]), f64(x["beta"]),
                            h0=f64(x["h0"]))
    # v and b were rounded to float32 after the beta scaling: compare at 1e-5
    assert rel(o, ro) <= 1e-5 and rel(ht, rh) <= 1e-5


# ---------------------------------------------------------------- forward, bfloat16 inputs
@pytest.mark.parametrize("T", [1, 63, 64, 65, 300])
def test_bf16_lengths(T):
    check(torch.bfloat16, 1, T, 2, 128, 128, h0=True)


@pytest.mark.parametrize("seed", [0, 1])
def test_bf16_seeds(seed):
    check(torch.bfloat16, 2, 700, 2, 128, 128, h0=False, seed=seed)


def test_bf16_chaining_matches_one_call():
    x = make_inputs(custom("dplr", 1, 400, 2, 128, 128, dtype=torch.bfloat16, h0=True), seed=4)
    d = {k: v.to(DEV) for k, v in x.items() if isinstance(v, torch.Tensor) and v.dim() == 4}
    h0 = x["h0"].to(DEV)
    names = ("q", "k", "v", "a", "b", "g")
    sl = lambda t, a, b: t[:, a:b].contiguous()
    o1, h1 = dplr_chunk_fwd(*(sl(d[n], 0, 200) for n in names), h0)
    o2, h2 = dplr_chunk_fwd(*(sl(d[n], 200, 400) for n in names), h1)
    torch.cuda.synchronize()
    ro, rh = run_oracle(x)
    oc = torch.cat([o1, o2], 1).double().cpu().numpy()
    assert rel(oc, ro) <= 5e-3 and rel(h2.double().cpu().numpy(), rh) <= 5e-3


def test_deterministic():
    x = make_inputs(custom("dplr", 2, 300, 2, 128, 128, dtype=torch.bfloat16, h0=True), seed=5)
    a, b = run_gpu(x), run_gpu(x)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_full_dplr_b2t8192h16d128_every_head():
    w = WORKLOADS["dplr_bf16_b2t8192h16d128"]
    x = make_inputs(w, seed=0)
    o, ht = run_gpu(x)
    assert np.isfinite(o).all() and np.isfinite(ht).all()
    ro, rh = run_oracle(x)
    eo = np.array([[rel(o[b, :, h], ro[b, :, h]) for h in range(w.H)] for b in range(w.B)])
    eh = np.array([[rel(ht[b, h], rh[b, h]) for h in range(w.H)] for b in range(w.B)])
    summary = f"dplr_bf16_b2t8192h16d128: worst head o {eo.max():.3e}, ht {eh.max():.3e}"
    print("parity:", summary)
    assert eo.max() <= 5e-3 and eh.max() <= 5e-3, summary


# ---------------------------------------------------------------- transition norms
def _norm_inputs(x):
    a, b = f64(x["a"]), f64(x["b"])
    na, nb = np.linalg.norm(a, axis=-1), np.linalg.norm(b, axis=-1)
    eta = na * nb
    c = (a * b).sum(-1) / eta
    return a, b, eta, c


def _check_norms(x, sample):
    d = {k: v.to(DEV) for k, v in x.items() if isinstance(v, torch.Tensor)}
    rho, nrm, mx = dplr_factor_norms(d["a"], d["b"], d["g"])
    torch.cuda.synchronize()
    rho, nrm, mx = rho.double().cpu().numpy(), nrm.double().cpu().numpy(), mx.double().cpu().numpy()
    a, b, eta, c = _norm_inputs(x)
    r_ref = spectral.rho_closed_form(eta, c)
    assert np.max(np.abs(rho - r_ref) / r_ref) <= 1e-5
    alpha = np.exp(f64(x["g"]))
    idx = tuple(np.asarray(ix) for ix in zip(*sample))
    exact = spectral.factor_norm_exact(alpha[idx], a[idx], b[idx])
    ratio = nrm[idx] / exact
    assert np.abs(ratio - 1).max() <= 2e-5, (ratio.min(), ratio.max())
    assert mx[0] == rho.max() and mx[1] == nrm.max()
    return rho, nrm, mx


def test_factor_norms_small():
    x = make_inputs(custom("dplr", 2, 100, 3, 128, 128, dtype=torch.float32), seed=2)
    rng = np.random.default_rng(0)
    sample = [(rng.integers(2), rng.integers(100), rng.integers(3)) for _ in range(64)]
    _check_norms(x, sample)


def test_factor_norms_dk64_scalar_gate_values():
    """Scalar gate: ||alpha (I - b a^T)|| = alpha rho exactly (eq. (4) scaled)."""
    x = make_inputs(custom("dplr", 1, 50, 2, 64, 64, dtype=torch.float32), seed=3)
    g = x["g"][..., 0].contiguous()
    d = {k: v.to(DEV) for k, v in x.items() if isinstance(v, torch.Tensor)}
    rho, nrm, _ = dplr_factor_norms(d["a"], d["b"], g.to(DEV))
    torch.cuda.synchronize()
    alpha = np.exp(f64(g))
    assert np.max(np.abs(nrm.double().cpu().numpy() / (alpha * rho.double().cpu().numpy()) - 1)) <= 2e-5


def test_factor_norms_full_workload():
    """The norm report of the DPLR workload B2 T8192 H16 d128: max rho > 1 and max factor norm > 1."""
    x = make_inputs(WORKLOADS["dplr_bf16_b2t8192h16d128"], seed=0)
    rng = np.random.default_rng(1)
    sample = [(rng.integers(2), rng.integers(8192), rng.integers(16)) for _ in range(32)]
    rho, nrm, mx = _check_norms(x, sample)
    assert mx[0] > 1.0 and mx[1] > 1.0


# ---------------------------------------------------------------- packed variable-length batches
@pytest.mark.parametrize("dtype,dk,dv", [(torch.float32, 64, 64), (torch.bfloat16, 128, 128)])
def test_packed_sequences(dtype, dk, dv):
    """cu_seqlens: ragged lengths below, at and above a 32-token chunk, an empty sequence and a
    one-token one, against the oracle on each sequence alone; no state crosses a boundary."""
    lens, H = [100, 32, 0, 1, 193, 37], 2
    parts = [make_inputs(custom("dplr", 1, max(n, 1), H, dk, dv, dtype=dtype, h0=True), seed=30 + i)
             for i, n in enumerate(lens)]
    rows = ("q", "k", "v", "a", "b", "g")
    x = {name: torch.cat([p_[name][:, :n] for p_, n in zip(parts, lens)], 1).contiguous() for name in rows}
    x["h0"] = torch.cat([p_["h0"] for p_ in parts], 0).contiguous()
    cu = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device=DEV)
    d = {k: v.to(DEV) for k, v in x.items()}
    o, ht = dplr_chunk_fwd(d["q"], d["k"], d["v"], d["a"], d["b"], d["g"], d["h0"], cu_seqlens=cu)
    torch.cuda.synchronize()
    o, ht = o.double().cpu().numpy(), ht.double().cpu().numpy()
    starts = np.concatenate([[0], np.cumsum(lens)])
    for i, (p_, n) in enumerate(zip(parts, lens)):
        if n == 0:
            assert np.array_equal(ht[i], f64(p_["h0"])[0]), i
            continue
        ro, rh = run_oracle({name: (p_[name][:, :n] if name in rows else p_[name]) for name in p_})
        assert rel(o[:, starts[i]:starts[i + 1]], ro) <= TOL[dtype], i
        assert rel(ht[i], rh[0]) <= TOL[dtype], i


"""Pins of the float64 oracle's reverse mode (``oracle.recurrence_bwd``).

The backward oracle is checked against things that are not itself:

* central finite differences of the forward oracle, entry by entry, on every
  input at T = 64 and on sampled entries across several checkpoint segments;
* the chunk backward of page "Kimi Delta Attention backward", restated in
  numpy (``chunk_forms.kda_chunk_bwd_form``) for several chunk sizes;
* the closed-form gradients of the GLA parallel form (page "Gated Linear
  Attention", section 6.3) when beta = 0;
* the DPLR chunk backward of page "Diagonal Plus Low Rank", section 3,
  restated in numpy (``chunk_forms.dplr_chunk_bwd_form``, with its readings);
* the eq. (7) clip of page "How to make GDN2 more stable": after it every
  factor norm (numpy SVD) is at most 1, eq. (6)'s KDA case is left alone, and
  the clip's chain rule agrees with central differences;
* and mutated copies of the reverse mode (a dropped term, a wrong sign, the
  gate gradient taken against the wrong state) fail the finite-difference pin.
"""
import numpy as np
import pytest

import oracle
from chunk_forms import gla_parallel_grads, kda_chunk_bwd_form

rng = np.random.default_rng


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _case(seed, B=1, T=64, H=1, dk=8, dv=8, scalar_gate=False):
    r = rng(seed)
    x = dict(
        q=_unit(r.standard_normal((B, T, H, dk))),
        k=_unit(r.standard_normal((B, T, H, dk))),
        v=r.standard_normal((B, T, H, dv)),
        beta=1 / (1 + np.exp(-r.standard_normal((B, T, H)))),
        g=-np.log1p(np.exp(r.standard_normal((B, T, H) if scalar_gate else (B, T, H, dk)))) * 0.1,
        h0=0.1 * r.standard_normal((B, H, dv, dk)),
        a=_unit(r.standard_normal((B, T, H, dk))),
    )
    x["b"] = (0.5 + r.random((B, T, H, 1))) * _unit(x["a"] + 0.3 * r.standard_normal((B, T, H, dk)))
    do = r.standard_normal((B, T, H, dv))
    dht = r.standard_normal((B, H, dv, dk))
    return x, do, dht


VARIANTS = {
    # name: (input names, forward, backward, gradient names)
    "kda": (("q", "k", "v", "g", "beta", "h0"),
            lambda x: oracle.kda_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], threads=1),
            lambda x, do, dht: oracle.kda_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], do, x["h0"], dht)),
    "gdn": (("q", "k", "v", "g", "beta", "h0"),
            lambda x: oracle.gdn_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], threads=1),
            lambda x, do, dht: oracle.gdn_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], do, x["h0"], dht)),
    "deltanet": (("q", "k", "v", "beta", "h0"),
                 lambda x: oracle.deltanet_fwd(x["q"], x["k"], x["v"], x["beta"], x["h0"], threads=1),
                 lambda x, do, dht: oracle.deltanet_bwd(x["q"], x["k"], x["v"], x["beta"], do, x["h0"], dht)),
    "gla": (("q", "k", "v", "g", "h0"),
            lambda x: oracle.gla_fwd(x["q"], x["k"], x["v"], x["g"], x["h0"], threads=1),
            lambda x, do, dht: oracle.gla_bwd(x["q"], x["k"], x["v"], x["g"], do, x["h0"], dht)),
    "dplr": (("q", "k", "v", "a", "b", "g", "h0"),
             lambda x: oracle.dplr_fwd(x["q"], x["k"], x["v"], x["a"], x["b"], x["g"], x["h0"], threads=1),
             lambda x, do, dht: oracle.dplr_bwd(x["q"], x["k"], x["v"], x["a"], x["b"], x["g"], do, x["h0"], dht)),
}


def _loss(fwd, x, do, dht):
    o, ht = fwd(x)
    return float((o * do).sum() + (ht * dht).sum())


def _fd(fwd, x, do, dht, name, idx, eps=1e-6):
    xp = {n: a.copy() for n, a in x.items()}
    xm = {n: a.copy() for n, a in x.items()}
    xp[name][idx] += eps
    xm[name][idx] -= eps
    return (_loss(fwd, xp, do, dht) - _loss(fwd, xm, do, dht)) / (2 * eps)


def _grad_key(name):
    return "dh0" if name == "h0" else "d" + name


@pytest.mark.parametrize("variant", list(VARIANTS))
def test_finite_differences_every_entry_t64(variant):
    """Every gradient entry equals a central difference of the forward oracle (T = 64)."""
    names, fwd, bwd = VARIANTS[variant]
    x, do, dht = _case(1, T=64, dk=6, dv=5, scalar_gate=(variant == "gdn"))
    grads = bwd(x, do, dht)
    for name in names:
        fd = np.zeros_like(x[name])
        for idx in np.ndindex(*x[name].shape):
            fd[idx] = _fd(fwd, x, do, dht, name, idx)
        got = grads[_grad_key(name)]
        err = np.linalg.norm(got - fd) / np.linalg.norm(fd)
        assert err <= 2e-7, f"{variant} d{name}: {err:.2e}"


def test_finite_differences_across_segments():
    """T = 200 spans four checkpoint segments of the reverse sweep: sampled entries vs central differences."""
    names, fwd, bwd = VARIANTS["kda"]
    x, do, dht = _case(2, B=2, T=200, H=2, dk=6, dv=5)
    grads = bwd(x, do, dht)
    r = rng(3)
    for name in names:
        for _ in range(12):
            idx = tuple(int(r.integers(s)) for s in x[name].shape)
            fd = _fd(fwd, x, do, dht, name, idx)
            assert abs(grads[_grad_key(name)][idx] - fd) <= 1e-6 * max(1.0, abs(fd)), (name, idx)


@pytest.mark.parametrize("C", [16, 32, 64])
@pytest.mark.parametrize("variant", ["kda", "deltanet", "gla"])
def test_chunk_backward_of_the_page_equals_reverse_mode(C, variant):
    """The page's chunk backward (restated in numpy) equals the token reverse mode."""
    x, do, dht = _case(4, T=150, dk=8, dv=6)
    q, k, v, g, beta, h0 = (x[n][0, :, 0] if n != "h0" else x[n][0, 0] for n in ("q", "k", "v", "g", "beta", "h0"))
    dO, dHt = do[0, :, 0], dht[0, 0]
    if variant == "deltanet":
        g = np.zeros_like(g)
    scale_v = variant != "gla"
    if variant == "gla":
        beta = np.zeros_like(beta)
    ref = kda_chunk_bwd_form(q, k, v, g, beta, dO, h0, dHt, C=C, scale_v=scale_v)
    if variant == "kda":
        got = oracle.kda_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], do, x["h0"], dht)
    elif variant == "deltanet":
        got = oracle.deltanet_bwd(x["q"], x["k"], x["v"], x["beta"], do, x["h0"], dht)
    else:
        got = oracle.gla_bwd(x["q"], x["k"], x["v"], x["g"], do, x["h0"], dht)
    keys = ["dq", "dk", "dv", "dh0"] + (["dg"] if variant != "deltanet" else []) + \
        (["dbeta"] if variant != "gla" else [])
    for key in keys:
        g_ = got[key][0, :, 0] if key != "dh0" else got[key][0, 0]
        np.testing.assert_allclose(g_, ref[key], rtol=1e-9, atol=1e-11, err_msg=key)


def test_gla_parallel_closed_form_gradients():
    """beta = 0: reverse mode equals the closed-form gradients of the GLA parallel form."""
    x, do, _ = _case(5, T=90, dk=7, dv=4)
    got = oracle.gla_bwd(x["q"], x["k"], x["v"], x["g"], do)
    dq, dk, dv, dg = gla_parallel_grads(x["q"][0, :, 0], x["k"][0, :, 0], x["v"][0, :, 0], x["g"][0, :, 0],
                                        do[0, :, 0])
    for key, ref in (("dq", dq), ("dk", dk), ("dv", dv), ("dg", dg)):
        np.testing.assert_allclose(got[key][0, :, 0], ref, rtol=1e-10, atol=1e-12, err_msg=key)


def test_gdn_gate_gradient_is_channel_sum():
    """A scalar gate's gradient is the sum over channels of the per-channel gradient at equal decays."""
    x, do, dht = _case(6, T=70, scalar_gate=True)
    got = oracle.gdn_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], do, x["h0"], dht)
    gch = np.repeat(x["g"][..., None], x["q"].shape[-1], axis=-1)
    ch = oracle.kda_bwd(x["q"], x["k"], x["v"], gch, x["beta"], do, x["h0"], dht)
    np.testing.assert_allclose(got["dg"], ch["dg"].sum(-1), rtol=1e-11, atol=1e-13)
    for key in ("dq", "dk", "dv", "dbeta", "dh0"):
        np.testing.assert_allclose(got[key], ch[key], rtol=1e-11, atol=1e-13)


def test_heads_subset_matches_full():
    x, do, dht = _case(7, B=2, T=80, H=3)
    full = oracle.kda_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], do, x["h0"], dht)
    part = oracle.kda_bwd(x["q"], x["k"], x["v"], x["g"], x["beta"], do, x["h0"], dht, heads=[(1, 2)])
    for key in ("dq", "dk", "dv", "dg", "dbeta"):
        np.testing.assert_array_equal(part[key][1, :, 2], full[key][1, :, 2])
    np.testing.assert_array_equal(part["dh0"][1, 2], full["dh0"][1, 2])


# --------------------------------------------------------------------------
# the finite-difference pin rejects plausible mistakes in a reverse mode
# --------------------------------------------------------------------------
def _mutant_bwd(q, k, v, g, beta, h0, do, dht, mode):
    """A Python copy of the KDA token reverse mode (one head) with one planted mistake."""
    T, dk = q.shape
    states = [h0.copy()]
    for t in range(T):
        al = np.exp(g[t])
        Sa = states[-1] * al[None, :]
        states.append(Sa - np.outer(Sa @ (beta[t] * k[t]), k[t]) + np.outer(beta[t] * v[t], k[t]))
    dS = dht.copy()
    out = {n: np.zeros_like(a) for n, a in (("dq", q), ("dk", k), ("dv", v), ("dg", g), ("dbeta", beta))}
    for t in reversed(range(T)):
        al, bt, vv = np.exp(g[t]), beta[t] * k[t], beta[t] * v[t]
        Sp, St = states[t], states[t + 1]
        dS = dS + np.outer(do[t], q[t])
        out["dq"][t] = St.T @ do[t]
        Sa = Sp * al[None, :]
        y = Sa @ bt
        dvv = dS @ k[t]
        dy = -dS @ k[t]
        da = -dS.T @ y
        dSa = dS + np.outer(dy, bt) if mode != "drop_dy_b" else dS
        db = Sa.T @ dy
        if mode == "sign_da":
            da = -da
        dal = (dSa * (St if mode == "gate_vs_new_state" else Sp)).sum(0)
        out["dg"][t] = al * dal
        out["dk"][t] = dS.T @ vv + da + beta[t] * db
        out["dv"][t] = beta[t] * dvv
        out["dbeta"][t] = db @ k[t] + dvv @ v[t]
        dS = dSa * al[None, :]
    out["dh0"] = dS
    return out


@pytest.mark.parametrize("mode", ["drop_dy_b", "sign_da", "gate_vs_new_state"])
def test_fd_pin_catches_planted_mistakes(mode):
    names, fwd, bwd = VARIANTS["kda"]
    x, do, dht = _case(8, T=24, dk=5, dv=4)
    one = lambda n: x[n][0, :, 0] if n != "h0" else x[n][0, 0]
    args = [one(n) for n in ("q", "k", "v", "g", "beta", "h0")] + [do[0, :, 0], dht[0, 0]]
    ok = _mutant_bwd(*args, mode="none")
    ref = bwd(x, do, dht)
    for key in ("dq", "dk", "dv", "dg", "dbeta"):
        np.testing.assert_allclose(ok[key], ref[key][0, :, 0], rtol=1e-10, atol=1e-12)
    bad = _mutant_bwd(*args, mode=mode)
    worst = 0.0
    for name in ("k", "g"):
        for idx in np.ndindex(*x[name].shape):
            fd = _fd(fwd, x, do, dht, name, idx)
            worst = max(worst, abs(bad[_grad_key(name)][idx[1]][idx[3]] - fd))
    assert worst > 1e-4


# --------------------------------------------------------------------------
# DPLR: the page's chunk backward and the eq. (7) clip
# --------------------------------------------------------------------------
@pytest.mark.parametrize("C", [16, 32, 64])
def test_dplr_chunk_backward_of_the_page_equals_reverse_mode(C):
    from chunk_forms import dplr_chunk_bwd_form
    x, do, dht = _case(9, T=150, dk=8, dv=6)
    one = lambda n: x[n][0, :, 0]
    ref = dplr_chunk_bwd_form(one("q"), one("k"), one("v"), one("a"), one("b"), one("g"), do[0, :, 0],
                              x["h0"][0, 0], dht[0, 0], C=C)
    got = oracle.dplr_bwd(x["q"], x["k"], x["v"], x["a"], x["b"], x["g"], do, x["h0"], dht)
    for key in ("dq", "dk", "dv", "da", "db", "dg", "dh0"):
        g_ = got[key][0, :, 0] if key != "dh0" else got[key][0, 0]
        np.testing.assert_allclose(g_, ref[key], rtol=1e-9, atol=1e-11, err_msg=key)


def test_clip_bounds_every_factor_norm_by_one():
    """Eq. (7): after g -> min(g, -log rho) every ||Diag(alpha)(I - b a^T)||_2 <= 1 (numpy SVD)."""
    x, _, _ = _case(10, T=50, dk=8)
    a, b = x["a"][0, :, 0], 1.6 * x["b"][0, :, 0]
    g = x["g"][0, :, 0] * 0.2                      # weak decay: the unclipped factors exceed 1
    before = oracle.factor_norm_exact(np.exp(g), a, b)
    after = oracle.factor_norm_exact(np.exp(oracle.clip_gate(g, a, b)), a, b)
    assert before.max() > 1.05
    assert after.max() <= 1 + 1e-12


def test_clip_leaves_kda_mapping_and_small_channels_alone():
    """Eq. (6): a = k unit, b = beta k with beta <= 2 gives rho = 1, so the clip changes nothing;
    in general only channels above -log rho change."""
    x, _, _ = _case(11, T=40, dk=8)
    k, beta, g = x["k"][0, :, 0], x["beta"][0, :, 0], x["g"][0, :, 0]
    np.testing.assert_array_equal(oracle.clip_gate(g, k, 2 * beta[:, None] * k), g)
    a, b = x["a"][0, :, 0], x["b"][0, :, 0]
    gc = oracle.clip_gate(g, a, b)
    lim = -np.log(oracle.rho_of(a, b))[:, None]
    np.testing.assert_array_equal(gc[g <= lim], g[g <= lim])
    assert np.all(gc[g > lim] == np.broadcast_to(lim, g.shape)[g > lim])


def test_dplr_clip_backward_finite_differences():
    """dplr_bwd(clip=True) against central differences of dplr_fwd(clip=True) on every entry."""
    x, do, dht = _case(12, T=40, dk=5, dv=4)
    x["b"] = 1.5 * x["b"]                          # rho well above 1 on many tokens: the clip is active
    names = ("q", "k", "v", "a", "b", "g", "h0")
    fwd = lambda y: oracle.dplr_fwd(y["q"], y["k"], y["v"], y["a"], y["b"], y["g"], y["h0"], clip=True, threads=1)
    grads = oracle.dplr_bwd(x["q"], x["k"], x["v"], x["a"], x["b"], x["g"], do, x["h0"], dht, clip=True)
    gc = oracle.clip_gate(x["g"], x["a"], x["b"])
    assert (gc < x["g"]).mean() > 0.2               # the clip acts on a good share of the channels
    for name in names:
        fd = np.zeros_like(x[name])
        for idx in np.ndindex(*x[name].shape):
            fd[idx] = _fd(fwd, x, do, dht, name, idx)
        err = np.linalg.norm(grads[_grad_key(name)] - fd) / np.linalg.norm(fd)
        assert err <= 1e-6, f"d{name}: {err:.2e}"

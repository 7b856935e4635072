"""Pins of the float64 oracle against facts the pages and mathematics fix.

Each test checks the token-recurrence oracle (or a spectral-norm routine)
against something that is not the oracle itself: a closed form, a
hand-derived worked example, an invariant of the delta rule, or an
independent derivation (the pages' chunk forms).  A plausible slip in the
oracle -- a dropped beta, a decay applied after the rank-one term instead of
before, a transposed state, a wrong sign -- fails at least one of them
(``test_pins_catch_planted_mistakes`` checks that on mutated copies).
"""
import math
import os

import numpy as np
import pytest

import oracle
from chunk_forms import dplr_chunk_form, dplr_wy_product, kda_chunk_form, kda_record_form

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng = np.random.default_rng


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _rand(seed, B=1, T=37, H=2, dk=8, dv=6):
    r = rng(seed)
    q = _unit(r.standard_normal((B, T, H, dk)))
    k = _unit(r.standard_normal((B, T, H, dk)))
    v = r.standard_normal((B, T, H, dv))
    beta = 1 / (1 + np.exp(-r.standard_normal((B, T, H))))
    g = -np.log1p(np.exp(r.standard_normal((B, T, H, dk)))) * 0.1
    h0 = 0.1 * r.standard_normal((B, H, dv, dk))
    return q, k, v, beta, g, h0


def _read_golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            key, rest = line.split(":")
            vals[key.strip()] = np.array([float(x) for x in rest.split()])
    return vals


# --------------------------------------------------------------------------
# worked example (hand-derived from the definition)
# --------------------------------------------------------------------------
def test_tiny_worked_example():
    gv = _read_golden("tiny_kda_worked.txt")
    k = gv["k"].reshape(1, 2, 1, 2)
    q = gv["q"].reshape(1, 2, 1, 2)
    v = gv["v"].reshape(1, 2, 1, 2)
    beta = gv["beta"].reshape(1, 2, 1)
    g = np.log(gv["alpha"]).reshape(1, 2, 1, 2)
    h0 = gv["h0"].reshape(1, 1, 2, 2)
    o, ht = oracle.kda_fwd(q, k, v, g, beta, h0)
    np.testing.assert_allclose(o.reshape(-1), gv["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(ht.reshape(-1), gv["ht"], rtol=0, atol=1e-14)


# --------------------------------------------------------------------------
# closed forms for the special cases
# --------------------------------------------------------------------------
def test_linear_attention_closed_form():
    """g = 0, beta = 0, vv = v: O = (Q K^T * M) V + Q h0^T (GLA page, 3.2-3.3)."""
    q, k, v, _, _, h0 = _rand(1, B=2, T=29, H=3)
    o, ht = oracle.recurrence(q, k, v, g=None, beta=None, scale_v=False, h0=h0)
    T = q.shape[1]
    M = np.tril(np.ones((T, T)))
    for b in range(q.shape[0]):
        for h in range(q.shape[2]):
            Q, K, V = q[b, :, h], k[b, :, h], v[b, :, h]
            ref = ((Q @ K.T) * M) @ V + Q @ h0[b, h].T
            np.testing.assert_allclose(o[b, :, h], ref, rtol=0, atol=1e-12)
            np.testing.assert_allclose(ht[b, h], h0[b, h] + V.T @ K, rtol=0, atol=1e-12)


def test_gla_parallel_closed_form():
    """beta = 0, vv = v, per-channel decay (GLA page, 5.1 recurrence, 5.2 chunk form).

    o_t = sum_{i<=t} v_i sum_j k_ij q_tj exp(G_tj - G_ij) + h0 Diag(exp(G_t)) q_t,
    G the inclusive running sum of g from the sequence start.
    """
    q, k, v, _, g, h0 = _rand(2, B=1, T=23, H=2)
    o, ht = oracle.gla_fwd(q, k, v, g, h0=h0)
    T = q.shape[1]
    for h in range(q.shape[2]):
        Q, K, V, G = q[0, :, h], k[0, :, h], v[0, :, h], np.cumsum(g[0, :, h], axis=0)
        decay = np.exp(G[:, None, :] - G[None, :, :])            # [t, i, j]
        scores = np.einsum("tj,ij,tij->ti", Q, K, decay) * np.tril(np.ones((T, T)))
        ref = scores @ V + np.einsum("vj,tj->tv", h0[0, h], Q * np.exp(G))
        np.testing.assert_allclose(o[0, :, h], ref, rtol=0, atol=1e-12)
        ref_ht = h0[0, h] * np.exp(G[-1]) + V.T @ (K * np.exp(G[-1] - G))
        np.testing.assert_allclose(ht[0, h], ref_ht, rtol=0, atol=1e-12)


def test_delta_rule_write():
    """Delta rule: for unit k_t, S_t k_t = (1 - beta_t) S_{t-1} Diag(alpha_t) k_t + beta_t v_t.

    Follows from (I - beta k k^T) k = (1 - beta) k (DeltaNet page, 4.1) and
    fixes both that beta scales v and that Diag(alpha) acts before the
    rank-one correction.  With q = k the output o_t is S_t k_t.
    """
    q, k, v, beta, g, h0 = _rand(3, B=1, T=17, H=1)
    o, _ = oracle.kda_fwd(k, k, v, g, beta, h0)
    for t in (0, 1, 5, 16):
        if t == 0:
            Sprev = h0[0, 0]
        else:
            _, hp = oracle.kda_fwd(k[:, :t], k[:, :t], v[:, :t], g[:, :t], beta[:, :t], h0)
            Sprev = hp[0, 0]
        kt = k[0, t, 0]
        ref = (1 - beta[0, t, 0]) * (Sprev * np.exp(g[0, t, 0])[None, :]) @ kt + beta[0, t, 0] * v[0, t, 0]
        np.testing.assert_allclose(o[0, t, 0], ref, rtol=0, atol=1e-12)


def test_deltanet_beta_one_memorises():
    """beta = 1, alpha = 1, orthonormal keys: S k_i = v_i for every written key."""
    d = 8
    r = rng(4)
    Qm, _ = np.linalg.qr(r.standard_normal((d, d)))
    k = Qm.T[None, :, None, :]                    # T = d orthonormal keys
    v = r.standard_normal((1, d, 1, 5))
    _, ht = oracle.deltanet_fwd(k, k, v, np.ones((1, d, 1)))
    np.testing.assert_allclose(ht[0, 0] @ Qm, v[0, :, 0].T, rtol=0, atol=1e-12)


def test_gdn_scalar_equals_broadcast_channel():
    """GDN's scalar decay equals a per-channel decay with equal channels (GDN2 page eq. (1), D = gamma I)."""
    q, k, v, beta, g, h0 = _rand(5, B=1, T=19, H=2)
    gs = g[..., 0]
    o1, h1 = oracle.gdn_fwd(q, k, v, gs, beta, h0)
    o2, h2 = oracle.kda_fwd(q, k, v, np.repeat(gs[..., None], q.shape[-1], -1), beta, h0)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-14)
    np.testing.assert_allclose(h1, h2, rtol=0, atol=1e-14)


def test_kda_is_dplr_with_mapping():
    """KDA = DPLR with a = k, b = beta k, v = beta v' (DPLR page, relation to KDA)."""
    q, k, v, beta, g, h0 = _rand(6, B=1, T=21, H=2)
    o1, h1 = oracle.kda_fwd(q, k, v, g, beta, h0)
    o2, h2 = oracle.dplr_fwd(q, k, beta[..., None] * v, k, beta[..., None] * k, g, h0)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(h1, h2, rtol=0, atol=1e-13)


# --------------------------------------------------------------------------
# the pages' chunk forms equal the recurrence, for every chunk size
# --------------------------------------------------------------------------
@pytest.mark.parametrize("C", [1, 16, 32, 64])
def test_kda_chunk_form_equals_recurrence(C):
    q, k, v, beta, g, h0 = _rand(7, B=1, T=130, H=2, dk=16, dv=12)
    o, ht = oracle.kda_fwd(q, k, v, g, beta, h0)
    for h in range(2):
        oc, Sc = kda_chunk_form(q[0, :, h], k[0, :, h], v[0, :, h], g[0, :, h],
                                beta[0, :, h], h0[0, h], C=C)
        scale = np.abs(o[0, :, h]).max()
        np.testing.assert_allclose(oc, o[0, :, h], rtol=0, atol=1e-12 * scale)
        np.testing.assert_allclose(Sc, ht[0, h], rtol=0, atol=1e-12 * np.abs(ht).max())


@pytest.mark.parametrize("C,blk", [(64, 16), (64, 8), (32, 16), (16, 16)])
@pytest.mark.parametrize("variant", ["kda", "gdn", "deltanet", "gla"])
def test_record_form_equals_recurrence(C, blk, variant):
    """The regrouped products of the tensor-core kernels ([L ; P], the block back-substitution
    of Z'(I + L) = [I ; P], A = [-W ; Q<- - P W], D1 = Z V + A S^T = [V_new ; O]) reach the
    recurrence's result: the regrouping is exact, whatever the chunk and block sizes."""
    q, k, v, beta, g, h0 = _rand(11, B=1, T=150, H=2, dk=16, dv=12)
    scale_v = True
    if variant == "kda":
        o, ht = oracle.kda_fwd(q, k, v, g, beta, h0)
    elif variant == "gdn":
        o, ht = oracle.gdn_fwd(q, k, v, g[..., 0], beta, h0)
        g = np.repeat(g[..., :1], g.shape[-1], axis=-1)
    elif variant == "deltanet":
        o, ht = oracle.deltanet_fwd(q, k, v, beta, h0)
        g = np.zeros_like(g)
    else:
        o, ht = oracle.gla_fwd(q, k, v, g, h0)
        beta = np.zeros_like(beta)
        scale_v = False
    for h in range(2):
        oc, Sc = kda_record_form(q[0, :, h], k[0, :, h], v[0, :, h], g[0, :, h], beta[0, :, h], h0[0, h],
                                 C=C, blk=blk, scale_v=scale_v)
        np.testing.assert_allclose(oc, o[0, :, h], rtol=0, atol=1e-12 * np.abs(o).max())
        np.testing.assert_allclose(Sc, ht[0, h], rtol=0, atol=1e-12 * np.abs(ht).max())


@pytest.mark.parametrize("C", [16, 64])
def test_gla_chunk_form_equals_recurrence(C):
    """beta = 0 with vv = v: the KDA chunk form collapses to GLA's (GLA page 5.2)."""
    q, k, v, _, g, h0 = _rand(8, B=1, T=100, H=1, dk=8, dv=8)
    o, ht = oracle.gla_fwd(q, k, v, g, h0)
    oc, Sc = kda_chunk_form(q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], None,
                            h0[0, 0], C=C, scale_v=False)
    np.testing.assert_allclose(oc, o[0, :, 0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(Sc, ht[0, 0], rtol=0, atol=1e-12)


@pytest.mark.parametrize("C", [8, 64])
def test_dplr_chunk_form_equals_recurrence(C):
    r = rng(9)
    q, k, v, _, g, h0 = _rand(9, B=1, T=90, H=1, dk=12, dv=10)
    a = _unit(r.standard_normal((1, 90, 1, 12)))
    b = 0.8 * _unit(a + 0.3 * r.standard_normal((1, 90, 1, 12)))
    o, ht = oracle.dplr_fwd(q, k, v, a, b, g, h0)
    oc, Sc = dplr_chunk_form(q[0, :, 0], k[0, :, 0], v[0, :, 0], a[0, :, 0], b[0, :, 0],
                             g[0, :, 0], h0[0, 0], C=C)
    np.testing.assert_allclose(oc, o[0, :, 0], rtol=0, atol=1e-11)
    np.testing.assert_allclose(Sc, ht[0, 0], rtol=0, atol=1e-11)


def test_wy_product_equals_bruteforce():
    """P^C from the w recursion equals the explicit product of C factors (DPLR page, section 2)."""
    r = rng(10)
    C, d = 12, 6
    a = _unit(r.standard_normal((C, d)))
    b = 0.9 * _unit(r.standard_normal((C, d)))
    alpha = np.exp(-0.2 * r.random((C, d)))
    P = np.eye(d)
    for i in range(C):
        P = P @ np.diag(alpha[i]) @ (np.eye(d) - np.outer(b[i], a[i]))
    np.testing.assert_allclose(dplr_wy_product(a, b, alpha), P, rtol=0, atol=1e-13)
    # and the oracle's state transition is that product: with v = 0, ht = h0 P
    h0 = r.standard_normal((1, 1, 4, d))
    z = np.zeros((1, C, 1, d))
    _, ht = oracle.dplr_fwd(z, z, np.zeros((1, C, 1, 4)), a[None, :, None], b[None, :, None],
                            np.log(alpha)[None, :, None], h0)
    np.testing.assert_allclose(ht[0, 0], h0[0, 0] @ P, rtol=0, atol=1e-13)


# --------------------------------------------------------------------------
# state chaining (resume) and threading
# --------------------------------------------------------------------------
def test_h0_chaining_equals_one_call():
    q, k, v, beta, g, h0 = _rand(11, B=2, T=50, H=2)
    o, ht = oracle.kda_fwd(q, k, v, g, beta, h0)
    o1, h1 = oracle.kda_fwd(q[:, :21], k[:, :21], v[:, :21], g[:, :21], beta[:, :21], h0)
    o2, h2 = oracle.kda_fwd(q[:, 21:], k[:, 21:], v[:, 21:], g[:, 21:], beta[:, 21:], h1)
    np.testing.assert_allclose(np.concatenate([o1, o2], 1), o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(h2, ht, rtol=0, atol=1e-13)


def test_heads_subset_and_threads_agree():
    q, k, v, beta, g, h0 = _rand(12, B=2, T=30, H=3)
    o, ht = oracle.kda_fwd(q, k, v, g, beta, h0, threads=1)
    o4, ht4 = oracle.kda_fwd(q, k, v, g, beta, h0, threads=4)
    np.testing.assert_array_equal(o, o4)
    np.testing.assert_array_equal(ht, ht4)
    os_, hs = oracle.kda_fwd(q, k, v, g, beta, h0, heads=[(1, 2)])
    np.testing.assert_array_equal(os_[1, :, 2], o[1, :, 2])
    np.testing.assert_array_equal(hs[1, 2], ht[1, 2])


# --------------------------------------------------------------------------
# spectral norm closed form (GDN2 page)
# --------------------------------------------------------------------------
def test_spectral_golden_points():
    rows = []
    with open(os.path.join(GOLDEN, "spectral_norm_points.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append([float(x) for x in line.split()])
    rows = np.array(rows)
    np.testing.assert_allclose(oracle.rho_closed_form(rows[:, 0], rows[:, 1]), rows[:, 2],
                               rtol=0, atol=1e-14)


def test_spectral_closed_form_matches_svd():
    """Eq. (4) against numpy's SVD of the explicit matrix I - eta k j^T."""
    r = rng(13)
    for d in (2, 3, 8, 64):
        for _ in range(20):
            kk, jj = _unit(r.standard_normal(d)), _unit(r.standard_normal(d))
            eta = 3 * r.random()
            m = np.eye(d) - eta * np.outer(kk, jj)
            ref = np.linalg.svd(m, compute_uv=False)[0]
            assert abs(oracle.rho_closed_form(eta, kk @ jj) - ref) < 1e-12


def test_spectral_bounds_eq5_eq6():
    """Eq. (5): for c < 1 and eta > 0, rho > max(eta, 2) - 1 >= 1.  Eq. (6): rho <= 1 iff c = 1 and eta <= 2, or eta = 0."""
    etas = np.linspace(0, 4, 81)
    for c in np.linspace(-1, 0.999, 50):
        rho = oracle.rho_closed_form(etas[1:], c)
        assert np.all(rho > np.maximum(etas[1:], 2) - 1)
        assert np.all(rho > 1)
    rho1 = oracle.rho_closed_form(etas, 1.0)
    np.testing.assert_allclose(rho1, np.maximum(etas, 2) - 1, atol=1e-12)
    assert np.all((rho1 <= 1 + 1e-12) == (etas <= 2))
    assert oracle.rho_closed_form(0.0, 0.3) == 1.0


def test_factor_norm_exact():
    """Diag(alpha) = I reduces the factor to I - b a^T, whose norm is eq. (4); eq. (9) gives the same 2x2 core."""
    r = rng(14)
    d = 16
    a = _unit(r.standard_normal((5, d)))
    kk = _unit(r.standard_normal((5, d)))
    eta = 2 * r.random(5)
    c = np.einsum("ij,ij->i", kk, a)
    got = oracle.factor_norm_exact(np.ones((5, d)), a, eta[:, None] * kk)
    np.testing.assert_allclose(got, oracle.rho_closed_form(eta, c), atol=1e-12)
    for e, cc in zip(eta, c):
        Bm = np.array([[1 - e * cc, 0.0], [-e * math.sqrt(1 - cc * cc), 1.0]])
        assert abs(np.linalg.svd(Bm, compute_uv=False)[0] - oracle.rho_closed_form(e, cc)) < 1e-12
    # a contracting diagonal can only shrink the norm
    alpha = np.exp(-r.random((5, d)))
    assert np.all(oracle.factor_norm_exact(alpha, a, eta[:, None] * kk) <= got + 1e-12)


# --------------------------------------------------------------------------
# the unit-lower-triangular inverse (DeltaNet page, 4.2)
# --------------------------------------------------------------------------
def test_neumann_doubling_and_block_inverse():
    """(I + L)^{-1} = sum_{n<N} (-L)^n; its doubling S_{k+1} = S_k (I + G_k), G_{k+1} = G_k^2;
    block form 2: B_ij = -A_ii^{-1} sum_{k=j}^{i-1} A_ik B_kj.  (The page prints the doubling step
    as S_{k+1} = S_{k+1}(I + G_k); the self-reference is read as S_k.)"""
    r = rng(15)
    N = 64
    L = np.tril(r.standard_normal((N, N)) * 0.2, -1)
    A = np.eye(N) + L
    ref = np.linalg.inv(A)
    neu = sum(np.linalg.matrix_power(-L, n) for n in range(N))
    np.testing.assert_allclose(neu, ref, atol=1e-10)
    S, G = np.eye(N) - L, L @ L          # S_1, G_1 = (-L)^2
    for _ in range(5):                   # up to 2^6 = 64 terms
        S, G = S @ (np.eye(N) + G), G @ G
    np.testing.assert_allclose(S, ref, atol=1e-10)
    nb, bs = 4, 16
    Bk = np.zeros((N, N))
    blk = lambda M, i, j: M[i * bs:(i + 1) * bs, j * bs:(j + 1) * bs]
    for i in range(nb):
        blk(Bk, i, i)[:] = np.linalg.inv(blk(A, i, i))
    for i in range(nb):
        for j in range(i):
            acc = sum(blk(A, i, kk) @ blk(Bk, kk, j) for kk in range(j, i))
            blk(Bk, i, j)[:] = -blk(Bk, i, i) @ acc
    np.testing.assert_allclose(Bk, ref, atol=1e-10)


def test_deltanet_inverse_entries_in_unit_interval():
    """Entries of (I + Diag(beta)(K K^T * M_{-1}))^{-1} lie in [-1, 1] for unit keys, beta in [0, 1]
    (GDN2 page, linked claim about DeltaNet's core inverse)."""
    r = rng(16)
    M1 = np.tril(np.ones((64, 64)), -1)
    worst = 0.0
    for d in (2, 16, 128):
        for _ in range(5):
            K = _unit(r.standard_normal((64, d)))
            beta = r.random(64)
            X = np.eye(64) + np.diag(beta) @ ((K @ K.T) * M1)
            worst = max(worst, np.abs(np.linalg.inv(X)).max())
    assert worst <= 1 + 1e-9


# --------------------------------------------------------------------------
# the pins above are sensitive: planted mistakes in a copy of the oracle fail
# --------------------------------------------------------------------------
def _mutant_recurrence(q, k, v, g, beta, h0, mode):
    """A Python copy of the recurrence with one planted mistake (per single head)."""
    T, dk = q.shape
    S = h0.copy()
    o = np.zeros((T, v.shape[1]))
    for t in range(T):
        al = np.exp(g[t])
        bt = beta[t] * k[t]
        vv = beta[t] * v[t] if mode != "no_beta_on_v" else v[t]
        if mode == "decay_after":
            S = (S - np.outer(S @ bt, k[t])) * al[None, :] + np.outer(vv, k[t])
        elif mode == "sign":
            Sa = S * al[None, :]
            S = Sa + np.outer(Sa @ bt, k[t]) + np.outer(vv, k[t])
        elif mode == "transposed_state":
            Sa = S * al[:, None] if S.shape[0] == S.shape[1] else S * al[None, :]
            S = Sa - np.outer(Sa @ bt, k[t]) + np.outer(vv, k[t])
        else:
            Sa = S * al[None, :]
            S = Sa - np.outer(Sa @ bt, k[t]) + np.outer(vv, k[t])
        o[t] = S @ q[t]
    return o, S


@pytest.mark.parametrize("mode", ["no_beta_on_v", "decay_after", "sign", "transposed_state"])
def test_pins_catch_planted_mistakes(mode):
    """The delta-rule-write and chunk-form pins reject each planted mistake."""
    q, k, v, beta, g, h0 = _rand(17, B=1, T=40, H=1, dk=8, dv=8)
    args = (q[0, :, 0], k[0, :, 0], v[0, :, 0], g[0, :, 0], beta[0, :, 0], h0[0, 0])
    o_ok, _ = _mutant_recurrence(*args, mode="none")
    o_ref, _ = oracle.kda_fwd(q, k, v, g, beta, h0)
    np.testing.assert_allclose(o_ok, o_ref[0, :, 0], atol=1e-12)   # the unmutated copy agrees
    o_bad, S_bad = _mutant_recurrence(*args, mode=mode)
    oc, Sc = kda_chunk_form(*args[:5], h0=args[5], C=16)
    assert np.abs(o_bad - oc).max() > 1e-3

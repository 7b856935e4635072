"""Spectral norms of the per-step transition factors -- TEST INFRASTRUCTURE.

Page "How to make GDN2 more stable":

* eq. (4) / eq. (12): for unit vectors k, j and eta >= 0,
  ||I - eta k j^T||_2 = (eta + sqrt(eta^2 - 4 eta c + 4)) / 2 with c = k^T j.
* eq. (7): the stabilising clip replaces D by min(D, 1/rho) with that rho;
  in log space g -> min(g, -log rho), token by token.

``rho_closed_form`` is eq. (4) written out.  ``factor_norm_exact`` is the
spectral norm of the full factor Diag(alpha)(I - b a^T) of the DPLR recurrence
(page "Diagonal Plus Low Rank", section 2), for which the page states no closed
form; it takes the largest singular value from numpy's SVD.
"""
from __future__ import annotations

import numpy as np


def rho_closed_form(eta, c):
    """Eq. (4): spectral norm of I - eta k j^T for unit k, j with c = k^T j."""
    eta = np.asarray(eta, dtype=np.float64)
    c = np.asarray(c, dtype=np.float64)
    return (eta + np.sqrt(eta * eta - 4.0 * eta * c + 4.0)) / 2.0


def factor_norm_exact(alpha, a, b):
    """Largest singular value of Diag(alpha) (I - b a^T).

    alpha, a, b: [..., d].  Returns an array of shape [...].
    """
    alpha = np.asarray(alpha, dtype=np.float64)
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    d = a.shape[-1]
    eye = np.eye(d)
    m = alpha[..., :, None] * (eye - b[..., :, None] * a[..., None, :])
    return np.linalg.svd(m, compute_uv=False)[..., 0]


def rho_of(a, b):
    """Eq. (4) for general a, b: ||I - b a^T||_2 with eta = |a||b|, c = a.b / eta (c = 1 at eta = 0).

    a, b: [..., d].  Returns rho [...].
    """
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    eta = np.linalg.norm(a, axis=-1) * np.linalg.norm(b, axis=-1)
    s = (a * b).sum(-1)
    c = np.where(eta > 0, s / np.where(eta > 0, eta, 1.0), 1.0)
    return rho_closed_form(eta, c)


def clip_gate(g, a, b):
    """Eq. (7) in log space: g' = min(g, -log rho) per token, rho = ||I - b a^T||_2.

    g: [..., d] per-channel log-decay; a, b: [..., d].  Returns g' [..., d].
    """
    g = np.asarray(g, dtype=np.float64)
    return np.minimum(g, -np.log(rho_of(a, b))[..., None])


def clip_gate_bwd(g, a, b, dg_clipped):
    """Chain rule of :func:`clip_gate`: gradients with respect to g, a and b.

    Where g < -log rho the gradient passes to g; elsewhere it goes to
    -log rho, and from there to a and b through the derivative of eq. (4):
    with eta = |a||b|, s = a.b and R = sqrt(eta^2 - 4 s + 4),
    d rho/d a = ((1 + eta/R) d eta/d a - 2 b / R) / 2, d eta/d a = |b| a / |a|,
    and symmetrically for b.  Returns (dg, da, db).
    """
    g = np.asarray(g, dtype=np.float64)
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    dgc = np.asarray(dg_clipped, dtype=np.float64)
    rho = rho_of(a, b)
    keep = g < -np.log(rho)[..., None]
    dg = np.where(keep, dgc, 0.0)
    d_neglog = np.where(keep, 0.0, dgc).sum(-1)              # dL / d(-log rho)
    na = np.linalg.norm(a, axis=-1, keepdims=True)
    nb = np.linalg.norm(b, axis=-1, keepdims=True)
    eta = na * nb
    s = (a * b).sum(-1, keepdims=True)
    R = np.sqrt(eta * eta - 4.0 * s + 4.0)
    deta_da = nb * a / np.where(na > 0, na, 1.0)
    deta_db = na * b / np.where(nb > 0, nb, 1.0)
    drho_da = 0.5 * ((1.0 + eta / R) * deta_da - 2.0 * b / R)
    drho_db = 0.5 * ((1.0 + eta / R) * deta_db - 2.0 * a / R)
    scale = (-d_neglog / rho)[..., None]                      # dL/d rho = -dL/d(-log rho) / rho
    return dg, scale * drho_da, scale * drho_db

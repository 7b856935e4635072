"""Spectral norms of the per-step transition factors -- TEST INFRASTRUCTURE.

Page "How to make GDN2 more stable":

* eq. (4) / eq. (12): for unit vectors k, j and eta >= 0,
  ||I - eta k j^T||_2 = (eta + sqrt(eta^2 - 4 eta c + 4)) / 2 with c = k^T j.
* eq. (7): the stabilising clip replaces D by min(D, 1/rho) with that rho.

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

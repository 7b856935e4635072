"""Float64 numpy restatements of the pages' chunk forms (test helpers only).

These exist to pin the token-recurrence oracle against an independent
derivation: the chunkwise algebra that the pages derive from the same
recurrence.  Each function follows one page's equations in their order and
notation; neither the oracle nor the CUDA library uses them.
"""
from __future__ import annotations

import numpy as np


def _masks(C):
    M = np.tril(np.ones((C, C)))          # inclusive lower mask
    return M, M - np.eye(C)               # M and M_{-1} = M - I


def kda_chunk_form(q, k, v, g, beta, h0=None, C=64, scale_v=True):
    """KDA chunk forward as page "Kimi Delta Attention backward" recaps it.

    Per chunk [t]: Gamma = exp(in-chunk cumsum of g); Q<- = Q*Gamma,
    K<- = K*Gamma, K-> = K/Gamma; X~ = I + Diag(beta)(K<- K->^T * M_{-1});
    A~ = X~^{-1}; W = A~ Diag(beta) K<-; U = A~ Diag(beta) V;
    V_new = U - W S^T; O = Q<- S^T + (Q<- K->^T * M) V_new;
    S <- S Diag(gamma^C) + V_new^T K-> Diag(gamma^C).
    With scale_v False, U = A~ V (beta does not scale v) -- the GLA-style
    reading used when beta is 0.

    Inputs per single (batch, head): q, k [T, dk]; v [T, dv]; g [T, dk] log
    decay (None -> 0); beta [T] (None -> 0); h0 [dv, dk].
    """
    T, dk = q.shape
    dv = v.shape[1]
    g = np.zeros((T, dk)) if g is None else g
    beta = np.zeros(T) if beta is None else beta
    S = np.zeros((dv, dk)) if h0 is None else h0.copy()
    o = np.zeros((T, dv))
    for s in range(0, T, C):
        e = min(s + C, T)
        n = e - s
        M, M1 = _masks(n)
        Gam = np.exp(np.cumsum(g[s:e], axis=0))
        Ql, Kl, Kr = q[s:e] * Gam, k[s:e] * Gam, k[s:e] / Gam
        Db = np.diag(beta[s:e])
        Xt = np.eye(n) + Db @ ((Kl @ Kr.T) * M1)
        At = np.linalg.inv(Xt)
        W = At @ Db @ Kl
        U = At @ Db @ v[s:e] if scale_v else At @ v[s:e]
        Vnew = U - W @ S.T
        o[s:e] = Ql @ S.T + ((Ql @ Kr.T) * M) @ Vnew
        gC = Gam[-1]
        S = S * gC[None, :] + (Vnew.T @ Kr) * gC[None, :]
    return o, S


def dplr_chunk_form(q, k, v, a, b, g, h0=None, C=64):
    """Gated DPLR chunk forward of page "Diagonal Plus Low Rank", section 2.

    E = (I + (B<- A->^T * M_{-1}))^{-1}; W = E B<-;
    C = -E (B<- K->^T * M_{-1}) V;
    S^C = S Diag(g^C) + V^T K-> Diag(g^C) + (C - W S^T)^T A-> Diag(g^C);
    O = Q<- S^T + (Q<- K->^T * M) V + (Q<- A->^T * M)(C - W S^T).
    """
    T, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dv, dk)) if h0 is None else h0.copy()
    o = np.zeros((T, dv))
    for s in range(0, T, C):
        e = min(s + C, T)
        n = e - s
        M, M1 = _masks(n)
        Gam = np.exp(np.cumsum(g[s:e], axis=0))
        Ql, Kr = q[s:e] * Gam, k[s:e] / Gam
        Ar, Bl = a[s:e] / Gam, b[s:e] * Gam
        E = np.linalg.inv(np.eye(n) + (Bl @ Ar.T) * M1)
        W = E @ Bl
        Cm = -E @ ((Bl @ Kr.T) * M1) @ v[s:e]
        V2 = Cm - W @ S.T
        gC = Gam[-1]
        o[s:e] = Ql @ S.T + ((Ql @ Kr.T) * M) @ v[s:e] + ((Ql @ Ar.T) * M) @ V2
        S = (S + v[s:e].T @ Kr + V2.T @ Ar) * gC[None, :]
    return o, S


def dplr_wy_product(a, b, alpha):
    """P^C of one chunk through the w recursion (page "Diagonal Plus Low Rank").

    w^r = (I - sum_{i<r} w^i (a^i / gamma^i)^T) (gamma^r * b^r) and
    P^C = (I - sum_i w^i (a^i / gamma^i)^T) Diag(gamma^C), gamma^r the
    running product of alpha.
    """
    C, d = a.shape
    gam = np.cumprod(alpha, axis=0)
    w = np.zeros((C, d))
    for r in range(C):
        acc = np.eye(d)
        for i in range(r):
            acc -= np.outer(w[i], a[i] / gam[i])
        w[r] = acc @ (gam[r] * b[r])
    acc = np.eye(d)
    for i in range(C):
        acc -= np.outer(w[i], a[i] / gam[i])
    return acc @ np.diag(gam[-1])

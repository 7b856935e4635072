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


def kda_record_form(q, k, v, g, beta, h0=None, C=64, blk=16, scale_v=True):
    """The regrouping of the KDA chunk form that the tensor-core kernels evaluate.

    Derived from the recap on page "Kimi Delta Attention backward": per chunk,
    with L = Diag(beta)(K<- K->^T * M_{-1}) and P = Q<- K->^T * M,
      Z' (I + L) = [I ; P]   solved by back-substitution over blk-column blocks
                             (page "DeltaNet" 4.2, block form, on the
                             transposed system): Z'_c = ([I ; P]_c -
                             sum_{c' > c} Z'_{c'} L_{c'c}) (I + L_cc)^{-1};
      Z = Z' Diag(beta) = [T ; P T]  with T = A~ Diag(beta);
      [W ; P W] = Z K<-,   A = [-W ; Q<- - P W];
      D1 = Z V + A S^T = [U - W S^T ; P U + (Q<- - P W) S^T] = [V_new ; O];
      S <- (S + V_new^T K->) Diag(gamma^C).
    With scale_v False (beta does not scale v) U = A~ V: V is multiplied by
    Z' instead of Z.  Inputs as kda_chunk_form.
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
        L = np.diag(beta[s:e]) @ ((Kl @ Kr.T) * M1)
        P = (Ql @ Kr.T) * M
        R = np.vstack([np.eye(n), P])
        Zp = np.zeros((2 * n, n))
        for c0 in reversed(range(0, n, blk)):
            c1 = min(c0 + blk, n)
            rhs = R[:, c0:c1] - Zp[:, c1:] @ L[c1:, c0:c1]
            Zp[:, c0:c1] = rhs @ np.linalg.inv(np.eye(c1 - c0) + L[c0:c1, c0:c1])
        Z = Zp @ np.diag(beta[s:e])
        WP = Z @ Kl
        A = np.vstack([-WP[:n], Ql - WP[n:]])
        D1 = (Z if scale_v else Zp) @ v[s:e] + A @ S.T
        o[s:e] = D1[n:]
        S = (S + D1[:n].T @ Kr) * Gam[-1][None, :]
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


def kda_chunk_bwd_form(q, k, v, g, beta, do, h0=None, dht=None, C=64, scale_v=True):
    """KDA chunk backward of page "Kimi Delta Attention backward" (one head).

    Forward per chunk as kda_chunk_form; backward per chunk, in reverse, with
    dS the gradient of the state after the chunk:
      dU = K-> Diag(gamma^C) dS^T + (Q<- K->^T * M)^T dO;   dW = -dU S_prev;
      dQ<- = dO S_prev + (dO V_new^T * M) K->;   dV = Diag(beta) A~^T dU;
      dA~ = dW K<-^T Diag(beta) + dU V^T Diag(beta);   dX~ = -A~^T dA~ A~^T;
      dK<- = Diag(beta) A~^T dW + (Diag(beta) dX~ * M_{-1}) K->;
      dK-> = V_new dS Diag(gamma^C) + (dO V_new^T * M)^T Q<- + (Diag(beta) dX~ * M_{-1})^T K<-;
      dK = dK<- * Gamma + dK-> / Gamma;   dQ = dQ<- * Gamma;
      dbeta = diag(A~^T dW K<-^T) + diag(A~^T dU V^T) + diag(dX~ (K<- K->^T * M_{-1})^T);
      dlogGamma = dQ * Q + (dK<- * Gamma) * K - (dK-> / Gamma) * K, last row + diag(S^T dS);
      dg = in-chunk suffix sum of dlogGamma;
      dS_prev = dS Diag(gamma^C) + dO^T Q<- - dU^T W.
    (The page's dS recursion, its dW with S_[t-1] and its dK-> with the
    output term of the final combination.)  With scale_v False (beta = 0,
    GLA) U = A~ V and the beta-terms of dV, dA~ and dbeta drop.
    Returns dq, dk, dv, dg, dbeta, dh0.
    """
    T, dk = q.shape
    dv = v.shape[1]
    g = np.zeros((T, dk)) if g is None else g
    beta = np.zeros(T) if beta is None else beta
    S = np.zeros((dv, dk)) if h0 is None else h0.copy()
    starts = list(range(0, T, C))
    prev = []
    for s in starts:                       # forward: states before each chunk
        e = min(s + C, T)
        n = e - s
        _, M1 = _masks(n)
        Gam = np.exp(np.cumsum(g[s:e], axis=0))
        Kl, Kr = k[s:e] * Gam, k[s:e] / Gam
        Db = np.diag(beta[s:e])
        At = np.linalg.inv(np.eye(n) + Db @ ((Kl @ Kr.T) * M1))
        W = At @ Db @ Kl
        U = At @ Db @ v[s:e] if scale_v else At @ v[s:e]
        prev.append(S.copy())
        S = (S + (U - W @ S.T).T @ Kr) * Gam[-1][None, :]
    out = {n: np.zeros_like(x) for n, x in (("dq", q), ("dk", k), ("dv", v), ("dg", g), ("dbeta", beta))}
    dS = np.zeros((dv, dk)) if dht is None else dht.copy()
    for idx in reversed(range(len(starts))):
        s = starts[idx]
        e = min(s + C, T)
        n = e - s
        M, M1 = _masks(n)
        Sp = prev[idx]
        Gam = np.exp(np.cumsum(g[s:e], axis=0))
        gC = Gam[-1]
        Q, K, V, dO = q[s:e], k[s:e], v[s:e], do[s:e]
        Ql, Kl, Kr = Q * Gam, K * Gam, K / Gam
        Db = np.diag(beta[s:e])
        N = (Kl @ Kr.T) * M1
        At = np.linalg.inv(np.eye(n) + Db @ N)
        W = At @ Db @ Kl
        U = At @ Db @ V if scale_v else At @ V
        Vn = U - W @ Sp.T
        P = (Ql @ Kr.T) * M
        St = (Sp + Vn.T @ Kr) * gC[None, :]
        dU = (Kr * gC[None, :]) @ dS.T + P.T @ dO
        dW = -dU @ Sp
        dOV = (dO @ Vn.T) * M
        dQl = dO @ Sp + dOV @ Kr
        dV = (Db @ At.T @ dU) if scale_v else At.T @ dU
        dAt = dW @ Kl.T @ Db + (dU @ V.T @ Db if scale_v else dU @ V.T)
        dXt = -At.T @ dAt @ At.T
        E = (Db @ dXt) * M1
        dKl = Db @ At.T @ dW + E @ Kr
        dKr = Vn @ dS * gC[None, :] + dOV.T @ Ql + E.T @ Kl
        dq = dQl * Gam
        dk_ = dKl * Gam + dKr / Gam
        dbeta = np.diag(At.T @ dW @ Kl.T) + np.diag(dXt @ N.T)
        if scale_v:
            dbeta = dbeta + np.diag(At.T @ dU @ V.T)
        dlg = dq * Q + dKl * Gam * K - dKr / Gam * K
        dlg[-1] += (St * dS).sum(0)
        out["dq"][s:e], out["dk"][s:e], out["dv"][s:e] = dq, dk_, dV
        out["dg"][s:e] = np.cumsum(dlg[::-1], axis=0)[::-1]
        out["dbeta"][s:e] = dbeta
        dS = dS * gC[None, :] + dO.T @ Ql - dU.T @ W
    out["dh0"] = dS
    return out


def gla_parallel_grads(q, k, v, g, do):
    """Gradients of the GLA parallel form o = (Q<- K->^T * M) V, whole sequence as one chunk.

    Page "Gated Linear Attention", section 6.3 with zero initial state and no
    final-state gradient: with A = (Q<- K->^T) * M and dA = (dO V^T) * M,
    dQ = (dA K->) * Gamma, dK = (dA^T Q<-) / Gamma, dV = A^T dO,
    dlogGamma = Q * dQ - K * dK and dg its suffix sum.
    """
    Gam = np.exp(np.cumsum(g, axis=0))
    M, _ = _masks(q.shape[0])
    Ql, Kr = q * Gam, k / Gam
    A = (Ql @ Kr.T) * M
    dA = (do @ v.T) * M
    dq = (dA @ Kr) * Gam
    dk = (dA.T @ Ql) / Gam
    dv = A.T @ do
    dlg = q * dq - k * dk
    return dq, dk, dv, np.cumsum(dlg[::-1], axis=0)[::-1]


def dplr_chunk_bwd_form(q, k, v, a, b, g, do, h0=None, dht=None, C=64):
    """Gated DPLR chunk backward of page "Diagonal Plus Low Rank", section 3 (one head).

    Forward per chunk as dplr_chunk_form, with F = I + (B<- A->^T * M_{-1}),
    E = F^{-1}, V_1 = V, V_2 = C - W S^T.  Backward per chunk, in reverse,
    dS the gradient of the state after the chunk:
      dC = dV_2 = A-> Diag(gamma^C) dS^T + (Q<- A->^T * M)^T dO;
      dV_1 = K-> Diag(gamma^C) dS^T + (Q<- K->^T * M)^T dO;   dW = -dC S_prev;
      dE = -dC V^T (B<- K->^T * M_{-1})^T + dW B<-^T;   dF = -E^T dE E^T;
      dQ<- = dO S_prev + (dO V_1^T * M) K-> + (dO V_2^T * M) A->;
      dB<- = E^T dW - (E^T dC V^T * M_{-1}) K-> + (dF * M_{-1}) A->;
      dK-> = (dO V_1^T * M)^T Q<- - (E^T dC V^T * M_{-1})^T B<- + V_1 dS Diag(gamma^C);
      dA-> = (dO V_2^T * M)^T Q<- + (dF * M_{-1})^T B<- + V_2 dS Diag(gamma^C);
      dV = dV_1 - (B<- K->^T * M_{-1})^T E^T dC;
      dq = dQ<- * Gamma, db = dB<- * Gamma, dk = dK-> / Gamma, da = dA-> / Gamma;
      dlogGamma = dQ<- * Q<- + dB<- * B<- - dK-> * K-> - dA-> * A->, last row + diag(S^T dS);
      dS_prev = dS Diag(gamma^C) + dO^T Q<- - dC^T W.
    Readings: dW against S_[t-1] (the page writes S_[t]); dB = dB<- * Gamma
    (the page writes dQ<-); dK-> and dA-> carry the state-update terms
    V_1 dS Diag(gamma^C) and V_2 dS Diag(gamma^C), which the page's lines omit.
    Returns dq, dk, dv, da, db, dg, dh0.
    """
    T, dk = q.shape
    dv = v.shape[1]
    S = np.zeros((dv, dk)) if h0 is None else h0.copy()
    starts = list(range(0, T, C))
    prev = []
    for s in starts:
        e = min(s + C, T)
        n = e - s
        _, M1 = _masks(n)
        Gam = np.exp(np.cumsum(g[s:e], axis=0))
        Kr, Ar, Bl = k[s:e] / Gam, a[s:e] / Gam, b[s:e] * Gam
        E = np.linalg.inv(np.eye(n) + (Bl @ Ar.T) * M1)
        W = E @ Bl
        Cm = -E @ ((Bl @ Kr.T) * M1) @ v[s:e]
        prev.append(S.copy())
        S = (S + v[s:e].T @ Kr + (Cm - W @ S.T).T @ Ar) * Gam[-1][None, :]
    out = {n: np.zeros_like(x) for n, x in (("dq", q), ("dk", k), ("dv", v), ("da", a), ("db", b), ("dg", g))}
    dS = np.zeros((dv, dk)) if dht is None else dht.copy()
    for idx in reversed(range(len(starts))):
        s = starts[idx]
        e = min(s + C, T)
        n = e - s
        M, M1 = _masks(n)
        Sp = prev[idx]
        Gam = np.exp(np.cumsum(g[s:e], axis=0))
        gC = Gam[-1]
        V, dO = v[s:e], do[s:e]
        Ql, Kr, Ar, Bl = q[s:e] * Gam, k[s:e] / Gam, a[s:e] / Gam, b[s:e] * Gam
        Nbk = (Bl @ Kr.T) * M1
        E = np.linalg.inv(np.eye(n) + (Bl @ Ar.T) * M1)
        W = E @ Bl
        Cm = -E @ Nbk @ V
        V2 = Cm - W @ Sp.T
        Pk, Pa = (Ql @ Kr.T) * M, (Ql @ Ar.T) * M
        St = (Sp + V.T @ Kr + V2.T @ Ar) * gC[None, :]
        dC = (Ar * gC[None, :]) @ dS.T + Pa.T @ dO
        dV1 = (Kr * gC[None, :]) @ dS.T + Pk.T @ dO
        dW = -dC @ Sp
        dE = -dC @ V.T @ Nbk.T + dW @ Bl.T
        dF = -E.T @ dE @ E.T
        O1, O2 = (dO @ V.T) * M, (dO @ V2.T) * M
        G = (E.T @ dC @ V.T) * M1
        dQl = dO @ Sp + O1 @ Kr + O2 @ Ar
        dBl = E.T @ dW - G @ Kr + (dF * M1) @ Ar
        dKr = O1.T @ Ql - G.T @ Bl + (V @ dS) * gC[None, :]
        dAr = O2.T @ Ql + (dF * M1).T @ Bl + (V2 @ dS) * gC[None, :]
        dV = dV1 - Nbk.T @ E.T @ dC
        dlg = dQl * Ql + dBl * Bl - dKr * Kr - dAr * Ar
        dlg[-1] += (St * dS).sum(0)
        out["dq"][s:e], out["db"][s:e] = dQl * Gam, dBl * Gam
        out["dk"][s:e], out["da"][s:e] = dKr / Gam, dAr / Gam
        out["dv"][s:e] = dV
        out["dg"][s:e] = np.cumsum(dlg[::-1], axis=0)[::-1]
        dS = dS * gC[None, :] + dO.T @ Ql - dC.T @ W
    out["dh0"] = dS
    return out

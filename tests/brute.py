"""Independent brute-force forms of the gated delta rule, used only to pin the oracle.

Neither form is the oracle's own arithmetic: the first accumulates the state as a product of
dense D x D matrices, the second is the chunked UT/WY algebra with a per-channel cumulative log
gate (the "chunked twin" the KDA module doc describes: k scaled by exp(-Gcum), q by exp(+Gcum)).
Both are plain numpy f64 for tiny D and T.

Per token the method is  S' = Diag(a) S;  u = v - S'^T k;  S <- S' + beta k u^T;  o = scale S^T q.
"""

from __future__ import annotations

import numpy as np


def dense_product_scan(q, k, v, g, beta, S0, scale):
    """Matrix form of one token: S <- (I - beta k k^T) Diag(a) S + beta k v^T, o = scale S^T q.
    Shapes: q, k, v, g [T, D]; beta [T]; S0 [D, D] in math layout (rows = key dim).
    Returns (o [T, D], S_T [D, D])."""
    T, D = q.shape
    S = S0.copy()
    eye = np.eye(D)
    o = np.zeros((T, D))
    for t in range(T):
        A = np.diag(np.exp(g[t]))
        P = eye - beta[t] * np.outer(k[t], k[t])
        S = P @ A @ S + beta[t] * np.outer(k[t], v[t])
        o[t] = scale * (S.T @ q[t])
    return o, S


def chunked_scan(q, k, v, g, beta, S0, scale, chunk):
    """Chunked UT/WY form.  Within a chunk with start state S0 and inclusive cumulative log gate
    Gc[t] = sum_{s<=t} g[s] (per channel), Gamma = exp(Gc):
        L[t, s]  = beta_t (k_t * Gamma_t) . (k_s / Gamma_s)       for s < t (strictly lower)
        Tm       = (I + L)^{-1}
        U        = Tm diag(beta) V,   W = Tm diag(beta) (K * Gamma)
        U'       = U - W S0
        O        = scale [ (Q * Gamma) S0 + tril_incl((Q * Gamma)(K / Gamma)^T) U' ]
        S_C      = Diag(Gamma_C) S0 + (K * Gamma_C / Gamma)^T U'
    Returns (o [T, D], S_T [D, D])."""
    T, D = q.shape
    S = S0.copy()
    o = np.zeros((T, D))
    for c0 in range(0, T, chunk):
        c1 = min(c0 + chunk, T)
        Q, K, V, G, B = q[c0:c1], k[c0:c1], v[c0:c1], g[c0:c1], beta[c0:c1]
        n = c1 - c0
        Gc = np.cumsum(G, axis=0)
        Gam = np.exp(Gc)
        Kp, Km, Qp = K * Gam, K / Gam, Q * Gam
        L = np.tril((B[:, None] * Kp) @ Km.T, -1)
        Tm = np.linalg.inv(np.eye(n) + L)
        U = Tm @ (B[:, None] * V)
        W = Tm @ (B[:, None] * Kp)
        Up = U - W @ S
        o[c0:c1] = scale * (Qp @ S + np.tril(Qp @ Km.T) @ Up)
        S = np.exp(Gc[-1])[:, None] * S + (K * np.exp(Gc[-1] - Gc)).T @ Up
    return o, S

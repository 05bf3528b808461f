"""Independent FP64 formulations of the gated delta rule, used to pin the
oracle.  Pure numpy; nothing here is imported by the oracle or by the CUDA
library.

* :func:`matrix_form` -- the recurrence written on S (V x K) with the explicit
  projector:  S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,
  o_t = S_t q_t * scale.  (The oracle works on h = S^T with a rank-one
  update instead.)
* :func:`chunked_form` -- the chunked (UT / WY) form of the project statement:
  chunk-local log-gate cumsum G; A = strictly-lower(diag(beta) * decay-masked
  K K^T); T = (I + A)^-1 by a library inverse; W = T diag(beta e^G) K;
  U = T diag(beta) V; v_new = U - W h; o = (Q e^G) h + causal(Q K^T * decay)
  v_new (diagonal included); h <- e^{G_last} h + K^T (v_new e^{G_last - G}).
* :func:`gla_closed_form` -- the beta-free recurrence evaluated as O(T^2)
  decay-masked attention plus the decayed initial state.
"""
from __future__ import annotations

import numpy as np


def _spans(B, T, cu):
    if cu is None:
        return [(b, 0, T) for b in range(B)]
    cu = [int(x) for x in cu]
    return [(0, cu[n], cu[n + 1]) for n in range(len(cu) - 1)]


def matrix_form(q, k, v, g, beta, h0, scale, cu=None):
    B, T, H, K = q.shape
    V = v.shape[-1]
    spans = _spans(B, T, cu)
    o = np.zeros((B, T, H, V))
    ht = np.zeros((len(spans), H, K, V))
    eye = np.eye(K)
    for n, (row, t0, t1) in enumerate(spans):
        for h in range(H):
            S = np.zeros((V, K)) if h0 is None else h0[n, h].T.copy()
            for t in range(t0, t1):
                a = np.exp(g[row, t, h])
                kt, vt = k[row, t, h], v[row, t, h]
                if beta is None:
                    S = a * S + np.outer(vt, kt)
                else:
                    b = beta[row, t, h]
                    S = a * S @ (eye - b * np.outer(kt, kt)) + b * np.outer(vt, kt)
                o[row, t, h] = (S @ q[row, t, h]) * scale
            ht[n, h] = S.T
    return o, ht


def chunked_form(q, k, v, g, beta, h0, scale, chunk, cu=None):
    B, T, H, K = q.shape
    V = v.shape[-1]
    spans = _spans(B, T, cu)
    o = np.zeros((B, T, H, V))
    ht = np.zeros((len(spans), H, K, V))
    for n, (row, t0, t1) in enumerate(spans):
        for hh in range(H):
            h = np.zeros((K, V)) if h0 is None else h0[n, hh].copy()
            for c0 in range(t0, t1, chunk):
                c1 = min(t1, c0 + chunk)
                L = c1 - c0
                Qc, Kc, Vc = q[row, c0:c1, hh], k[row, c0:c1, hh], v[row, c0:c1, hh]
                G = np.cumsum(g[row, c0:c1, hh])
                ii, jj = np.meshgrid(np.arange(L), np.arange(L), indexing="ij")
                # decay e^{G_i - G_j} only where i >= j (masked before exp)
                D = np.where(ii >= jj, G[:, None] - G[None, :], -np.inf)
                Gam = np.exp(D)
                if beta is None:
                    v_new = Vc
                else:
                    bc = beta[row, c0:c1, hh]
                    A = np.where(ii > jj, bc[:, None] * Gam * (Kc @ Kc.T), 0.0)
                    Tm = np.linalg.inv(np.eye(L) + A)
                    W = Tm @ ((bc * np.exp(G))[:, None] * Kc)
                    U = Tm @ (bc[:, None] * Vc)
                    v_new = U - W @ h
                Oc = (Qc * np.exp(G)[:, None]) @ h + ((Qc @ Kc.T) * Gam) @ v_new
                o[row, c0:c1, hh] = Oc * scale
                h = np.exp(G[-1]) * h + Kc.T @ (v_new * np.exp(G[-1] - G)[:, None])
            ht[n, hh] = h
    return o, ht


def gla_closed_form(q, k, v, g, h0, scale, cu=None):
    """beta-free: o_t = scale [e^{G_t} h0^T q_t + sum_{j<=t} e^{G_t-G_j}
    (q_t . k_j) v_j], ht = e^{G_T} h0 + sum_j e^{G_T - G_j} k_j v_j^T, with G
    the sequence-global inclusive cumsum of g."""
    B, T, H, K = q.shape
    V = v.shape[-1]
    spans = _spans(B, T, cu)
    o = np.zeros((B, T, H, V))
    ht = np.zeros((len(spans), H, K, V))
    for n, (row, t0, t1) in enumerate(spans):
        for hh in range(H):
            L = t1 - t0
            Qs, Ks, Vs = q[row, t0:t1, hh], k[row, t0:t1, hh], v[row, t0:t1, hh]
            G = np.cumsum(g[row, t0:t1, hh])
            ii, jj = np.meshgrid(np.arange(L), np.arange(L), indexing="ij")
            Dm = np.exp(np.where(ii >= jj, G[:, None] - G[None, :], -np.inf))
            out = ((Qs @ Ks.T) * Dm) @ Vs
            hz = np.zeros((K, V)) if h0 is None else h0[n, hh]
            out = out + np.exp(G)[:, None] * (Qs @ hz)
            o[row, t0:t1, hh] = out * scale
            GT = G[-1] if L else 0.0
            ht[n, hh] = np.exp(GT) * hz + Ks.T @ (np.exp(GT - G)[:, None] * Vs)
    return o, ht


def rel(x, ref):
    d = np.linalg.norm((x - ref).ravel())
    r = np.linalg.norm(ref.ravel())
    return d / r if r > 0 else d

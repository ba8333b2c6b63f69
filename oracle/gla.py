"""Gated linear attention (GLA) over a draft tree -- TEST INFRASTRUCTURE ONLY (oracle).

The review of SpecLA (pith.science 7ERME3HB), editorial analysis, names GLA
next to DeltaNet and Mamba as recurrences whose per-token factor records the
same verify / commit runtime would carry.  GLA's gate is per key channel (a
diagonal decay) and it has no delta-rule erasure.  In this library's layout
(S is d_v x d_k, row = value index) the recurrence, walked here in fp64 along
each node's own root-to-node path from S0, is

    S_t = S_parent(t) diag(alpha_t) + beta_t v_t k_t^T,    o_t = S_t q_t,

with alpha_t in (0, 1]^{d_k} (one gate per key channel) and beta_t a write
strength (beta = 1 is the plain GLA update).  Returned: out [B,N,H,dv], and
the factor record the commit consumes -- delta [B,H,N,dv] = beta_t v_t and
the per-channel cumulative log gate g [B,H,N,dk] = sum of log alpha_j over
j on path(t), root first.  ``commit`` walks the accepted root-first path.
"""
from __future__ import annotations

import numpy as np


def _path(parent_row, t):
    p = []
    while t >= 0:
        p.append(int(t))
        t = int(parent_row[t])
    return p[::-1]


def tree_verify(q, k, v, alpha, beta, parent, S0):
    """alpha [B,N,H,dk], beta [B,N,H]; other tensors as the GDN verifier."""
    q, k, v, alpha, beta, S0 = (np.asarray(x, np.float64) for x in (q, k, v, alpha, beta, S0))
    B, N, H, dk = q.shape
    dv = v.shape[-1]
    out = np.zeros((B, N, H, dv))
    delta = np.zeros((B, H, N, dv))
    g = np.zeros((B, H, N, dk))
    for b in range(B):
        for t in range(N):
            path = _path(parent[b], t)
            for h in range(H):
                S = S0[b, h].copy()
                gs = np.zeros(dk)
                for j in path:
                    S = S * alpha[b, j, h][None, :] + beta[b, j, h] * np.outer(v[b, j, h], k[b, j, h])
                    gs = gs + np.log(alpha[b, j, h])
                out[b, t, h] = S @ q[b, t, h]
                delta[b, h, t] = beta[b, t, h] * v[b, t, h]
                g[b, h, t] = gs
    return out, delta, g


def commit(k, v, alpha, beta, parent, S0, path):
    """State after walking the accepted root-first path ([B, Lmax], -1 padded) from S0."""
    k, v, alpha, beta, S0 = (np.asarray(x, np.float64) for x in (k, v, alpha, beta, S0))
    S = S0.copy()
    for b in range(S.shape[0]):
        for j in path[b]:
            if j < 0:
                break
            for h in range(S.shape[1]):
                S[b, h] = S[b, h] * alpha[b, j, h][None, :] + beta[b, j, h] * np.outer(v[b, j, h], k[b, j, h])
    return S

"""Decay-gated linear attention over a draft tree -- TEST INFRASTRUCTURE ONLY (oracle).

The factor record and commit of the SpecLA review (pith.science 7ERME3HB)
apply to other linear-attention recurrences; "Axiom & Free-Parameter Ledger"
and the editorial summary name DeltaNet, GLA and Mamba-style models.  This is
the scalar-decay recurrence without the delta-rule erasure (Mamba-2 /
RetNet-style), in fp64, walking each node's root-to-node path:

    S_t = alpha_t S_parent(t) + beta_t v_t k_t^T,   o_t = S_t q_t

with the same tensors as the GDN verifier (beta scales the write).  Returns
(out [B,N,H,dv], delta [B,H,N,dv] = beta_t v_t, g [B,H,N] = sum of log alpha
along the path), the factor record the library's commit consumes.
DeltaNet is the GDN recurrence with alpha = 1 and needs no separate oracle.
"""
from __future__ import annotations

import numpy as np


def tree_verify(q, k, v, alpha, beta, parent, S0):
    q, k, v, alpha, beta, S0 = (np.asarray(x, np.float64) for x in (q, k, v, alpha, beta, S0))
    B, N, H, dk = q.shape
    dv = v.shape[-1]
    out = np.zeros((B, N, H, dv))
    delta = np.zeros((B, H, N, dv))
    g = np.zeros((B, H, N))
    for b in range(B):
        for t in range(N):
            path = []
            u = t
            while u >= 0:
                path.append(u)
                u = int(parent[b, u])
            path.reverse()
            for h in range(H):
                S = S0[b, h].copy()
                gs = 0.0
                for j in path:
                    S = alpha[b, j, h] * S + beta[b, j, h] * np.outer(v[b, j, h], k[b, j, h])
                    gs += np.log(alpha[b, j, h])
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
                S[b, h] = alpha[b, j, h] * S[b, h] + beta[b, j, h] * np.outer(v[b, j, h], k[b, j, h])
    return S

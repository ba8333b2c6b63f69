"""Pins for the decay-gated linear-attention oracle (oracle/linear.py), CPU only:
the attention-form closed expression (a different algorithm from the path walk),
sibling isolation, and reduction to a plain scaled S0 read-out when beta = 0."""
import numpy as np

from oracle import linear as LA
from speculative_decoding_linear_gb300 import workloads as wl


def inputs(seed, N=9, B=2, H=2, d=6):
    w = wl.custom_workload(B, N, H, d, d, wl.random_tree(np.random.default_rng(seed), N, 4), seed=seed, dtype=wl.F32)
    return w, [w.widened(n) for n in ("q", "k", "v", "alpha", "beta", "S0")]


def test_attention_form_closed_expression():
    # o_t = e^{g_t} S0 q_t + sum_{j in path(t)} e^{g_t - g_j} beta_j (k_j . q_t) v_j
    w, (q, k, v, al, be, S0) = inputs(1)
    out, delta, g = LA.tree_verify(q, k, v, al, be, w.parent, S0)
    for b in range(w.B):
        for t in range(w.N):
            path = wl.root_path(w.parent[b], t)
            for h in range(w.H):
                gt = sum(np.log(al[b, j, h]) for j in path)
                ref = np.exp(gt) * S0[b, h] @ q[b, t, h]
                for i, j in enumerate(path):
                    gj = sum(np.log(al[b, u, h]) for u in path[:i + 1])
                    ref = ref + np.exp(gt - gj) * be[b, j, h] * (k[b, j, h] @ q[b, t, h]) * v[b, j, h]
                np.testing.assert_allclose(out[b, t, h], ref, rtol=1e-12, atol=1e-12)
                np.testing.assert_allclose(g[b, h, t], gt, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(delta, np.transpose(be[..., None] * v, (0, 2, 1, 3)), rtol=0, atol=0)


def test_beta_zero_reads_the_decayed_state():
    w, (q, k, v, al, be, S0) = inputs(2)
    out, _, g = LA.tree_verify(q, k, v, al, np.zeros_like(be), w.parent, S0)
    ref = np.exp(np.transpose(g, (0, 2, 1)))[..., None] * np.einsum("bhvk,bthk->bthv", S0, q)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)


def test_sibling_isolation():
    w, (q, k, v, al, be, S0) = inputs(3, N=12, B=1)
    o0, _, _ = LA.tree_verify(q, k, v, al, be, w.parent, S0)
    j = 4
    v2 = v.copy()
    v2[0, j] += 1.0
    o1, _, _ = LA.tree_verify(q, k, v2, al, be, w.parent, S0)
    desc = {j}
    for t in range(w.N):
        if w.parent[0, t] in desc:
            desc.add(t)
    for t in range(w.N):
        if t not in desc:
            np.testing.assert_array_equal(o0[0, t], o1[0, t])


def test_commit_is_the_walk_to_the_accepted_node():
    w, (q, k, v, al, be, S0) = inputs(4)
    S = LA.commit(k, v, al, be, w.parent, S0, w.path)
    out, _, _ = LA.tree_verify(q, k, v, al, be, w.parent, S0)
    for b in range(w.B):
        a = [j for j in w.path[b] if j >= 0][-1]
        for h in range(w.H):
            np.testing.assert_allclose(S[b, h] @ q[b, a, h], out[b, a, h], rtol=1e-12, atol=1e-13)

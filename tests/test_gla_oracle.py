"""Pins for the gated-linear-attention oracle (oracle/gla.py), CPU only.

Each pin fixes the oracle by something other than itself:
* a three-node tree worked by hand (tests/golden/gla_hand_tree3.json);
* the attention-form closed expression with the gates multiplied out as plain
  products (no logs, no state matrix: a different algorithm);
* scalar gates (every channel equal) reduce it to the decay-gated linear
  attention oracle, a separately pinned implementation;
* beta = 0 reads the channel-decayed S0;
* the commit from the factor record (S0 e^{g_a} + sum delta_j (k_j e^{g_a - g_j})^T,
  the form the library's commit evaluates) equals the walk, and S_a q_a = o_a;
* perturbing a node leaves every non-descendant's output bit-identical.
"""
import json
import os

import numpy as np
import pytest

from oracle import gla as GLA
from oracle import linear as LA
from speculative_decoding_linear_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "gla_hand_tree3.json")


def inputs(seed, N=9, B=2, H=2, dk=6, dv=5, maxdepth=4):
    rng = np.random.default_rng(seed)
    parent = np.stack([wl.random_tree(rng, N, maxdepth) for _ in range(B)])
    w = wl.make_gla_workload(0, seed=seed, B=B, parent=parent, N=N, H=H, dk=dk, dv=dv)
    return w, [w.widened(n) for n in ("q", "k", "v", "alpha", "beta", "S0")]


def test_hand_worked_three_node_tree():
    G = json.load(open(GOLDEN))
    parent = np.array([G["parent"]], np.int32)
    S0 = np.array(G["S0"])[None, None]                       # [1, 1, dv = 1, dk = 2]
    al = np.array(G["alpha"])[None, :, None]                  # [1, 3, 1, 2]
    be = np.array(G["beta"])[None, :, None]
    k = np.array(G["k"])[None, :, None]
    v = np.array(G["v"])[None, :, None]
    q = np.array(G["q"])[None, :, None]
    out, delta, g = GLA.tree_verify(q, k, v, al, be, parent, S0)
    np.testing.assert_allclose(out[0, :, 0], np.array(G["out"]), rtol=0, atol=1e-15)
    np.testing.assert_allclose(delta[0, 0], np.array(G["delta"]), rtol=0, atol=0)
    np.testing.assert_allclose(np.exp(g[0, 0]), np.array(G["g_exp"]), rtol=1e-15)
    for name, p in (("path_0_1", [0, 1]), ("path_2", [2, -1]), ("empty", [-1, -1])):
        S = GLA.commit(k, v, al, be, parent, S0, np.array([p], np.int32))
        np.testing.assert_allclose(S[0, 0], np.array(G["commit"][name]), rtol=0, atol=1e-15)


def test_attention_form_with_explicit_gate_products():
    # o_t = S0 (prod_{i in path(t)} alpha_i (.) q_t) + sum_{j in path(t)} beta_j v_j
    #       * sum_c q_t[c] k_j[c] prod_{i in path(t) after j} alpha_i[c]
    w, (q, k, v, al, be, S0) = inputs(1)
    out, _, g = GLA.tree_verify(q, k, v, al, be, w.parent, S0)
    for b in range(w.B):
        for t in range(w.N):
            path = wl.root_path(w.parent[b], t)
            for h in range(w.H):
                decay = np.ones(w.dk)
                for j in path:
                    decay = decay * al[b, j, h]
                ref = S0[b, h] @ (decay * q[b, t, h])
                for i, j in enumerate(path):
                    after = np.ones(w.dk)
                    for u in path[i + 1:]:
                        after = after * al[b, u, h]
                    ref = ref + be[b, j, h] * np.sum(q[b, t, h] * k[b, j, h] * after) * v[b, j, h]
                np.testing.assert_allclose(out[b, t, h], ref, rtol=1e-12, atol=1e-13)
                np.testing.assert_allclose(np.exp(g[b, h, t]), decay, rtol=1e-12)


def test_scalar_gates_reduce_to_decay_gated_linear_attention():
    w, (q, k, v, al, be, S0) = inputs(2)
    a1 = al[..., :1]                                          # one gate per node, copied to every channel
    out, delta, g = GLA.tree_verify(q, k, v, np.broadcast_to(a1, al.shape), be, w.parent, S0)
    o_ref, d_ref, g_ref = LA.tree_verify(q, k, v, a1[..., 0], be, w.parent, S0)
    np.testing.assert_allclose(out, o_ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(delta, d_ref, rtol=0, atol=0)
    np.testing.assert_allclose(g, np.broadcast_to(g_ref[..., None], g.shape), rtol=1e-13, atol=1e-14)


def test_beta_zero_reads_the_channel_decayed_state():
    w, (q, k, v, al, be, S0) = inputs(3)
    out, _, g = GLA.tree_verify(q, k, v, al, np.zeros_like(be), w.parent, S0)
    ref = np.einsum("bhvk,bthk->bthv", S0, np.exp(np.transpose(g, (0, 2, 1, 3))) * q)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("seed", [4, 5])
def test_commit_from_the_factor_record_equals_the_walk(seed):
    w, (q, k, v, al, be, S0) = inputs(seed, N=12, maxdepth=6)
    out, delta, g = GLA.tree_verify(q, k, v, al, be, w.parent, S0)
    S_walk = GLA.commit(k, v, al, be, w.parent, S0, w.path)
    for b in range(w.B):
        acc = [int(j) for j in w.path[b] if j >= 0]
        a = acc[-1]
        for h in range(w.H):
            S = S0[b, h] * np.exp(g[b, h, a])[None, :]
            for j in acc:
                S = S + np.outer(delta[b, h, j], k[b, j, h] * np.exp(g[b, h, a] - g[b, h, j]))
            np.testing.assert_allclose(S_walk[b, h], S, rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(S_walk[b, h] @ q[b, a, h], out[b, a, h], rtol=1e-12, atol=1e-13)
    empty = np.full_like(w.path, -1)
    assert np.array_equal(GLA.commit(k, v, al, be, w.parent, S0, empty), S0)


def test_sibling_isolation():
    w, (q, k, v, al, be, S0) = inputs(6, N=10)
    out, _, _ = GLA.tree_verify(q, k, v, al, be, w.parent, S0)
    b, node = 1, 3
    k2 = k.copy()
    k2[b, node] += 0.5
    al2 = al.copy()
    al2[b, node] *= 0.5
    out2, _, _ = GLA.tree_verify(q, k2, v, al2, be, w.parent, S0)
    desc = {t for t in range(w.N) if node in wl.root_path(w.parent[b], t)}
    for t in range(w.N):
        same = np.array_equal(out2[b, t], out[b, t])
        assert same == (t not in desc)
    assert np.array_equal(out2[0], out[0])

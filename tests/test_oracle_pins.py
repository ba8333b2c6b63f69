"""Pins for the fp64 oracle (CPU only).

Each test ties the oracle to something other than itself: a value worked by
hand, a closed form of the recurrence, an invariant the review pages state
(sibling isolation, commit equals the sequential state), a brute-force
alternative (explicit (I - beta k k^T) matrices carried node by node), or the
pages' own factorized verifier written out with a library triangular solve.
Together they fail on a dropped term, a wrong sign, a wrong index or parent,
a transposed state or a misplaced gate anywhere in the oracle.
"""
import json
import os

import numpy as np
import pytest
import scipy.linalg

from speculative_decoding_linear_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _inputs(w):
    return dict(q=w.widened("q"), k=w.widened("k"), v=w.widened("v"),
                alpha=w.alpha.astype(np.float64), beta=w.beta.astype(np.float64),
                parent=w.parent, S0=w.S0.astype(np.float64))


def _rel(a, b):
    return np.max(np.abs(a - b)) / max(np.sqrt(np.mean(b ** 2)), 1e-300)


# ---------------------------------------------------------------------------
# worked example
# ---------------------------------------------------------------------------
def test_hand_worked_tree(oracle_mod):
    g = json.load(open(os.path.join(GOLDEN, "hand_tree3_d2.json")))
    N, d = 3, 2
    k = np.array(g["k"], float).reshape(1, N, 1, d)
    v = np.array(g["v"], float).reshape(1, N, 1, d)
    q = np.array(g["q"], float).reshape(1, N, 1, d)
    a = np.array(g["alpha"], float).reshape(1, N, 1)
    b = np.array(g["beta"], float).reshape(1, N, 1)
    par = np.array(g["parent"], np.int32).reshape(1, N)
    S0 = np.array(g["S0"], float).reshape(1, 1, d, d)
    out, delta, gg = oracle_mod.tree_verify(q, k, v, a, b, par, S0)
    np.testing.assert_allclose(out[0, :, 0], np.array(g["out"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(delta[0, 0], np.array(g["delta"]), rtol=0, atol=1e-14)
    np.testing.assert_allclose(gg[0, 0] / np.log(0.5), np.array(g["g_over_ln_half"]), atol=1e-14)
    for key, want in g["commits"].items():
        nodes = [int(x) for x in key.split(",")] if key else []
        path = np.full((1, 2), -1, np.int32)
        path[0, : len(nodes)] = nodes
        S = oracle_mod.commit(k, v, a, b, par, S0, path)
        np.testing.assert_allclose(S[0, 0], np.array(want), rtol=0, atol=1e-14)


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------
def _path_gate(parent_row, alpha_bh, t):
    return np.prod([alpha_bh[j] for j in wl.root_path(parent_row, t)])


@pytest.mark.parametrize("seed", [0, 1])
def test_beta_zero_is_pure_decay(oracle_mod, seed):
    """beta = 0 removes every write: o_t = (prod of alpha over path(t)) S0 q_t, delta = 0."""
    w = wl.make_workload(wl.Spec("t", 2, 12, 2, 8, 6, wl.F32, "random", 4, "uniform_node", 0.3, seed))
    x = _inputs(w)
    x["beta"] = np.zeros_like(x["beta"])
    out, delta, g = oracle_mod.tree_verify(**x)
    for b in range(2):
        for h in range(2):
            for t in range(12):
                gate = _path_gate(w.parent[b], x["alpha"][b, :, h], t)
                want = gate * x["S0"][b, h] @ x["q"][b, t, h]
                np.testing.assert_allclose(out[b, t, h], want, rtol=1e-13, atol=1e-15)
                np.testing.assert_allclose(g[b, h, t], np.log(gate), rtol=1e-13)
    assert np.all(delta == 0)


def test_write_then_read_returns_value(oracle_mod):
    """beta_t = 1, |k_t| = 1 and q_t = k_t: S_t k_t = v_t whatever alpha and the state."""
    w = wl.make_workload(wl.Spec("t", 2, 16, 3, 16, 8, wl.F32, "random", 5, "uniform_node", 0.5, 7))
    x = _inputs(w)
    x["k"] = x["k"] / np.linalg.norm(x["k"], axis=-1, keepdims=True)
    x["q"] = x["k"].copy()
    x["beta"] = np.ones_like(x["beta"])
    out, _, _ = oracle_mod.tree_verify(**x)
    np.testing.assert_allclose(out, x["v"], rtol=0, atol=1e-12)


def test_query_orthogonal_to_all_keys(oracle_mod):
    """If q is orthogonal to every key on the path, writes are invisible: o_t = e^{g_t} S0 q_t."""
    rng = np.random.default_rng(3)
    w = wl.make_workload(wl.Spec("t", 1, 10, 2, 8, 5, wl.F32, "random", 3, "uniform_node", 0.4, 3))
    x = _inputs(w)
    x["k"][..., 0] = 0.0            # every key lives in span(e_1..e_7)
    x["q"] = np.zeros_like(x["q"])
    x["q"][..., 0] = rng.uniform(0.5, 2.0, x["q"].shape[:-1])
    out, _, _ = oracle_mod.tree_verify(**x)
    for h in range(2):
        for t in range(10):
            gate = _path_gate(w.parent[0], x["alpha"][0, :, h], t)
            np.testing.assert_allclose(out[0, t, h], gate * x["S0"][0, h] @ x["q"][0, t, h],
                                       rtol=1e-13, atol=1e-15)


# ---------------------------------------------------------------------------
# brute force: explicit matrices, one stored state per node
# ---------------------------------------------------------------------------
def _brute_states(x, b, h):
    """Carry an explicit state per node: S_t = alpha S_parent (I - beta k k^T) + beta v k^T."""
    N = x["parent"].shape[1]
    dk = x["k"].shape[-1]
    S = {}
    for t in range(N):
        p = x["parent"][b, t]
        Sp = x["S0"][b, h] if p < 0 else S[p]
        kt, vt = x["k"][b, t, h], x["v"][b, t, h]
        a, be = x["alpha"][b, t, h], x["beta"][b, t, h]
        S[t] = a * Sp @ (np.eye(dk) - be * np.outer(kt, kt)) + be * np.outer(vt, kt)
    return S


@pytest.mark.parametrize("cfg", [0, "forest", "chain"])
def test_brute_force_explicit_matrices(oracle_mod, cfg):
    if cfg == 0:
        w = wl.make_workload(0)
    elif cfg == "chain":
        w = wl.custom_workload(1, 7, 2, 6, 5, wl.chain_tree(7), seed=11, dtype=wl.F32)
    else:   # a forest: two roots hanging under S0
        w = wl.custom_workload(2, 7, 2, 6, 4, [-1, 0, -1, 1, 2, 0, 4], seed=12, dtype=wl.F32)
    x = _inputs(w)
    out, delta, _ = oracle_mod.tree_verify(**x)
    for b in range(w.B):
        for h in range(w.H):
            S = _brute_states(x, b, h)
            for t in range(w.N):
                np.testing.assert_allclose(out[b, t, h], S[t] @ x["q"][b, t, h], rtol=1e-12, atol=1e-13)
                p = w.parent[b, t]
                Sp = x["S0"][b, h] if p < 0 else S[p]
                # S_t = alpha_t S_parent + delta_t k_t^T defines delta_t
                np.testing.assert_allclose(np.outer(delta[b, h, t], x["k"][b, t, h]),
                                           S[t] - x["alpha"][b, t, h] * Sp, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------
# invariants stated by the pages
# ---------------------------------------------------------------------------
def _descendants(parent, j):
    out = {j}
    for t in range(j + 1, len(parent)):
        if parent[t] in out:
            out.add(t)
    return out


@pytest.mark.parametrize("victim", [1, 4, 9])
def test_sibling_isolation_bit_identical(oracle_mod, victim):
    """Perturbing one node changes its subtree and leaves every other node's output bit-identical."""
    w = wl.make_workload(wl.Spec("t", 1, 14, 2, 8, 8, wl.F32, "random", 4, "uniform_node", 0.2, 21))
    x = _inputs(w)
    out0, d0, g0 = oracle_mod.tree_verify(**x)
    y = {kk: vv.copy() for kk, vv in x.items()}
    y["k"][0, victim] += 0.3
    y["v"][0, victim] -= 0.7
    y["alpha"][0, victim] *= 0.5
    y["beta"][0, victim] = 0.9
    out1, d1, g1 = oracle_mod.tree_verify(**y)
    desc = _descendants(w.parent[0], victim)
    for t in range(w.N):
        if t in desc:
            assert np.max(np.abs(out1[0, t] - out0[0, t])) > 1e-6
        else:
            assert np.array_equal(out1[0, t], out0[0, t])
            assert np.array_equal(d1[0, :, t], d0[0, :, t])
            assert np.array_equal(g1[0, :, t], g0[0, :, t])


def test_relabelling_permutes_outputs(oracle_mod):
    """Another topological numbering of the same tree permutes the outputs bit-identically."""
    w = wl.make_workload(wl.Spec("t", 1, 12, 2, 8, 8, wl.F32, "random", 5, "uniform_node", 0.2, 5))
    x = _inputs(w)
    par = w.parent[0]
    # a different topological order: repeatedly take the highest-index ready node
    order, placed = [], set()
    while len(order) < w.N:
        ready = [t for t in range(w.N) if t not in placed and (par[t] < 0 or par[t] in placed)]
        order.append(ready[-1])
        placed.add(ready[-1])
    new_of = {old: new for new, old in enumerate(order)}
    perm = np.array(order)
    y = {kk: vv.copy() for kk, vv in x.items()}
    for name in ("q", "k", "v", "alpha", "beta"):
        y[name] = x[name][:, perm]
    y["parent"] = np.array([[-1 if par[o] < 0 else new_of[par[o]] for o in order]], np.int32)
    out0, d0, g0 = oracle_mod.tree_verify(**x)
    out1, d1, g1 = oracle_mod.tree_verify(**y)
    assert np.array_equal(out1, out0[:, perm])
    assert np.array_equal(d1, d0[:, :, perm])
    assert np.array_equal(g1, g0[:, :, perm])


def test_commit_equals_sequential_state(oracle_mod):
    w = wl.make_workload(3, B=4)
    x = _inputs(w)
    S_new = oracle_mod.commit(x["k"], x["v"], x["alpha"], x["beta"], w.parent, x["S0"], w.path)
    for b in range(w.B):
        L = int(np.sum(w.path[b] >= 0))
        for h in (0, 5):
            S = x["S0"][b, h].copy()
            for j in w.path[b, :L]:
                kt, vt = x["k"][b, j, h], x["v"][b, j, h]
                a, be = x["alpha"][b, j, h], x["beta"][b, j, h]
                S = a * S @ (np.eye(w.dk) - be * np.outer(kt, kt)) + be * np.outer(vt, kt)
            assert _rel(S_new[b, h], S) < 1e-12


def test_commit_reads_back_verified_output(oracle_mod):
    """The committed state of the accepted node a reproduces that node's verified output: S_new q_a = o_a."""
    w = wl.make_workload(2)
    x = _inputs(w)
    out, _, _ = oracle_mod.tree_verify(**x)
    S_new = oracle_mod.commit(x["k"], x["v"], x["alpha"], x["beta"], w.parent, x["S0"], w.path)
    L = int(np.sum(w.path[0] >= 0))
    a = w.path[0, L - 1]
    for h in range(w.H):
        np.testing.assert_allclose(S_new[0, h] @ x["q"][0, a, h], out[0, a, h], rtol=1e-12, atol=1e-13)


def test_empty_commit_is_identity(oracle_mod):
    w = wl.make_workload(1)
    x = _inputs(w)
    path = np.full_like(w.path, -1)
    S_new = oracle_mod.commit(x["k"], x["v"], x["alpha"], x["beta"], w.parent, x["S0"], path)
    assert np.array_equal(S_new, x["S0"])


# ---------------------------------------------------------------------------
# the pages' factorized verifier, written out with a library triangular solve
# ---------------------------------------------------------------------------
def factorized_reference(x, b, h):
    """A_tree = M (.) (K_b K_a^T), T = solve_tril(I - A_tree), U/W factors,
    O = Qhat S0^T - Attn (W S0^T) + Attn U, with the readings: K_b = diag(beta e^g) K,
    K_a = diag(e^-g) K, A_tree = -(strict mask (.) K_b K_a^T), Qhat = diag(e^g) Q,
    Attn = inclusive mask (.) e^{g_t - g_j} (.) Q K^T."""
    par = x["parent"][b]
    N = len(par)
    K, Q, V = x["k"][b, :, h], x["q"][b, :, h], x["v"][b, :, h]
    beta = x["beta"][b, :, h]
    g = np.array([np.sum(np.log(x["alpha"][b, wl.root_path(par, t), h])) for t in range(N)])
    strict = np.zeros((N, N))
    for t in range(N):
        for j in wl.root_path(par, t)[:-1]:
            strict[t, j] = 1.0
    incl = strict + np.eye(N)
    gamma = np.where(incl > 0, np.exp(np.subtract.outer(g, g) * (incl > 0)), 0.0)
    A_tree = -(strict * beta[:, None] * gamma * (K @ K.T))
    T = scipy.linalg.solve_triangular(np.eye(N) - A_tree, np.eye(N), lower=True)
    U = T @ (beta[:, None] * V)
    W = T @ ((beta * np.exp(g))[:, None] * K)
    Attn = incl * gamma * (Q @ K.T)
    S0 = x["S0"][b, h]
    Qhat = np.exp(g)[:, None] * Q
    O = Qhat @ S0.T - Attn @ (W @ S0.T) + Attn @ U
    Delta = U - W @ S0.T
    return O, Delta, g, T, incl


@pytest.mark.parametrize("cfg", [0, 2, 3])
def test_factorized_form_matches_walk(oracle_mod, cfg):
    w = wl.make_workload(cfg, B=2 if cfg == 3 else None)
    x = _inputs(w)
    out, delta, g = oracle_mod.tree_verify(**x)
    for b in range(w.B):
        for h in range(min(w.H, 3)):
            O, Delta, gf, T, incl = factorized_reference(x, b, h)
            assert _rel(out[b, :, h], O) < 1e-12
            assert _rel(delta[b, h], Delta) < 1e-12
            np.testing.assert_allclose(g[b, h], gf, rtol=1e-13)
            assert np.all(T[incl == 0] == 0.0)     # T lives on the inclusive ancestor mask
            # commit in factor form: S_a = e^{g_a} S0 + sum_{j in path(a)} e^{g_a - g_j} delta_j k_j^T
            L = int(np.sum(w.path[b] >= 0))
            if L:
                a = w.path[b, L - 1]
                S_f = np.exp(gf[a]) * x["S0"][b, h]
                for j in w.path[b, :L]:
                    S_f = S_f + np.exp(gf[a] - gf[j]) * np.outer(Delta[j], x["k"][b, j, h])
                S_new = oracle_mod.commit(x["k"][b:b + 1], x["v"][b:b + 1], x["alpha"][b:b + 1],
                                          x["beta"][b:b + 1], w.parent[b:b + 1], x["S0"][b:b + 1],
                                          w.path[b:b + 1])
                assert _rel(S_new[0, h], S_f) < 1e-12


# ---------------------------------------------------------------------------
# topology and invalid input
# ---------------------------------------------------------------------------
def test_tree_meta_binary_tree(oracle_mod):
    mask, depth = oracle_mod.tree_meta(wl.binary_tree_depth2()[None])
    assert mask[0].tolist() == [0, 0b1, 0b1, 0b11, 0b11, 0b101, 0b101]
    assert depth[0].tolist() == [0, 1, 1, 2, 2, 2, 2]


def test_tree_meta_chain_and_forest(oracle_mod):
    mask, depth = oracle_mod.tree_meta(wl.chain_tree(64)[None])
    assert [int(m) for m in mask[0]] == [(1 << t) - 1 for t in range(64)]
    assert depth[0].tolist() == list(range(64))
    mask, depth = oracle_mod.tree_meta(np.array([[-1, -1, 0, 1, 3]], np.int32))
    assert mask[0].tolist() == [0, 0, 0b1, 0b10, 0b1010]
    assert depth[0].tolist() == [0, 0, 1, 1, 2]


@pytest.mark.parametrize("bad", [[-1, 1, 0], [-1, 0, 5], [-2, 0, 1]])
def test_invalid_parent_rejected(oracle_mod, bad):
    w = wl.custom_workload(1, 3, 1, 4, 4, [-1, 0, 1], seed=1, dtype=wl.F32)
    x = _inputs(w)
    x["parent"] = np.array([bad], np.int32)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.tree_verify(**x)


@pytest.mark.parametrize("path", [[1, -1], [0, 0], [-1, 0], [0, 1, 2], [0, 3]])
def test_invalid_path_rejected(oracle_mod, path):
    w = wl.custom_workload(1, 3, 1, 4, 4, [-1, 0, 0], seed=1, dtype=wl.F32)
    x = _inputs(w)
    p = np.full((1, 3), -1, np.int32)
    p[0, : len(path)] = path
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.commit(x["k"], x["v"], x["alpha"], x["beta"], w.parent, x["S0"], p)

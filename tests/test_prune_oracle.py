"""Pins for the pruning oracle (oracle/prune.py), CPU only: a hand-worked tree,
closed-form limits (no margin and a large budget keep everything; a zero
margin keeps a single best child per node) and invariants on random trees."""
import numpy as np
import pytest

from oracle import prune as P
from speculative_decoding_linear_gb300 import workloads as wl

PARENT = np.array([-1, 0, 0, 1, 1, 2], np.int32)
LOGP = np.array([0.0, -0.1, -1.0, -0.2, -3.0, -0.1])


def test_hand_tree_margin():
    # path scores: 0, -0.1, -1.0, -0.3, -3.1, -1.1
    idx, par, n = P.prune(PARENT, LOGP, tau=0.5, budget=64)
    assert n == 3 and idx.tolist() == [0, 1, -1, 2, -1, -1] and par.tolist() == [-1, 0, 1]
    idx, par, n = P.prune(PARENT, LOGP, tau=1.0, budget=64)
    assert idx.tolist() == [0, 1, 2, 3, -1, 4] and par.tolist() == [-1, 0, 0, 1, 2]


def test_hand_tree_budget():
    idx, par, n = P.prune(PARENT, LOGP, tau=1.0, budget=3)
    assert idx.tolist() == [0, 1, -1, 2, -1, -1] and par.tolist() == [-1, 0, 1]
    idx, par, n = P.prune(PARENT, LOGP, tau=1.0, budget=4)
    assert idx.tolist() == [0, 1, 2, 3, -1, -1] and par.tolist() == [-1, 0, 0, 1]
    assert P.prune(PARENT, LOGP, tau=1.0, budget=0)[2] == 0


def _random(seed, n=40, depth=6):
    rng = np.random.default_rng(seed)
    parent = wl.random_tree(rng, n, depth)
    logp = -rng.exponential(1.0, n)
    return parent, logp


@pytest.mark.parametrize("seed", range(6))
def test_no_margin_large_budget_keeps_all(seed):
    parent, logp = _random(seed)
    idx, par, n = P.prune(parent, logp, tau=np.inf, budget=1000)
    assert n == len(parent) and idx.tolist() == list(range(len(parent))) and np.array_equal(par, parent)


@pytest.mark.parametrize("seed", range(6))
def test_zero_margin_keeps_one_best_child(seed):
    parent, logp = _random(seed)
    idx, par, n = P.prune(parent, logp, tau=0.0, budget=1000)
    kids = np.bincount(par[par >= 0], minlength=n) if n else np.zeros(0)
    assert np.all(kids <= 1) and np.count_nonzero(par < 0) == 1


@pytest.mark.parametrize("seed", range(8))
def test_closed_under_ancestors_and_budget(seed):
    parent, logp = _random(seed, n=50)
    rng = np.random.default_rng(100 + seed)
    tau, budget = float(rng.uniform(0, 3)), int(rng.integers(1, 50))
    idx, par, n = P.prune(parent, logp, tau, budget)
    assert n <= budget
    kept = np.nonzero(idx >= 0)[0]
    for u in kept:
        assert parent[u] < 0 or idx[parent[u]] >= 0
        assert par[idx[u]] == (idx[parent[u]] if parent[u] >= 0 else -1)
    assert all(par[i] < i for i in range(n))
    # brute force of the budget rule: no pruned survivor scores above a kept node
    s = P.path_scores(parent, logp)
    surv = [u for u in range(len(parent)) if s[u] >= np.float32(max(s[w] for w in range(len(parent)) if parent[w] == parent[u]) - np.float32(tau))]
    surv = [u for u in surv if all(v in surv for v in wl.root_path(parent, u))]
    if len(surv) > budget:
        assert min(s[kept]) >= max(s[u] for u in surv if idx[u] < 0)
    else:
        assert sorted(kept.tolist()) == sorted(surv)

"""Confidence-guided draft-tree pruning -- TEST INFRASTRUCTURE ONLY (oracle).

Plain Python definition of the pruning rule the library applies before
verification.  Source: "Pith review of SpecLA: Efficient Speculative Decoding
for Linear-Attention Models" (pith.science 7ERME3HB), which names
"confidence-guided tree pruning" with a tree margin tau_tree and a draft
budget (Referee Report, minor comment on Section 6.1) without defining them;
the reading used here:

* score(t) = sum of the drafter's log-probabilities along path(t) (each node's
  log-probability given its parent);
* margin: node t survives if score(t) >= max over its siblings s (nodes with
  the same parent, t included) of score(s) - tau, and its parent survives;
* budget: of the survivors, the `budget` nodes with the highest score are kept,
  ties going to the lower node index (log-probabilities are <= 0, so a parent
  never scores below its child and the kept set stays closed under ancestors);
* the kept nodes keep their relative order and are renumbered 0..n-1; their
  parents are renumbered with them (-1 stays -1).

Scores and comparisons are fp32 (the precision the library decides in), each
score formed root first as fl(logp_t + score(parent)), and the margin test as
score(t) >= fl(best - tau).

Returns (new_index [N] int32, -1 for pruned nodes; new_parent [n] int32; n).
"""
from __future__ import annotations

import numpy as np


def path_scores(parent, logp):
    parent = np.asarray(parent)
    logp = np.asarray(logp, dtype=np.float32)
    s = np.zeros(len(parent), dtype=np.float32)
    for t in range(len(parent)):
        s[t] = logp[t] + (s[parent[t]] if parent[t] >= 0 else np.float32(0.0))
    return s


def prune(parent, logp, tau, budget):
    parent = np.asarray(parent, dtype=np.int64)
    N = len(parent)
    s = path_scores(parent, logp)
    alive = np.zeros(N, dtype=bool)
    for t in range(N):
        sib = [u for u in range(N) if parent[u] == parent[t]]
        best = max(s[u] for u in sib)
        ok = s[t] >= np.float32(best - np.float32(tau))
        alive[t] = ok and (parent[t] < 0 or alive[parent[t]])
    order = sorted((u for u in range(N) if alive[u]), key=lambda u: (-s[u], u))
    kept = sorted(order[:max(0, budget)])
    new_index = np.full(N, -1, dtype=np.int32)
    for i, u in enumerate(kept):
        new_index[u] = i
    new_parent = np.array([new_index[parent[u]] if parent[u] >= 0 else -1 for u in kept], dtype=np.int32)
    return new_index, new_parent, len(kept)

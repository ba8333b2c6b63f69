"""Seeded synthetic inputs for tree verification and accepted-path commit.

This module only *draws inputs*: draft-tree topologies, queries/keys/values,
gates, initial recurrent states and accepted paths.  It holds none of the
verifier's or the commit's arithmetic.  The CUDA path's tests, the benchmark
and the oracle's tests all take their inputs from here, so both sides of every
parity check see the same bits.

Shapes and distributions follow the single-GDN-layer workload of the SpecLA
review pages (pith.science 7ERME3HB, "Referee Report", major comment 1: one GDN
layer shaped like GDN-1.3B, h_v = 8, d_k = d_v = 256, fp32 recurrent state):

* q, k ~ N(0, 1), L2-normalised per (token, head), then rounded to bf16
  (round-to-nearest-even); v ~ N(0, 1) rounded to bf16.  The tiny case keeps
  q/k/v in fp32.
* beta = sigmoid(U(-2, 2)); alpha = exp(-softplus(U(-3, 1))), in [0.27, 0.95].
* S0 ~ N(0, 0.1) for the tiny case, N(0, 0.05) otherwise; layout [B, H, d_v, d_k].
* Draft trees: node 0 is a root (parent -1); node i >= 1 picks its parent
  uniformly among the earlier nodes whose depth is below the maximum depth.
* Accepted paths: root-first node lists, padded with -1, shape [B, Lmax].

Random numbers come from numpy's ``default_rng`` (PCG64) with a fixed draw
order: trees, then q, k, v, then the alpha and beta pre-activations, then S0,
then accepted paths.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

BF16 = "bf16"
F32 = "f32"


# ---------------------------------------------------------------------------
# dtype helpers (conversions only)
# ---------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest, ties to even); return the uint16 bit patterns."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounding = ((b >> 16) & 1) + 0x7FFF
    return ((b + rounding) >> 16).astype(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float64 exactly."""
    u = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# topologies
# ---------------------------------------------------------------------------
def chain_tree(n: int) -> np.ndarray:
    """parent_idx of a linear chain: node t hangs under t-1, node 0 under the committed state."""
    return (np.arange(n, dtype=np.int32) - 1).astype(np.int32)


def binary_tree_depth2() -> np.ndarray:
    """Full binary draft tree of depth 2 (7 nodes), nodes numbered breadth-first."""
    return np.array([-1, 0, 0, 1, 1, 2, 2], dtype=np.int32)


def random_tree(rng: np.random.Generator, n: int, maxdepth: int) -> np.ndarray:
    """Node 0 is the root; node i picks its parent uniformly among earlier nodes of depth < maxdepth
    (with maxdepth 0 every node is a root)."""
    parent = np.full(n, -1, dtype=np.int32)
    depth = np.zeros(n, dtype=np.int64)
    for i in range(1, n):
        eligible = np.nonzero(depth[:i] < maxdepth)[0]
        if len(eligible) == 0:          # maxdepth 0: every node is a root (a forest)
            continue
        p = int(eligible[rng.integers(len(eligible))])
        parent[i] = p
        depth[i] = depth[p] + 1
    return parent


def narrow_tree(n: int, chains: int, trunk: int) -> np.ndarray:
    """Deep, narrow draft tree: a trunk of ``trunk`` nodes (0 .. trunk-1) and ``chains`` chains
    hanging from its last node, numbered chain by chain; the last chain takes the remainder."""
    assert 1 <= trunk <= n and chains >= 1
    parent = chain_tree(trunk).tolist()
    rest = n - trunk
    per = rest // chains
    for c in range(chains):
        length = per if c < chains - 1 else rest - per * (chains - 1)
        for i in range(length):
            parent.append(trunk - 1 if i == 0 else len(parent) - 1)
    return np.asarray(parent, dtype=np.int32)


def node_depths(parent: np.ndarray) -> np.ndarray:
    """Depth of every node of a topologically ordered parent array (roots have depth 0)."""
    d = np.zeros(len(parent), dtype=np.int64)
    for i, p in enumerate(parent):
        d[i] = 0 if p < 0 else d[p] + 1
    return d


def root_path(parent: np.ndarray, node: int) -> list:
    """Node list from the root down to ``node`` (inclusive)."""
    out = []
    t = int(node)
    while t >= 0:
        out.append(t)
        t = int(parent[t])
    return out[::-1]


def _pad_path(path: list, lmax: int) -> np.ndarray:
    row = np.full(lmax, -1, dtype=np.int32)
    row[: len(path)] = path
    return row


# ---------------------------------------------------------------------------
# workload specs
# ---------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Spec:
    name: str
    B: int
    N: int
    H: int
    dk: int
    dv: int
    dtype: str            # q/k/v storage type: "bf16" or "f32"
    tree: str             # "binary7", "chain" or "random"
    maxdepth: int         # maximum node depth (root = 0)
    path_rule: str        # "fixed", "prefix", "uniform_node", "uniform_len"
    s0_std: float
    seed: int
    hidden: int = 0       # > 0 for the full-layer workload

    @property
    def lmax(self) -> int:
        return self.maxdepth + 1


# The five synthetic workloads: tiny oracle check, chain verify, tree verify,
# batched tree verify + commit, full GDN layer decode step.
SPECS = {
    0: Spec("tiny_binary7_d16", 1, 7, 1, 16, 16, F32, "binary7", 2, "fixed", 0.1, 0),
    1: Spec("chain8_b1_h8_d256", 1, 8, 8, 256, 256, BF16, "chain", 7, "prefix", 0.05, 1),
    2: Spec("tree32_depth6_b1_h8_d256", 1, 32, 8, 256, 256, BF16, "random", 6, "uniform_node", 0.05, 2),
    3: Spec("tree64_depth8_b16_h8_d256", 16, 64, 8, 256, 256, BF16, "random", 8, "uniform_len", 0.05, 3),
    4: Spec("layer_tree64_depth8_b64_hid2048", 64, 64, 8, 256, 256, BF16, "random", 8, "uniform_node", 0.05, 4,
            hidden=2048),
}


@dataclasses.dataclass
class Workload:
    spec: Spec
    B: int
    N: int
    H: int
    dk: int
    dv: int
    dtype: str
    q: np.ndarray          # bf16 bits (uint16) or float32, [B, N, H, dk]
    k: np.ndarray          # same, [B, N, H, dk]
    v: np.ndarray          # same, [B, N, H, dv]
    alpha: np.ndarray      # float32 [B, N, H]
    beta: np.ndarray       # float32 [B, N, H]
    parent: np.ndarray     # int32 [B, N]
    S0: np.ndarray         # float32 [B, H, dv, dk]
    path: np.ndarray       # int32 [B, Lmax], root first, -1 padded

    def widened(self, name: str) -> np.ndarray:
        """float64 copy of q/k/v/alpha/beta/S0 exactly as stored (bf16 or fp32 values)."""
        x = getattr(self, name)
        if x.dtype == np.uint16:
            return bf16_bits_to_f64(x)
        return x.astype(np.float64)


def _unit_rows(x: np.ndarray) -> np.ndarray:
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _store(x: np.ndarray, dtype: str) -> np.ndarray:
    x32 = x.astype(np.float32)
    return f32_to_bf16_bits(x32) if dtype == BF16 else x32


def draw_trees(rng: np.random.Generator, spec: Spec, B: int) -> np.ndarray:
    if spec.tree == "binary7":
        return np.stack([binary_tree_depth2() for _ in range(B)])
    if spec.tree == "chain":
        return np.stack([chain_tree(spec.N) for _ in range(B)])
    return np.stack([random_tree(rng, spec.N, spec.maxdepth) for _ in range(B)])


def draw_paths(rng: np.random.Generator, spec: Spec, parent: np.ndarray) -> np.ndarray:
    B = parent.shape[0]
    out = np.full((B, spec.lmax), -1, dtype=np.int32)
    for b in range(B):
        par = parent[b]
        if spec.path_rule == "fixed":            # root -> left -> left
            path = [0, 1, 3]
        elif spec.path_rule == "prefix":         # accepted prefix of a chain, L ~ U{0..N}
            L = int(rng.integers(0, spec.N + 1))
            path = list(range(L))
        elif spec.path_rule == "uniform_node":   # root to a uniformly chosen node
            path = root_path(par, int(rng.integers(spec.N)))
        elif spec.path_rule == "uniform_len":    # L ~ U{1..8}, then a node of depth L-1
            depth = node_depths(par)
            while True:
                L = int(rng.integers(1, 9))
                cands = np.nonzero(depth == L - 1)[0]
                if len(cands):
                    break
            path = root_path(par, int(cands[rng.integers(len(cands))]))
        else:
            raise ValueError(spec.path_rule)
        out[b] = _pad_path(path, spec.lmax)
    return out


def make_workload(cfg, seed: Optional[int] = None, B: Optional[int] = None) -> Workload:
    """Draw one instance of workload ``cfg`` (an index into SPECS or a Spec).

    ``seed`` overrides the spec's seed (used for extra layer instances and
    fuzzing); ``B`` overrides the batch size.
    """
    spec = SPECS[cfg] if isinstance(cfg, int) else cfg
    B = spec.B if B is None else B
    rng = np.random.default_rng(spec.seed if seed is None else seed)
    N, H, dk, dv = spec.N, spec.H, spec.dk, spec.dv
    parent = draw_trees(rng, spec, B).astype(np.int32)
    q = _unit_rows(rng.standard_normal((B, N, H, dk)))
    k = _unit_rows(rng.standard_normal((B, N, H, dk)))
    v = rng.standard_normal((B, N, H, dv))
    a_pre = rng.uniform(-3.0, 1.0, (B, N, H))
    b_pre = rng.uniform(-2.0, 2.0, (B, N, H))
    alpha = np.exp(-np.logaddexp(0.0, a_pre)).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-b_pre))).astype(np.float32)
    S0 = (rng.standard_normal((B, H, dv, dk)) * spec.s0_std).astype(np.float32)
    path = draw_paths(rng, spec, parent)
    return Workload(spec, B, N, H, dk, dv, spec.dtype,
                    _store(q, spec.dtype), _store(k, spec.dtype), _store(v, spec.dtype),
                    alpha, beta, parent, S0, path)


def custom_workload(B: int, N: int, H: int, dk: int, dv: int, parent: np.ndarray, seed: int,
                    dtype: str = BF16, s0_std: float = 0.05, path: Optional[np.ndarray] = None,
                    lmax: Optional[int] = None) -> Workload:
    """Workload with a caller-chosen topology (edge cases, fuzzing).

    ``parent`` is [N] (shared by every batch element) or [B, N].  When no
    ``path`` is given, each batch element accepts root -> a uniformly drawn node.
    """
    parent = np.asarray(parent, dtype=np.int32)
    if parent.ndim == 1:
        parent = np.broadcast_to(parent, (B, N)).copy()
    rng = np.random.default_rng(seed)
    q = _unit_rows(rng.standard_normal((B, N, H, dk)))
    k = _unit_rows(rng.standard_normal((B, N, H, dk)))
    v = rng.standard_normal((B, N, H, dv))
    a_pre = rng.uniform(-3.0, 1.0, (B, N, H))
    b_pre = rng.uniform(-2.0, 2.0, (B, N, H))
    alpha = np.exp(-np.logaddexp(0.0, a_pre)).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-b_pre))).astype(np.float32)
    S0 = (rng.standard_normal((B, H, dv, dk)) * s0_std).astype(np.float32)
    depth = np.stack([node_depths(parent[b]) for b in range(B)])
    if lmax is None:
        lmax = int(depth.max()) + 1
    if path is None:
        path = np.full((B, lmax), -1, dtype=np.int32)
        for b in range(B):
            path[b] = _pad_path(root_path(parent[b], int(rng.integers(N))), lmax)
    spec = Spec("custom", B, N, H, dk, dv, dtype, "custom", int(depth.max()), "custom", s0_std, seed)
    return Workload(spec, B, N, H, dk, dv, dtype, _store(q, dtype), _store(k, dtype), _store(v, dtype),
                    alpha, beta, parent, S0, np.asarray(path, dtype=np.int32))


# ---------------------------------------------------------------------------
# full GDN layer decode step
# ---------------------------------------------------------------------------
WEIGHT_STD = 0.02


@dataclasses.dataclass
class LayerWorkload:
    """Inputs of one GDN layer decode step over B draft trees.

    Row blocks of W_in, in order: q (H d_k), k (H d_k), v (H d_v), output gate
    z (H d_v), alpha pre-activation a (H), beta pre-activation b (H).  Conv
    channels are the q | k | v rows; conv_w tap 0 is the oldest position.
    """
    spec: Spec
    B: int
    N: int
    H: int
    dk: int
    dv: int
    hidden: int
    X: np.ndarray           # bf16 bits [B, N, hidden]
    W_in: np.ndarray        # bf16 bits [2 H dk + 2 H dv + 2 H, hidden]
    conv_w: np.ndarray      # float32 [H (2 dk + dv), 4]
    conv_state: np.ndarray  # float32 [B, 3, H (2 dk + dv)], oldest row first
    W_o: np.ndarray         # bf16 bits [hidden, H dv]
    parent: np.ndarray      # int32 [B, N]
    S0: np.ndarray          # float32 [B, H, dv, dk]
    path: np.ndarray        # int32 [B, Lmax]

    @property
    def conv_channels(self) -> int:
        return self.H * (2 * self.dk + self.dv)

    @property
    def in_rows(self) -> int:
        return 2 * self.H * self.dk + 2 * self.H * self.dv + 2 * self.H

    def widened(self, name: str) -> np.ndarray:
        x = getattr(self, name)
        if x.dtype == np.uint16:
            return bf16_bits_to_f64(x)
        return x.astype(np.float64)


def make_layer_workload(cfg=4, seed: Optional[int] = None, B: Optional[int] = None, N: Optional[int] = None,
                        H: Optional[int] = None, dk: Optional[int] = None, dv: Optional[int] = None,
                        hidden: Optional[int] = None, maxdepth: Optional[int] = None,
                        tree: Optional[str] = None) -> LayerWorkload:
    """Draw one full-layer workload (SPECS[4] by default; any field may be overridden).

    X ~ N(0, 1) and the weights ~ N(0, 0.02), rounded to bf16; conv weights
    ~ N(0, 0.02) in fp32; the committed conv history ~ N(0, (0.02 sqrt(hidden))^2),
    the spread of a projected N(0, 1) hidden row; S0 ~ N(0, s0_std).  Draw
    order: trees, X, W_in, conv_w, conv history, W_o, S0, accepted paths.
    """
    base = SPECS[cfg] if isinstance(cfg, int) else cfg
    spec = dataclasses.replace(
        base, B=base.B if B is None else B, N=base.N if N is None else N, H=base.H if H is None else H,
        dk=base.dk if dk is None else dk, dv=base.dv if dv is None else dv,
        hidden=base.hidden if hidden is None else hidden,
        maxdepth=base.maxdepth if maxdepth is None else maxdepth, tree=base.tree if tree is None else tree)
    rng = np.random.default_rng(spec.seed if seed is None else seed)
    B, N, H, dk, dv, hid = spec.B, spec.N, spec.H, spec.dk, spec.dv, spec.hidden
    parent = draw_trees(rng, spec, B).astype(np.int32)
    C = H * (2 * dk + dv)
    rows = 2 * H * dk + 2 * H * dv + 2 * H
    X = f32_to_bf16_bits(rng.standard_normal((B, N, hid)).astype(np.float32))
    W_in = f32_to_bf16_bits((rng.standard_normal((rows, hid)) * WEIGHT_STD).astype(np.float32))
    conv_w = (rng.standard_normal((C, 4)) * WEIGHT_STD).astype(np.float32)
    conv_state = (rng.standard_normal((B, 3, C)) * (WEIGHT_STD * np.sqrt(hid))).astype(np.float32)
    W_o = f32_to_bf16_bits((rng.standard_normal((hid, H * dv)) * WEIGHT_STD).astype(np.float32))
    S0 = (rng.standard_normal((B, H, dv, dk)) * spec.s0_std).astype(np.float32)
    path = draw_paths(rng, spec, parent)
    return LayerWorkload(spec, B, N, H, dk, dv, hid, X, W_in, conv_w, conv_state, W_o, parent, S0, path)


# ---------------------------------------------------------------------------
# gated linear attention (per-channel gates)
# ---------------------------------------------------------------------------
def make_gla_workload(cfg=3, seed: Optional[int] = None, B: Optional[int] = None, parent: Optional[np.ndarray] = None,
                      **override) -> Workload:
    """A tree workload whose gate alpha is per key channel, [B, N, H, dk] (every other input as
    ``make_workload``).  Each gate channel is drawn like the scalar gates: alpha = exp(-softplus(U(-3, 1))).
    ``parent`` ([B, N]) replaces the drawn trees (then paths go root -> a uniformly drawn node);
    ``override`` replaces Spec fields (N, H, dk, dv, dtype, maxdepth).  Draw order: trees, q, k, v,
    alpha pre-activations, beta pre-activations, S0, paths."""
    base = SPECS[cfg] if isinstance(cfg, int) else cfg
    spec = dataclasses.replace(base, name="gla_" + base.name, **({"B": B} if B is not None else {}), **override)
    B = spec.B
    rng = np.random.default_rng(spec.seed if seed is None else seed)
    N, H, dk, dv = spec.N, spec.H, spec.dk, spec.dv
    par = draw_trees(rng, spec, B).astype(np.int32) if parent is None else np.asarray(parent, np.int32)
    q = _unit_rows(rng.standard_normal((B, N, H, dk)))
    k = _unit_rows(rng.standard_normal((B, N, H, dk)))
    v = rng.standard_normal((B, N, H, dv))
    a_pre = rng.uniform(-3.0, 1.0, (B, N, H, dk))
    b_pre = rng.uniform(-2.0, 2.0, (B, N, H))
    alpha = np.exp(-np.logaddexp(0.0, a_pre)).astype(np.float32)
    beta = (1.0 / (1.0 + np.exp(-b_pre))).astype(np.float32)
    S0 = (rng.standard_normal((B, H, dv, dk)) * spec.s0_std).astype(np.float32)
    if parent is None:
        path = draw_paths(rng, spec, par)
    else:
        depth = np.stack([node_depths(par[b]) for b in range(B)])
        lmax = int(depth.max()) + 1
        path = np.stack([_pad_path(root_path(par[b], int(rng.integers(N))), lmax) for b in range(B)])
    return Workload(spec, B, N, H, dk, dv, spec.dtype, _store(q, spec.dtype), _store(k, spec.dtype),
                    _store(v, spec.dtype), alpha, beta, par, S0, path.astype(np.int32))

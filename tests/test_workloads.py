"""Input generator: determinism, shapes, distributions and tree rules (CPU only)."""
import numpy as np
import pytest

from speculative_decoding_linear_gb300 import workloads as wl


def test_bf16_rounding_ties_to_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 0.0], np.float32)
    assert wl.f32_to_bf16_bits(x).tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x0000]
    assert np.array_equal(wl.bf16_bits_to_f64(np.array([0x3F80, 0xC020], np.uint16)), [1.0, -2.5])


@pytest.mark.parametrize("cfg", [0, 1, 2, 3])
def test_specs_shapes_and_determinism(cfg):
    a, b = wl.make_workload(cfg), wl.make_workload(cfg)
    s = wl.SPECS[cfg]
    assert a.q.shape == (s.B, s.N, s.H, s.dk) and a.v.shape == (s.B, s.N, s.H, s.dv)
    assert a.S0.shape == (s.B, s.H, s.dv, s.dk) and a.path.shape == (s.B, s.lmax)
    for name in ("q", "k", "v", "alpha", "beta", "parent", "S0", "path"):
        assert np.array_equal(getattr(a, name), getattr(b, name))
    assert (a.q.dtype == np.uint16) == (s.dtype == wl.BF16)


def test_distributions():
    w = wl.make_workload(3)
    assert w.alpha.min() > 0.26 and w.alpha.max() < 0.96
    assert w.beta.min() > 0.11 and w.beta.max() < 0.89
    nq = np.linalg.norm(w.widened("q"), axis=-1)
    assert np.all(np.abs(nq - 1) < 1e-2)           # unit rows up to bf16 rounding
    assert abs(np.std(w.S0) - 0.05) < 1e-3


@pytest.mark.parametrize("cfg", [2, 3])
def test_random_tree_rules(cfg):
    w = wl.make_workload(cfg)
    s = wl.SPECS[cfg]
    for b in range(w.B):
        par = w.parent[b]
        assert par[0] == -1 and np.all(par[1:] >= 0) and np.all(par[1:] < np.arange(1, s.N))
        d = wl.node_depths(par)
        assert d.max() <= s.maxdepth
        L = int(np.sum(w.path[b] >= 0))
        assert L >= 1
        nodes = w.path[b, :L]
        assert par[nodes[0]] == -1 and all(par[nodes[i]] == nodes[i - 1] for i in range(1, L))
        assert np.all(w.path[b, L:] == -1)
        if cfg == 3:
            assert 1 <= L <= 8


def test_tiny_and_chain_topologies():
    w0 = wl.make_workload(0)
    assert w0.parent[0].tolist() == [-1, 0, 0, 1, 1, 2, 2]
    assert w0.path[0].tolist() == [0, 1, 3]
    w1 = wl.make_workload(1)
    assert w1.parent[0].tolist() == list(range(-1, 7))
    L = int(np.sum(w1.path[0] >= 0))
    assert w1.path[0, :L].tolist() == list(range(L))


def test_narrow_tree_shape():
    p = wl.narrow_tree(64, 4, 8)
    assert len(p) == 64 and p[0] == -1
    assert all(0 <= p[t] < t for t in range(1, 64))
    kids = np.bincount(p[p >= 0], minlength=64)
    assert kids[7] == 4 and np.count_nonzero(kids >= 2) == 1
    assert wl.node_depths(p).max() == 7 + 14

"""Oracle -- TEST INFRASTRUCTURE ONLY.

A plain, slow fp64 CPU implementation of what the GDN tree verifier and the
accepted-path commit compute, used to prove the CUDA library right.  Only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import it.  It shares no code with the CUDA library.

* ``tree_meta``     -- strict-ancestor bitmask and depth of every draft node.
* ``tree_verify``   -- walks each node's root-to-node path with the gated delta
                       rule from S0 and returns o_t = S_t q_t, the innovation
                       delta_t and the cumulative log gate g_t (gdn_oracle.c).
* ``commit``        -- walks the accepted root-first path and returns its state.
* ``layer``         -- the full GDN layer decode step (oracle/layer.py).

Sources: "Pith review of SpecLA: Efficient Speculative Decoding for
Linear-Attention Models" (pith.science 7ERME3HB): "Core claim", "Load-bearing
premise", "What would settle it"; the recurrence is the gated delta rule of the
Gated DeltaNet paper that review cites.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

BAD_ARG, BAD_TREE, BAD_PATH = -1, -2, -3


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile gdn_oracle.c with gcc into oracle/_build/liboracle.so (fp64, no FP contraction)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.check_call(cmd)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I = ctypes.c_int
            lib.oracle_tree_meta.argtypes = [I, I, P, P, P]
            lib.oracle_tree_verify.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P, P, P, P, P, I]
            lib.oracle_commit.argtypes = [I, I, I, I, I, P, P, P, P, P, P, P, I, P, I]
            for f in (lib.oracle_tree_meta, lib.oracle_tree_verify, lib.oracle_commit):
                f.restype = I
            _lib = lib
    return _lib


def _f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def _i32(x):
    return np.ascontiguousarray(x, dtype=np.int32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc):
    if rc != 0:
        raise OracleError({BAD_ARG: "bad argument", BAD_TREE: "invalid parent_idx",
                           BAD_PATH: "invalid accepted path"}.get(rc, str(rc)))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def tree_meta(parent):
    """parent [B,N] -> (mask [B,N] uint64 strict-ancestor bits, depth [B,N] int32)."""
    parent = _i32(parent)
    B, N = parent.shape
    mask = np.zeros((B, N), dtype=np.uint64)
    depth = np.zeros((B, N), dtype=np.int32)
    _check(_load().oracle_tree_meta(B, N, _ptr(parent), _ptr(mask), _ptr(depth)))
    return mask, depth


def tree_verify(q, k, v, alpha, beta, parent, S0, want=None, nthreads=None):
    """Per-node outputs by walking each root-to-node path with the gated delta rule.

    q, k [B,N,H,dk]; v [B,N,H,dv]; alpha, beta [B,N,H]; parent [B,N]; S0 [B,H,dv,dk].
    Returns (out [B,N,H,dv], delta [B,H,N,dv], g [B,H,N]) in float64.  With
    ``want`` ([B,N] bool) only the selected nodes are evaluated (others stay 0).
    """
    q, k, v, alpha, beta, S0 = map(_f64, (q, k, v, alpha, beta, S0))
    parent = _i32(parent)
    B, N, H, dk = q.shape
    dv = v.shape[-1]
    assert k.shape == (B, N, H, dk) and v.shape == (B, N, H, dv)
    assert alpha.shape == (B, N, H) and beta.shape == (B, N, H) and parent.shape == (B, N)
    assert S0.shape == (B, H, dv, dk)
    out = np.zeros((B, N, H, dv))
    delta = np.zeros((B, H, N, dv))
    g = np.zeros((B, H, N))
    w = None if want is None else np.ascontiguousarray(want, dtype=np.uint8)
    rc = _load().oracle_tree_verify(B, N, H, dk, dv, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                                    _ptr(beta), _ptr(parent), _ptr(S0), _ptr(w), _ptr(out),
                                    _ptr(delta), _ptr(g), nthreads or default_threads())
    _check(rc)
    return out, delta, g


def commit(k, v, alpha, beta, parent, S0, path, nthreads=None):
    """State after walking the accepted root-first path (-1 padded, [B, Lmax]) from S0."""
    k, v, alpha, beta, S0 = map(_f64, (k, v, alpha, beta, S0))
    parent = _i32(parent)
    path = _i32(path)
    B, N, H, dk = k.shape
    dv = v.shape[-1]
    S_new = np.zeros_like(S0)
    rc = _load().oracle_commit(B, N, H, dk, dv, _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta),
                               _ptr(parent), _ptr(S0), _ptr(path), path.shape[1], _ptr(S_new),
                               nthreads or default_threads())
    _check(rc)
    return S_new

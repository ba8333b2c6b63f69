"""Thin Python binding of libgdnspec.so (the C ABI in include/gdnspec.h).

Argument marshalling only: every function here forwards device pointers,
sizes and the current CUDA stream to the entry point of the same name and
turns a negative status into :class:`GdnError`.  All arithmetic runs in the
library's CUDA kernels; there is no CPU fallback -- if the compiled library is
missing, importing it raises.

Tensors are PyTorch CUDA tensors (PyTorch is used for device memory and
streams only); plain integer device addresses are accepted as well.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

_lib = None
_lock = threading.Lock()

OK, ERR_ARG, ERR_TREE, ERR_PATH, ERR_TIMEOUT, ERR_CUDA, ERR_DEVICE, ERR_CAPACITY = 0, -1, -2, -3, -4, -5, -6, -7
DTYPE_BF16, DTYPE_F32 = 0, 1

# (name, restype, argtypes) for every extern "C" symbol of include/gdnspec.h
_P, _I, _S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "gdn_factors_bytes": (_I, [_I, _I, _I, _I, _I, _I, ctypes.POINTER(_S)]),
    "gdn_workspace_bytes": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(_S)]),
    "gdn_tree_mask": (_I, [_P, _I, _I, _P, _P, _P]),
    "gdn_tree_verify": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "gdn_tree_verify_noalloc": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "gdn_chain_verify": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "gdn_commit": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P]),
    "gdn_commit_tree_verify": (_I, [_P, _P, _I, _P, _I, _P, _P, _P, _I, _P, _P, _P, _P, _P, _P,
                                    _I, _I, _I, _I, _I, _P]),
    "gdn_commit_chain_verify": (_I, [_P, _P, _I, _P, _I, _P, _P, _P, _I, _P, _P, _P, _P,
                                     _I, _I, _I, _I, _I, _P]),
    "gdn_layer_record_bytes": (_I, [_I, _I, _I, _I, _I, _I, ctypes.POINTER(_S)]),
    "gdn_layer_workspace_bytes": (_I, [_I, _I, _I, _I, _I, _I, ctypes.POINTER(_S)]),
    "gdn_layer_tree_step": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _P, _P, _P,
                                 _I, _I, _I, _I, _I, _I, _P]),
    "gdn_layer_token_step": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _P,
                                  _I, _I, _I, _I, _I, _I, _P]),
    "gdn_layer_stage_events": (_I, [_P, _I]),
    "gdn_model_workspace_bytes": (_I, [_I, _I, _I, _I, _I, _I, _I, ctypes.POINTER(_S)]),
    "gdn_model_tree_step": (_I, [_I, _P, _P, _P, _P, _P, _P, _P, _P, _I, _P, _I, _P, _P, _P,
                                 _I, _I, _I, _I, _I, _I, _P]),
    "gdn_prune_tree": (_I, [_P, _P, ctypes.c_float, _I, _P, _P, _P, _I, _I, _P]),
    "gdn_hybrid_workspace_bytes": (_I, [_I, _I, _I, _I, _I, _P]),
    "gdn_hybrid_tree_verify": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "gdn_replay_tree_verify": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "gdn_replay_commit": (_I, [_P, _P, _I, _P, _P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _P]),
    "gdn_snapshot_tree_verify": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "gdn_snapshot_commit": (_I, [_P, _P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _P]),
    "gdn_linear_tree_verify": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "gdn_gla_factors_bytes": (_I, [_I, _I, _I, _I, _I, _I, ctypes.POINTER(_S)]),
    "gdn_gla_workspace_bytes": (_I, [_I, _I, _I, _I, _I, ctypes.POINTER(_S)]),
    "gdn_gla_tree_verify": (_I, [_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P]),
    "gdn_gla_commit": (_I, [_P, _P, _P, _I, _P, _I, _I, _I, _I, _I, _I, _P]),
    "gdn_set_launch_overlap": (_I, [_I]),
    "gdn_set_wait_limit_ns": (_I, [ctypes.c_ulonglong]),
    "gdn_selftest_stuck_wait": (_I, [_P]),
    "gdn_last_error": (_I, [_P]),
    "gdn_strerror": (ctypes.c_char_p, [_I]),
}


class GdnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__("%s: %s (status %d)" % (where, strerror(code), code))


def library_path() -> str:
    return _build.LIB


def lib(build_if_missing: bool = True) -> ctypes.CDLL:
    """The loaded libgdnspec.so.  Builds it when absent (nvcc required); raises if it cannot."""
    global _lib
    loaded = _lib              # once loaded, every call returns it without taking the lock
    if loaded is not None:
        return loaded
    with _lock:
        if _lib is None:
            path = _build.LIB
            if build_if_missing and not _build.up_to_date():
                _build.build()
            if not os.path.exists(path):
                raise ImportError("libgdnspec.so not found at %s: the CUDA library is required "
                                  "(there is no CPU fallback)" % path)
            L = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().gdn_strerror(int(code)).decode()


def _check(rc: int, where: str):
    if rc != OK:
        raise GdnError(rc, where)


def _ptr(x):
    if type(x) is torch.Tensor or isinstance(x, torch.Tensor):
        if x.is_cuda and x.is_contiguous():
            return x.data_ptr()
        raise ValueError("expected a contiguous CUDA tensor")
    if x is None:
        return None
    if isinstance(x, int):
        return x
    raise TypeError(type(x))


# The current stream as a raw handle without building a Stream object (a few
# microseconds per call otherwise, more than a chain verification on the GPU).
_raw_current_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream):
    if stream is None:
        if _raw_current_stream is not None:
            return _raw_current_stream(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def dtype_code(t) -> int:
    if t in (torch.bfloat16, "bf16"):
        return DTYPE_BF16
    if t in (torch.float32, "f32"):
        return DTYPE_F32
    raise ValueError("q/k/v must be bf16 or fp32, got %s" % (t,))


# ---------------------------------------------------------------------------
# sizes
# ---------------------------------------------------------------------------
def gdn_factors_bytes(B, N, H, dk, dv, dtype) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().gdn_factors_bytes(B, N, H, dk, dv, dtype_code(dtype) if not isinstance(dtype, int)
                                   else dtype, ctypes.byref(out)), "gdn_factors_bytes")
    return out.value


def gdn_workspace_bytes(B, N, H, dk, dv) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().gdn_workspace_bytes(B, N, H, dk, dv, ctypes.byref(out)), "gdn_workspace_bytes")
    return out.value


def empty_factors(B, N, H, dk, dv, dtype, device="cuda"):
    """Caller-owned factor buffer (uint8 tensor) of the size the library asks for."""
    return torch.empty(gdn_factors_bytes(B, N, H, dk, dv, dtype), dtype=torch.uint8, device=device)


def empty_workspace(B, N, H, dk, dv, device="cuda"):
    return torch.empty(gdn_workspace_bytes(B, N, H, dk, dv), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------------------
# entry points (same names as the C ABI)
# ---------------------------------------------------------------------------
def _dims(q, v):
    B, N, H, dk = q.shape
    return B, N, H, dk, v.shape[-1]


def gdn_tree_mask(parent_idx, mask, depth, stream=None):
    B, N = parent_idx.shape
    _check(lib().gdn_tree_mask(_ptr(parent_idx), B, N, _ptr(mask), _ptr(depth), _stream(stream)),
           "gdn_tree_mask")


def gdn_tree_verify(q, k, v, alpha, beta, parent_idx, S0, out, factors, workspace, stream=None):
    B, N, H, dk, dv = _dims(q, v)
    _check(lib().gdn_tree_verify(_ptr(q), _ptr(k), _ptr(v), dtype_code(q.dtype), _ptr(alpha),
                                 _ptr(beta), _ptr(parent_idx), _ptr(S0), _ptr(out), _ptr(factors),
                                 _ptr(workspace), B, N, H, dk, dv, _stream(stream)),
           "gdn_tree_verify")


def gdn_tree_verify_noalloc(q, k, v, alpha, beta, parent_idx, S0, out, factors, stream=None):
    """gdn_tree_verify without a workspace argument: for callers that cannot allocate device
    memory (a framework that owns all device memory, or a decode loop that must not allocate).
    The workspace is a fixed 32 MiB scratch array inside the library, shared by all calls on a
    device; calls overlapping on the GPU race on it.  See include/gdnspec.h."""
    B, N, H, dk, dv = _dims(q, v)
    _check(lib().gdn_tree_verify_noalloc(_ptr(q), _ptr(k), _ptr(v), dtype_code(q.dtype), _ptr(alpha),
                                         _ptr(beta), _ptr(parent_idx), _ptr(S0), _ptr(out),
                                         _ptr(factors), B, N, H, dk, dv, _stream(stream)),
           "gdn_tree_verify_noalloc")


def gdn_chain_verify(q, k, v, alpha, beta, S0, out, factors, stream=None):
    B, N, H, dk, dv = _dims(q, v)
    _check(lib().gdn_chain_verify(_ptr(q), _ptr(k), _ptr(v), dtype_code(q.dtype), _ptr(alpha),
                                  _ptr(beta), _ptr(S0), _ptr(out), _ptr(factors), B, N, H, dk, dv,
                                  _stream(stream)), "gdn_chain_verify")


def gdn_commit(S0, factors, accepted_path, S_new, N, dtype, stream=None):
    B, H, dv, dk = S0.shape
    _check(lib().gdn_commit(_ptr(S0), _ptr(factors), _ptr(accepted_path), accepted_path.shape[1],
                            _ptr(S_new), B, N, H, dk, dv, dtype_code(dtype), _stream(stream)),
           "gdn_commit")


def gdn_commit_tree_verify(S, prev_factors, N_prev, prev_path, q, k, v, alpha, beta, parent_idx,
                           out, factors, workspace, stream=None):
    B, N, H, dk, dv = _dims(q, v)
    _check(lib().gdn_commit_tree_verify(_ptr(S), _ptr(prev_factors), N_prev, _ptr(prev_path),
                                        prev_path.shape[1], _ptr(q), _ptr(k), _ptr(v),
                                        dtype_code(q.dtype), _ptr(alpha), _ptr(beta),
                                        _ptr(parent_idx), _ptr(out), _ptr(factors), _ptr(workspace),
                                        B, N, H, dk, dv, _stream(stream)), "gdn_commit_tree_verify")


def gdn_commit_chain_verify(S, prev_factors, N_prev, prev_path, q, k, v, alpha, beta, out, factors,
                            stream=None):
    B, N, H, dk, dv = _dims(q, v)
    _check(lib().gdn_commit_chain_verify(_ptr(S), _ptr(prev_factors), N_prev, _ptr(prev_path),
                                         prev_path.shape[1], _ptr(q), _ptr(k), _ptr(v),
                                         dtype_code(q.dtype), _ptr(alpha), _ptr(beta), _ptr(out),
                                         _ptr(factors), B, N, H, dk, dv, _stream(stream)),
           "gdn_commit_chain_verify")


def gdn_layer_record_bytes(B, N, H, hidden, dk, dv) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().gdn_layer_record_bytes(B, N, H, hidden, dk, dv, ctypes.byref(out)), "gdn_layer_record_bytes")
    return out.value


def gdn_layer_workspace_bytes(B, N, H, hidden, dk, dv) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().gdn_layer_workspace_bytes(B, N, H, hidden, dk, dv, ctypes.byref(out)),
           "gdn_layer_workspace_bytes")
    return out.value


def gdn_layer_tree_step(X, W_in, conv_w, W_o, parent_idx, S, conv_state, prev_record, N_prev, prev_path,
                        out, record, workspace, H, dk, dv, stream=None):
    """One GDN layer decode step over B draft trees (see include/gdnspec.h).  prev_record and
    prev_path are both None when there is no pending commit."""
    B, N, hidden = X.shape
    Lmax = 0 if prev_path is None else prev_path.shape[1]
    _check(lib().gdn_layer_tree_step(_ptr(X), _ptr(W_in), _ptr(conv_w), _ptr(W_o), _ptr(parent_idx), _ptr(S),
                                     _ptr(conv_state), _ptr(prev_record), int(N_prev), _ptr(prev_path), Lmax,
                                     _ptr(out), _ptr(record), _ptr(workspace), B, N, H, hidden, dk, dv,
                                     _stream(stream)), "gdn_layer_tree_step")


def gdn_layer_token_step(X, W_in, conv_w, W_o, parent_idx, S0, conv_state, S_nodes, t, out, record, workspace,
                         H, dk, dv, stream=None):
    """Decode node t of every tree on its own from its parent's materialised state (see
    include/gdnspec.h); S_nodes is [N, B, H, dv, dk] fp32."""
    B, N, hidden = X.shape
    _check(lib().gdn_layer_token_step(_ptr(X), _ptr(W_in), _ptr(conv_w), _ptr(W_o), _ptr(parent_idx), _ptr(S0),
                                      _ptr(conv_state), _ptr(S_nodes), int(t), _ptr(out), _ptr(record),
                                      _ptr(workspace), B, N, H, hidden, dk, dv, _stream(stream)),
           "gdn_layer_token_step")


def gdn_layer_stage_events(events):
    """Turn the layer step's per-kernel timing hook on with 6 torch.cuda.Event objects (timing
    enabled, each recorded at least once so that its CUDA event exists), or off with None (see
    include/gdnspec.h)."""
    if events is None:
        _check(lib().gdn_layer_stage_events(None, 0), "gdn_layer_stage_events")
        return
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event if hasattr(e, "cuda_event") else int(e) for e in events])
    _check(lib().gdn_layer_stage_events(ctypes.cast(arr, ctypes.c_void_p), len(events)), "gdn_layer_stage_events")


def gdn_model_workspace_bytes(L, B, N, H, hidden, dk, dv) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().gdn_model_workspace_bytes(L, B, N, H, hidden, dk, dv, ctypes.byref(out)),
           "gdn_model_workspace_bytes")
    return out.value


def _ptr_array(xs):
    if xs is None:
        return None
    arr = (ctypes.c_void_p * len(xs))(*[_ptr(x) for x in xs])
    return ctypes.cast(arr, ctypes.c_void_p), arr      # keep the array alive with the call


def gdn_model_tree_step(X, W_in, conv_w, W_o, parent_idx, S, conv_state, prev_records, N_prev, prev_path, out,
                        records, workspace, H, dk, dv, stream=None):
    """L layers back to back (see include/gdnspec.h); the per-layer arguments are lists of L tensors."""
    B, N, hidden = X.shape
    L = len(W_in)
    arrs = [_ptr_array(x) for x in (W_in, conv_w, W_o, S, conv_state, prev_records, records)]
    ptrs = [a[0] if a is not None else None for a in arrs]
    Lmax = 0 if prev_path is None else prev_path.shape[1]
    _check(lib().gdn_model_tree_step(L, _ptr(X), ptrs[0], ptrs[1], ptrs[2], _ptr(parent_idx), ptrs[3], ptrs[4],
                                     ptrs[5], int(N_prev), _ptr(prev_path), Lmax, _ptr(out), ptrs[6],
                                     _ptr(workspace), B, N, H, hidden, dk, dv, _stream(stream)),
           "gdn_model_tree_step")


def gdn_prune_tree(parent_idx, logp, tau, budget, new_index, new_parent, n_kept, stream=None):
    """Confidence-guided pruning of B draft trees (see include/gdnspec.h)."""
    B, N = parent_idx.shape
    _check(lib().gdn_prune_tree(_ptr(parent_idx), _ptr(logp), float(tau), int(budget), _ptr(new_index),
                                _ptr(new_parent), _ptr(n_kept), B, N, _stream(stream)), "gdn_prune_tree")


def gdn_hybrid_workspace_bytes(B, N, H, dk, dv) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().gdn_hybrid_workspace_bytes(B, N, H, dk, dv, ctypes.byref(out)), "gdn_hybrid_workspace_bytes")
    return out.value


def gdn_hybrid_tree_verify(q, k, v, alpha, beta, parent_idx, S0, out, factors, workspace, stream=None):
    """Chain-decomposed tree verification (see include/gdnspec.h); same outputs and factor record as
    gdn_tree_verify.  workspace: gdn_hybrid_workspace_bytes(...) bytes (None when that is 0)."""
    B, N, H, dk, dv = _dims(q, v)
    _check(lib().gdn_hybrid_tree_verify(_ptr(q), _ptr(k), _ptr(v), dtype_code(q.dtype), _ptr(alpha), _ptr(beta),
                                        _ptr(parent_idx), _ptr(S0), _ptr(out), _ptr(factors),
                                        _ptr(workspace), B, N, H, dk, dv,
                                        _stream(stream)), "gdn_hybrid_tree_verify")


def gdn_replay_tree_verify(q, k, v, alpha, beta, parent_idx, S0, out, stream=None):
    """Baseline: replay every root-to-leaf path token by token (see include/gdnspec.h)."""
    B, N, H, dk, dv = _dims(q, v)
    _check(lib().gdn_replay_tree_verify(_ptr(q), _ptr(k), _ptr(v), dtype_code(q.dtype), _ptr(alpha), _ptr(beta),
                                        _ptr(parent_idx), _ptr(S0), _ptr(out), B, N, H, dk, dv, _stream(stream)),
           "gdn_replay_tree_verify")


def gdn_replay_commit(k, v, alpha, beta, parent_idx, S0, accepted_path, S_new, stream=None):
    """Baseline: replay the accepted tokens from S0 into S_new (see include/gdnspec.h)."""
    B, N, H, dk, dv = _dims(k, v)
    _check(lib().gdn_replay_commit(_ptr(k), _ptr(v), dtype_code(k.dtype), _ptr(alpha), _ptr(beta), _ptr(parent_idx),
                                   _ptr(S0), _ptr(accepted_path), accepted_path.shape[1], _ptr(S_new), B, N, H, dk,
                                   dv, _stream(stream)), "gdn_replay_commit")


def gdn_snapshot_tree_verify(q, k, v, alpha, beta, parent_idx, S0, out, S_nodes, stream=None):
    """Baseline: build and store every draft node's state, node by node (see include/gdnspec.h);
    S_nodes is [N, B, H, dv, dk] fp32."""
    B, N, H, dk, dv = _dims(q, v)
    _check(lib().gdn_snapshot_tree_verify(_ptr(q), _ptr(k), _ptr(v), dtype_code(q.dtype), _ptr(alpha), _ptr(beta),
                                          _ptr(parent_idx), _ptr(S0), _ptr(out), _ptr(S_nodes), B, N, H, dk, dv,
                                          _stream(stream)), "gdn_snapshot_tree_verify")


def gdn_snapshot_commit(S_nodes, S0, parent_idx, accepted_path, S_new, stream=None):
    """Baseline: the accepted node's stored state becomes the committed state (see include/gdnspec.h)."""
    N, B, H, dv, dk = S_nodes.shape
    _check(lib().gdn_snapshot_commit(_ptr(S_nodes), _ptr(S0), _ptr(parent_idx), _ptr(accepted_path),
                                     accepted_path.shape[1], _ptr(S_new), B, N, H, dk, dv, _stream(stream)),
           "gdn_snapshot_commit")


def gdn_linear_tree_verify(q, k, v, alpha, beta, parent_idx, S0, out, factors, workspace, stream=None):
    """Decay-gated linear attention (no delta-rule erasure) over a draft tree; see include/gdnspec.h."""
    B, N, H, dk, dv = _dims(q, v)
    _check(lib().gdn_linear_tree_verify(_ptr(q), _ptr(k), _ptr(v), dtype_code(q.dtype), _ptr(alpha), _ptr(beta),
                                        _ptr(parent_idx), _ptr(S0), _ptr(out), _ptr(factors), _ptr(workspace),
                                        B, N, H, dk, dv, _stream(stream)), "gdn_linear_tree_verify")


def gdn_gla_factors_bytes(B, N, H, dk, dv, dtype) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().gdn_gla_factors_bytes(B, N, H, dk, dv, dtype_code(dtype) if not isinstance(dtype, int) else dtype,
                                       ctypes.byref(out)), "gdn_gla_factors_bytes")
    return out.value


def gdn_gla_workspace_bytes(B, N, H, dk, dv) -> int:
    out = ctypes.c_size_t(0)
    _check(lib().gdn_gla_workspace_bytes(B, N, H, dk, dv, ctypes.byref(out)), "gdn_gla_workspace_bytes")
    return out.value


def gdn_gla_tree_verify(q, k, v, alpha, beta, parent_idx, S0, out, factors, workspace, stream=None):
    """Gated linear attention (per-channel gates alpha [B,N,H,dk]) over draft trees; see include/gdnspec.h."""
    B, N, H, dk, dv = _dims(q, v)
    _check(lib().gdn_gla_tree_verify(_ptr(q), _ptr(k), _ptr(v), dtype_code(q.dtype), _ptr(alpha), _ptr(beta),
                                     _ptr(parent_idx), _ptr(S0), _ptr(out), _ptr(factors), _ptr(workspace),
                                     B, N, H, dk, dv, _stream(stream)), "gdn_gla_tree_verify")


def gdn_gla_commit(S0, factors, accepted_path, S_new, N, dtype, stream=None):
    """Accepted-path commit from a GLA factor record (see include/gdnspec.h)."""
    B, H, dv, dk = S0.shape
    _check(lib().gdn_gla_commit(_ptr(S0), _ptr(factors), _ptr(accepted_path), accepted_path.shape[1], _ptr(S_new),
                                B, N, H, dk, dv, dtype_code(dtype), _stream(stream)), "gdn_gla_commit")


def gla_factor_views(buf, B, N, H, dk, dv, dtype):
    """(delta [B,H,N,dv] f32, key [B,H,N,dk], g [B,H,N,dk] f32, parent [B,N] i32) views of a GLA factor buffer."""
    esz = 4 if dtype_code(dtype) == DTYPE_F32 else 2
    BHN = B * H * N
    o_key = _align(BHN * dv * 4)
    o_g = _align(o_key + BHN * dk * esz)
    o_par = _align(o_g + BHN * dk * 4)
    kt = torch.float32 if esz == 4 else torch.bfloat16
    delta = buf[: BHN * dv * 4].view(torch.float32).view(B, H, N, dv)
    key = buf[o_key: o_key + BHN * dk * esz].view(kt).view(B, H, N, dk)
    g = buf[o_g: o_g + BHN * dk * 4].view(torch.float32).view(B, H, N, dk)
    par = buf[o_par: o_par + B * N * 4].view(torch.int32).view(B, N)
    return delta, key, g, par


def gdn_set_launch_overlap(enable: bool) -> bool:
    """Process-wide switch; returns the previous setting (see include/gdnspec.h)."""
    return bool(lib().gdn_set_launch_overlap(1 if enable else 0))


def gdn_set_wait_limit_ns(ns: int):
    """Limit of every bounded device wait on the current device (see include/gdnspec.h)."""
    _check(lib().gdn_set_wait_limit_ns(int(ns)), "gdn_set_wait_limit_ns")


def gdn_selftest_stuck_wait(stream=None):
    """Launch a wait that nothing completes; gdn_last_error then reports GDN_ERR_TIMEOUT."""
    _check(lib().gdn_selftest_stuck_wait(_stream(stream)), "gdn_selftest_stuck_wait")


def gdn_last_error(stream=None) -> int:
    return lib().gdn_last_error(_stream(stream))


# ---------------------------------------------------------------------------
# factor-buffer views (host-side reinterpretation of the documented layout)
# ---------------------------------------------------------------------------
def _align(x, a=256):
    return (x + a - 1) // a * a


def factor_views(buf, B, N, H, dk, dv, dtype):
    """(delta [B,H,N,dv] f32, key [B,H,N,dk], g [B,H,N] f32, parent [B,N] i32) views of a factor buffer."""
    esz = 4 if dtype_code(dtype) == DTYPE_F32 else 2
    BHN = B * H * N
    o_key = _align(BHN * dv * 4)
    o_g = _align(o_key + BHN * dk * esz)
    o_par = _align(o_g + BHN * 4)
    kt = torch.float32 if esz == 4 else torch.bfloat16
    delta = buf[: BHN * dv * 4].view(torch.float32).view(B, H, N, dv)
    key = buf[o_key: o_key + BHN * dk * esz].view(kt).view(B, H, N, dk)
    g = buf[o_g: o_g + BHN * 4].view(torch.float32).view(B, H, N)
    par = buf[o_par: o_par + B * N * 4].view(torch.int32).view(B, N)
    return delta, key, g, par


def layer_record_views(buf, B, N, H, hidden, dk, dv):
    """(Y [B*N, rows] fp32 projections, factor-buffer slice) views of a layer record."""
    rows = 2 * H * dk + 2 * H * dv + 2 * H
    ldy = (rows + 3) // 4 * 4
    y_bytes = B * N * ldy * 4
    Y = buf[:y_bytes].view(torch.float32).view(B * N, ldy)[:, :rows]
    fac = buf[_align(y_bytes):]
    return Y, fac


def layer_workspace_views(buf, B, N, H, hidden, dk, dv):
    """q, k [B,N,H,dk], v, o [B,N,H,dv], alpha, beta [B,N,H] fp32; the bf16 hi/lo terms of q and k
    (qhi, qlo, khi, klo [B,N,H,dk]); y_hi, y_lo [B*N, H*dv] bf16.  When the single-kernel verifier runs
    (d_k = d_v = 256) the fp32 q and k rows are not written: q is carried by its hi/lo terms and the
    keys go straight to the factor record."""
    BN = B * N
    sizes = [("q", BN * H * dk * 4), ("k", BN * H * dk * 4), ("v", BN * H * dv * 4), ("alpha", BN * H * 4),
             ("beta", BN * H * 4), ("o", BN * H * dv * 4), ("qhi", BN * H * dk * 2), ("khi", BN * H * dk * 2),
             ("qlo", BN * H * dk * 2), ("klo", BN * H * dk * 2), ("yhi", BN * H * dv * 2),
             ("ylo", BN * H * dv * 2)]
    out, off = {}, 0
    for name, n in sizes:
        out[name] = buf[off:off + n]
        off = _align(off + n)
    f32 = lambda x, *shape: x.view(torch.float32).view(*shape)
    bf = lambda x: x.view(torch.bfloat16).view(B, N, H, dk)
    return dict(q=f32(out["q"], B, N, H, dk), k=f32(out["k"], B, N, H, dk), v=f32(out["v"], B, N, H, dv),
                qhi=bf(out["qhi"]), qlo=bf(out["qlo"]), khi=bf(out["khi"]), klo=bf(out["klo"]),
                alpha=f32(out["alpha"], B, N, H), beta=f32(out["beta"], B, N, H), o=f32(out["o"], B, N, H, dv),
                yhi=out["yhi"].view(torch.bfloat16).view(BN, H * dv),
                ylo=out["ylo"].view(torch.bfloat16).view(BN, H * dv))

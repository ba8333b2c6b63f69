"""The C-ABI library builds, loads without a GPU and exports every declared symbol (CPU only).

Only host-side logic runs here: size queries and argument validation that
returns before any CUDA call.  No kernel is launched.
"""
import ctypes
import os
import re
import subprocess

import pytest
import torch

from speculative_decoding_linear_gb300 import build as gbuild
from speculative_decoding_linear_gb300 import gdnspec

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gdnspec.h")


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|const char\s*\*)\s*(gdn_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def L():
    gbuild.build()
    return gdnspec.lib()


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert len(names) >= 10
    out = subprocess.run(["nm", "-D", "--defined-only", gbuild.LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT\s+(gdn_\w+)", out))
    for n in names:
        assert n in exported, n
        assert hasattr(L, n)
    assert set(names) == set(gdnspec.SIGNATURES), "binding and header disagree"


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert gdnspec.strerror(code) != "unknown status"
    assert gdnspec.strerror(-99) == "unknown status"


def test_factor_and_workspace_sizes(L):
    B, N, H, dk, dv = 16, 64, 8, 256, 256
    nb = gdnspec.gdn_factors_bytes(B, N, H, dk, dv, "bf16")
    delta = B * H * N * dv * 4
    key = B * H * N * dk * 2
    assert nb >= delta + key + B * H * N * 4 + B * N * 4
    assert nb % 256 == 0
    assert gdnspec.gdn_factors_bytes(B, N, H, dk, dv, "f32") > nb
    ws = gdnspec.gdn_workspace_bytes(B, N, H, dk, dv)
    assert ws >= B * H * (2 * N * N * 4)
    buf = torch.zeros(nb, dtype=torch.uint8)
    d, k, g, p = gdnspec.factor_views(buf, B, N, H, dk, dv, "bf16")
    assert d.shape == (B, H, N, dv) and k.shape == (B, H, N, dk) and g.shape == (B, H, N) and p.shape == (B, N)
    assert p.data_ptr() + p.numel() * 4 <= buf.data_ptr() + nb


@pytest.mark.parametrize("shape", [(1, 65, 8, 256, 256), (1, 0, 8, 256, 256), (0, 8, 8, 256, 256),
                                   (1, 8, 8, 24, 256), (1, 8, 8, 256, 512), (1, 8, 0, 256, 256)])
def test_bad_shapes_rejected(L, shape):
    out = ctypes.c_size_t(0)
    assert L.gdn_factors_bytes(*shape, 0, ctypes.byref(out)) == gdnspec.ERR_ARG
    assert L.gdn_workspace_bytes(*shape, ctypes.byref(out)) == gdnspec.ERR_ARG
    B, N, H, dk, dv = shape
    p = 4096   # aligned non-null dummy address: validation fails before any dereference
    assert L.gdn_tree_verify(p, p, p, 0, p, p, p, p, p, p, p, B, N, H, dk, dv, None) == gdnspec.ERR_ARG
    assert L.gdn_chain_verify(p, p, p, 0, p, p, p, p, p, B, N, H, dk, dv, None) == gdnspec.ERR_ARG


def test_null_misaligned_and_overlap_rejected(L):
    p, B, N, H, d = 4096, 1, 8, 8, 256
    args = [p, p, p, 0, p, p, p, p, p, p, p, B, N, H, d, d, None]
    for i in range(11):
        bad = list(args)
        bad[i] = None if i != 3 else 7      # null pointer (or an unknown dtype code)
        assert L.gdn_tree_verify(*bad) == gdnspec.ERR_ARG
    bad = list(args)
    bad[0] = p + 8                           # misaligned q
    assert L.gdn_tree_verify(*bad) == gdnspec.ERR_ARG
    # out overlapping the factor buffer
    bad = list(args)
    bad[8], bad[9] = 1 << 20, (1 << 20) + 256
    assert L.gdn_tree_verify(*bad) == gdnspec.ERR_ARG
    # commit: Lmax out of range, partial overlap of S0 / S_new
    assert L.gdn_commit(p, p, p, 0, p, B, N, H, d, d, 0, None) == gdnspec.ERR_ARG
    assert L.gdn_commit(p, p, p, 65, p, B, N, H, d, d, 0, None) == gdnspec.ERR_ARG
    assert L.gdn_commit(1 << 20, p, p, 4, (1 << 20) + 4096, B, N, H, d, d, 0, None) == gdnspec.ERR_ARG
    # fused: prev factors overlapping the new factor buffer
    assert L.gdn_commit_tree_verify(p, 1 << 20, N, p, 4, p, p, p, 0, p, p, p, p, (1 << 20) + 256, p,
                                    B, N, H, d, d, None) == gdnspec.ERR_ARG
    assert L.gdn_tree_mask(p, 1, 65, p, p, None) == gdnspec.ERR_ARG


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU failure mode")
def test_valid_call_without_gpu_fails_loudly(L):
    p = 4096
    rc = L.gdn_tree_verify(p, p, p, 0, p, p, p, p, p, 1 << 24, 1 << 26, 1, 8, 8, 256, 256, None)
    assert rc in (gdnspec.ERR_CUDA, gdnspec.ERR_DEVICE)

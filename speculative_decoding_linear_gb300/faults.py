"""Host-side fault injection for testing that parity checks catch corrupted factors.

A fault is planted on the host, never on the GPU: one innovation row of a
factor buffer is copied to host memory, changed there, and copied back before
the commit that reads it.  The commit is linear in each innovation (S_a =
e^{g_a} S0 + sum_{j on path(a)} e^{g_a - g_j} delta_j k_j^T), so adding c to
every entry of delta_j moves the committed state of that (sequence, head) by
exactly e^{g_a - g_j} c 1 k_j^T -- the amount a parity check must report.
"""
from __future__ import annotations

import numpy as np


def corrupt_delta_row(factors, B, N, H, dk, dv, dtype, b, h, node, amount):
    """Add `amount` to every entry of delta[b, h, node, :] of a factor buffer (device tensor of bytes),
    through a host round trip.  Returns the row before the change (numpy)."""
    import torch
    from . import gdnspec
    delta, _, _, _ = gdnspec.factor_views(factors, B, N, H, dk, dv, dtype)
    row = delta[b, h, node].cpu().numpy().copy()
    bad = (row.astype(np.float64) + amount).astype(np.float32)
    delta[b, h, node].copy_(torch.from_numpy(bad))
    return row

"""Sequence sharding of a batch across ranks (one process per GPU).

Every (sequence, head) of a verification or commit is independent of every
other -- the verifier's masks, solves and contractions never mix sequences
(review of SpecLA, pith.science 7ERME3HB, "Core claim") -- so a batch of B
draft trees splits across ranks by sequence with no exchange on the data
path: rank r takes a contiguous block of sequences, runs the same library
calls on its block, and the gathered outputs are the one-rank outputs.

This module holds only the partition and the slicing of host-side inputs; it
contains none of the method's arithmetic.
"""
from __future__ import annotations

import dataclasses

import numpy as np


def sequence_range(B: int, world: int, rank: int) -> tuple:
    """[lo, hi) of the sequences rank `rank` of `world` owns: contiguous blocks whose sizes differ by at
    most one, the larger blocks first.  Ranks beyond B get an empty block."""
    if world < 1 or not 0 <= rank < world or B < 0:
        raise ValueError("bad partition request: B=%d world=%d rank=%d" % (B, world, rank))
    base, extra = divmod(B, world)
    lo = rank * base + min(rank, extra)
    hi = lo + base + (1 if rank < extra else 0)
    return lo, hi


# per-sequence arrays of the two workload kinds (leading axis = sequence)
_TREE_FIELDS = ("q", "k", "v", "alpha", "beta", "parent", "S0", "path")
_LAYER_FIELDS = ("X", "conv_state", "parent", "S0", "path")


def shard_workload(w, world: int, rank: int):
    """The rank's block of a Workload or LayerWorkload: per-sequence arrays sliced along the batch axis,
    shared weights kept as they are, B and spec.B set to the block size."""
    lo, hi = sequence_range(w.B, world, rank)
    fields = _LAYER_FIELDS if hasattr(w, "W_in") else _TREE_FIELDS
    sliced = {f: np.ascontiguousarray(getattr(w, f)[lo:hi]) for f in fields}
    spec = dataclasses.replace(w.spec, B=hi - lo)
    return dataclasses.replace(w, spec=spec, B=hi - lo, **sliced)


def gather_order(B: int, world: int) -> list:
    """Per rank, the global sequence indices of its block, in rank order (concatenating the ranks'
    outputs in this order gives the batch order)."""
    return [list(range(*sequence_range(B, world, r))) for r in range(world)]

"""Generic fp64 ragged-dot forms (test infrastructure; see ``oracle/__init__``).

"Group-GEMM in XLA", Part 1 ("The Ragged-Dot Operation") and Part 3
("Contracting"):

* non-contracting: lhs [m, k] x rhs [G, k, n] -> out [m, n]; ``group_sizes``
  partitions the rows of lhs into contiguous groups and the rows of group g
  multiply rhs[g]. Rows past sum(group_sizes) belong to no group and are zero.
* contracting: lhs [m, K_total] x rhs [K_total, n] -> out [G, m, n]; group g
  reduces only over its slice [prefix_exclusive[g], prefix_inclusive[g]) of the
  contracted axis and writes out[g].

Plain loops over groups with numpy matmul as the per-group step.
"""
from __future__ import annotations

import numpy as np


def prefix_sums(group_sizes):
    """(exclusive, inclusive) prefix sums of the group sizes."""
    gs = np.asarray(group_sizes, dtype=np.int64)
    inc = np.cumsum(gs)
    exc = inc - gs
    return exc, inc


def ragged_dot(lhs, rhs, group_sizes):
    lhs = np.asarray(lhs, dtype=np.float64)
    rhs = np.asarray(rhs, dtype=np.float64)
    m, k = lhs.shape
    G, k2, n = rhs.shape
    assert k == k2 and len(group_sizes) == G
    exc, inc = prefix_sums(group_sizes)
    out = np.zeros((m, n), dtype=np.float64)
    for g in range(G):
        lo, hi = int(exc[g]), int(inc[g])
        out[lo:hi] = lhs[lo:hi] @ rhs[g]
    return out


def ragged_dot_contracting(lhs, rhs, group_sizes):
    lhs = np.asarray(lhs, dtype=np.float64)
    rhs = np.asarray(rhs, dtype=np.float64)
    m, kt = lhs.shape
    kt2, n = rhs.shape
    assert kt == kt2
    G = len(group_sizes)
    exc, inc = prefix_sums(group_sizes)
    out = np.zeros((G, m, n), dtype=np.float64)
    for g in range(G):
        lo, hi = int(exc[g]), int(inc[g])
        out[g] = lhs[:, lo:hi] @ rhs[lo:hi, :]
    return out

"""Test helpers: quantised inputs built on the host with the oracle's quantiser
(so no oracle input ever comes from the CUDA path), the parity tolerance, and
sample-index builders for full-size parity."""
from __future__ import annotations

import numpy as np

import oracle
from moe_ragged_contraction_gb300 import inputs as I


def quantised_operand(rows: int, M: int, seed: int, stream: int, dist: str = "normal",
                      block_rows: int = 256):
    """Seeded fp32 operand [rows, M] quantised tokenwise on the host, block by
    block (the fp32 array is never held whole)."""
    q = np.empty((rows, M), dtype=np.uint8)
    s = np.empty((rows, M // 32), dtype=np.uint8)
    for r0 in range(0, rows, block_rows):
        r1 = min(rows, r0 + block_rows)
        x = I.host_operand(r1 - r0, M, seed, stream, dist, row0=r0)
        q[r0:r1], s[r0:r1] = oracle.quantize_tokenwise(x)
    return q, s


def workload_inputs(name: str):
    """(A, sA, B, sB, offs) for a named workload, quantised on the host."""
    w = I.WORKLOADS[name]
    A, sA = quantised_operand(w.N, w.M, w.seed, 0, w.dist)
    B, sB = quantised_operand(w.K, w.M, w.seed, 1, w.dist)
    offs = I.offsets(I.group_sizes(name))
    return A, sA, B, sB, offs


def tolerance_violations(gpu_bits, ref_bits, absacc):
    """Elements violating |gpu - ref| <= 1e-2 |ref| + 1e-3 sqrt(sum |a b|)."""
    g = oracle.bf16_bits_to_f64(gpu_bits)
    r = oracle.bf16_bits_to_f64(ref_bits)
    tol = 1e-2 * np.abs(r) + 1e-3 * np.sqrt(absacc)
    bad = ~(np.abs(g - r) <= tol)  # NaN counts as a violation
    return bad


def same_bits_signless_zero(a, b):
    """Bitwise equality with +0 == -0."""
    a = np.where((a & 0x7FFF) == 0, 0, a)
    b = np.where((b & 0x7FFF) == 0, 0, b)
    return np.array_equal(a, b)


def sample_indices(E, N, K, rng, rows=8, cols=8, rand=4096, tiling=None, corner_experts=8):
    """Per expert: `rows` full output rows (first, last, random), `cols` full
    columns (likewise) and `rand` random elements. Given the library's tiling
    (a dict with kn, tn, tiles_m, tiles_n as mxfp8_wgrad_tile_config reports
    it), also every element of the four corner tiles of the output (the first
    and last tile of the first and last tile row: the last ones are clipped at
    the output's edges) for `corner_experts` experts (the first, the last and
    random others; all of them when E is at most that). Returns int32 arrays
    (g, n, k)."""
    gs, ns, ks = [], [], []
    corners = []
    if tiling is not None:
        # tile extents along n (output rows) and k (output columns)
        tr, tc = (tiling["tn"], 256) if tiling["kn"] else (256, tiling["tn"])
        rt = sorted({0, (N - 1) // tr})
        ct = sorted({0, (K - 1) // tc})
        for a in rt:
            for b in ct:
                nn = np.arange(a * tr, min(N, (a + 1) * tr))
                kk = np.arange(b * tc, min(K, (b + 1) * tc))
                corners.append((np.repeat(nn, kk.size), np.tile(kk, nn.size)))
    cg = set(range(E)) if E <= corner_experts else {0, E - 1, *rng.choice(E, corner_experts - 2, replace=False).tolist()}
    for g in range(E):
        rsel = sorted({0, N - 1, *rng.integers(0, N, max(0, rows - 2)).tolist()})
        csel = sorted({0, K - 1, *rng.integers(0, K, max(0, cols - 2)).tolist()})
        for n in rsel:
            gs.append(np.full(K, g)); ns.append(np.full(K, n)); ks.append(np.arange(K))
        for k in csel:
            gs.append(np.full(N, g)); ns.append(np.arange(N)); ks.append(np.full(N, k))
        gs.append(np.full(rand, g)); ns.append(rng.integers(0, N, rand)); ks.append(rng.integers(0, K, rand))
        for nn, kk in (corners if g in cg else []):
            gs.append(np.full(nn.size, g)); ns.append(nn); ks.append(kk)
    cat = lambda v: np.concatenate(v).astype(np.int32)  # noqa: E731
    return cat(gs), cat(ns), cat(ks)

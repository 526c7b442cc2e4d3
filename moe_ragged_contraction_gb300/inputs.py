"""Seeded synthetic inputs: routings (group sizes / offsets) and fp32 operands.

This module holds no arithmetic of the method itself (no quantisation, no
contraction). It is the one module that both the CUDA path's tests/benchmark
and the CPU oracle's tests draw inputs from.

Workloads follow "Ragged MXFP8 Weight Gradients: A FlyDSL Grouped GEMM on
MI355X": section 2 names the expert shapes ("16B": N=1408, K=2048, 8 local
experts; "671B": N=4096 or 7168, 32 experts), section 1 gives the routing
properties (busiest expert 1.2-1.7x the mean, empty experts possible,
32-aligned boundaries) and section 7 the synthetic linear-ramp routing with the
busiest expert at 1.5x the mean, plus the 32-aligned-but-not-128-aligned
boundary variant.

Recipes (numpy ``default_rng(seed)``):

* ``tiny`` (seed 1000): one expert (drawn uniformly) is empty; the other three
  get 32 * multinomial(32, [1/3]*3) tokens.
* ``16B`` (1001) / ``16Bp`` (1002): linear ramp t_g = mean * linspace(0.5, 1.5, E),
  rounded to 128 and then moved by +32 (even g) / -32 (odd g), so no size is a
  multiple of 128; the residual goes to the largest group; a seeded
  permutation places the sizes on experts.
* ``671Bgu`` (1003): 30 non-empty experts with Zipf weights r^-s (r = 1..30),
  s found by bisection so that max/mean = 1.7 (mean = M/E); largest-remainder
  rounding to 32-token units; a seeded permutation places them and leaves two
  experts empty.
* ``671Bd`` (1004): 31 non-empty experts on a linear ramp whose maximum is
  1.5 * M/E, in 32-token units; every other size is forced to an odd number of
  units; the residual goes to the last ramp entry; a seeded permutation places
  them and leaves one expert empty.

* ``manyE160`` (1005) / ``manyE512`` (1006): many experts with few tokens each,
  balanced routing in 32-token units ("Group-GEMM in XLA", Part 4: balanced
  group sizes; expert counts and feature sizes of its micro-benchmark classes
  with 160 and 512 experts, token counts raised to whole 32-token scale
  blocks: 64 and 32 tokens per expert).

Operands: dY [M,N] and X [M,K] are drawn directly as their token-contiguous
transposes A_f32 [N,M] and B_f32 [K,M]; N(0,1) for every workload but
``671Bd``, which draws Student-t with 3 degrees of freedom, generated from its
definition z0 / sqrt((z1^2 + z2^2 + z3^2) / 3) with independent normals.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    E: int
    N: int
    K: int
    M: int
    seed: int
    dist: str  # "normal" or "student_t3"
    description: str

    @property
    def flop(self) -> int:
        return 2 * self.N * self.K * self.M


WORKLOADS = {
    "tiny": Workload("tiny", 4, 128, 256, 1024, 1000, "normal",
                     "E=4 N=128 K=256 M=1024, one empty expert, multinomial routing"),
    "16B": Workload("16B", 8, 1408, 2048, 32768, 1001, "normal",
                    "16B shape: E=8 N=1408 K=2048 M=32768 (mean 4096 tok/expert), ramp routing max/mean~1.5, 32- not 128-aligned"),
    "16Bp": Workload("16Bp", 8, 1408, 2048, 196608, 1002, "normal",
                     "16B shape production: E=8 N=1408 K=2048 M=196608 (mean 24576 tok/expert), ramp routing max/mean~1.5"),
    "671Bgu": Workload("671Bgu", 32, 4096, 7168, 262144, 1003, "normal",
                       "671B up/gate: E=32 N=4096 K=7168 M=262144, Zipf routing max/mean~1.7, two empty experts"),
    "671Bd": Workload("671Bd", 32, 7168, 2048, 524288, 1004, "student_t3",
                      "671B down: E=32 N=7168 K=2048 M=524288, ramp routing max/mean~1.5, odd 32-multiples, one empty, Student-t(3) operands"),
    # many experts, few tokens each (scheduling and output-write stress)
    "manyE160": Workload("manyE160", 160, 1536, 5120, 10240, 1005, "normal",
                         "many-expert stress: E=160 N=1536 K=5120 M=10240, balanced routing, 64 tokens per expert"),
    "manyE512": Workload("manyE512", 512, 512, 2048, 16384, 1006, "normal",
                         "many-expert stress: E=512 N=512 K=2048 M=16384, balanced routing, 32 tokens per expert"),
}


# ----------------------------------------------------------------- routing

def _sizes_tiny(w: Workload, rng) -> np.ndarray:
    empty = int(rng.integers(w.E))
    counts = rng.multinomial(w.M // 32, [1.0 / (w.E - 1)] * (w.E - 1))
    sizes = np.zeros(w.E, dtype=np.int64)
    others = [g for g in range(w.E) if g != empty]
    sizes[others] = 32 * counts
    return sizes


def _sizes_ramp_offset(w: Workload, rng) -> np.ndarray:
    mean = w.M / w.E
    t = mean * np.linspace(0.5, 1.5, w.E)
    base = 128 * np.round(t / 128.0).astype(np.int64)
    shift = np.where(np.arange(w.E) % 2 == 0, 32, -32)
    sizes = base + shift
    sizes[int(np.argmax(sizes))] += w.M - int(sizes.sum())
    return sizes[rng.permutation(w.E)]


def _largest_remainder(weights: np.ndarray, units: int) -> np.ndarray:
    exact = units * weights / weights.sum()
    fl = np.floor(exact).astype(np.int64)
    rest = units - int(fl.sum())
    order = np.argsort(-(exact - fl), kind="stable")
    fl[order[:rest]] += 1
    return fl


def _sizes_zipf(w: Workload, rng, n_nonempty=30, ratio=1.7) -> np.ndarray:
    r = np.arange(1, n_nonempty + 1, dtype=np.float64)
    target = w.E / ratio  # sum_r r^-s such that max/mean (mean = M/E) == ratio

    lo, hi = 0.0, 4.0
    for _ in range(200):
        s = 0.5 * (lo + hi)
        if np.sum(r ** -s) > target:
            lo = s
        else:
            hi = s
    s = 0.5 * (lo + hi)
    units = _largest_remainder(r ** -s, w.M // 32)
    sizes = np.zeros(w.E, dtype=np.int64)
    perm = rng.permutation(w.E)
    sizes[perm[:n_nonempty]] = 32 * units
    return sizes


def _sizes_ramp_odd(w: Workload, rng, n_nonempty=31, ratio=1.5) -> np.ndarray:
    units_total = w.M // 32
    mx = ratio * (w.M / w.E) / 32.0  # maximum in 32-token units
    n = n_nonempty
    # t_i = a + b*i, i = 0..n-1, with t_{n-1} = mx and sum t = units_total
    b = (n * mx - units_total) / (n * (n - 1) / 2.0)
    a = mx - b * (n - 1)
    u = np.round(a + b * np.arange(n)).astype(np.int64)
    for i in range(0, n, 2):  # every other size: an odd number of 32-token units
        if u[i] % 2 == 0:
            u[i] -= 1
    u[-1] += units_total - int(u.sum())
    if u[-1] % 2 == 0:  # keep the last (even-indexed) entry odd: trade one unit
        u[-1] -= 1
        u[-2] += 1
    sizes = np.zeros(w.E, dtype=np.int64)
    perm = rng.permutation(w.E)
    sizes[perm[:n]] = 32 * u
    return sizes


def _sizes_balanced(w: Workload, rng) -> np.ndarray:
    return balanced_sizes(w.E, w.M)


_RECIPES = {
    "tiny": _sizes_tiny,
    "16B": _sizes_ramp_offset,
    "16Bp": _sizes_ramp_offset,
    "671Bgu": _sizes_zipf,
    "671Bd": _sizes_ramp_odd,
    "manyE160": _sizes_balanced,
    "manyE512": _sizes_balanced,
}


def with_tokens(name: str, M: int) -> str:
    """Registers (once) and returns the name of a copy of workload `name` with
    M tokens instead of its own, routed by the same recipe: the same expert
    shapes and routing pattern at a smaller size (profiler captures)."""
    from dataclasses import replace

    if M % 32 or M < 32 * WORKLOADS[name].E:
        raise ValueError(f"M={M} must be a multiple of 32 and give every expert at least 32 tokens")
    new = f"{name}@M{M}"
    if new not in WORKLOADS:
        w = WORKLOADS[name]
        WORKLOADS[new] = replace(w, name=new, M=M, description=f"{w.description}; scaled to M={M} tokens")
        _RECIPES[new] = _RECIPES[name]
    return new


def with_experts(name: str, E: int) -> str:
    """Registers (once) and returns the name of a copy of workload `name` with
    E experts and the same mean tokens per expert, routed evenly (every
    expert gets the mean run, in 32-token units): the expert shapes and run
    lengths of the workload at a fraction of its size (profiler captures)."""
    from dataclasses import replace

    w = WORKLOADS[name]
    if E < 1:
        raise ValueError("E must be >= 1")
    M = max(32, int(round(w.M / w.E / 32.0)) * 32) * E
    new = f"{name}@E{E}"
    if new not in WORKLOADS:
        WORKLOADS[new] = replace(w, name=new, E=E, M=M,
                                 description=f"{w.description}; {E} experts with its mean run of {M // E} tokens each")
        _RECIPES[new] = _sizes_balanced
    return new


def group_sizes(name: str) -> np.ndarray:
    """Per-expert token counts (int64 [E]); multiples of 32 summing to M."""
    w = WORKLOADS[name]
    sizes = _RECIPES[name](w, np.random.default_rng(w.seed))
    assert int(sizes.sum()) == w.M and np.all(sizes % 32 == 0) and np.all(sizes >= 0)
    return sizes


def offsets(sizes) -> np.ndarray:
    """Inclusive group ends (int32 [E]) from group sizes."""
    return np.cumsum(np.asarray(sizes, dtype=np.int64)).astype(np.int32)


def balanced_sizes(E: int, M: int, align: int = 32) -> np.ndarray:
    """Deterministic balanced routing ("Group-GEMM in XLA", Part 4): base share
    per group with the remainder going to the first groups, in ``align`` units."""
    units = M // align
    base, rem = divmod(units, E)
    sizes = np.full(E, base, dtype=np.int64)
    sizes[:rem] += 1
    return sizes * align


def random_sizes(E: int, M: int, rng, empty_frac: float = 0.25, align: int = 32) -> np.ndarray:
    """Random 32-aligned group sizes summing to at most M (used for edge tests)."""
    units = M // align
    w = rng.random(E)
    w[rng.random(E) < empty_frac] = 0.0
    if w.sum() == 0:
        return np.zeros(E, dtype=np.int64)
    cut = rng.integers(units // 2, units + 1)
    return _largest_remainder(w, int(cut)) * align


# ---------------------------------------------------------------- operands

_CHUNK_ROWS = 16


def _fill_rows(seed: int, stream: int, dist: str, row0: int, out: np.ndarray) -> None:
    """Fill out[:, :] (rows row0.. of a [R,M] operand) deterministically: each
    block of _CHUNK_ROWS rows has its own generator (seed, stream, block)."""
    rows = out.shape[0]
    for r in range(0, rows, _CHUNK_ROWS):
        blk = (row0 + r) // _CHUNK_ROWS
        assert (row0 + r) % _CHUNK_ROWS == 0
        rng = np.random.default_rng(np.random.SeedSequence(seed, spawn_key=(stream, blk)))
        view = out[r:r + _CHUNK_ROWS]
        if dist == "normal":
            rng.standard_normal(out=view, dtype=np.float32)
        elif dist == "student_t3":
            z0 = rng.standard_normal(view.shape, dtype=np.float32)
            c = np.zeros(view.shape, dtype=np.float32)
            for _ in range(3):
                z = rng.standard_normal(view.shape, dtype=np.float32)
                c += z * z
            np.divide(z0, np.sqrt(c / np.float32(3.0)), out=view)
        else:
            raise ValueError(dist)


def host_operand(rows: int, M: int, seed: int, stream: int, dist: str = "normal",
                 row0: int = 0, nthreads: int | None = None) -> np.ndarray:
    """fp32 [rows, M] slice (rows row0..row0+rows) of a seeded operand; stream 0
    is A = dY^T, stream 1 is B = X^T. Deterministic for any thread count."""
    assert row0 % _CHUNK_ROWS == 0
    out = np.empty((rows, M), dtype=np.float32)
    nthreads = nthreads or max(1, len(os.sched_getaffinity(0)))
    blocks = list(range(0, rows, _CHUNK_ROWS))
    if len(blocks) <= 1 or nthreads == 1:
        _fill_rows(seed, stream, dist, row0, out)
        return out
    with cf.ThreadPoolExecutor(nthreads) as ex:
        list(ex.map(lambda r: _fill_rows(seed, stream, dist, row0 + r, out[r:r + _CHUNK_ROWS]), blocks))
    return out


def device_operand(rows: int, M: int, seed: int, stream: int, dist: str = "normal",
                   device="cuda", chunk_rows: int = 256):
    """fp32 [rows, M] seeded operand generated on the GPU with torch's CUDA
    generator (same distributions as ``host_operand``, different stream of
    numbers). Used by the benchmark, whose inputs need no oracle."""
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(seed * 1000003 + stream)
    out = torch.empty((rows, M), dtype=torch.float32, device=device)
    for r in range(0, rows, chunk_rows):
        view = out[r:r + chunk_rows]
        if dist == "normal":
            view.normal_(generator=gen)
        elif dist == "student_t3":
            z0 = torch.randn(view.shape, generator=gen, device=device)
            c = torch.zeros_like(z0)
            for _ in range(3):
                z = torch.randn(view.shape, generator=gen, device=device)
                c += z * z
            torch.div(z0, torch.sqrt(c / 3.0), out=view)
        else:
            raise ValueError(dist)
    return out

"""GPU parity of the MXFP8 grouped GEMM with ragged rows (the forward /
data-gradient form of the expert layer) against the CPU oracle, through the
C ABI: full outputs on small cases (ragged row boundaries, empty groups,
padding rows, partial K-steps, partial tiles), sampled elements on the 16B
expert shape, exact-representable cases bit for bit, bit-reproducibility and
every tiling giving the same bits."""
import numpy as np
import pytest
import torch

import oracle
import moe_ragged_contraction_gb300 as mx
from moe_ragged_contraction_gb300 import inputs as I

from _util import quantised_operand, same_bits_signless_zero, tolerance_violations

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx.build()
    mx.load()
    mx.device_status(clear=True)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def weights(E, N, K, seed):
    W = np.empty((E, N, K), np.uint8)
    sW = np.empty((E, N, K // 32), np.uint8)
    for g in range(E):
        W[g], sW[g] = quantised_operand(N, K, seed=seed, stream=10 + g)
    return W, sW


def run(X, sX, W, sW, offs):
    M, K = X.shape
    E, N, _ = W.shape
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    out.view(torch.int16).fill_(-1)  # NaN: an unwritten element shows
    mx.grouped_gemm(dev(X), dev(sX), dev(W), dev(sW), dev(np.asarray(offs, np.int32)), out=out)
    torch.cuda.synchronize()
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("E,M,N,K,sizes", [
    (4, 1000, 256, 512, [300, 0, 457, 200]),     # ragged rows, an empty group, 43 padding rows
    (1, 512, 128, 256, [512]),                  # one group: a dense GEMM
    (3, 700, 200, 96, [1, 511, 150]),           # one-row group, N not a tile multiple, K = 96 (3 of 4 MMAs)
    (2, 640, 1408, 1408, [333, 307]),           # K = 11 K-steps, N = 1408
    (16, 900, 64, 128, None),                   # many small groups
])
def test_grouped_gemm_matches_oracle(E, M, N, K, sizes):
    rng = np.random.default_rng(E * 100 + M)
    if sizes is None:
        cuts = np.sort(rng.integers(0, M + 1, E))
        offs = cuts.astype(np.int32)
    else:
        offs = np.cumsum(sizes).astype(np.int32)
    X, sX = quantised_operand(M, K, seed=M + N, stream=0)
    W, sW = weights(E, N, K, seed=M + N)
    got = run(X, sX, W, sW, offs)
    assert mx.device_status(clear=True) == 0
    ref, _, aacc = oracle.grouped_gemm(X, sX, W, sW, offs, E, M, N, K, want_acc=True)
    bad = tolerance_violations(got, ref, aacc)
    assert not bad.any(), f"{bad.sum()} of {bad.size} out of tolerance; first {np.argwhere(bad)[:5].tolist()}"
    assert np.all(got[int(offs[-1]):] == 0), "padding rows not +0"


def test_grouped_gemm_exact_integers():
    """Values in [-2, 2] with unit scales: every partial sum is an exact
    integer in fp32, so the GPU must give the oracle's bits."""
    rng = np.random.default_rng(5)
    E, M, N, K = 3, 600, 320, 1024
    vals = np.array([0x38, 0x40, 0xB8, 0xC0, 0x00], np.uint8)
    X = vals[rng.integers(0, 5, (M, K))]
    W = vals[rng.integers(0, 5, (E, N, K))]
    sX = np.full((M, K // 32), 127, np.uint8)
    sW = np.full((E, N, K // 32), 127, np.uint8)
    offs = np.array([123, 123, 590], np.int32)
    got = run(X, sX, W, sW, offs)
    ref = oracle.grouped_gemm(X, sX, W, sW, offs, E, M, N, K)
    assert same_bits_signless_zero(got, ref)


def test_grouped_gemm_tilings_and_reproducible():
    E, M, N, K = 3, 800, 448, 640
    X, sX = quantised_operand(M, K, seed=7, stream=0)
    W, sW = weights(E, N, K, seed=7)
    offs = np.array([250, 251, 777], np.int32)
    outs = []
    try:
        for tn in (0, 128, 224, 256, 320, 352, 416, 448):
            mx.set_tile_rows(tn)
            for store in (0, 1):  # TMA stores where their staging fits / direct stores
                mx.set_epilogue_store(store)
                outs.append(run(X, sX, W, sW, offs))
    finally:
        mx.set_tile_rows(0)
        mx.set_epilogue_store(0)
    outs.append(run(X, sX, W, sW, offs))
    for o in outs[1:]:
        assert np.array_equal(outs[0], o)


def test_grouped_gemm_16B_expert_shape_sampled():
    """The 16B expert layer's forward product (hidden 2048 -> 1408 per expert)
    on the 16B routing: sampled full rows and random elements vs the oracle,
    whole output finite, reproducible."""
    w = I.WORKLOADS["16B"]
    E, M, N, K = w.E, w.M, w.N, w.K
    offs = I.offsets(I.group_sizes("16B"))
    X, sX = quantised_operand(M, K, seed=w.seed, stream=2)
    W, sW = weights(E, N, K, seed=w.seed)
    dX, dsX, dW, dsW, doffs = dev(X), dev(sX), dev(W), dev(sW), dev(offs)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    out.view(torch.int16).fill_(-1)
    mx.grouped_gemm(dX, dsX, dW, dsW, doffs, out=out)
    out2 = mx.grouped_gemm(dX, dsX, dW, dsW, doffs)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    assert torch.isfinite(out.float()).all()
    rng = np.random.default_rng(11)
    rows = np.concatenate([[0, M - 1], rng.integers(0, M, 14), offs[:-1] - 1, offs[:-1]]).astype(np.int64)
    t = np.repeat(rows, N)
    n = np.tile(np.arange(N), rows.size)
    t = np.concatenate([t, rng.integers(0, M, 4096)])
    n = np.concatenate([n, rng.integers(0, N, 4096)])
    ref, _, aacc = oracle.grouped_gemm(X, sX, W, sW, offs, E, M, N, K, points=(t, n), want_acc=True)
    got = out.view(torch.int16)[torch.from_numpy(t).cuda(), torch.from_numpy(n).cuda()].cpu().numpy().view(np.uint16)
    bad = tolerance_violations(got, ref, aacc)
    assert not bad.any(), f"{bad.sum()} of {bad.size} sampled elements out of tolerance"


@pytest.mark.parametrize("E,M,N,K,sizes", [
    (3, 64, 256, 64, [0, 0, 0]),          # every group empty: the whole output is padding
    (1, 1, 32, 32, [1]),                  # one row, one partial K-step (one k = 32 MMA)
    (2, 160, 8, 160, [150, 10]),          # the narrowest output (N = 8), K-step of 32 + partial
    (5, 2000, 264, 96, None),             # M not a multiple of 32, random group boundaries
    (2, 512, 1408, 2048, [511, 1]),       # a one-row group after a 511-row group
])
def test_grouped_gemm_edge_shapes(E, M, N, K, sizes):
    rng = np.random.default_rng(E * 7 + M + N + K)
    if sizes is None:
        offs = np.sort(rng.integers(0, M + 1, E)).astype(np.int32)
    else:
        offs = np.cumsum(sizes).astype(np.int32)
    X, sX = quantised_operand(M, K, seed=M + K, stream=0)
    W, sW = weights(E, N, K, seed=M + K)
    outs = []
    try:
        for store in (0, 1):
            mx.set_epilogue_store(store)
            outs.append(run(X, sX, W, sW, offs))
    finally:
        mx.set_epilogue_store(0)
    assert np.array_equal(outs[0], outs[1])
    assert mx.device_status(clear=True) == 0
    ref, _, aacc = oracle.grouped_gemm(X, sX, W, sW, offs, E, M, N, K, want_acc=True)
    bad = tolerance_violations(outs[0], ref, aacc)
    assert not bad.any(), f"{bad.sum()} of {bad.size} out of tolerance"
    assert np.all(outs[0][int(offs[-1]):] == 0), "padding rows not +0"


@pytest.mark.parametrize("name,product", [
    ("671Bgu", "forward"), ("671Bgu", "dgrad"), ("671Bd", "forward"), ("671Bd", "dgrad"),
])
def test_grouped_gemm_671B_layer_shapes_sampled(name, product):
    """The 671B expert layers' forward and data-gradient products at full
    size, on the workload's routing, in the launch the grouped-GEMM benchmark
    times: forward X [M, K] x W [E, N, K]^T, data gradient dY [M, N] x
    W^T [E, K, N]^T. Sampled elements against the oracle (full rows at both
    ends, at every group boundary and at random, plus 4,096 random elements),
    the whole NaN-poisoned output finite, two runs identical."""
    w = I.WORKLOADS[name]
    E, M = w.E, w.M
    rows_w, cols = (w.N, w.K) if product == "forward" else (w.K, w.N)  # W [E, rows_w, cols], contraction over cols
    offs = I.offsets(I.group_sizes(name))
    block = max(256, (1 << 24) // cols // 16 * 16)  # rows per host-generated block (a multiple of 16)
    X, sX = quantised_operand(M, cols, seed=w.seed, stream=30 if product == "forward" else 31, dist=w.dist,
                              block_rows=block)
    W = np.empty((E, rows_w, cols), np.uint8)
    sW = np.empty((E, rows_w, cols // 32), np.uint8)
    for g in range(E):
        W[g], sW[g] = quantised_operand(rows_w, cols, seed=w.seed, stream=40 + g, block_rows=block)
    dX, dsX, dW, dsW, doffs = dev(X), dev(sX), dev(W), dev(sW), dev(offs)
    mx.device_status(clear=True)
    out = torch.empty((M, rows_w), dtype=torch.bfloat16, device="cuda")
    out.view(torch.int16).fill_(-1)
    mx.grouped_gemm(dX, dsX, dW, dsW, doffs, out=out)
    out2 = torch.empty_like(out)
    out2.view(torch.int16).fill_(-1)
    mx.grouped_gemm(dX, dsX, dW, dsW, doffs, out=out2)
    torch.cuda.synchronize()
    assert mx.device_status(clear=True) == 0
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16)), "not bit-reproducible"
    del out2
    assert torch.isfinite(out.float()).all(), "unwritten (NaN-poisoned) or non-finite elements"
    rng = np.random.default_rng(w.seed + (0 if product == "forward" else 1))
    live = offs[:-1][(offs[:-1] > 0) & (offs[:-1] < M)]
    rows = np.unique(np.concatenate([[0, M - 1], rng.integers(0, M, 8), live - 1, live])).astype(np.int64)
    t = np.concatenate([np.repeat(rows, rows_w), rng.integers(0, M, 4096)])
    n = np.concatenate([np.tile(np.arange(rows_w), rows.size), rng.integers(0, rows_w, 4096)])
    ref, _, aacc = oracle.grouped_gemm(X, sX, W, sW, offs, E, M, rows_w, cols, points=(t, n), want_acc=True)
    got = out.view(torch.int16)[torch.from_numpy(t).cuda(), torch.from_numpy(n).cuda()].cpu().numpy().view(np.uint16)
    bad = tolerance_violations(got, ref, aacc)
    assert not bad.any(), f"{bad.sum()} of {bad.size} sampled elements out of tolerance"

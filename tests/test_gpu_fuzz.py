"""Randomised shapes and routings against the oracle (full outputs): the
weight gradient, the grouped GEMM with ragged rows, and the path over scale
blocks written by the quantiser (against the regular path's bits).

Seeded draws of E, N, K, M and of the routing (empty experts, runs that start
and end inside a 128-token step, tokens left past the last run), each under
the library's own tiling and under a forced orientation and tile width, with
realistic quantised operands. Every output element is compared with the
oracle within the parity tolerance (NaN-poisoned outputs, so an unwritten
element shows), empty experts are exact +0, and the forced tiling gives the
same bits as the library's own (each output element sums the same 32-token
block products in the same order whatever the tiling)."""
import numpy as np
import pytest
import torch

import oracle
import moe_ragged_contraction_gb300 as mx

from _util import quantised_operand, tolerance_violations

pytestmark = pytest.mark.gpu

CASES = 16


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx.build()
    mx.load()
    mx.device_status(clear=True)
    yield
    mx.set_tile_orientation(0)
    mx.set_tile_rows(0)


def draw_case(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 41))
    N = int(rng.integers(1, 90)) * 8
    K = int(rng.integers(1, 110)) * 8
    M = int(rng.integers(1, 129)) * 32
    # runs in 32-token units: some empty, the rest random, a random tail left unused
    units = M // 32
    used = int(rng.integers(units // 2, units + 1))
    w = rng.random(E) * (rng.random(E) > 0.2)
    if w.sum() == 0:
        sizes = np.zeros(E, np.int64)
    else:
        sizes = np.floor(w / w.sum() * used).astype(np.int64)
    offs = (np.cumsum(sizes) * 32).astype(np.int32)
    # forced tiling for the second run: an orientation and an admissible width
    orient = int(rng.integers(1, 3))
    tn = int(rng.integers(1, 29)) * 16
    return E, N, K, M, offs, orient, tn


def run(A, sA, B, sB, offs, E, N, K):
    d = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (A, sA, B, sB, offs)]
    out = torch.empty((E, N, K), dtype=torch.bfloat16, device="cuda")
    out.view(torch.int16).fill_(-1)
    mx.wgrad_grouped(*d, out=out)
    torch.cuda.synchronize()
    assert mx.device_status(clear=True) == 0
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


@pytest.mark.parametrize("seed", range(CASES))
def test_random_shape_against_oracle(seed):
    E, N, K, M, offs, orient, tn = draw_case(1000 + seed)
    A, sA = quantised_operand(N, M, seed=2000 + seed, stream=0, block_rows=64)
    B, sB = quantised_operand(K, M, seed=2000 + seed, stream=1, block_rows=64)
    try:
        mx.set_tile_orientation(0)
        mx.set_tile_rows(0)
        got = run(A, sA, B, sB, offs, E, N, K)
        mx.set_tile_orientation(orient)
        mx.set_tile_rows(tn)
        forced = run(A, sA, B, sB, offs, E, N, K)
    finally:
        mx.set_tile_orientation(0)
        mx.set_tile_rows(0)
    ref, _, aacc = oracle.wgrad(A, sA, B, sB, offs, E, N, K, M, want_acc=True)
    bad = tolerance_violations(got, ref, aacc)
    assert not bad.any(), f"E={E} N={N} K={K} M={M}: {bad.sum()} elements out of tolerance"
    assert np.array_equal(got, forced), f"E={E} N={N} K={K} M={M}: orientation {orient}, tn {tn} gave other bits"
    lo = 0
    for g in range(E):
        if int(offs[g]) == lo:
            assert not got[g].any(), f"empty expert {g} not exact +0"
        lo = int(offs[g])


def draw_gemm_case(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 17))
    M = int(rng.integers(1, 1500))
    N = int(rng.integers(1, 80)) * 8
    K = int(rng.integers(1, 25)) * 32
    used = int(rng.integers(M // 2, M + 1))
    w = rng.random(E) * (rng.random(E) > 0.2)
    sizes = np.zeros(E, np.int64) if w.sum() == 0 else np.floor(w / w.sum() * used).astype(np.int64)
    return E, M, N, K, np.cumsum(sizes).astype(np.int32)


@pytest.mark.parametrize("seed", range(8))
def test_random_grouped_gemm_against_oracle(seed):
    """The grouped GEMM with ragged rows (groups cut at any row) on random
    shapes: within the parity tolerance of the oracle, rows past the last group
    exact +0."""
    E, M, N, K, offs = draw_gemm_case(3000 + seed)
    X, sX = quantised_operand(M, K, seed=4000 + seed, stream=0, block_rows=16)
    W = np.empty((E, N, K), np.uint8)
    sW = np.empty((E, N, K // 32), np.uint8)
    for e in range(E):
        W[e], sW[e] = quantised_operand(N, K, seed=5000 + seed, stream=1 + e, block_rows=16)
    d = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (X, sX, W, sW, offs)]
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    out.view(torch.int16).fill_(-1)
    mx.grouped_gemm(*d, out=out)
    torch.cuda.synchronize()
    assert mx.device_status(clear=True) == 0
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    ref, _, aacc = oracle.grouped_gemm(X, sX, W, sW, offs, E, M, N, K, want_acc=True)
    bad = tolerance_violations(got, ref, aacc)
    assert not bad.any(), f"E={E} M={M} N={N} K={K}: {bad.sum()} elements out of tolerance"
    assert not got[int(offs[-1]):].any(), "rows past the last group not +0"


@pytest.mark.parametrize("seed", range(6))
def test_random_scale_block_path_same_bits(seed):
    """The quantiser that writes scale-factor blocks and the weight gradient
    over them (mxfp8_quantize_transpose_bf16_sf, mxfp8_wgrad_grouped_sf) on
    random shapes and routings, for the library's tiling and for a random
    other one: the regular entry point's bits on the same quantised operands."""
    rng = np.random.default_rng(6000 + seed)
    E = int(rng.integers(1, 25))
    N = int(rng.integers(1, 700))
    K = int(rng.integers(1, 90)) * 8
    M = int(rng.integers(1, 97)) * 32
    units = M // 32
    used = int(rng.integers(units // 2, units + 1))
    w = rng.random(E) * (rng.random(E) > 0.2)
    sizes = np.zeros(E, np.int64) if w.sum() == 0 else np.floor(w / w.sum() * used).astype(np.int64)
    offs = torch.from_numpy((np.cumsum(sizes) * 32).astype(np.int32)).cuda()
    g = torch.Generator(device="cuda")
    g.manual_seed(7000 + seed)
    dy = torch.randn(M, N, device="cuda", generator=g).to(torch.bfloat16)
    x = torch.randn(M, K, device="cuda", generator=g).to(torch.bfloat16)
    cfg = mx.tile_config(E, N, K, M)
    tilings = [(cfg["kn"], cfg["tn"]), (int(rng.integers(0, 2)), int(rng.integers(1, 29)) * 16)]
    ref = None
    for kn, tn in tilings:
        sA = torch.empty((N, M // 32), dtype=torch.uint8, device="cuda")
        sB = torch.empty((K, M // 32), dtype=torch.uint8, device="cuda")
        A, sfA, _ = mx.quantize_transpose_bf16_sf(dy, tn if kn else 256, s=sA)
        B, sfB, _ = mx.quantize_transpose_bf16_sf(x, 256 if kn else tn, s=sB)
        if ref is None:
            ref = mx.wgrad_grouped(A, sA, B, sB, offs)
        got = torch.empty_like(ref)
        got.view(torch.int16).fill_(-1)
        mx.wgrad_grouped_sf(A, sfA, B, sfB, offs, kn, tn, out=got)
        torch.cuda.synchronize()
        assert mx.device_status(clear=True) == 0
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), \
            f"E={E} N={N} K={K} M={M} kn={kn} tn={tn}: not the regular entry point's bits"

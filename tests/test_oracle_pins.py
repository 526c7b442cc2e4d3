"""Pins for the CPU oracle: each test ties the oracle to something other than
itself (a library decode or rounding routine, exact rational arithmetic, a
hand-computed value, a closed form, a dense-GEMM special case, or the worked
example printed on the XLA page), so that a dropped term, a wrong sign or
index, or a transposed operand in the oracle fails at least one of them."""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import ragged_dot as rd

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------- helpers

def torch_e4m3(codes):
    t = torch.tensor(np.asarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_e8m0(codes):
    t = torch.tensor(np.asarray(codes, dtype=np.uint8))
    return t.view(torch.float8_e8m0fnu).to(torch.float64).numpy()


_BF16_FINITE = None


def bf16_table():
    """All finite non-negative bf16 values (bits 0x0000..0x7F7F) as fp64, sorted."""
    global _BF16_FINITE
    if _BF16_FINITE is None:
        bits = np.arange(0, 0x7F80, dtype=np.uint32)
        vals = (bits << 16).view(np.float32).astype(np.float64)
        _BF16_FINITE = (bits.astype(np.uint16), vals)
    return _BF16_FINITE


def bf16_nearest_exact(x: Fraction) -> int:
    """Brute-force round-to-nearest-even of an exact rational to bf16 bits, by
    search over the table of all finite bf16 values."""
    bits, vals = bf16_table()
    neg = x < 0
    ax = -x if neg else x
    sign = 0x8000 if neg else 0
    if ax == 0:
        return sign
    i = int(np.searchsorted(vals, float(ax)))
    cands = [j for j in (i - 2, i - 1, i, i + 1) if 0 <= j < len(vals)]
    best = None
    for j in cands:
        d = abs(Fraction(vals[j]) - ax)
        key = (d, int(bits[j]) & 1)  # tie -> even mantissa (LSB 0)
        if best is None or key < best[0]:
            best = (key, j)
    j = best[1]
    if j == len(vals) - 1 and ax > Fraction(vals[j]):
        # above the largest finite value: overflow to inf once past the halfway point
        top = Fraction(vals[j])
        ulp = top - Fraction(vals[j - 1])
        if ax >= top + ulp / 2:
            return sign | 0x7F80
    return sign | int(bits[j])


def q_operand(rng, R, M, lo=0, hi=256, scale_lo=120, scale_hi=135):
    """Random finite E4M3 codes and E8M0 scales (no NaN codes)."""
    q = rng.integers(lo, hi, size=(R, M), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x7E
    s = rng.integers(scale_lo, scale_hi, size=(R, M // 32), dtype=np.uint8)
    return q, s


# --------------------------------------------------------------- P-h decode tables

def test_e4m3_decode_matches_torch(oracle_mod):
    codes = np.arange(256)
    ref = torch_e4m3(codes)
    got = np.array([oracle_mod.dec_e4m3(c) for c in codes])
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan_ref)
    assert nan_ref.sum() == 2  # 0x7F and 0xFF only
    assert np.array_equal(got[~nan_ref], ref[~nan_ref])
    # spot values: 448 is the largest finite value (the scale rule divides by it)
    assert oracle_mod.dec_e4m3(0x7E) == 448.0
    assert oracle_mod.dec_e4m3(0x38) == 1.0 and oracle_mod.dec_e4m3(0xB8) == -1.0
    assert oracle_mod.dec_e4m3(0x01) == 2.0 ** -9 and oracle_mod.dec_e4m3(0x07) == 7 * 2.0 ** -9
    assert oracle_mod.dec_e4m3(0x08) == 2.0 ** -6


def test_e8m0_decode_matches_torch(oracle_mod):
    codes = np.arange(256)
    ref = torch_e8m0(codes)
    got = np.array([oracle_mod.dec_e8m0(c) for c in codes])
    assert np.isnan(got[255]) and np.isnan(ref[255])
    assert np.array_equal(got[:255], ref[:255])
    assert oracle_mod.dec_e8m0(0x7F) == 1.0 and oracle_mod.dec_e8m0(0x80) == 2.0
    assert oracle_mod.dec_e8m0(0x00) == 2.0 ** -127


# --------------------------------------------------------------- bf16 rounding

def test_bf16_rne_matches_torch_on_fp32_values(oracle_mod):
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(1e3),
        rng.standard_normal(2000).astype(np.float32) * np.float32(1e-38),   # bf16 subnormals
        np.clip(rng.standard_normal(2000) * 3e38, -3.4e38, 3.4e38).astype(np.float32),  # near overflow
        np.array([0.0, -0.0, 1.0, -1.0, 3.3895314e38, 3.4e38], dtype=np.float32),
    ])
    x = x[np.isfinite(x)]
    ref = torch.tensor(x).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    got = np.array([oracle_mod.bf16_rne(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_rne_exact_on_fp64_values(oracle_mod):
    """Values that fp32 cannot hold (so no library routine applies): brute-force
    nearest-even search over every finite bf16 value, in exact rationals."""
    rng = np.random.default_rng(11)
    xs = list(rng.standard_normal(300) * 10.0 ** rng.integers(-45, 39, 300))
    # exact ties between neighbours: 1 + 2^-8 (tie -> 1.0), 1 + 3*2^-8 (tie -> 1+2^-6)
    xs += [1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 2.0 ** -134, 3 * 2.0 ** -134,
           2.0 ** -140, 448.0 ** 2 * 2.0 ** -254, 1e300, -1e300]
    for x in xs:
        assert oracle_mod.bf16_rne(x) == bf16_nearest_exact(Fraction(x)), x
    assert oracle_mod.bf16_rne(float("nan")) == 0x7FC0


# --------------------------------------------------------------- P-a exact brute force

def exact_wgrad(A, sA, B, sB, offs, E, N, K, M):
    fa = {c: Fraction(float(torch_e4m3([c])[0])) for c in range(256) if (c & 0x7F) != 0x7F}
    out = np.zeros((E, N, K), dtype=np.uint16)
    exact = {}
    for g in range(E):
        lo = 0 if g == 0 else int(offs[g - 1])
        hi = int(offs[g])
        for n in range(N):
            for k in range(K):
                acc = Fraction(0)
                for t in range(lo, hi):
                    a = fa[int(A[n, t])] * Fraction(2) ** (int(sA[n, t // 32]) - 127)
                    b = fa[int(B[k, t])] * Fraction(2) ** (int(sB[k, t // 32]) - 127)
                    acc += a * b
                exact[(g, n, k)] = acc
                out[g, n, k] = bf16_nearest_exact(acc)
    return out, exact


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_wgrad_exact_bruteforce(oracle_mod, seed):
    rng = np.random.default_rng(100 + seed)
    E = int(rng.integers(1, 4))
    N = int(rng.integers(1, 5))
    K = int(rng.integers(1, 5))
    M = 32 * int(rng.integers(1, 5))
    A, sA = q_operand(rng, N, M)
    B, sB = q_operand(rng, K, M)
    cuts = np.sort(rng.integers(0, M // 32 + 1, size=E)) * 32
    offs = cuts.astype(np.int32)
    got, acc, _ = oracle_mod.wgrad(A, sA, B, sB, offs, E, N, K, M, want_acc=True)
    ref, exact = exact_wgrad(A, sA, B, sB, offs, E, N, K, M)
    zero_eq = (got & 0x7FFF) == 0
    assert np.array_equal(np.where(zero_eq, 0, got), np.where((ref & 0x7FFF) == 0, 0, ref))
    for (g, n, k), v in exact.items():
        assert abs(Fraction(acc[g, n, k]) - v) <= abs(v) * Fraction(1, 2 ** 50)


def test_wgrad_rejects_bad_offsets(oracle_mod):
    rng = np.random.default_rng(5)
    A, sA = q_operand(rng, 2, 64)
    B, sB = q_operand(rng, 2, 64)
    for offs in ([32, 16], [48, 64], [32, 96], [-32, 64]):
        with pytest.raises(ValueError):
            oracle_mod.wgrad(A, sA, B, sB, np.array(offs, np.int32), 2, 2, 2, 64)


# --------------------------------------------------------------- P-b hand-computed

def _const_case(a_code, b_code, offs, E=2, M=64, sa=None):
    A = np.full((1, M), a_code, np.uint8)
    B = np.full((1, M), b_code, np.uint8)
    sA = np.full((1, M // 32), 0x7F, np.uint8) if sa is None else np.array([sa], np.uint8)
    sB = np.full((1, M // 32), 0x7F, np.uint8)
    return A, sA, B, sB, np.array(offs, np.int32), E, 1, 1, M


def test_hand_case_1(oracle_mod):
    out = oracle_mod.wgrad(*_const_case(0x38, 0x40, [32, 64]))
    assert oracle_mod.bf16_bits_to_f64(out).ravel().tolist() == [64.0, 64.0]  # 32 * 1 * 2


def test_hand_case_2_block_scale(oracle_mod):
    out = oracle_mod.wgrad(*_const_case(0x38, 0x40, [32, 64], sa=[0x7F, 0x80]))
    assert oracle_mod.bf16_bits_to_f64(out).ravel().tolist() == [64.0, 128.0]


def test_hand_case_3_empty_first(oracle_mod):
    out = oracle_mod.wgrad(*_const_case(0x38, 0x40, [0, 64]))
    assert oracle_mod.bf16_bits_to_f64(out).ravel().tolist() == [0.0, 128.0]
    assert out.ravel()[0] == 0x0000


def test_hand_case_4_underflow_to_zero(oracle_mod):
    # one token pair 448 * 448 with both scales 2^-127: 448^2 * 2^-254, nonzero in
    # fp64, zero after bf16 rounding (below half the smallest bf16 subnormal)
    A = np.zeros((1, 32), np.uint8); A[0, 0] = 0x7E
    B = np.zeros((1, 32), np.uint8); B[0, 0] = 0x7E
    sA = np.zeros((1, 1), np.uint8); sB = np.zeros((1, 1), np.uint8)
    out, acc, _ = oracle_mod.wgrad(A, sA, B, sB, np.array([32], np.int32), 1, 1, 1, 32, want_acc=True)
    assert acc[0, 0, 0] == 448.0 ** 2 * 2.0 ** -254 and acc[0, 0, 0] > 0
    assert out[0, 0, 0] == 0x0000


def test_hand_negative_and_mixed(oracle_mod):
    # A = -1 (0xB8) for 32 tokens of expert 0, +0.5 (0x30) after; B = 2 (0x40)
    M = 64
    A = np.concatenate([np.full(32, 0xB8), np.full(32, 0x30)]).astype(np.uint8)[None]
    B = np.full((1, M), 0x40, np.uint8)
    s = np.full((1, 2), 0x7F, np.uint8)
    out = oracle_mod.wgrad(A, s, B, s, np.array([32, 64], np.int32), 2, 1, 1, M)
    assert oracle_mod.bf16_bits_to_f64(out).ravel().tolist() == [-64.0, 32.0]


# --------------------------------------------------------------- P-c empty experts

def test_empty_experts_exact_zero(oracle_mod):
    rng = np.random.default_rng(3)
    M, N, K = 128, 3, 5
    A, sA = q_operand(rng, N, M)
    B, sB = q_operand(rng, K, M)
    for offs in ([0, 0, 0], [0, 64, 64, 128], [128, 128], [0, 0, 128]):
        E = len(offs)
        out = oracle_mod.wgrad(A, sA, B, sB, np.array(offs, np.int32), E, N, K, M)
        for g in range(E):
            lo = 0 if g == 0 else offs[g - 1]
            if offs[g] == lo:
                assert np.all(out[g] == 0x0000)
            else:
                assert np.any(out[g] != 0)


# --------------------------------------------------------------- P-d invariant, P-f dense special cases

def test_sum_over_experts_equals_dense(oracle_mod):
    rng = np.random.default_rng(9)
    E, N, K, M = 5, 17, 23, 640
    A, sA = q_operand(rng, N, M)
    B, sB = q_operand(rng, K, M)
    sizes = np.array([96, 0, 224, 64, 160])
    offs = np.cumsum(sizes).astype(np.int32)  # ends at 544 < M: tail ignored
    _, acc, _ = oracle_mod.wgrad(A, sA, B, sB, offs, E, N, K, M, want_acc=True)
    Ad = oracle_mod.decode_operand(A, sA)[:, :offs[-1]]
    Bd = oracle_mod.decode_operand(B, sB)[:, :offs[-1]]
    dense = Ad @ Bd.T
    assert np.allclose(acc.sum(axis=0), dense, rtol=1e-12, atol=1e-300)
    # each expert alone is the dense product over its own token slice (transposes
    # would swap the [N,K] axes and fail on N != K)
    lo = 0
    for g in range(E):
        hi = int(offs[g])
        ref = Ad[:, lo:hi] @ Bd[:, lo:hi].T
        assert acc[g].shape == ref.shape
        assert np.allclose(acc[g], ref, rtol=1e-12, atol=1e-300)
        lo = hi


def test_integer_data_exact(oracle_mod):
    """Integer-valued data with power-of-two scales: fp64 sums are exact, and
    the result equals numpy's integer matmul exactly."""
    rng = np.random.default_rng(12)
    N, K, M = 9, 13, 256
    ints = np.array([-2, -1, 0, 1, 2])
    codes = {-2: 0xC0, -1: 0xB8, 0: 0x00, 1: 0x38, 2: 0x40}
    Ai = rng.choice(ints, size=(N, M)); Bi = rng.choice(ints, size=(K, M))
    A = np.vectorize(codes.get)(Ai).astype(np.uint8)
    B = np.vectorize(codes.get)(Bi).astype(np.uint8)
    s = np.full((N, M // 32), 0x7F, np.uint8); t = np.full((K, M // 32), 0x7F, np.uint8)
    offs = np.array([96, 256], np.int32)
    out, acc, _ = oracle_mod.wgrad(A, s, B, t, offs, 2, N, K, M, want_acc=True)
    assert np.array_equal(acc[0], (Ai[:, :96] @ Bi[:, :96].T).astype(np.float64))
    assert np.array_equal(acc[1], (Ai[:, 96:] @ Bi[:, 96:].T).astype(np.float64))
    ref_bits = torch.tensor(acc.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    assert np.array_equal(out, ref_bits)


def test_single_expert_is_dense_gemm(oracle_mod):
    rng = np.random.default_rng(13)
    N, K, M = 11, 7, 320
    A, sA = q_operand(rng, N, M)
    B, sB = q_operand(rng, K, M)
    out, acc, _ = oracle_mod.wgrad(A, sA, B, sB, np.array([M], np.int32), 1, N, K, M, want_acc=True)
    dense = oracle_mod.decode_operand(A, sA) @ oracle_mod.decode_operand(B, sB).T
    assert np.allclose(acc[0], dense, rtol=1e-12, atol=0)
    ref_bits = torch.tensor(dense.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    # fp64 -> fp32 -> bf16 can double-round; allow one ulp, and require most equal
    diff = np.abs(out.astype(np.int32) - ref_bits.astype(np.int32))
    assert diff.max() <= 1 and (diff == 0).mean() > 0.95


def test_equal_groups_are_batched_gemm(oracle_mod):
    rng = np.random.default_rng(14)
    E, N, K, L = 4, 6, 10, 96
    M = E * L
    A, sA = q_operand(rng, N, M)
    B, sB = q_operand(rng, K, M)
    offs = (np.arange(1, E + 1) * L).astype(np.int32)
    _, acc, _ = oracle_mod.wgrad(A, sA, B, sB, offs, E, N, K, M, want_acc=True)
    Ad = oracle_mod.decode_operand(A, sA).reshape(N, E, L)
    Bd = oracle_mod.decode_operand(B, sB).reshape(K, E, L)
    ref = np.einsum("nel,kel->enk", Ad, Bd)
    assert np.allclose(acc, ref, rtol=1e-12, atol=0)


def test_abs_sum_output(oracle_mod):
    rng = np.random.default_rng(15)
    N, K, M = 4, 5, 128
    A, sA = q_operand(rng, N, M)
    B, sB = q_operand(rng, K, M)
    _, _, aacc = oracle_mod.wgrad(A, sA, B, sB, np.array([M], np.int32), 1, N, K, M, want_acc=True)
    ref = np.abs(oracle_mod.decode_operand(A, sA)) @ np.abs(oracle_mod.decode_operand(B, sB)).T
    assert np.allclose(aacc[0], ref, rtol=1e-12, atol=0)


def test_points_match_full(oracle_mod):
    rng = np.random.default_rng(16)
    E, N, K, M = 3, 8, 12, 256
    A, sA = q_operand(rng, N, M)
    B, sB = q_operand(rng, K, M)
    offs = np.array([64, 64, 224], np.int32)
    full = oracle_mod.wgrad(A, sA, B, sB, offs, E, N, K, M)
    g = rng.integers(0, E, 50); n = rng.integers(0, N, 50); k = rng.integers(0, K, 50)
    pts = oracle_mod.wgrad_points(A, sA, B, sB, offs, E, N, K, M, g, n, k)
    assert np.array_equal(pts, full[g, n, k])


# --------------------------------------------------------------- P-g worked example

def test_xla_worked_example():
    with open(os.path.join(GOLDEN, "ragged_dot_worked_example.json")) as f:
        ex = json.load(f)
    lhs = np.array(ex["lhs"]); rhs = np.array(ex["rhs"]); gs = ex["group_sizes"]
    out = rd.ragged_dot(lhs, rhs, gs)
    assert np.allclose(out, np.array(ex["ragged_dot"]), rtol=0, atol=1e-12)
    con = rd.ragged_dot_contracting(out.T, lhs, gs)  # out_g = Y[g]^T lhs[g]
    assert np.allclose(con, np.array(ex["contracting_YT_lhs"]), rtol=0, atol=1e-12)


def test_contracting_form_matches_wgrad(oracle_mod):
    """The MXFP8 wgrad is the contracting ragged dot on dequantised operands:
    lhs = dY^T [N, M], rhs = X [M, K]."""
    rng = np.random.default_rng(17)
    E, N, K, M = 3, 5, 6, 192
    A, sA = q_operand(rng, N, M)
    B, sB = q_operand(rng, K, M)
    sizes = [64, 0, 128]
    offs = np.cumsum(sizes).astype(np.int32)
    _, acc, _ = oracle_mod.wgrad(A, sA, B, sB, offs, E, N, K, M, want_acc=True)
    ref = rd.ragged_dot_contracting(oracle_mod.decode_operand(A, sA), oracle_mod.decode_operand(B, sB).T, sizes)
    assert np.allclose(acc, ref, rtol=1e-12, atol=0)


# --------------------------------------------------------------- P-i quantiser

def test_quantiser_scale_rule_and_rounding(oracle_mod):
    rng = np.random.default_rng(21)
    R, M = 16, 2048
    x = rng.standard_normal((R, M)).astype(np.float32) * np.float32(10.0) ** rng.integers(-8, 8, (R, 1)).astype(np.float32)
    q, s = oracle_mod.quantize_tokenwise(x)
    xb = x.reshape(R, M // 32, 32).astype(np.float64)
    amax = np.abs(xb).max(axis=2)
    # the page's rule: scale = 2^ceil(log2(amax / 448))
    e_ref = np.array([[math.ceil(math.log2(a / 448.0)) for a in row] for row in amax])
    assert np.array_equal(s.astype(np.int64) - 127, e_ref)
    # elements: x * 2^-e rounded to E4M3 by torch's fp32 -> float8_e4m3fn cast (RNE)
    y = (xb * np.exp2(-e_ref)[:, :, None]).astype(np.float32).reshape(R, M)
    ref = torch.tensor(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)


def test_quantiser_round_trip_on_grid(oracle_mod):
    rng = np.random.default_rng(22)
    R, M = 8, 512
    codes = rng.integers(0, 0x7E, size=(R, M), dtype=np.uint8) | (rng.integers(0, 2, (R, M), dtype=np.uint8) << 7)
    codes[:, ::32] = 0x7E  # each block holds +448 * 2^e exactly -> scale exponent e
    e = rng.integers(-20, 20, size=(R, M // 32))
    x = (torch_e4m3(codes) * np.repeat(np.exp2(e), 32, axis=1)).astype(np.float32)
    q, s = oracle_mod.quantize_tokenwise(x)
    assert np.array_equal(s.astype(np.int64) - 127, e)
    assert np.array_equal(q, codes)


def test_quantiser_amax_boundary_and_zero_block(oracle_mod):
    x = np.zeros((3, 64), np.float32)
    x[0, :32] = 0.0                       # all-zero block -> byte 0, data 0
    x[0, 32] = 448.0 * 2.0 ** 3           # amax exactly 448*2^3 -> e = 3, not 4
    x[1, 0] = np.nextafter(np.float32(448.0), np.float32(1e9))  # just above 448 -> e = 1
    x[1, 32] = -448.0
    x[2, 0] = np.float32(1e-44)           # fp32 subnormal amax -> clamped to e = -127
    x[2, 32] = -0.0
    q, s = oracle_mod.quantize_tokenwise(x)
    assert s[0, 0] == 0x00 and np.all(q[0, :32] == 0)
    assert int(s[0, 1]) - 127 == 3 and q[0, 32] == 0x7E
    assert int(s[1, 0]) - 127 == 1
    assert int(s[1, 1]) - 127 == 0 and q[1, 32] == 0xFE
    assert int(s[2, 0]) == 0
    assert int(s[2, 1]) == 0 and q[2, 32] == 0x80  # -0.0 keeps its sign


def test_quantiser_nonfinite_block(oracle_mod):
    x = np.ones((1, 64), np.float32)
    x[0, 5] = np.nan
    x[0, 40] = np.inf
    q, s = oracle_mod.quantize_tokenwise(x)
    assert s[0, 0] == 0xFF and s[0, 1] == 0xFF
    assert np.all(q == 0x7F)


# --------------------------------------------------------------- non-contracting grouped GEMM

def q_weights(rng, E, N, K):
    W = np.empty((E, N, K), np.uint8)
    sW = np.empty((E, N, K // 32), np.uint8)
    for g in range(E):
        W[g], sW[g] = q_operand(rng, N, K)
    return W, sW


def exact_grouped_gemm(X, sX, W, sW, offs, E, M, N, K):
    fa = {c: Fraction(float(torch_e4m3([c])[0])) for c in range(256) if (c & 0x7F) != 0x7F}
    out = np.zeros((M, N), dtype=np.uint16)
    lo = 0
    for g in range(E):
        hi = int(offs[g])
        for t in range(lo, hi):
            for n in range(N):
                acc = Fraction(0)
                for k in range(K):
                    x = fa[int(X[t, k])] * Fraction(2) ** (int(sX[t, k // 32]) - 127)
                    w = fa[int(W[g, n, k])] * Fraction(2) ** (int(sW[g, n, k // 32]) - 127)
                    acc += x * w
                out[t, n] = bf16_nearest_exact(acc)
        lo = hi
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_grouped_gemm_exact_bruteforce(oracle_mod, seed):
    """Exact rational sums rounded to bf16, on tiny ragged inputs whose group
    boundaries are arbitrary rows (not multiples of 32), with an empty group
    and padding rows past the last group."""
    rng = np.random.default_rng(300 + seed)
    E = int(rng.integers(2, 4))
    M = int(rng.integers(3, 9))
    N = int(rng.integers(1, 4))
    K = 32 * int(rng.integers(1, 3))
    X, sX = q_operand(rng, M, K)
    W, sW = q_weights(rng, E, N, K)
    cuts = np.sort(rng.integers(0, M + 1, size=E))
    cuts[0] = min(cuts[0], cuts[1])  # keep non-decreasing
    offs = cuts.astype(np.int32)
    got = oracle_mod.grouped_gemm(X, sX, W, sW, offs, E, M, N, K)
    ref = exact_grouped_gemm(X, sX, W, sW, offs, E, M, N, K)
    zero = lambda a: np.where((a & 0x7FFF) == 0, 0, a)  # noqa: E731
    assert np.array_equal(zero(got), zero(ref))
    assert np.all(got[int(offs[-1]):] == 0)


def test_grouped_gemm_is_ragged_dot_of_dequantised(oracle_mod):
    """The grouped GEMM is the generic non-contracting ragged dot (per-group
    numpy matmul) on operands dequantised through the library decode tables:
    lhs = X [M, K], rhs[g] = W[g]^T [K, N]."""
    rng = np.random.default_rng(31)
    E, M, N, K = 3, 50, 7, 96
    X, sX = q_operand(rng, M, K)
    W, sW = q_weights(rng, E, N, K)
    sizes = [17, 0, 29]  # 4 padding rows at the end
    offs = np.cumsum(sizes).astype(np.int32)
    _, acc, aacc = oracle_mod.grouped_gemm(X, sX, W, sW, offs, E, M, N, K, want_acc=True)

    def deq(q, s):
        return torch_e4m3(q.reshape(-1)).reshape(q.shape) * np.repeat(torch_e8m0(s.reshape(-1)).reshape(s.shape), 32, axis=-1)

    Xd = deq(X, sX)
    Wd = np.stack([deq(W[g], sW[g]) for g in range(E)])
    ref = rd.ragged_dot(Xd, np.transpose(Wd, (0, 2, 1)), sizes)
    assert np.allclose(acc, ref, rtol=1e-12, atol=0)
    ref_abs = rd.ragged_dot(np.abs(Xd), np.abs(np.transpose(Wd, (0, 2, 1))), sizes)
    assert np.allclose(aacc, ref_abs, rtol=1e-12, atol=0)


def test_grouped_gemm_single_group_is_dense(oracle_mod):
    rng = np.random.default_rng(32)
    M, N, K = 40, 9, 64
    X, sX = q_operand(rng, M, K)
    W, sW = q_weights(rng, 1, N, K)
    _, acc, _ = oracle_mod.grouped_gemm(X, sX, W, sW, np.array([M], np.int32), 1, M, N, K, want_acc=True)
    dense = oracle_mod.decode_operand(X, sX) @ oracle_mod.decode_operand(W[0], sW[0]).T
    assert np.allclose(acc, dense, rtol=1e-12, atol=0)


def test_grouped_gemm_points_and_rejects(oracle_mod):
    rng = np.random.default_rng(33)
    E, M, N, K = 3, 30, 5, 64
    X, sX = q_operand(rng, M, K)
    W, sW = q_weights(rng, E, N, K)
    offs = np.array([7, 7, 26], np.int32)
    full = oracle_mod.grouped_gemm(X, sX, W, sW, offs, E, M, N, K)
    t = rng.integers(0, M, 40); n = rng.integers(0, N, 40)
    pts = oracle_mod.grouped_gemm(X, sX, W, sW, offs, E, M, N, K, points=(t, n))
    assert np.array_equal(pts, full[t, n])
    with pytest.raises(ValueError):
        oracle_mod.grouped_gemm(X, sX, W, sW, np.array([7, 5, 26], np.int32), E, M, N, K)  # decreasing
    with pytest.raises(ValueError):
        oracle_mod.grouped_gemm(X, sX, W, sW, np.array([7, 9, 31], np.int32), E, M, N, K)  # past M

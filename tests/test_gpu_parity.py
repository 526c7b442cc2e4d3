"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.

Bars: bit-exact on exactly-representable cases and on the quantiser; within
|gpu - oracle| <= 1e-2 |oracle| + 1e-3 sqrt(sum |a b|) elsewhere;
bit-reproducible run to run; every output element written (NaN-poisoned
outputs); padding past the last group never read into the result; empty
experts exact +0.0."""
import numpy as np
import pytest
import torch

import oracle
import moe_ragged_contraction_gb300 as mx
from moe_ragged_contraction_gb300 import inputs as I

from _util import (quantised_operand, same_bits_signless_zero, tolerance_violations)

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


def run_gpu(A, sA, B, sB, offs, E, N, K, poison=True, workspace=None):
    out = torch.empty((E, N, K), dtype=torch.bfloat16, device="cuda")
    if poison:
        out.view(torch.int16).fill_(-1)  # 0xFFFF: bf16 NaN, so an unwritten element shows
    mx.wgrad_grouped(dev(A), dev(sA), dev(B), dev(sB), dev(np.asarray(offs, np.int32)), out=out,
                     workspace=workspace)
    torch.cuda.synchronize()
    return out.view(torch.int16).cpu().numpy().view(np.uint16)


def rand_operand(rng, R, M, scale_lo=118, scale_hi=136):
    q = rng.integers(0, 256, size=(R, M), dtype=np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x7E
    s = rng.integers(scale_lo, scale_hi, size=(R, M // 32), dtype=np.uint8)
    return q, s


def check_tol(got, A, sA, B, sB, offs, E, N, K, M):
    ref, acc, aacc = oracle.wgrad(A, sA, B, sB, offs, E, N, K, M, want_acc=True)
    bad = tolerance_violations(got, ref, aacc)
    assert not bad.any(), f"{bad.sum()} of {bad.size} elements out of tolerance; first at {np.argwhere(bad)[:5].tolist()}"
    lo = 0
    for g in range(E):
        if int(offs[g]) == lo:
            assert np.all(got[g] == 0x0000), f"empty expert {g} not exact +0"
        lo = int(offs[g])
    return ref


# ------------------------------------------------------------------ quantiser

@pytest.mark.parametrize("R,M,dist", [(128, 1024, "normal"), (37, 4096, "student_t3"), (1, 32, "normal")])
def test_quantiser_bit_exact(R, M, dist):
    x = I.host_operand(R, M, seed=77, stream=0, dist=dist)
    x[:, :32] *= np.float32(1e-30)  # tiny values: subnormal E4M3 codes
    if R > 2:
        x[1, 64:96] = 0.0
        x[2, 0:32] = np.float32(448.0 * 2.0 ** 5)
    q_ref, s_ref = oracle.quantize_tokenwise(x)
    q, s = mx.quantize_tokenwise(dev(x))
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)


def test_quantiser_nonfinite():
    x = np.ones((2, 64), np.float32)
    x[0, 3] = np.nan
    x[1, 40] = -np.inf
    q_ref, s_ref = oracle.quantize_tokenwise(x)
    q, s = mx.quantize_tokenwise(dev(x))
    assert np.array_equal(s.cpu().numpy(), s_ref) and np.array_equal(q.cpu().numpy(), q_ref)


# ------------------------------------------------------------------ exact cases

def int_operand(rng, R, M, vals, codes):
    v = rng.choice(vals, size=(R, M))
    return np.vectorize(codes.get)(v).astype(np.uint8)


def test_exact_tier1_integers_unit_scales():
    """Values in [-2, 2], unit scales, groups <= 1024 tokens: every partial sum
    is an integer below 2^12, so any fp32 accumulation order is exact."""
    rng = np.random.default_rng(1)
    codes = {-2: 0xC0, -1: 0xB8, 0: 0x00, 1: 0x38, 2: 0x40}
    E, N, K, M = 5, 256, 512, 2048
    A = int_operand(rng, N, M, list(codes), codes)
    B = int_operand(rng, K, M, list(codes), codes)
    sA = np.full((N, M // 32), 0x7F, np.uint8)
    sB = np.full((K, M // 32), 0x7F, np.uint8)
    offs = np.cumsum([0, 416, 1024, 96, 480]).astype(np.int32)  # one empty, 32-aligned, ragged
    got = run_gpu(A, sA, B, sB, offs, E, N, K)
    ref = oracle.wgrad(A, sA, B, sB, offs, E, N, K, M)
    assert same_bits_signless_zero(got, ref)
    assert np.all(got[0] == 0)


def test_exact_tier2_scaled_integers():
    """Integers in [-16, 16] (E4M3-exact) with per-block scales 2^[-2, 2]:
    products are multiples of 2^-4 and |sums| < 2^20, exact in fp32."""
    rng = np.random.default_rng(2)
    vals = list(range(-16, 17))
    t = torch.tensor(np.array(vals, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    codes = dict(zip(vals, t.tolist()))
    E, N, K, M = 3, 128, 256, 1024
    A = int_operand(rng, N, M, vals, codes)
    B = int_operand(rng, K, M, vals, codes)
    sA = rng.integers(125, 130, size=(N, M // 32), dtype=np.uint8)
    sB = rng.integers(125, 130, size=(K, M // 32), dtype=np.uint8)
    offs = np.array([320, 640, 1024], np.int32)
    got = run_gpu(A, sA, B, sB, offs, E, N, K)
    ref, acc, _ = oracle.wgrad(A, sA, B, sB, offs, E, N, K, M, want_acc=True)
    assert np.all(np.abs(acc) < 2.0 ** 20)
    assert same_bits_signless_zero(got, ref), f"{np.sum(got != ref)} elements differ"


# ------------------------------------------------------------------ tolerance parity

def test_tiny_workload_full():
    w = I.WORKLOADS["tiny"]
    A, sA = quantised_operand(w.N, w.M, w.seed, 0, w.dist)
    B, sB = quantised_operand(w.K, w.M, w.seed, 1, w.dist)
    offs = I.offsets(I.group_sizes("tiny"))
    got = run_gpu(A, sA, B, sB, offs, w.E, w.N, w.K)
    check_tol(got, A, sA, B, sB, offs, w.E, w.N, w.K, w.M)


@pytest.mark.parametrize("E,N,K,M,sizes", [
    (1, 128, 256, 128, [128]),                        # one tile, one K-step
    (1, 128, 256, 96, [96]),                          # single partial K-step
    (2, 128, 256, 256, [32, 224]),                    # 32-token group, boundary mid K-step
    (3, 320, 640, 1536, [608, 0, 928]),               # N, K not tile multiples
    (4, 1408, 1152, 2048, [800, 352, 0, 896]),        # 11 row tiles, K = 4.5 col tiles
    (1, 40, 8, 512, [512]),                           # tiny N and K
    (2, 256, 256, 4096, [4064, 32]),                  # long group, then a 32-token group
    (3, 128, 256, 1024, [0, 0, 0]),                   # all experts empty
    (64, 128, 256, 4096, None),                       # many experts, small groups
])
def test_edge_shapes(E, N, K, M, sizes):
    rng = np.random.default_rng(E * 1000 + N + K + M)
    A, sA = quantised_operand(N, M, seed=E * 1000 + N, stream=0)
    B, sB = quantised_operand(K, M, seed=E * 1000 + N, stream=1)
    if sizes is None:
        sizes = I.random_sizes(E, M, rng)
    offs = np.cumsum(sizes).astype(np.int32)
    got = run_gpu(A, sA, B, sB, offs, E, N, K)
    check_tol(got, A, sA, B, sB, offs, E, N, K, M)


def test_varied_scales_move_rows_and_columns():
    """Operands whose magnitude varies per row over 2^-6..2^6 before
    quantisation, so scales vary per (row, 32-token block) on both operands: a
    misplaced scale would shift whole rows or columns, far outside the
    tolerance."""
    rng = np.random.default_rng(31)
    E, N, K, M = 2, 256, 512, 1024
    xa = I.host_operand(N, M, seed=31, stream=0) * np.exp2(rng.integers(-6, 7, (N, 1))).astype(np.float32)
    xb = I.host_operand(K, M, seed=31, stream=1) * np.exp2(rng.integers(-6, 7, (K, 1))).astype(np.float32)
    A, sA = oracle.quantize_tokenwise(xa)
    B, sB = oracle.quantize_tokenwise(xb)
    assert len(np.unique(sA)) > 10 and len(np.unique(sB)) > 10
    offs = np.array([480, 1024], np.int32)
    got = run_gpu(A, sA, B, sB, offs, E, N, K)
    check_tol(got, A, sA, B, sB, offs, E, N, K, M)


def test_extreme_dynamic_range():
    """Uniformly random E4M3 codes (all magnitudes, subnormals included) with
    independent scales over 2^-9..2^8 per 32-token block: sums cancel by up to
    five orders of magnitude, so the bound is the one fp32 accumulation itself
    gives. The tensor core adds each k = 32 block product into the fp32
    accumulator; with L tokens that is at most L/32 + 32 roundings of a partial
    sum bounded by sum|ab|, each at most 2^-24 of it, plus the final bf16
    rounding (at most one bf16 ulp apart from the oracle's exact rounding):
        |gpu - oracle| <= 2^-7 |oracle| + (L/32 + 32) 2^-24 sum|ab|."""
    rng = np.random.default_rng(32)
    E, N, K, M = 4, 384, 768, 2048
    A, sA = rand_operand(rng, N, M)
    B, sB = rand_operand(rng, K, M)
    sizes = np.array([800, 352, 0, 896])
    offs = np.cumsum(sizes).astype(np.int32)
    got = run_gpu(A, sA, B, sB, offs, E, N, K)
    ref, acc, aacc = oracle.wgrad(A, sA, B, sB, offs, E, N, K, M, want_acc=True)
    L = sizes[:, None, None].astype(np.float64)
    bound = 2.0 ** -7 * np.abs(oracle.bf16_bits_to_f64(ref)) + (L / 32 + 32) * 2.0 ** -24 * aacc
    err = np.abs(oracle.bf16_bits_to_f64(got) - oracle.bf16_bits_to_f64(ref))
    assert np.all(err <= bound)
    assert np.all(got[2] == 0)


# ------------------------------------------------------------------ properties

def test_bit_reproducible_and_workspace_variant():
    rng = np.random.default_rng(41)
    E, N, K, M = 6, 384, 768, 3072
    A, sA = rand_operand(rng, N, M)
    B, sB = rand_operand(rng, K, M)
    offs = np.cumsum(I.random_sizes(E, M, rng)).astype(np.int32)
    runs = [run_gpu(A, sA, B, sB, offs, E, N, K) for _ in range(3)]
    assert all(np.array_equal(runs[0], r) for r in runs[1:])
    ws = torch.empty(mx.workspace_bytes(E, N, K, M), dtype=torch.uint8, device="cuda")
    assert np.array_equal(runs[0], run_gpu(A, sA, B, sB, offs, E, N, K, workspace=ws))


def test_padding_garbage_never_read():
    """NaN data and NaN scales past the last group give the same bits as the
    same call on operands cut down to their real token width."""
    E, N, K, M = 3, 256, 512, 2048
    A, sA = quantised_operand(N, M, seed=51, stream=0)
    B, sB = quantised_operand(K, M, seed=51, stream=1)
    offs = np.array([416, 416, 1376], np.int32)
    Mc = int(offs[-1])
    cut = run_gpu(A[:, :Mc].copy(), sA[:, :Mc // 32].copy(), B[:, :Mc].copy(), sB[:, :Mc // 32].copy(),
                  offs, E, N, K)
    A2, sA2, B2, sB2 = A.copy(), sA.copy(), B.copy(), sB.copy()
    A2[:, Mc:] = 0x7F; B2[:, Mc:] = 0xFF
    sA2[:, Mc // 32:] = 0xFF; sB2[:, Mc // 32:] = 0xFF
    got = run_gpu(A2, sA2, B2, sB2, offs, E, N, K)
    assert np.array_equal(got, cut)
    check_tol(got, A, sA, B, sB, offs, E, N, K, M)


def test_invalid_offsets_are_clamped_and_flagged():
    E, N, K, M = 4, 128, 256, 1024
    A, sA = quantised_operand(N, M, seed=61, stream=0)
    B, sB = quantised_operand(K, M, seed=61, stream=1)
    mx.device_status(clear=True)
    bad = np.array([300, 200, 5000, 1024], np.int32)  # unaligned, decreasing, beyond M
    got = run_gpu(A, sA, B, sB, bad, E, N, K)
    st = mx.device_status(clear=True)
    assert st & 1 and st & 2 and st & 4 and not st & 8
    clamped = np.array([288, 288, 1024, 1024], np.int32)
    check_tol(got, A, sA, B, sB, clamped, E, N, K, M)
    assert mx.device_status(clear=True) == 0


# ------------------------------------------------------------------ tilings

@pytest.fixture
def tiling_reset():
    yield
    mx.set_tile_orientation(0)
    mx.set_tile_rows(0)
    mx.set_epilogue_store(0)


# (orientation mode, forced tile rows): the model's choice per orientation,
# one-MMA tiles, two-MMA tiles (the second 16 columns wide, or 192), narrow
# tiles; the drain that holds a warp's row as bf16 pairs with five (272, 288,
# 320), six (352) and seven (416, 448) chunks, whole and partial last ones
TILINGS = [(1, 0), (2, 0), (1, 256), (2, 448), (1, 272), (2, 160), (1, 48), (1, 320), (1, 352), (1, 448),
           (2, 352), (1, 416), (2, 416), (2, 288)]
# epilogue stores: TMA stores through shared memory where their staging fits
# (tn = 48, 256, 320, 352 with its half-chunk stored directly, 448; both
# orientations), direct stores
STORES = (0, 1)


@pytest.mark.parametrize("E,N,K,M,sizes", [
    (4, 1408, 1152, 2048, [800, 352, 0, 896]),        # N, K not multiples of any tile
    (3, 320, 640, 1536, [608, 0, 928]),               # ragged on both sides
    (1, 40, 8, 512, [512]),                           # tiles far larger than the output
    (2, 136, 264, 1024, [544, 480]),                  # odd tile counts
    (2, 1408, 2048, 2048, [1120, 928]),               # the 16B expert shape
])
def test_tilings_bit_identical(E, N, K, M, sizes, tiling_reset):
    """Every tiling accumulates each output element from the same 32-token
    block products in the same order, so all of them must agree bit for bit,
    and match the oracle."""
    A, sA = quantised_operand(N, M, seed=E * 7 + N, stream=0)
    B, sB = quantised_operand(K, M, seed=E * 7 + N, stream=1)
    offs = np.cumsum(sizes).astype(np.int32)
    outs, names = [], []
    for mode, tn in TILINGS:
        mx.set_tile_orientation(mode)
        mx.set_tile_rows(tn)
        cfg = mx.tile_config(E, N, K, M)
        assert cfg["kn"] == mode - 1 and (tn == 0 or cfg["tn"] == tn)
        for store in STORES:
            mx.set_epilogue_store(store)
            outs.append(run_gpu(A, sA, B, sB, offs, E, N, K))
            names.append(f"mode={mode} tn={tn} store={store}")
    for name, o in zip(names[1:], outs[1:]):
        assert np.array_equal(outs[0], o), f"tiling {name} differs"
    check_tol(outs[0], A, sA, B, sB, offs, E, N, K, M)


def test_tilings_exact_integers(tiling_reset):
    """Integer-valued operands whose sums are exact in fp32: every tiling
    rounds the exact sum to bf16 and gives the oracle's bits exactly."""
    rng = np.random.default_rng(71)
    E, N, K, M = 3, 200, 344, 1536
    vals = np.array([0x38, 0x40, 0xB8, 0xC0, 0x00], np.uint8)  # +-1, +-2, 0 in E4M3
    A = vals[rng.integers(0, 5, (N, M))]
    B = vals[rng.integers(0, 5, (K, M))]
    sA = np.full((N, M // 32), 127, np.uint8)
    sB = np.full((K, M // 32), 127, np.uint8)
    offs = np.array([224, 224, 1536], np.int32)
    ref = oracle.wgrad(A, sA, B, sB, offs, E, N, K, M)
    for mode, tn in TILINGS:
        mx.set_tile_orientation(mode)
        mx.set_tile_rows(tn)
        for store in STORES:
            mx.set_epilogue_store(store)
            got = run_gpu(A, sA, B, sB, offs, E, N, K)
            assert same_bits_signless_zero(got, ref), f"tiling mode={mode} tn={tn} store={store}"


# ------------------------------------------------------------------ extremes of the plan

def test_max_expert_count():
    """E = 2048 (the largest supported): the plan, the scale gather and the
    schedule at their largest expert count, with empty and 32-token experts."""
    E, N, K = 2048, 64, 128
    rng = np.random.default_rng(91)
    sizes = 32 * rng.integers(0, 3, E)
    M = int(sizes.sum()) + 64  # 64 tokens of padding past the last group
    A, sA = quantised_operand(N, M, seed=91, stream=0)
    B, sB = quantised_operand(K, M, seed=91, stream=1)
    offs = np.cumsum(sizes).astype(np.int32)
    got = run_gpu(A, sA, B, sB, offs, E, N, K)
    check_tol(got, A, sA, B, sB, offs, E, N, K, M)


def test_unaligned_scale_planes():
    """Scale planes that start at odd byte addresses (views into larger
    buffers) give the same bits as aligned ones."""
    E, N, K, M = 3, 256, 384, 1536
    A, sA = quantised_operand(N, M, seed=93, stream=0)
    B, sB = quantised_operand(K, M, seed=93, stream=1)
    offs = np.array([416, 416, 1504], np.int32)
    ref = run_gpu(A, sA, B, sB, offs, E, N, K)

    def odd_view(a, shift):
        buf = torch.empty(a.size + 64, dtype=torch.uint8, device="cuda")
        v = buf[shift:shift + a.size].view(a.shape)
        v.copy_(torch.from_numpy(np.ascontiguousarray(a)))
        return v

    out = torch.empty((E, N, K), dtype=torch.bfloat16, device="cuda")
    out.view(torch.int16).fill_(-1)
    mx.wgrad_grouped(dev(A), odd_view(sA, 1), dev(B), odd_view(sB, 3), dev(offs), out=out)
    torch.cuda.synchronize()
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------ fused quantise + transpose

def _bf16_bits(x32):
    """fp32 -> bf16 bit patterns (round to nearest even), NaN kept NaN."""
    b = np.ascontiguousarray(x32, dtype=np.float32).view(np.uint32)
    r = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
    r[np.isnan(x32)] = 0x7FC0
    return r


@pytest.mark.parametrize("M,R", [(1024, 256), (96, 200), (64, 13), (2048, 1408)])
def test_quantize_transpose_bit_exact(M, R):
    """bf16 [M, R] token-major -> E4M3 [R, M] + E8M0 [R, M/32]: bit-identical
    to the oracle's quantiser applied to the transpose (bf16 values are exact
    in fp32). Covers a partial token tile (M % 64 == 32), partial feature tiles,
    rows not a multiple of 8 (scalar loads), tiny, zero and non-finite blocks."""
    rng = np.random.default_rng(M + R)
    x = (rng.standard_normal((M, R)) * np.exp2(rng.integers(-8, 9, (1, R)))).astype(np.float32)
    x[:32, 0] = 0.0
    x[32:64, min(1, R - 1)] *= np.float32(1e-38)
    if R > 3 and M >= 96:
        x[64:96, 2] = np.float32(448.0 * 2.0 ** 7)
        x[40, 3] = np.inf
    bits = _bf16_bits(x)
    x_exact = (bits.astype(np.uint32) << 16).view(np.float32)  # the values the bf16 bits hold
    q_ref, s_ref = oracle.quantize_tokenwise(np.ascontiguousarray(x_exact.T))
    xt = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    q, s = mx.quantize_transpose_bf16(xt)
    torch.cuda.synchronize()
    assert np.array_equal(s.cpu().numpy(), s_ref)
    assert np.array_equal(q.cpu().numpy(), q_ref)

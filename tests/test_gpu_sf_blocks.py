"""GPU tests of the scale-factor-block path: the fused quantiser that writes
the scales straight into the tensor core's block layout, and the weight
gradient that reads them (mxfp8_quantize_transpose_bf16_sf,
mxfp8_wgrad_grouped_sf), through the C ABI.

* The quantiser's E4M3 bytes and scale plane equal the oracle's quantiser on
  the transposed input, and its blocks hold exactly the oracle's scales at the
  positions the layout defines (zeros past the rows and tokens).
* The weight gradient over the blocks gives the same bits as the regular
  entry point over the planes (every output element sums the same 32-token
  block products in the same order), for runs that start inside a 128-token
  step, empty experts and token padding, both tile orientations and several
  tile widths; and it is within the parity tolerance of the oracle.
* At the 16B, 671B down and 671B up/gate shapes (full size, the library's own tiling) the
  two entry points agree bit for bit over the whole output."""
import numpy as np
import pytest
import torch

import oracle
import moe_ragged_contraction_gb300 as mx
from moe_ragged_contraction_gb300 import inputs as I

from _util import tolerance_violations

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx.build()
    mx.load()
    mx.device_status(clear=True)


def bf16_host(rows, cols, seed, stream, dist="normal"):
    """Seeded token-major operand [rows (tokens), cols] rounded to bf16 (host)."""
    x = I.host_operand(((rows + 15) // 16) * 16, cols, seed, stream, dist)[:rows]
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16)


def expected_blocks(plane, R, M, tile_rows):
    """The layout written out in numpy from a scale plane [R][M/32]."""
    T = tile_rows
    tiles = (R + T - 1) // T
    steps = (M + 127) // 128
    nblk = (T + 127) // 128
    buf = np.zeros((tiles, steps, nblk, 512), np.uint8)
    padded = np.zeros((tiles * T, steps * 4), np.uint8)
    padded[:R, :M // 32] = plane
    for t in range(tiles):
        for h in range(nblk):
            rows = np.arange(128)
            tr = 128 * h + rows
            ok = tr < T
            src = padded[t * T + tr[ok]]                      # [valid rows][steps*4]
            r = rows[ok]
            for g in range(steps):
                for kb in range(4):
                    buf[t, g, h, (r % 32) * 16 + (r // 32) * 4 + kb] = src[:, 4 * g + kb]
    return buf.reshape(-1)


@pytest.mark.parametrize("M,R,tile_rows", [(1056, 300, 256), (1024, 704, 352), (2048, 416, 416), (160, 37, 448),
                                           (4096, 128, 128)])
def test_quantizer_writes_blocks(M, R, tile_rows):
    x = bf16_host(M, R, seed=M + R, stream=5)
    ref_q, ref_s = oracle.quantize_tokenwise(np.ascontiguousarray(x.float().numpy().T))
    xd = x.cuda()
    s = torch.empty((R, M // 32), dtype=torch.uint8, device="cuda")
    nbytes = mx.sf_blocks_bytes(R, M, tile_rows)
    sf = torch.full((nbytes,), 0xAB, dtype=torch.uint8, device="cuda")  # every byte must be written
    q, sf, s = mx.quantize_transpose_bf16_sf(xd, tile_rows, sf=sf, s=s)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), ref_q)
    assert np.array_equal(s.cpu().numpy(), ref_s)
    assert np.array_equal(sf.cpu().numpy(), expected_blocks(ref_s, R, M, tile_rows))
    # without the plane: the same bytes and blocks
    q2, sf2, _ = mx.quantize_transpose_bf16_sf(xd, tile_rows)
    torch.cuda.synchronize()
    assert torch.equal(q2, q) and torch.equal(sf2, sf)


def operands_sf(dy, x, kn, tn):
    """A, B with both their planes and their blocks for tiling (kn, tn)."""
    rows_a, rows_b = (tn, 256) if kn else (256, tn)
    M, N = dy.shape
    K = x.shape[1]
    sA = torch.empty((N, M // 32), dtype=torch.uint8, device="cuda")
    sB = torch.empty((K, M // 32), dtype=torch.uint8, device="cuda")
    A, sfA, _ = mx.quantize_transpose_bf16_sf(dy, rows_a, s=sA)
    B, sfB, _ = mx.quantize_transpose_bf16_sf(x, rows_b, s=sB)
    return A, sA, sfA, B, sB, sfB


@pytest.mark.parametrize("E,N,K,M,sizes,kn,tn", [
    (4, 384, 768, 3072, [416, 0, 1056, 96], 0, 256),        # starts at 416, 1472: inside a 128-token step
    (4, 384, 768, 3072, [416, 0, 1056, 96], 1, 352),        # the other orientation, two MMAs per chunk
    (6, 256, 512, 4096, [32, 1024, 0, 2016, 96, 160], 0, 416),
    (3, 1408, 2048, 2048, [1504, 480, 64], 1, 352),         # the 16B expert shape
    (5, 200, 136, 1600, [64, 320, 0, 864, 288], 0, 128),   # ragged N and K, partial tiles
    (2, 128, 256, 1024, [0, 0], 0, 256),                    # every expert empty
])
def test_wgrad_sf_same_bits_as_regular(E, N, K, M, sizes, kn, tn):
    offs = np.cumsum(sizes).astype(np.int32)
    dy = bf16_host(M, N, seed=E + N, stream=6).cuda()
    x = bf16_host(M, K, seed=E + K, stream=7).cuda()
    A, sA, sfA, B, sB, sfB = operands_sf(dy, x, kn, tn)
    doffs = torch.from_numpy(offs).cuda()
    ref = torch.empty((E, N, K), dtype=torch.bfloat16, device="cuda")
    ref.view(torch.int16).fill_(-1)
    mx.wgrad_grouped(A, sA, B, sB, doffs, out=ref)
    got = torch.empty_like(ref)
    got.view(torch.int16).fill_(-1)
    mx.wgrad_grouped_sf(A, sfA, B, sfB, doffs, kn, tn, out=got)
    torch.cuda.synchronize()
    assert mx.device_status(clear=True) == 0
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), "not the regular entry point's bits"
    bits = got.view(torch.int16).cpu().numpy().view(np.uint16)
    o_ref, _, aacc = oracle.wgrad(A.cpu().numpy(), sA.cpu().numpy(), B.cpu().numpy(), sB.cpu().numpy(), offs,
                                  E, N, K, M, want_acc=True)
    assert not tolerance_violations(bits, o_ref, aacc).any()
    lo = 0
    for g in range(E):
        if int(offs[g]) == lo:
            assert not np.any(bits[g]), f"empty expert {g} not exact +0"
        lo = int(offs[g])


@pytest.mark.parametrize("name", ["16B", "671Bd", "671Bgu"])
def test_wgrad_sf_full_size(name):
    """Full-size operands generated on the GPU, quantised once with both the
    plane and the blocks for the library's own tiling: the two entry points
    agree bit for bit over the whole output, and no element is left unwritten."""
    w = I.WORKLOADS[name]
    cfg = mx.tile_config(w.E, w.N, w.K, w.M)
    kn, tn = cfg["kn"], cfg["tn"]
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed)
    dy = torch.randn(w.M, w.N, device="cuda", generator=g).to(torch.bfloat16)
    x = torch.randn(w.M, w.K, device="cuda", generator=g).to(torch.bfloat16)
    A, sA, sfA, B, sB, sfB = operands_sf(dy, x, kn, tn)
    del dy, x
    offs = torch.from_numpy(I.offsets(I.group_sizes(name))).cuda()
    ref = mx.wgrad_grouped(A, sA, B, sB, offs)
    got = torch.empty_like(ref)
    got.view(torch.int16).fill_(-1)
    mx.wgrad_grouped_sf(A, sfA, B, sfB, offs, kn, tn, out=got)
    torch.cuda.synchronize()
    assert mx.device_status(clear=True) == 0
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
    assert torch.isfinite(got.float()).all()

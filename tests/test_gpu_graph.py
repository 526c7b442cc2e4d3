"""The library's calls captured in CUDA graphs and replayed.

With a caller-provided workspace (mxfp8_wgrad_grouped_ws) a call allocates
nothing, so its two launches (the plan / scale re-layout kernel, then the main
kernel as its programmatic dependent, cooperative where the producers meet at
expert boundaries) can be recorded in a graph. The graph reads the operands,
scales and offs from the same device buffers on every replay, so new contents
and a new routing copied into them are picked up. Checked: every replay gives
the same bits as an eager call on the same inputs, the small case stays within
the parity tolerance of the oracle, and the device status word stays clear.
The entry points that keep scratch per stream (mxfp8_wgrad_grouped,
mxfp8_grouped_gemm) refuse to grow it while their stream is captured and are
captured after one eager call on that stream."""
import numpy as np
import pytest
import torch

import oracle
import moe_ragged_contraction_gb300 as mx

from _util import quantised_operand, tolerance_violations

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx.build()
    mx.load()
    mx.device_status(clear=True)


def random_operand(rows, M, gen):
    """E4M3 codes of magnitude at most 15 (no NaN bytes) with scales 2^-3 .. 2^3, generated on the GPU."""
    mag = torch.randint(0, 0x58, (rows, M), dtype=torch.uint8, device="cuda", generator=gen)
    sign = torch.randint(0, 2, (rows, M), dtype=torch.uint8, device="cuda", generator=gen) << 7
    s = torch.randint(124, 131, (rows, M // 32), dtype=torch.uint8, device="cuda", generator=gen)
    return mag | sign, s


def routing(E, M, gen):
    """Inclusive ends of E runs of 32-token multiples (some empty) covering at most M tokens."""
    w = torch.rand(E, generator=gen, device="cuda").cpu().numpy() + 0.05
    w[0] = 0.0                                   # one empty expert
    sizes = np.floor(w / w.sum() * (M // 32)).astype(np.int64) * 32
    return np.cumsum(sizes).astype(np.int32)


def eager(A, sA, B, sB, offs, ws, E, N, K):
    out = torch.empty((E, N, K), dtype=torch.bfloat16, device="cuda")
    mx.wgrad_grouped(A, sA, B, sB, offs, out=out, workspace=ws)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("E,N,K,M", [
    (5, 384, 768, 3072),        # small: one or two passes, no pass barrier
    (4, 7168, 2048, 65536),     # the 671B down expert shape: 128 tiles per expert, pass barrier on
])
def test_graph_replay_same_bits_as_eager(E, N, K, M):
    gen = torch.Generator(device="cuda")
    gen.manual_seed(E * 1000 + N)
    A, sA = random_operand(N, M, gen)
    B, sB = random_operand(K, M, gen)
    offs = torch.from_numpy(routing(E, M, gen)).cuda()
    ws = torch.empty(mx.workspace_bytes(E, N, K, M), dtype=torch.uint8, device="cuda")
    out = torch.empty((E, N, K), dtype=torch.bfloat16, device="cuda")

    mx.wgrad_grouped(A, sA, B, sB, offs, out=out, workspace=ws)  # attributes and module set up outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mx.wgrad_grouped(A, sA, B, sB, offs, out=out, workspace=ws)
    torch.cuda.synchronize()
    assert mx.device_status(clear=True) == 0

    for rep in range(3):
        if rep:
            # new operand contents and a new routing in the same buffers
            a2, s2 = random_operand(N, M, gen)
            A.copy_(a2)
            sA.copy_(s2)
            offs.copy_(torch.from_numpy(routing(E, M, gen)).cuda())
        out.view(torch.int16).fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        assert mx.device_status(clear=True) == 0
        ref = eager(A, sA, B, sB, offs, ws, E, N, K)
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"replay {rep} differs from the eager call"


def test_graph_replay_matches_oracle():
    E, N, K, M = 6, 256, 512, 2048
    sizes = [32, 0, 704, 480, 96, 736]
    A, sA = quantised_operand(N, M, seed=77, stream=0)
    B, sB = quantised_operand(K, M, seed=77, stream=1)
    offs = np.cumsum(sizes).astype(np.int32)
    d = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (A, sA, B, sB, offs)]
    ws = torch.empty(mx.workspace_bytes(E, N, K, M), dtype=torch.uint8, device="cuda")
    out = torch.empty((E, N, K), dtype=torch.bfloat16, device="cuda")
    mx.wgrad_grouped(*d, out=out, workspace=ws)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        mx.wgrad_grouped(*d, out=out, workspace=ws)
    out.view(torch.int16).fill_(-1)
    g.replay()
    torch.cuda.synchronize()
    assert mx.device_status(clear=True) == 0
    bits = out.view(torch.int16).cpu().numpy().view(np.uint16)
    ref, _, aacc = oracle.wgrad(A, sA, B, sB, offs, E, N, K, M, want_acc=True)
    assert not tolerance_violations(bits, ref, aacc).any()
    assert not bits[1].any(), "empty expert not exact +0"


def test_plain_entry_point_under_capture():
    """The plain entry point's scratch cache does not allocate while its stream
    is captured: a first call on a capturing stream fails with MXFP8_ENOWS and
    records nothing; after the same call has run once eagerly on that stream,
    capture reuses the cached scratch and replays give the eager bits."""
    E, N, K, M = 3, 256, 512, 2048
    sizes = [512, 0, 1504]
    A, sA = quantised_operand(N, M, seed=78, stream=0)
    B, sB = quantised_operand(K, M, seed=78, stream=1)
    offs = np.cumsum(sizes).astype(np.int32)
    d = [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in (A, sA, B, sB, offs)]
    out = torch.empty((E, N, K), dtype=torch.bfloat16, device="cuda")
    ref = mx.wgrad_grouped(*d)  # library state set up on the default stream
    torch.cuda.synchronize()

    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with pytest.raises(mx.Mxfp8Error, match="being captured"):
        with torch.cuda.graph(g, stream=s):
            mx.wgrad_grouped(*d, out=out)
    torch.cuda.synchronize()

    with torch.cuda.stream(s):
        mx.wgrad_grouped(*d, out=out)
    torch.cuda.synchronize()
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g2, stream=s):
        mx.wgrad_grouped(*d, out=out)
    out.view(torch.int16).fill_(-1)
    g2.replay()
    torch.cuda.synchronize()
    assert mx.device_status(clear=True) == 0
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_grouped_gemm_under_capture():
    """The grouped GEMM with ragged rows (the layer's forward product) captured
    after one eager call on the capturing stream: replays with new rows of X
    and a new routing in the captured buffers give the eager bits, and rows
    past the last group stay +0."""
    E, M, N, K = 4, 1000, 384, 512
    gen = torch.Generator(device="cuda")
    gen.manual_seed(4242)
    X, sX = random_operand(M, K, gen)
    W = torch.empty((E, N, K), dtype=torch.uint8, device="cuda")
    sW = torch.empty((E, N, K // 32), dtype=torch.uint8, device="cuda")
    for e in range(E):
        W[e], sW[e] = random_operand(N, K, gen)
    offs = torch.tensor([200, 200, 650, 960], dtype=torch.int32, device="cuda")  # an empty group, 40 padding rows
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        mx.grouped_gemm(X, sX, W, sW, offs, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        mx.grouped_gemm(X, sX, W, sW, offs, out=out)
    for rep in range(2):
        if rep:
            x2, s2 = random_operand(M, K, gen)
            X.copy_(x2)
            sX.copy_(s2)
            offs.copy_(torch.tensor([96, 480, 480, 992], dtype=torch.int32, device="cuda"))
        out.view(torch.int16).fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        assert mx.device_status(clear=True) == 0
        ref = mx.grouped_gemm(X, sX, W, sW, offs)
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), f"replay {rep} differs from the eager call"
        last = int(offs[-1])
        assert not out[last:].view(torch.int16).any(), "padding rows not +0"

"""The plan the prep kernel builds for the main kernel's static schedule, read
back from the workspace of mxfp8_wgrad_grouped_ws: per expert its clamped
start, length, K-steps on the global 128-token grid and first grid step, and
the experts in longest-first order (equal lengths in expert order), against a
host restatement of those rules on the 16B routings and random ones."""
import numpy as np
import pytest
import torch

import moe_ragged_contraction_gb300 as mx
from moe_ragged_contraction_gb300 import inputs as I

pytestmark = pytest.mark.gpu

PLAN_HDR = 8


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx.build()
    mx.load()
    mx.device_status(clear=True)


def grid_steps(offs):
    starts = np.concatenate([[0], offs[:-1]]).astype(np.int64)
    lens = offs.astype(np.int64) - starts
    return np.where(lens > 0, (starts + lens + 127) // 128 - starts // 128, 0), lens


def routings():
    yield "16B", I.offsets(I.group_sizes("16B")), 1408, 2048, 32768
    yield "16Bp", I.offsets(I.group_sizes("16Bp")), 1408, 2048, 196608
    rng = np.random.default_rng(11)
    for j in range(4):
        E = int(rng.integers(3, 13))
        M = 32 * int(rng.integers(256, 1025))
        sizes = np.floor(rng.dirichlet(np.ones(E) * 0.7) * (M // 32)).astype(np.int64) * 32
        yield f"random{j}", np.cumsum(sizes).astype(np.int32), 1408, 2048, M


@pytest.mark.parametrize("case", list(routings()), ids=lambda c: c[0])
def test_plan_entries_and_order(case):
    name, offs, N, K, M = case
    E = len(offs)
    # the plan does not depend on the operands: random E4M3 codes (no NaN bytes) and scales
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    A = torch.randint(0, 0x7F, (N, M), dtype=torch.uint8, device="cuda", generator=g)
    B = torch.randint(0, 0x7F, (K, M), dtype=torch.uint8, device="cuda", generator=g)
    sA = torch.full((N, M // 32), 127, dtype=torch.uint8, device="cuda")
    sB = torch.full((K, M // 32), 127, dtype=torch.uint8, device="cuda")
    ws = torch.zeros(mx.workspace_bytes(E, N, K, M), dtype=torch.uint8, device="cuda")
    mx.wgrad_grouped(A, sA, B, sB, torch.from_numpy(offs).cuda(), workspace=ws)
    torch.cuda.synchronize()
    assert mx.device_status(clear=True) == 0
    plan = ws[: 4 * (PLAN_HDR + 5 * E)].cpu().numpy().view(np.int32)
    assert plan[0] == (M + 127) // 128 and plan[1] == E
    ex = plan[PLAN_HDR: PLAN_HDR + 4 * E].reshape(E, 4)
    starts = np.concatenate([[0], offs[:-1]]).astype(np.int64)
    steps, lens = grid_steps(offs)
    assert np.array_equal(ex[:, 0], starts) and np.array_equal(ex[:, 1], lens)
    assert np.array_equal(ex[:, 2], steps) and np.array_equal(ex[:, 3], starts // 128)
    order = plan[PLAN_HDR + 4 * E: PLAN_HDR + 5 * E].tolist()
    assert order == sorted(range(E), key=lambda e: (-lens[e], e)), f"{name}: order {order}"

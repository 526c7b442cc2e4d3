"""Full-size parity on every named workload, in the launch configuration the
benchmark times (the plain C-ABI call): sampled output elements against the
oracle (8 full rows, 8 full columns, the four corner tiles of the
library's tiling and 4,096 random elements of every expert), the
whole output checked for unwritten / non-finite elements, bit-reproducibility
over two runs, and exact zeros for empty experts."""
import numpy as np
import pytest
import torch

import oracle
import moe_ragged_contraction_gb300 as mx
from moe_ragged_contraction_gb300 import inputs as I

from _util import sample_indices, tolerance_violations, workload_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    mx.build()
    mx.load()


@pytest.mark.parametrize("name", ["tiny", "16B", "16Bp", "671Bgu", "671Bd", "manyE160", "manyE512"])
def test_workload_parity(name):
    w = I.WORKLOADS[name]
    A, sA, B, sB, offs = workload_inputs(name)
    dA, dsA, dB, dsB = (torch.from_numpy(a).cuda() for a in (A, sA, B, sB))
    doffs = torch.from_numpy(offs).cuda()
    mx.device_status(clear=True)
    out = torch.empty((w.E, w.N, w.K), dtype=torch.bfloat16, device="cuda")
    out.view(torch.int16).fill_(-1)
    mx.wgrad_grouped(dA, dsA, dB, dsB, doffs, out=out)
    out2 = torch.empty_like(out)
    out2.view(torch.int16).fill_(-1)
    mx.wgrad_grouped(dA, dsA, dB, dsB, doffs, out=out2)
    torch.cuda.synchronize()
    assert mx.device_status(clear=True) == 0
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16)), "not bit-reproducible"
    assert torch.isfinite(out.float()).all(), "unwritten (NaN-poisoned) or non-finite elements"
    sizes = I.group_sizes(name)
    for g in np.nonzero(sizes == 0)[0]:
        assert not out[g].view(torch.int16).any(), f"empty expert {g} not exact +0"

    rng = np.random.default_rng(w.seed)
    g, n, k = sample_indices(w.E, w.N, w.K, rng, tiling=mx.tile_config(w.E, w.N, w.K, w.M))
    keep = sizes[g] > 0
    g, n, k = g[keep], n[keep], k[keep]
    ref, _, aacc = oracle.wgrad_points(A, sA, B, sB, offs, w.E, w.N, w.K, w.M, g, n, k, want_acc=True)
    got = out.view(torch.int16)[torch.from_numpy(g).long().cuda(), torch.from_numpy(n).long().cuda(),
                                 torch.from_numpy(k).long().cuda()].cpu().numpy().view(np.uint16)
    bad = tolerance_violations(got, ref, aacc)
    assert not bad.any(), f"{bad.sum()} of {bad.size} sampled elements out of tolerance"

"""Failure detection without a GPU fault: a host-side test hook makes the
first pipeline stage declare more bytes than it receives, so that stage's
bounded wait runs out. The kernel must stop its pipeline, raise
MXFP8_DEV_WAIT_TIMEOUT in the device status word and return; the context must
stay usable (a following normal call is correct and leaves the status clear).
Runs in a child process with a 50 ms wait limit."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import ctypes, sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1]); sys.path.insert(0, sys.argv[1] + "/tests")
import oracle
import moe_ragged_contraction_gb300 as mx
from _util import quantised_operand, tolerance_violations
lib = mx.load()
lib.mxfp8_test_stall_next_call.argtypes = [ctypes.c_int]
E, N, K, M = 3, 256, 512, 1024
A, sA = quantised_operand(N, M, seed=7, stream=0)
B, sB = quantised_operand(K, M, seed=7, stream=1)
offs = np.array([320, 640, 1024], np.int32)
d = [torch.from_numpy(a).cuda() for a in (A, sA, B, sB, offs)]
mx.device_status(clear=True)
out = torch.empty((E, N, K), dtype=torch.bfloat16, device="cuda")
lib.mxfp8_test_stall_next_call(1)
mx.wgrad_grouped(*d, out=out)
torch.cuda.synchronize()
st = mx.device_status(clear=True)
assert st & 8, f"expected the wait-timeout bit, status={st}"
out.view(torch.int16).fill_(-1)
mx.wgrad_grouped(*d, out=out)
torch.cuda.synchronize()
assert mx.device_status(clear=True) == 0
ref, _, aacc = oracle.wgrad(A, sA, B, sB, offs, E, N, K, M, want_acc=True)
got = out.view(torch.int16).cpu().numpy().view(np.uint16)
assert not tolerance_violations(got, ref, aacc).any()
print("OK")
'''


def test_wait_timeout_reported_and_context_survives():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, MXFP8_WAIT_LIMIT_MS="50")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and "OK" in r.stdout, r.stdout + r.stderr

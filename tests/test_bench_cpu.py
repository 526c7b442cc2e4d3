"""The benchmark's CPU-side pieces: the reference arm (the oracle timed on a
bounded sample) prints the contract's line with the same `config` object as
the GPU arm, and the pooled rows it draws from are exactly the corresponding
rows of the seeded operands."""
import json
import os
import subprocess
import sys

import numpy as np

import bench
import oracle
from moe_ragged_contraction_gb300 import inputs as I

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--config", "tiny",
                        "--steps", "3", "--warmup", "3", "--ref-step-seconds", "0.5"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["steps"] == 3 and line["warmup"] == 3
    assert line["config"] == bench.bench_config("tiny", 1)
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["value"] > 0
    assert line["spread"]["timed_steps"]["n"] == 3


def test_host_pool_rows_are_operand_rows():
    w = I.WORKLOADS["tiny"]
    Ap, sAp, Bp, sBp, offs = bench._host_pool("tiny")
    rn, rk = bench.pool_rows(w)
    A, sA = oracle.quantize_tokenwise(I.host_operand(w.N, w.M, w.seed, 0, w.dist))
    B, sB = oracle.quantize_tokenwise(I.host_operand(w.K, w.M, w.seed, 1, w.dist))
    assert np.array_equal(Ap, A[rn]) and np.array_equal(sAp, sA[rn])
    assert np.array_equal(Bp, B[rk]) and np.array_equal(sBp, sB[rk])
    assert np.array_equal(offs, I.offsets(I.group_sizes("tiny")))


def test_default_workload_is_the_largest():
    big = max(I.WORKLOADS.values(), key=lambda w: (w.flop, (w.N + w.K) * w.M))
    assert bench.DEFAULT_CONFIG == big.name

"""Seeded input recipes: routing properties the workloads promise (32-aligned
sizes summing to M, skew, empty experts, non-128-aligned boundaries) and
determinism of the operand generators."""
import numpy as np
import pytest

from moe_ragged_contraction_gb300 import inputs as I


@pytest.mark.parametrize("name", list(I.WORKLOADS))
def test_routing_basic(name):
    w = I.WORKLOADS[name]
    s = I.group_sizes(name)
    assert s.shape == (w.E,) and int(s.sum()) == w.M
    assert np.all(s % 32 == 0) and np.all(s >= 0)
    offs = I.offsets(s)
    assert offs.dtype == np.int32 and offs[-1] == w.M and np.all(np.diff(offs) >= 0)
    assert np.array_equal(I.group_sizes(name), s)  # deterministic


def test_routing_specifics():
    assert I.group_sizes("tiny").tolist() == [0, 352, 320, 352]
    s16 = I.group_sizes("16B")
    assert sorted(s16.tolist()) == [2080, 2656, 3232, 3808, 4384, 4960, 5536, 6112]
    for name in ("16B", "16Bp"):
        s = I.group_sizes(name)
        w = I.WORKLOADS[name]
        assert np.all(s % 128 != 0)  # 32-aligned, never 128-aligned
        assert 1.2 <= s.max() / (w.M / w.E) <= 1.7
    gu = I.group_sizes("671Bgu")
    assert (gu == 0).sum() == 2 and abs(gu.max() / (262144 / 32) - 1.7) < 0.01
    d = I.group_sizes("671Bd")
    assert (d == 0).sum() == 1 and 1.2 <= d.max() / (524288 / 32) <= 1.7
    assert ((d // 32) % 2 == 1).sum() >= 8  # odd multiples of 32


def test_balanced_sizes():
    s = I.balanced_sizes(3, 32 * 10)
    assert s.tolist() == [128, 96, 96]


def test_host_operand_deterministic_any_threads():
    a = I.host_operand(40, 256, seed=5, stream=0, nthreads=1)
    b = I.host_operand(40, 256, seed=5, stream=0, nthreads=4)
    assert np.array_equal(a, b)
    c = I.host_operand(24, 256, seed=5, stream=0, row0=16, nthreads=3)
    assert np.array_equal(a[16:40], c)
    d = I.host_operand(40, 256, seed=5, stream=1)
    assert not np.array_equal(a, d)
    assert abs(a.mean()) < 0.05 and abs(a.std() - 1) < 0.05


def test_host_operand_student_t():
    t = I.host_operand(64, 4096, seed=3, stream=0, dist="student_t3")
    assert np.isfinite(t).all()
    # Student-t(3): variance 3, heavy tails
    assert 2.0 < t.var() < 5.0 and np.abs(t).max() > 10

"""The bench's algorithmic byte counts, the numerators of its GB/s figures.

Each closed form is checked two ways: against a per-rank enumeration of
what every emulated rank reads and writes in each phase (stage, fold,
publish, gather), and against the multiples of S the scope table prints for
eight ranks (LL8: eps = 2; LL128: eps = 128 / 120).  S is bytes per rank;
for the all-gather it is the gathered output per rank."""
from __future__ import annotations

import pytest

import bench

MIB = 2**20


def _enumerate(kind: str, n: int, s: float, eps: float) -> float:
    """Walk the ranks phase by phase and add up every read and write."""
    part = s / n  # one rank's partition of a scattered buffer
    total = 0.0
    for r in range(n):
        if kind == "allgather":
            # rank r stages its contribution s / n as lines
            total += part + part * eps
        else:
            # rank r stages its whole input as lines
            total += s + s * eps
    for r in range(n):
        if kind == "oneshot":
            # every rank reads all N images in full and writes its output
            total += n * s * eps + s
        elif kind == "twoshot":
            # owner r reads partition r of every image, publishes it as lines,
            # then every rank reads every published partition and writes S
            total += n * part * eps + part * eps
        elif kind == "reducescatter":
            # owner r reads partition r of every image and writes it out
            total += n * part * eps + part
        elif kind == "allgather":
            # every rank reads every source's lines and writes S
            total += n * part * eps + s
    if kind == "twoshot":
        for r in range(n):
            total += n * part * eps + s
    return total


@pytest.mark.parametrize("n", [1, 2, 4, 8])
@pytest.mark.parametrize("eps", [bench.EPS_LL8, bench.EPS_LL128, 1.0])
def test_closed_forms_match_a_per_rank_enumeration(n, eps):
    s = 3 * MIB
    assert bench.bytes_allreduce_oneshot(n, s, eps) == pytest.approx(
        _enumerate("oneshot", n, s, eps), rel=1e-12)
    assert bench.bytes_allreduce_twoshot(n, s, eps) == pytest.approx(
        _enumerate("twoshot", n, s, eps), rel=1e-12)
    assert bench.bytes_reduce_scatter(n, s, eps) == pytest.approx(
        _enumerate("reducescatter", n, s, eps), rel=1e-12)
    assert bench.bytes_all_gather(n, s, eps) == pytest.approx(
        _enumerate("allgather", n, s, eps), rel=1e-12)


def test_multiples_of_s_printed_for_eight_ranks():
    s = 1.0
    assert bench.bytes_allreduce_oneshot(8, s, bench.EPS_LL8) == pytest.approx(160.0)
    assert bench.bytes_allreduce_twoshot(8, s, bench.EPS_LL128) == pytest.approx(42.67, abs=5e-3)
    assert bench.bytes_reduce_scatter(8, s, bench.EPS_LL128) == pytest.approx(26.07, abs=5e-3)
    assert bench.bytes_all_gather(8, s, bench.EPS_LL128) == pytest.approx(18.6, abs=5e-3)


def test_bench_workload_bytes():
    s = 256 * MIB
    # 11.45 GB of issue-level bytes per 8 x 256 MiB all-reduce, 4.29 GB floor
    assert bench.bytes_allreduce_twoshot(8, s, bench.EPS_LL128) == pytest.approx(11.45e9, rel=1e-3)
    assert bench.unique_bytes_allreduce(8, s) == 2 * 8 * s == 4294967296
    assert bench.bytes_reduce_scatter(8, s, bench.EPS_LL128) == pytest.approx(7.00e9, rel=1e-3)
    assert bench.bytes_all_gather(8, s, bench.EPS_LL128) == pytest.approx(4.99e9, rel=1e-3)


@pytest.mark.parametrize("eps", [bench.EPS_LL128, 1.0])
def test_three_launches_add_up_and_floors_stay_below(eps):
    n, s = 8, 256 * MIB
    k = bench.kernel_bytes_allreduce_twoshot(n, s, eps)
    f = bench.kernel_floor_bytes_allreduce_twoshot(n, s, eps)
    assert sum(k) == pytest.approx(bench.bytes_allreduce_twoshot(n, s, eps), rel=1e-12)
    assert all(fi <= ki for fi, ki in zip(f, k))
    # the gather's N readers of a published line share one DRAM read
    assert k[2] - f[2] == pytest.approx((n - 1) * s * eps, rel=1e-12)
    # one launch: the floor is below every stream-ordered launch's sum
    assert bench.unique_bytes_allreduce(n, s) < sum(f)

"""Sentinel readiness (flash-comm §3.1) on the GPU against the oracle, bit for
bit: every collective, both launch paths, every re-arm mode, consecutive
epochs and graph replay, withheld packs published late while consumers poll,
and inputs that contain the reserved pattern 0xFFFF (delivered by copies as
the canonical quiet NaN, folded like any other NaN)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import buffers, empty_dev, from_dev, read_lines, to_dev

pytestmark = pytest.mark.gpu

SENT = 2
ALL_ONES = np.uint64(0xFFFFFFFFFFFFFFFF)


@pytest.fixture(scope="module")
def cd():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import collective_datapath_gb300 as m

    return m


def plant_reserved(xs, seed, frac=0.01):
    """Overwrite a seeded 1 % of every input with the reserved pattern."""
    g = np.random.Generator(np.random.Philox(seed))
    out = []
    for x in xs:
        y = x.copy()
        if y.size:
            y[g.integers(0, y.size, max(1, int(frac * y.size)))] = 0xFFFF
        out.append(y)
    return out


def expected(name, xs, count=None, v=None):
    san = [oracle.sent_sanitize(x) for x in xs]
    if name == "ALLREDUCE":
        return oracle.allreduce(xs)
    if name == "REDUCE_SCATTER":
        return oracle.reduce_scatter(xs)
    if name == "ALLGATHER":
        return oracle.all_gather(san, count)
    if name == "ALLTOALL":
        return oracle.all_to_all(san)
    if name == "REDUCE_SCATTER_V":
        return oracle.reduce_scatter_v(xs, v)
    if name == "ALLGATHER_V":
        return oracle.all_gather_v(san, v)
    return oracle.all_to_all_v(san, v)


def check(cd, coll, outs, want, n):
    code, rank, line = coll.status()
    assert code == cd.COLL_OK, f"device status {code} rank {rank} line {line}"
    for r in range(n):
        got = from_dev(outs[r])[:want[r].size]
        if not np.array_equal(got, want[r]):
            bad = np.flatnonzero(got != want[r])
            raise AssertionError(f"rank {r}: {bad.size} mismatches, first at {bad[0]}: "
                                 f"got {got[bad[0]]:#06x} want {want[r][bad[0]]:#06x}")


def run_with(cd, coll, xs, ins, outs):
    for r in range(len(xs)):
        ins[r].copy_(to_dev(xs[r]))
    coll.run(ins, outs)


@pytest.mark.parametrize("algo", [1, 2])
@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("T", [1, 8, 32, 128])
def test_decode_allreduce_sentinel(cd, T, path, algo):
    n, count = 8, T * 4096
    coll = cd.Collective(cd.ALLREDUCE, n, count, encoding=SENT, algorithm=algo, path=path)
    xs, ins, outs = buffers(coll, n, seed=20, tag=T)
    for e in range(2):                                   # both slots
        xs = plant_reserved([synth.normal_bf16(20 + e, count, T, r) for r in range(n)], T + e)
        run_with(cd, coll, xs, ins, outs)
        check(cd, coll, outs, oracle.allreduce(xs), n)


CASES = [
    ("ALLREDUCE", 3, 1000), ("ALLREDUCE", 8, 24), ("ALLREDUCE", 1, 4096),
    ("REDUCE_SCATTER", 8, 8 * 3000), ("REDUCE_SCATTER", 5, 5 * 56 + 16),
    ("ALLGATHER", 8, 8 * 2048), ("ALLGATHER", 4, 4 * 104 + 8),
    ("ALLTOALL", 8, 8 * 960), ("ALLTOALL", 4, 256),
]


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("name,n,count", CASES)
def test_layout_collectives_sentinel(cd, name, n, count, path):
    triple = getattr(cd, name)
    for algo in ((1, 2) if name == "ALLREDUCE" else (0,)):
        coll = cd.Collective(triple, n, count, encoding=SENT, path=path, algorithm=algo)
        xs, ins, outs = buffers(coll, n, seed=21, dist="bits", tag=count)
        xs = plant_reserved(xs, count)
        for _ in range(2):
            run_with(cd, coll, xs, ins, outs)
            check(cd, coll, outs, expected(name, xs, count), n)


@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("name", ["REDUCE_SCATTER_V", "ALLGATHER_V", "ALLTOALL_V"])
def test_v_collectives_sentinel(cd, name, path):
    n = 8
    base = [b // 2 for b in synth.zipf_split(1 << 20, n)]
    v = [synth.rotate_right(base, p + 1) for p in range(n)] if name == "ALLTOALL_V" else base
    count = 0 if name == "ALLTOALL_V" else sum(base)
    coll = cd.Collective(getattr(cd, name), n, count, encoding=SENT, path=path, vcounts=v)
    xs, ins, outs = buffers(coll, n, seed=22, dist="bits", tag=len(name))
    xs = plant_reserved(xs, 5)
    for _ in range(2):
        run_with(cd, coll, xs, ins, outs)
        check(cd, coll, outs, expected(name, xs, v=v), n)


def test_staged_packs_match_the_oracle_encoding(cd):
    """coll_stage writes exactly the oracle's packs (sanitised inputs) into
    slot 1; the unused slot 0 still holds the pattern everywhere."""
    import torch

    n, count = 4, 4 * 1000
    coll = cd.Collective(cd.ALLREDUCE, n, count, encoding=SENT, path=cd.COLL_PATH_STREAMED)
    xs, ins, outs = buffers(coll, n, seed=23, dist="bits")
    xs = plant_reserved(xs, 23, frac=0.05)
    for r in range(n):
        ins[r].copy_(to_dev(xs[r]))
        coll.stage(r, ins[r])
    torch.cuda.synchronize()
    for r in range(n):
        for k in range(n):
            raw, lines, lb = read_lines(coll, 0, 1, r, k)
            assert lb == 8
            b, ln = oracle.shard_begin(count, n, k), oracle.shard_len(count, n, k)
            assert np.array_equal(raw.view(np.uint64), oracle.sent_encode(xs[r][b:b + ln]))
            other, _, _ = read_lines(coll, 0, 0, r, k)
            assert np.all(other.view(np.uint64) == ALL_ONES)
    coll.run(None, outs)
    check(cd, coll, outs, oracle.allreduce(xs), n)


@pytest.mark.parametrize("algo", [1, 2])
@pytest.mark.parametrize("reset", [0, 1, 3])
@pytest.mark.parametrize("path", [1, 2])
def test_packs_rearmed_after_run(cd, algo, reset, path):
    """After the consumers are done, every pack of the consumed slot holds the
    pattern again: right after the run for the last-reader (0) and kernel (1)
    modes, after the next run for the deferred mode (3)."""
    n, count = 8, 8 * 512
    coll = cd.Collective(cd.ALLREDUCE, n, count, encoding=SENT, algorithm=algo,
                         reset_mode=reset, path=path)
    xs, ins, outs = buffers(coll, n, seed=24)
    coll.run(ins, outs)                                  # epoch 1 -> slot 1
    check(cd, coll, outs, oracle.allreduce(xs), n)
    if reset == 3:
        raw, _, _ = read_lines(coll, 0, 1, 0, 0)         # not yet re-armed
        assert not np.any(raw.view(np.uint64) == ALL_ONES)
        coll.run(ins, outs)                              # epoch 2 -> slot 0, re-arms slot 1
        check(cd, coll, outs, oracle.allreduce(xs), n)
    for region in ((0, 1) if algo == 2 else (0,)):
        for r in range(n):
            for k in range(n if region == 0 else 1):
                raw, _, _ = read_lines(coll, region, 1, r, k)
                assert np.all(raw.view(np.uint64) == ALL_ONES), f"region {region} {r} {k}"


@pytest.mark.parametrize("reset", [0, 1, 3])
@pytest.mark.parametrize("path", [1, 2])
def test_consecutive_epochs_sentinel(cd, reset, path):
    n, count = 8, 8 * 2000
    for algo in (1, 2):
        coll = cd.Collective(cd.ALLREDUCE, n, count, encoding=SENT, path=path, algorithm=algo,
                             reset_mode=reset)
        _, ins, outs = buffers(coll, n, seed=25)
        for e in range(1, 7):
            xs = [synth.normal_bf16(250 + e, count, r) for r in range(n)]
            run_with(cd, coll, xs, ins, outs)
            check(cd, coll, outs, oracle.allreduce(xs), n)
            assert coll.epoch() == e + 1


def test_graph_replay_sentinel(cd):
    import torch

    n, count = 8, 8 * 512
    coll = cd.Collective(cd.ALLREDUCE, n, count, encoding=SENT, path=cd.COLL_PATH_FUSED)
    _, ins, outs = buffers(coll, n, seed=26)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        coll.run(ins, outs, stream=s)
    for rep in range(4):
        xs = [synth.normal_bf16(260 + rep, count, r) for r in range(n)]
        for r in range(n):
            ins[r].copy_(to_dev(xs[r]))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        check(cd, coll, outs, oracle.allreduce(xs), n)
    assert coll.epoch() == 5


def test_unpublished_pack_times_out_with_status(cd):
    import torch

    n, count = 4, 4 * 480
    coll = cd.Collective(cd.ALLREDUCE, n, count, encoding=SENT, path=cd.COLL_PATH_STREAMED,
                         algorithm=cd.COLL_ONESHOT, timeout_ns=2_000_000)
    xs, ins, outs = buffers(coll, n, seed=27)
    lines = torch.tensor([5], dtype=torch.int64, device="cuda")
    kind = torch.tensor([0], dtype=torch.int32, device="cuda")
    poison = torch.tensor([0], dtype=torch.int16, device="cuda")
    for r in range(n):
        if r == 1:
            cd.coll_stage_withheld(coll.spec, r, ins[r], lines, kind, poison)
        else:
            coll.stage(r, ins[r])
    coll.run(None, outs)
    code, rank, line = coll.status()
    assert code == cd.COLL_ERR_TIMEOUT and rank == 1 and line >= 0
    coll.run(ins, outs)                                  # the next epoch works
    check(cd, coll, outs, oracle.allreduce(xs), n)


def test_unpublished_pack_in_a_copy_phase_times_out_with_status(cd):
    """A stream-ordered all-gather copies packs through the pipelined
    sentinel copy: a pack that rank 1 never publishes ends the wait at the
    bound with COLL_ERR_TIMEOUT naming rank 1, and the next epoch works."""
    import torch

    n, count = 4, 4 * 480
    coll = cd.Collective(cd.ALLGATHER, n, count, encoding=SENT, path=cd.COLL_PATH_STREAMED,
                         timeout_ns=2_000_000)
    xs, ins, outs = buffers(coll, n, seed=29)
    lines = torch.tensor([5], dtype=torch.int64, device="cuda")
    kind = torch.tensor([0], dtype=torch.int32, device="cuda")
    poison = torch.tensor([0], dtype=torch.int16, device="cuda")
    for r in range(n):
        if r == 1:
            cd.coll_stage_withheld(coll.spec, r, ins[r], lines, kind, poison)
        else:
            coll.stage(r, ins[r])
    coll.run(None, outs)
    code, rank, line = coll.status()
    assert code == cd.COLL_ERR_TIMEOUT and rank == 1 and line >= 0
    coll.run(ins, outs)                                  # the next epoch works
    check(cd, coll, outs, oracle.all_gather(xs, count), n)


def real_lines(cd, coll, n_seg):
    base, _, lb = cd.coll_staging_layout(coll.spec, 0, 0, 0, 0)
    out = []
    for k in range(n_seg):
        off, lines, _ = cd.coll_staging_layout(coll.spec, 0, 0, 0, k)
        l0 = (off - base) // lb
        out.append(np.arange(l0, l0 + lines, dtype=np.int64))
    return np.concatenate(out)


@pytest.mark.parametrize("algo,epochs", [(1, 64), (2, 64)])
def test_late_packs_rejected_until_published(cd, algo, epochs):
    """8 ranks x [16 x 7168] normal(0,1): each epoch a seeded 10 % of every
    rank's packs still hold the pattern when the consumers start and are
    published late, in a seeded order, by producer CTAs of the same launch.
    Consumers wait for exactly those packs; the result is the oracle's."""
    import torch

    n, count = 8, 16 * 7168
    coll = cd.Collective(cd.ALLREDUCE, n, count, encoding=SENT, algorithm=algo,
                         path=cd.COLL_PATH_FUSED, timeout_ns=500_000_000)
    real = real_lines(cd, coll, n)
    assert real.size == count // 4
    ins = [empty_dev(count) for _ in range(n)]
    outs = [empty_dev(count) for _ in range(n)]
    for e in range(1, epochs + 1):
        xs = plant_reserved([synth.normal_bf16(28, count, e, r) for r in range(n)], e)
        orders = []
        for r in range(n):
            ins[r].copy_(to_dev(xs[r]))
            idx, order, kind, poison = synth.stale_plan(28, real.size, 0.10, e, r)
            cd.coll_stage_withheld(coll.spec, r, ins[r], torch.from_numpy(real[idx]).cuda(),
                                   torch.from_numpy(kind).cuda(),
                                   torch.from_numpy(poison.view(np.int16)).cuda())
            orders.append(torch.from_numpy(real[order]).cuda())
        cd.coll_run_late(coll.spec, ins, outs, orders)
        check(cd, coll, outs, oracle.allreduce(xs), n)
        assert coll.epoch() == e + 1
    assert cd.coll_get_rejections(coll.spec) > 0

"""Bandwidth regime at full size: 8 ranks, bf16 uniform[-4,4], 32 / 128 /
256 MiB per rank, LL128 lines (and sentinel packs), on the launch paths the
bench times: the composed one-launch path and the stream-ordered launches.

Every element of every rank's output is compared with the oracle.  The
oracle folds the full inputs once per size with its reduce-scatter (one
fold per element, in rank order; its partitions laid end to end are the
all-reduce result, which is the same expression for every rank); the
all-gather and all-to-all outputs are the oracle's own copies.  Expected
values are moved to the device and compared there with torch.equal (a
library comparison, not this package's code).  Composed-against-streamed
equality is kept as an extra check, never as the main one."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

N = 8
MAX_ELEMS = 128 * 1024 * 1024  # 256 MiB of bf16 per rank


@pytest.fixture(scope="module")
def cd():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import collective_datapath_gb300 as m

    return m


@pytest.fixture(scope="module")
def host_inputs(cd):
    xs = [synth.uniform_bf16(4, MAX_ELEMS, -4.0, 4.0, 4, r) for r in range(N)]
    # no input holds the sentinel's reserved pattern, so the sentinel
    # encoding's sanitisation leaves them unchanged
    assert not any(bool((x == 0xFFFF).any()) for x in xs)
    return xs


@pytest.fixture(scope="module")
def inputs(host_inputs):
    import torch

    return [torch.from_numpy(x.view(np.int16)).cuda() for x in host_inputs]


def dev(x: np.ndarray):
    import torch

    return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).cuda()


@pytest.fixture(scope="module")
def fold(host_inputs):
    """fold(count): the oracle's all-reduce of the first `count` elements of
    every rank (on the device), computed once per size."""
    cache = {}

    def get(count: int):
        if count not in cache:
            parts = oracle.reduce_scatter([x[:count] for x in host_inputs])
            full = np.concatenate(parts)
            assert full.size == count
            cache[count] = dev(full)
        return cache[count]

    yield get
    cache.clear()


def check(got, want, what: str) -> None:
    """Every element of `got` equals `want` (device tensors)."""
    import torch

    assert got.numel() >= want.numel(), what
    g = got[:want.numel()]
    if not torch.equal(g, want):
        bad = torch.nonzero(g != want)
        i = int(bad[0, 0])
        raise AssertionError(f"{what}: {bad.shape[0]} elements differ from the oracle, "
                             f"first at {i} (got {int(g[i]) & 0xFFFF:#06x}, "
                             f"want {int(want[i]) & 0xFFFF:#06x})")


def release():
    import torch

    torch.cuda.synchronize()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mib", [32, 128, 256])
def test_bandwidth_allreduce_twoshot_ll128(cd, inputs, fold, mib):
    import torch

    count = mib * 1024 * 1024 // 2
    coll = cd.Collective(cd.ALLREDUCE, N, count, encoding=cd.COLL_LL128,
                         algorithm=cd.COLL_TWOSHOT, path=cd.COLL_PATH_STREAMED)
    ins = [x[:count] for x in inputs]
    outs = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(N)]
    for epoch in range(2):                   # two epochs: both staging slots
        for o in outs:
            o.fill_(0x5A5A)
        coll.run(ins, outs)
        code, rank, line = coll.status()
        assert code == cd.COLL_OK, (code, rank, line)
        for r in range(N):
            check(outs[r], fold(count), f"epoch {epoch} rank {r}")
    del coll, outs
    release()


@pytest.mark.parametrize("mib", [32, 256])
def test_bandwidth_reduce_scatter_and_all_gather(cd, inputs, fold, mib):
    """Stream-ordered reduce-scatter (shard r = partition r of the oracle's
    fold), all-gather of those shards (= the oracle's all-reduce: AG after RS
    is AR), and the all-reduce itself (oneshot at 32 MiB, twoshot at 256)."""
    import torch

    count = mib * 1024 * 1024 // 2
    m = count // N
    want = fold(count)
    ins = [x[:count] for x in inputs]
    rs = cd.Collective(cd.REDUCE_SCATTER, N, count, encoding=cd.COLL_LL128,
                       path=cd.COLL_PATH_STREAMED)
    shards = [torch.empty(m, dtype=torch.int16, device="cuda") for _ in range(N)]
    rs.run(ins, shards)
    assert rs.status()[0] == cd.COLL_OK
    del rs
    for r in range(N):
        check(shards[r], want[r * m:(r + 1) * m], f"reduce-scatter shard {r}")
    ag = cd.Collective(cd.ALLGATHER, N, count, encoding=cd.COLL_LL128,
                       path=cd.COLL_PATH_STREAMED)
    gathered = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(N)]
    ag.run(shards, gathered)
    assert ag.status()[0] == cd.COLL_OK
    del ag, shards
    for d in range(N):
        check(gathered[d], want, f"all-gather of the shards, rank {d}")
    del gathered
    ar = cd.Collective(cd.ALLREDUCE, N, count, encoding=cd.COLL_LL128,
                       algorithm=cd.COLL_ONESHOT if mib == 32 else cd.COLL_TWOSHOT,
                       path=cd.COLL_PATH_STREAMED)
    outs = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(N)]
    ar.run(ins, outs)
    assert ar.status()[0] == cd.COLL_OK
    for d in range(N):
        check(outs[d], want, f"all-reduce rank {d}")
    del ar, outs
    release()


@pytest.mark.parametrize("mib,staging_mib", [(32, 0), (128, 0), (256, 0), (256, 8), (256, 4)])
def test_bandwidth_allreduce_composed_twoshot(cd, inputs, fold, mib, staging_mib):
    """The one-launch twoshot (the bench's launch) at full size, every element
    of every rank against the oracle over two epochs; also with the staging
    images bounded to a few MiB, chunks cycling through them.  Extra check:
    byte-identical to the stream-ordered twoshot."""
    import torch

    count = mib * 1024 * 1024 // 2
    want = fold(count)
    ins = [x[:count] for x in inputs]
    comp = cd.Collective(cd.ALLREDUCE, N, count, encoding=cd.COLL_LL128,
                         algorithm=cd.COLL_TWOSHOT, path=cd.COLL_PATH_COMPOSED,
                         staging_bytes=staging_mib << 20)
    outs = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(N)]
    for epoch in range(2):
        for o in outs:
            o.fill_(0x5A5A)
        comp.run(ins, outs)
        code, rank, line = comp.status()
        assert code == cd.COLL_OK, (code, rank, line)
        for r in range(N):
            check(outs[r], want, f"epoch {epoch} rank {r}")
    del comp
    ref = cd.Collective(cd.ALLREDUCE, N, count, encoding=cd.COLL_LL128,
                        algorithm=cd.COLL_TWOSHOT, path=cd.COLL_PATH_STREAMED)
    tmp = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(N)]
    ref.run(ins, tmp)
    assert ref.status()[0] == cd.COLL_OK
    for r in range(N):
        assert torch.equal(outs[r], tmp[r]), f"rank {r}: composed and streamed differ"
    del ref, tmp, outs
    release()


@pytest.mark.parametrize("mib", [32, 256])
def test_bandwidth_composed_all_gather(cd, host_inputs, inputs, mib):
    """All-gather (gathered output `mib` MiB per rank), composed and streamed:
    every destination against the oracle's all-gather."""
    import torch

    count = mib * 1024 * 1024 // 2
    m = count // N
    want = oracle.all_gather([x[:m] for x in host_inputs], count)
    for path in (cd.COLL_PATH_COMPOSED, cd.COLL_PATH_STREAMED):
        coll = cd.Collective(cd.ALLGATHER, N, count, encoding=cd.COLL_LL128, path=path)
        ins = [inputs[r][:coll.elems(r)[0]] for r in range(N)]
        outs = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(N)]
        for epoch in range(2):
            for o in outs:
                o.fill_(0x5A5A)
            coll.run(ins, outs)
            code, rank, line = coll.status()
            assert code == cd.COLL_OK, (path, code, rank, line)
            for d in range(N):
                check(outs[d], dev(want[d]), f"path {path} epoch {epoch} rank {d}")
        del coll, outs
    del want
    release()


@pytest.mark.parametrize("mib", [32, 256])
def test_bandwidth_composed_reduce_scatter_and_all_to_all(cd, host_inputs, inputs, fold, mib):
    """Reduce-scatter and all-to-all, composed and streamed: every shard
    against the oracle's fold, every all-to-all output against the oracle's
    all-to-all."""
    import torch

    count = mib * 1024 * 1024 // 2
    m = count // N
    want = fold(count)
    ins = [x[:count] for x in inputs]
    for path in (cd.COLL_PATH_COMPOSED, cd.COLL_PATH_STREAMED):
        rs = cd.Collective(cd.REDUCE_SCATTER, N, count, encoding=cd.COLL_LL128, path=path)
        shards = [torch.empty(m, dtype=torch.int16, device="cuda") for _ in range(N)]
        for epoch in range(2):
            for sh in shards:
                sh.fill_(0x5A5A)
            rs.run(ins, shards)
            assert rs.status()[0] == cd.COLL_OK
            for r in range(N):
                check(shards[r], want[r * m:(r + 1) * m], f"path {path} epoch {epoch} shard {r}")
        del rs, shards
    a2a_want = oracle.all_to_all([x[:count] for x in host_inputs])
    for path in (cd.COLL_PATH_COMPOSED, cd.COLL_PATH_STREAMED):
        a2a = cd.Collective(cd.ALLTOALL, N, count, encoding=cd.COLL_LL128, path=path)
        outs = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(N)]
        for epoch in range(2):
            for o in outs:
                o.fill_(0x5A5A)
            a2a.run(ins, outs)
            assert a2a.status()[0] == cd.COLL_OK
            for d in range(N):
                check(outs[d], dev(a2a_want[d]), f"all-to-all path {path} epoch {epoch} rank {d}")
        del a2a, outs
    del a2a_want
    release()


@pytest.mark.parametrize("mib", [32, 256])
def test_bandwidth_allreduce_sentinel_twoshot(cd, inputs, fold, mib):
    """Sentinel packs, twoshot, on the stream-ordered path the policy runs at
    these sizes (pipelined sentinel fold and copy, deferred re-arm), over two
    epochs: every rank against the oracle's fold (no input holds the reserved
    pattern, so sanitisation changes nothing)."""
    import torch

    count = mib * 1024 * 1024 // 2
    want = fold(count)
    ins = [x[:count] for x in inputs]
    coll = cd.Collective(cd.ALLREDUCE, N, count, encoding=cd.COLL_SENT,
                         algorithm=cd.COLL_TWOSHOT, path=cd.COLL_PATH_STREAMED)
    outs = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(N)]
    for epoch in range(2):
        for o in outs:
            o.fill_(0x5A5A)
        coll.run(ins, outs)
        code, rank, line = coll.status()
        assert code == cd.COLL_OK, (code, rank, line)
        for r in range(N):
            check(outs[r], want, f"epoch {epoch} rank {r}")
    del coll, outs
    release()

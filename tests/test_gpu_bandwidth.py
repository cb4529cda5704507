"""Bandwidth regime at full size: 8 ranks, bf16 uniform[-4,4], 32 / 128 /
256 MiB per rank, LL128 lines, streamed launch path (the configuration the
bench times).  The oracle cannot fold 2 GiB per rank in seconds, so outputs
are checked on sampled positions (random, plus every partition edge and
LL128 row edge near them) against the oracle's fold of those positions, and
in full against properties that hold at any size: every all-reduce copy is
identical, and all-gather(reduce-scatter(x)) equals all-reduce(x)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import from_dev

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
def inputs(cd):
    import torch

    dev = []
    for r in range(N):
        x = synth.uniform_bf16(4, MAX_ELEMS, -4.0, 4.0, 4, r)
        dev.append(torch.from_numpy(x.view(np.int16)).cuda())
        del x
    return dev


def sample_positions(count: int, seed: int) -> np.ndarray:
    g = np.random.Generator(np.random.Philox(seed))
    pos = set(g.integers(0, count, size=40000).tolist())
    m = oracle.shard_elems(count, N)
    for r in range(N + 1):
        for d in (-241, -240, -61, -60, -59, -1, 0, 1, 59, 60, 239, 240):
            v = r * m + d
            if 0 <= v < count:
                pos.add(v)
    pos.update([0, count - 1])
    return np.array(sorted(pos), dtype=np.int64)


def sampled_reference(inputs, count, pos):
    import torch

    idx = torch.from_numpy(pos).cuda()
    cols = [inputs[r][:count][idx].cpu().numpy().view(np.uint16) for r in range(N)]
    return oracle.allreduce(cols)[0]


@pytest.mark.parametrize("mib", [32, 128, 256])
def test_bandwidth_allreduce_twoshot_ll128(cd, inputs, mib):
    import torch

    count = mib * 1024 * 1024 // 2
    coll = cd.Collective(cd.ALLREDUCE, N, count, encoding=cd.COLL_LL128,
                         algorithm=cd.COLL_TWOSHOT, path=cd.COLL_PATH_STREAMED)
    ins = [x[:count] for x in inputs]
    outs = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(N)]
    for _ in range(2):                       # two epochs: both staging slots
        coll.run(ins, outs)
    code, rank, line = coll.status()
    assert code == cd.COLL_OK, (code, rank, line)
    for r in range(1, N):
        assert torch.equal(outs[r], outs[0]), f"copy {r} differs"
    pos = sample_positions(count, mib)
    want = sampled_reference(inputs, count, pos)
    got = outs[0][torch.from_numpy(pos).cuda()].cpu().numpy().view(np.uint16)
    assert np.array_equal(got, want)
    del coll, outs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mib", [32, 256])
def test_bandwidth_reduce_scatter_and_all_gather(cd, inputs, mib):
    import torch

    count = mib * 1024 * 1024 // 2
    m = count // N
    ins = [x[:count] for x in inputs]
    rs = cd.Collective(cd.REDUCE_SCATTER, N, count, encoding=cd.COLL_LL128,
                       path=cd.COLL_PATH_STREAMED)
    shards = [torch.empty(m, dtype=torch.int16, device="cuda") for _ in range(N)]
    rs.run(ins, shards)
    assert rs.status()[0] == cd.COLL_OK
    del rs
    ag = cd.Collective(cd.ALLGATHER, N, count, encoding=cd.COLL_LL128,
                       path=cd.COLL_PATH_STREAMED)
    gathered = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(N)]
    ag.run(shards, gathered)
    assert ag.status()[0] == cd.COLL_OK
    del ag
    # sampled against the oracle: RS shard r holds the fold of partition r
    pos = sample_positions(count, 7 + mib)
    want = sampled_reference(inputs, count, pos)
    got = gathered[3][torch.from_numpy(pos).cuda()].cpu().numpy().view(np.uint16)
    assert np.array_equal(got, want)
    for r in range(N):
        sel = pos[(pos >= r * m) & (pos < (r + 1) * m)]
        g = shards[r][torch.from_numpy(sel - r * m).cuda()].cpu().numpy().view(np.uint16)
        assert np.array_equal(g, want[np.searchsorted(pos, sel)])
    # all-gather copies are identical, and equal all-reduce in full
    for r in range(1, N):
        assert torch.equal(gathered[r], gathered[0])
    del shards
    ar = cd.Collective(cd.ALLREDUCE, N, count, encoding=cd.COLL_LL128,
                       algorithm=cd.COLL_ONESHOT if mib == 32 else cd.COLL_TWOSHOT,
                       path=cd.COLL_PATH_STREAMED)
    outs = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(2)]
    ar_outs = outs + [torch.empty(count, dtype=torch.int16, device="cuda")
                      for _ in range(N - 2)]
    ar.run(ins, ar_outs)
    assert ar.status()[0] == cd.COLL_OK
    assert torch.equal(ar_outs[5], gathered[0])
    del ar, ar_outs, outs, gathered
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mib,staging_mib", [(32, 0), (256, 0), (256, 8), (256, 4)])
def test_bandwidth_allreduce_composed_twoshot(cd, inputs, mib, staging_mib):
    """The one-launch twoshot at full size: sampled against the oracle, and
    byte-identical to the stream-ordered twoshot on every element; also with
    the staging images bounded to a few MiB, chunks cycling through them."""
    import torch

    count = mib * 1024 * 1024 // 2
    ins = [x[:count] for x in inputs]
    comp = cd.Collective(cd.ALLREDUCE, N, count, encoding=cd.COLL_LL128,
                         algorithm=cd.COLL_TWOSHOT, path=cd.COLL_PATH_COMPOSED,
                         staging_bytes=staging_mib << 20)
    outs = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(N)]
    for _ in range(2):
        comp.run(ins, outs)
    code, rank, line = comp.status()
    assert code == cd.COLL_OK, (code, rank, line)
    pos = sample_positions(count, 50 + mib)
    want = sampled_reference(inputs, count, pos)
    got = outs[0][torch.from_numpy(pos).cuda()].cpu().numpy().view(np.uint16)
    assert np.array_equal(got, want)
    del comp
    ref = cd.Collective(cd.ALLREDUCE, N, count, encoding=cd.COLL_LL128,
                        algorithm=cd.COLL_TWOSHOT, path=cd.COLL_PATH_STREAMED)
    ref_out = torch.empty(count, dtype=torch.int16, device="cuda")
    tmp = [ref_out] + [torch.empty(count, dtype=torch.int16, device="cuda")
                       for _ in range(N - 1)]
    ref.run(ins, tmp)
    assert ref.status()[0] == cd.COLL_OK
    for r in range(N):
        assert torch.equal(outs[r], ref_out), f"rank {r}"
    del ref, tmp, outs
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mib", [32, 256])
def test_bandwidth_composed_all_gather(cd, inputs, mib):
    """The one-launch all-gather at full size (gathered output `mib` MiB per
    rank): byte-identical to the stream-ordered all-gather, and every
    destination holds each source's segment in its partition."""
    import torch

    count = mib * 1024 * 1024 // 2
    res = {}
    for path in (cd.COLL_PATH_COMPOSED, cd.COLL_PATH_STREAMED):
        coll = cd.Collective(cd.ALLGATHER, N, count, encoding=cd.COLL_LL128, path=path)
        ins = [inputs[r][:coll.elems(r)[0]] for r in range(N)]
        outs = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(N)]
        for _ in range(2):
            coll.run(ins, outs)
        code, rank, line = coll.status()
        assert code == cd.COLL_OK, (path, code, rank, line)
        res[path] = outs
        del coll
    m = count // N
    for d in range(N):
        assert torch.equal(res[cd.COLL_PATH_COMPOSED][d], res[cd.COLL_PATH_STREAMED][d])
        for p in (0, N - 1):
            assert torch.equal(res[cd.COLL_PATH_COMPOSED][d][p * m:(p + 1) * m], inputs[p][:m])
    del res
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mib", [32, 256])
def test_bandwidth_composed_reduce_scatter_and_all_to_all(cd, inputs, mib):
    """The one-launch reduce-scatter (sampled against the oracle, and equal
    to the stream-ordered one on every element) and all-to-all (equal to the
    stream-ordered one on every element)."""
    import torch

    count = mib * 1024 * 1024 // 2
    m = count // N
    ins = [x[:count] for x in inputs]
    results = {}
    for path in (cd.COLL_PATH_COMPOSED, cd.COLL_PATH_STREAMED):
        rs = cd.Collective(cd.REDUCE_SCATTER, N, count, encoding=cd.COLL_LL128, path=path)
        shards = [torch.empty(m, dtype=torch.int16, device="cuda") for _ in range(N)]
        for _ in range(2):
            rs.run(ins, shards)
        assert rs.status()[0] == cd.COLL_OK
        del rs
        results[("rs", path)] = shards
    pos = sample_positions(count, 90 + mib)
    want = sampled_reference(inputs, count, pos)
    for r in range(N):
        sel = pos[(pos >= r * m) & (pos < (r + 1) * m)]
        got = results[("rs", cd.COLL_PATH_COMPOSED)][r][torch.from_numpy(sel - r * m).cuda()]
        assert np.array_equal(got.cpu().numpy().view(np.uint16), want[np.searchsorted(pos, sel)])
        assert torch.equal(results[("rs", cd.COLL_PATH_COMPOSED)][r],
                           results[("rs", cd.COLL_PATH_STREAMED)][r])
    del results
    outs = {}
    for path in (cd.COLL_PATH_COMPOSED, cd.COLL_PATH_STREAMED):
        a2a = cd.Collective(cd.ALLTOALL, N, count, encoding=cd.COLL_LL128, path=path)
        o = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(N)]
        for _ in range(2):
            a2a.run(ins, o)
        assert a2a.status()[0] == cd.COLL_OK
        del a2a
        outs[path] = o
    for d in range(N):
        assert torch.equal(outs[cd.COLL_PATH_COMPOSED][d], outs[cd.COLL_PATH_STREAMED][d])
        # block p of destination d is block d of source p
        for p in (0, 3, N - 1):
            assert torch.equal(outs[cd.COLL_PATH_COMPOSED][d][p * m:(p + 1) * m],
                               ins[p][d * m:(d + 1) * m])
    del outs
    torch.cuda.empty_cache()

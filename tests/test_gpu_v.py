"""Variable-length collectives (reduce-scatter V, all-gather V, all-to-all V)
on the GPU against the oracle, element by element.  Sizes follow the
variable-length experiment of the Purlin paper (Figure 13 and appendix
Eq. (4)): 8 ranks, a Zipf split with exponent 0.125 of a power-of-two total
T, all-to-all V rotating each source's split right by (source + 1)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import buffers, from_dev, to_dev

pytestmark = pytest.mark.gpu

N = 8


@pytest.fixture(scope="module")
def cd():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import collective_datapath_gb300 as m

    return m


def split(total_bytes, n=N):
    return [b // 2 for b in synth.zipf_split(total_bytes, n)]


def vectors(name, total_bytes, n=N):
    base = split(total_bytes, n)
    if name == "ALLTOALL_V":
        return [synth.rotate_right(base, p + 1) for p in range(n)]
    return base


def expected(name, ins, v):
    if name == "REDUCE_SCATTER_V":
        return oracle.reduce_scatter_v(ins, v)
    if name == "ALLGATHER_V":
        return oracle.all_gather_v(ins, v)
    return oracle.all_to_all_v(ins, v)


def check(cd, name, v, n, seed, staged=False, epochs=2, **opts):
    count = 0 if name == "ALLTOALL_V" else int(sum(v))
    coll = cd.Collective(getattr(cd, name), n, count, vcounts=v, **opts)
    ins_h, ins_d, outs_d = buffers(coll, n, seed, dist="bits" if name != "REDUCE_SCATTER_V"
                                   else "normal", tag=len(name))
    want = expected(name, ins_h, v)
    for epoch in range(epochs):                      # both staging slots
        if staged:
            for r in range(n):
                coll.stage(r, ins_d[r])
            coll.run(None, outs_d)
        else:
            coll.run(ins_d, outs_d)
        code, rank, line = coll.status()
        assert code == cd.COLL_OK, (code, rank, line)
        for r in range(n):
            got = from_dev(outs_d[r])[:want[r].size]
            assert np.array_equal(got, want[r]), f"epoch {epoch} rank {r}"
    coll.close()


NAMES = ["REDUCE_SCATTER_V", "ALLGATHER_V", "ALLTOALL_V"]


@pytest.mark.parametrize("name", NAMES)
@pytest.mark.parametrize("enc", [0, 1])
@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("total", [1 << 20, 1 << 22])
def test_v_collective_zipf_matches_oracle(cd, name, enc, path, total):
    check(cd, name, vectors(name, total), N, 11, encoding=enc, path=path)


@pytest.mark.parametrize("name", NAMES)
def test_v_collective_zipf_64mib_streamed_ll128(cd, name):
    check(cd, name, vectors(name, 64 << 20), N, 12, encoding=1, path=2)


@pytest.mark.parametrize("name", NAMES)
def test_v_collective_staged_and_fused_ll8_rearm_modes(cd, name):
    for mode in (0, 1, 3):
        check(cd, name, vectors(name, 1 << 18), N, 13 + mode, staged=True, epochs=3,
              encoding=0, path=1, reset_mode=mode)


@pytest.mark.parametrize("name,n,v", [
    ("REDUCE_SCATTER_V", 3, [8, 0, 488]),
    ("ALLGATHER_V", 4, [64, 8, 0, 1208]),
    ("ALLTOALL_V", 3, [[8, 0, 240], [0, 0, 16], [128, 64, 8]]),
    ("ALLTOALL_V", 2, [[0, 0], [0, 0]]),
])
@pytest.mark.parametrize("enc", [0, 1])
def test_v_collective_ragged_and_empty_partitions(cd, name, n, v, enc):
    check(cd, name, v, n, 14, encoding=enc, path=2)
    check(cd, name, v, n, 15, encoding=enc, path=1)


# ---- the composed launch by columns ------------------------------------------

@pytest.mark.parametrize("name", NAMES)
@pytest.mark.parametrize("total", [1 << 20, 1 << 22, 64 << 20])
def test_v_collective_zipf_composed(cd, name, total):
    """One launch by columns: column (chunk c, partition x) stages every
    source's lines of partition x, then folds them into owner x's output
    (reduce-scatter V) or copies them out (all-gather V: source x's one
    piece to every destination at the sum of the earlier sources' lengths;
    all-to-all V: each source's own piece, of its own length, into block p
    of destination x).  Columns past a partition's end are skipped."""
    check(cd, name, vectors(name, total), N, 16, encoding=1, path=3)


@pytest.mark.parametrize("name,n,v", [
    ("REDUCE_SCATTER_V", 3, [8, 0, 488]),
    ("ALLGATHER_V", 4, [64, 8, 0, 1208]),
    ("ALLTOALL_V", 3, [[8, 0, 240], [0, 0, 16], [128, 64, 8]]),
    ("ALLTOALL_V", 2, [[0, 0], [0, 0]]),
    ("ALLTOALL_V", 4, [[0, 4096, 8, 0], [8, 0, 0, 7800], [0, 0, 0, 0], [64, 120, 56, 0]]),
])
def test_v_collective_composed_ragged_and_empty_partitions(cd, name, n, v):
    check(cd, name, v, n, 17, encoding=1, path=3)


@pytest.mark.parametrize("name", ["REDUCE_SCATTER_V", "ALLGATHER_V"])
def test_v_collective_composed_queue_schedule(cd, name, monkeypatch):
    """The task-queue schedule of the composed launch serves the reduce-
    scatter and all-gather V from the same segment fields."""
    monkeypatch.setenv("COLL_COMPOSED_SHAPE", "32,5,1,2,-1,1")
    check(cd, name, vectors(name, 1 << 22), N, 18, encoding=1, path=3)


def test_alltoall_v_refuses_the_queue_schedule(cd, monkeypatch):
    monkeypatch.setenv("COLL_COMPOSED_SHAPE", "32,5,1,2,-1,1")
    v = vectors("ALLTOALL_V", 1 << 20)
    coll = cd.Collective(cd.ALLTOALL_V, N, 0, vcounts=v, encoding=1, path=3)
    _, ins_d, outs_d = buffers(coll, N, 3, dist="bits")
    with pytest.raises(cd.CollError) as e:
        coll.run(ins_d, outs_d)
    assert e.value.status == cd.COLL_ERR_UNSUPPORTED
    coll.close()


@pytest.mark.parametrize("name", ["REDUCE_SCATTER_V", "ALLTOALL_V"])
@pytest.mark.parametrize("slots", [2, 9])
def test_v_collective_composed_bounded_staging(cd, name, slots):
    """Bounded staging (Purlin §4.1): each CTA owns a chunk slot of every
    rank image and reuses it column after column, lines carrying epoch + the
    column index (§4.2).  New inputs every epoch, so a stale line taken from
    an earlier cycle or run would show in the result."""
    v = vectors(name, 1 << 22)
    count = 0 if name == "ALLTOALL_V" else int(sum(v))
    coll = cd.Collective(getattr(cd, name), N, count, vcounts=v, encoding=1, path=3,
                         staging_bytes=slots * N * 16 * 128)
    _, ins_d, outs_d = buffers(coll, N, 19, dist="bits")
    last = coll.epoch()
    for e in range(4):
        sizes = [coll.elems(r)[0] for r in range(N)]
        xs = [synth.random_bits16(600 + e, sizes[r], N, r) if name == "ALLTOALL_V"
              else synth.normal_bf16(600 + e, sizes[r], N, r) for r in range(N)]
        for r in range(N):
            ins_d[r][:sizes[r]].copy_(to_dev(xs[r]))
        coll.run(ins_d, outs_d)
        code, rank, line = coll.status()
        assert code == cd.COLL_OK, (code, rank, line)
        want = expected(name, xs, v)
        for r in range(N):
            assert np.array_equal(from_dev(outs_d[r])[:want[r].size], want[r]), f"epoch {e} rank {r}"
        now = coll.epoch()
        assert (now - last) % 2 == 1, (last, now)
        last = now
    coll.close()

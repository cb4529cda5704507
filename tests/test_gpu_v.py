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
from tests.gpu_util import buffers, from_dev

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

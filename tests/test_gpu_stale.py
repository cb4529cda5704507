"""Self-synchronizing dual-buffer run with stale lines published late:
8 ranks x [16 x 7168] bf16 normal(0,1), 64 consecutive all-reduce epochs on
two staging slots, LL8 and LL128.  Each epoch a seeded 10% of every rank's
lines is left stale (readiness value of the previous epoch, of the slot's
previous occupant, or zero, over a poison payload) and published late, in a
seeded order, by producer CTAs of the same cooperative launch while the
consumers poll.  The consumers must reject every stale line and fold in rank
order whatever the publication order: the result equals the oracle's
all-reduce of the published inputs, bit for bit."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import empty_dev, from_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cd():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import collective_datapath_gb300 as m

    return m


def image_lines_of_real_lines(cd, coll, n_seg):
    """Image line index of every payload line of a rank image (slot 0, rank 0)."""
    base, _, lb = cd.coll_staging_layout(coll.spec, 0, 0, 0, 0)
    out = []
    for k in range(n_seg):
        off, lines, _ = cd.coll_staging_layout(coll.spec, 0, 0, 0, k)
        l0 = (off - base) // lb
        out.append(np.arange(l0, l0 + lines, dtype=np.int64))
    return np.concatenate(out)


@pytest.mark.parametrize("enc,algo,epochs", [(0, 1, 64), (1, 1, 64), (0, 2, 64), (1, 2, 64)])
def test_stale_lines_rejected_across_64_epochs(cd, enc, algo, epochs):
    import torch

    n, count = 8, 16 * 7168
    coll = cd.Collective(cd.ALLREDUCE, n, count, encoding=enc, algorithm=algo,
                         path=cd.COLL_PATH_FUSED, timeout_ns=500_000_000)
    real = image_lines_of_real_lines(cd, coll, n)
    assert real.size == (57344 if enc == 0 else 8 * 239)
    ins = [empty_dev(count) for _ in range(n)]
    outs = [empty_dev(count) for _ in range(n)]
    for e in range(1, epochs + 1):
        xs = [synth.normal_bf16(3, count, e, r) for r in range(n)]
        orders = []
        for r in range(n):
            ins[r].copy_(to_dev(xs[r]))
            idx, order, kind, poison = synth.stale_plan(3, real.size, 0.10, e, r)
            lines = torch.from_numpy(real[idx]).cuda()
            cd.coll_stage_withheld(coll.spec, r, ins[r], lines,
                                   torch.from_numpy(kind).cuda(),
                                   torch.from_numpy(poison.view(np.int16)).cuda())
            orders.append(torch.from_numpy(real[order]).cuda())
        cd.coll_run_late(coll.spec, ins, outs, orders)
        code, rank, line = coll.status()
        assert code == cd.COLL_OK, f"epoch {e}: status {code} rank {rank} line {line}"
        want = oracle.allreduce(xs)
        for r in range(n):
            got = from_dev(outs[r])
            assert np.array_equal(got, want[r]), f"epoch {e} rank {r}"
        assert coll.epoch() == e + 1
    # consumers did see stale lines and waited for them
    assert cd.coll_get_rejections(coll.spec) > 0

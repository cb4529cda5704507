"""MoE dispatch all-to-all (scatteredV -> transposedV copy) on the GPU against
the oracle: small cases in full (rows and counts), the full-size workload
(8 ranks x 4096 tokens x 7168 bf16, top-8 of 256 experts) row by row through
the oracle's listing of each output row's source, and host-made faults."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import from_dev, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cd():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import collective_datapath_gb300 as m

    return m


def make_moe(cd, n, tokens, hidden, k, experts, **kw):
    return cd.Collective(cd.MOE_DISPATCH, n, 0, encoding=cd.COLL_LL128, tokens=tokens,
                         hidden=hidden, topk=k, experts=experts, **kw)


def route(cd, coll, topk_dev):
    for r, t in enumerate(topk_dev):
        cd.coll_set_routing(coll.spec, r, t)


def counts_of(cd, coll, n, experts):
    import torch

    el = experts // n
    buf = torch.zeros(n * el * n + n, dtype=torch.int32, device="cuda")
    cd.coll_get_counts(coll.spec, buf)
    torch.cuda.synchronize()
    c = buf.cpu().numpy()
    return c[:n * el * n].reshape(n, el, n), c[n * el * n:]


@pytest.mark.parametrize("path", [2, 3, "3q"])
@pytest.mark.parametrize("n,tokens,hidden,k,experts,staged", [
    (4, 300, 64, 3, 16, False),
    (2, 128, 136, 2, 4, True),
    (8, 257, 7168, 8, 256, False),
    (3, 50, 120, 4, 9, True),
    (8, 33, 960, 8, 512, False),
    (1, 17, 64, 2, 2, False),
    # more than 32 choices per token (a copy warp's second register of rows)
    (4, 70, 256, 40, 64, False),
    (8, 40, 480, 64, 64, False),
    # 32 local experts per rank: a token's 20 choices often all on one rank
    (2, 90, 120, 20, 64, True),
])
def test_moe_dispatch_small_cases_match_the_oracle(cd, n, tokens, hidden, k, experts, staged,
                                                   path, monkeypatch):
    """Both launch forms: routing, stage and copy launches (2), and routing
    plus one launch (3) of columns (a source's token sub-block staged and
    copied by one CTA) or, "3q", of the queue of stage and copy tasks with a
    lag of 6 blocks; staged runs take the first form's copy."""
    import torch

    if path == "3q":
        monkeypatch.setenv("COLL_MOE_LAG", "6")
        path = 3
    coll = make_moe(cd, n, tokens, hidden, k, experts, path=path)
    xs = [synth.normal_bf16(5, tokens * hidden, n, r).reshape(tokens, hidden) for r in range(n)]
    tk = [synth.topk_experts(5, tokens, k, experts, n, r) for r in range(n)]
    ins = [to_dev(x.ravel()) for x in xs]
    topk_dev = [torch.from_numpy(t.ravel()).cuda() for t in tk]
    route(cd, coll, topk_dev)
    outs = [torch.zeros(coll.elems(r)[1], dtype=torch.int16, device="cuda") for r in range(n)]
    want, wcounts, wrows = oracle.moe_dispatch(xs, tk, experts)
    for epoch in range(2):                     # both staging slots
        if staged:
            for r in range(n):
                coll.stage(r, ins[r])
            coll.run(None, outs)
        else:
            coll.run(ins, outs)
        code, rank, line = coll.status()
        assert code == cd.COLL_OK, (code, rank, line)
        counts, rows = counts_of(cd, coll, n, experts)
        assert np.array_equal(counts, wcounts)
        assert np.array_equal(rows, wrows)
        for d in range(n):
            got = from_dev(outs[d])[:wrows[d] * hidden].reshape(-1, hidden)
            assert np.array_equal(got, want[d]), f"epoch {epoch} destination {d}"


@pytest.mark.parametrize("path", [2, 3])
@pytest.mark.parametrize("n,tokens,hidden,k,experts", [(4, 300, 64, 3, 16), (8, 129, 3584, 8, 256),
                                                      (2, 40, 8, 2, 4)])
def test_moe_dispatch_f32_rows(cd, n, tokens, hidden, k, experts, path):
    """fp32 rows (random bit patterns, NaN payloads included) dispatched byte
    for byte: the oracle's dispatch of the same bytes seen as 2 * hidden
    16-bit units, rows and counts, both launch forms, two epochs."""
    import torch

    coll = make_moe(cd, n, tokens, hidden, k, experts, path=path, dtype=cd.COLL_F32)
    xs = [synth.random_bits32(7, tokens * hidden, n, r) for r in range(n)]
    tk = [synth.topk_experts(7, tokens, k, experts, n, r) for r in range(n)]
    ins = [torch.from_numpy(x.view(np.int32)).cuda() for x in xs]
    topk_dev = [torch.from_numpy(t.ravel()).cuda() for t in tk]
    route(cd, coll, topk_dev)
    assert coll.elems(0) == (tokens * hidden, coll.elems(0)[1])
    outs = [torch.zeros(coll.elems(r)[1], dtype=torch.int32, device="cuda") for r in range(n)]
    want, wcounts, wrows = oracle.moe_dispatch(
        [x.view(np.uint16).reshape(tokens, 2 * hidden) for x in xs], tk, experts)
    for epoch in range(2):
        coll.run(ins, outs)
        code, rank, line = coll.status()
        assert code == cd.COLL_OK, (code, rank, line)
        counts, rows = counts_of(cd, coll, n, experts)
        assert np.array_equal(counts, wcounts)
        assert np.array_equal(rows, wrows)
        for d in range(n):
            got = outs[d].cpu().numpy().view(np.uint16)[:wrows[d] * 2 * hidden]
            assert np.array_equal(got.reshape(-1, 2 * hidden), want[d]), (epoch, d)


@pytest.mark.parametrize("path", [2, 3])
def test_moe_dispatch_8x4096x7168_full_size(cd, path):
    """8 ranks x 4096 tokens x 7168 bf16 normal(0,1), top-8 of 256 experts:
    every output row of every destination equals its source row as listed
    by the oracle, and the counts equal the oracle's (both launch forms)."""
    import torch

    n, tokens, hidden, k, experts = 8, 4096, 7168, 8, 256
    coll = make_moe(cd, n, tokens, hidden, k, experts, max_rows=40000, path=path)
    xs = [synth.normal_bf16(6, tokens * hidden, r) for r in range(n)]
    tk = [synth.topk_experts(6, tokens, k, experts, r) for r in range(n)]
    x_dev = torch.stack([torch.from_numpy(x.view(np.int16)) for x in xs]).cuda()  # [n, T*H]
    ins = [x_dev[r] for r in range(n)]
    topk_dev = [torch.from_numpy(t.ravel()).cuda() for t in tk]
    route(cd, coll, topk_dev)
    outs = [torch.empty(coll.elems(r)[1], dtype=torch.int16, device="cuda") for r in range(n)]
    coll.run(ins, outs)
    code, rank, line = coll.status()
    assert code == cd.COLL_OK, (code, rank, line)
    _, wcounts, wrows = oracle.moe_dispatch([x.reshape(tokens, hidden) for x in xs], tk,
                                            experts, with_rows=False)
    counts, rows = counts_of(cd, coll, n, experts)
    assert np.array_equal(counts, wcounts) and np.array_equal(rows, wrows)
    xr = x_dev.view(n, tokens, hidden)
    for d in range(n):
        sr, st = oracle.moe_row_sources(tk, experts, d)
        expect = xr[torch.from_numpy(sr).long().cuda(), torch.from_numpy(st).long().cuda()]
        got = outs[d][:sr.size * hidden].view(sr.size, hidden)
        assert torch.equal(got, expect), f"destination {d}"


def test_moe_out_of_range_expert_latches_invalid(cd):
    import torch

    n, tokens, hidden, k, experts = 2, 64, 32, 2, 4
    coll = make_moe(cd, n, tokens, hidden, k, experts)
    tk = [synth.topk_experts(7, tokens, k, experts, r) for r in range(n)]
    tk[1][10, 1] = 99                           # host-made fault: not an expert
    ins = [to_dev(synth.normal_bf16(7, tokens * hidden, r)) for r in range(n)]
    topk_dev = [torch.from_numpy(t.ravel()).cuda() for t in tk]  # must outlive the run
    route(cd, coll, topk_dev)
    outs = [torch.zeros(coll.elems(r)[1], dtype=torch.int16, device="cuda") for r in range(n)]
    coll.run(ins, outs)
    code, rank, line = coll.status()
    assert code == cd.COLL_ERR_INVALID and rank == 1 and line == 10 * k + 1


def test_moe_more_rows_than_capacity_latches_nomem(cd):
    import torch

    n, tokens, hidden, k, experts = 2, 64, 32, 2, 4
    coll = make_moe(cd, n, tokens, hidden, k, experts, max_rows=10)
    tk = [synth.topk_experts(8, tokens, k, experts, r) for r in range(n)]
    ins = [to_dev(synth.normal_bf16(8, tokens * hidden, r)) for r in range(n)]
    topk_dev = [torch.from_numpy(t.ravel()).cuda() for t in tk]  # must outlive the run
    route(cd, coll, topk_dev)
    outs = [torch.zeros(coll.elems(r)[1], dtype=torch.int16, device="cuda") for r in range(n)]
    coll.run(ins, outs)
    code, rank, line = coll.status()
    assert code == cd.COLL_ERR_NOMEM and line > 10

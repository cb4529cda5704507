"""GPU parity: every collective, both encodings, both launch paths, against
the CPU oracle, bit for bit (tolerance 0 ulp: the fold order is fixed and the
accumulation is fp32 with one rounding)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import buffers, empty_dev, from_dev, make, read_lines, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cd():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import collective_datapath_gb300 as m

    return m


def expected(cd, triple, ins, count):
    if triple == cd.ALLREDUCE:
        return oracle.allreduce(ins)
    if triple == cd.REDUCE_SCATTER:
        return oracle.reduce_scatter(ins)
    if triple == cd.ALLGATHER:
        return oracle.all_gather(ins, count)
    return oracle.all_to_all(ins)


def check(coll, outs, want, n):
    import collective_datapath_gb300 as cd

    code, rank, line = coll.status()
    assert code == cd.COLL_OK, f"device status {code} rank {rank} line {line}"
    for r in range(n):
        got = from_dev(outs[r])[:want[r].size]
        if not np.array_equal(got, want[r]):
            bad = np.flatnonzero(got != want[r])
            raise AssertionError(f"rank {r}: {bad.size} mismatches, first at {bad[0]}: "
                                 f"got {got[bad[0]]:#06x} want {want[r][bad[0]]:#06x}")


def test_oneshot_two_ranks_512_elements(cd):
    """2 ranks x 512 bf16 uniform[-1,1] seed 0, LL8, oneshot, one epoch."""
    n, count = 2, 512
    coll = make(cd, cd.ALLREDUCE, n, count, encoding=cd.COLL_LL8,
                algorithm=cd.COLL_ONESHOT, path=cd.COLL_PATH_FUSED)
    xs = [synth.uniform_bf16(0, count, -1.0, 1.0, 1, p) for p in range(n)]
    ins = [to_dev(x) for x in xs]
    outs = [empty_dev(count) for _ in range(n)]
    coll.run(ins, outs)
    check(coll, outs, oracle.allreduce(xs), n)
    assert coll.epoch() == 2


@pytest.mark.parametrize("algo", [1, 2])
@pytest.mark.parametrize("path", [1, 2])
@pytest.mark.parametrize("T", [1, 2, 4, 8, 16, 32, 64, 128])
def test_decode_allreduce_8_ranks(cd, T, path, algo):
    """8 ranks x [T x 4096] normal(0,1), LL8, oneshot and twoshot; all 8
    output copies identical and equal to the oracle."""
    n, count = 8, T * 4096
    coll = make(cd, cd.ALLREDUCE, n, count, encoding=cd.COLL_LL8, algorithm=algo,
                path=path)
    xs, ins, outs = buffers(coll, n, seed=2, tag=T)
    coll.run(ins, outs)
    want = oracle.allreduce(xs)
    check(coll, outs, want, n)
    first = from_dev(outs[0])
    for r in range(1, n):
        assert np.array_equal(from_dev(outs[r]), first)


CASES = [
    ("ALLREDUCE", 8, 8 * 1000, 1, 1), ("ALLREDUCE", 8, 8 * 1000, 1, 2),
    ("ALLREDUCE", 3, 1000, 0, 1), ("ALLREDUCE", 3, 1000, 1, 2),
    ("ALLREDUCE", 8, 24, 0, 1), ("ALLREDUCE", 1, 4096, 0, 2), ("ALLREDUCE", 1, 4096, 1, 1),
    ("REDUCE_SCATTER", 8, 8 * 3000, 0, 1), ("REDUCE_SCATTER", 8, 8 * 3000, 1, 2),
    ("REDUCE_SCATTER", 5, 5 * 56 + 16, 1, 1),
    ("ALLGATHER", 8, 8 * 2048, 0, 2), ("ALLGATHER", 8, 8 * 2048, 1, 1),
    ("ALLGATHER", 4, 4 * 104 + 8, 1, 2),
    ("ALLTOALL", 8, 8 * 960, 1, 2), ("ALLTOALL", 8, 8 * 960, 0, 1), ("ALLTOALL", 4, 256, 1, 1),
]


@pytest.mark.parametrize("name,n,count,enc,path", CASES)
def test_layout_collectives(cd, name, n, count, enc, path):
    triple = getattr(cd, name)
    for algo in ((1, 2) if name == "ALLREDUCE" else (0,)):
        coll = make(cd, triple, n, count, encoding=enc, path=path, algorithm=algo)
        xs, ins, outs = buffers(coll, n, seed=4, dist="bits" if name != "REDUCE_SCATTER" and
                                name != "ALLREDUCE" else "normal", tag=count)
        coll.run(ins, outs)
        check(coll, outs, expected(cd, triple, xs, count), n)


@pytest.mark.parametrize("enc", [0, 1])
def test_staged_lines_match_the_oracle_encoding(cd, enc):
    """coll_stage writes exactly the oracle's LL8 / LL128 lines (epoch 1,
    slot 1), one segment per partition of the scattered input."""
    n, count = 4, 4 * 1000
    coll = make(cd, cd.ALLREDUCE, n, count, encoding=enc, path=cd.COLL_PATH_STREAMED)
    xs, ins, outs = buffers(coll, n, seed=5, dist="bits")
    for r in range(n):
        coll.stage(r, ins[r])
    import torch

    torch.cuda.synchronize()
    for r in range(n):
        for k in range(n):
            raw, lines, lb = read_lines(coll, 0, 1, r, k)
            b, ln = oracle.shard_begin(count, n, k), oracle.shard_len(count, n, k)
            seg = xs[r][b:b + ln]
            want = (oracle.ll8_encode(seg, 1).view(np.uint8) if enc == 0
                    else oracle.ll128_encode(seg, 1))
            assert np.array_equal(raw, want), f"rank {r} segment {k}"
    coll.run(None, outs)
    check(coll, outs, oracle.allreduce(xs), n)


@pytest.mark.parametrize("algo", [1, 2])
@pytest.mark.parametrize("reset", [0, 1, 3])
@pytest.mark.parametrize("path", [1, 2])
def test_flags_rearmed_after_run(cd, algo, reset, path):
    """LL8 re-arm: every flag word of a consumed slot is 0 afterwards -- the
    slot of the run itself for the last-reader (0) and kernel (1) modes; for
    the deferred mode (3) the slot of the previous run, re-armed while the
    next run uses the other slot."""
    n, count = 8, 8 * 512
    coll = make(cd, cd.ALLREDUCE, n, count, encoding=0, algorithm=algo,
                reset_mode=reset, path=path)
    xs, ins, outs = buffers(coll, n, seed=6)
    coll.run(ins, outs)                      # epoch 1 -> slot 1
    check(coll, outs, oracle.allreduce(xs), n)
    if reset == 3:
        coll.run(ins, outs)                  # epoch 2 -> slot 0, re-arms slot 1
        check(coll, outs, oracle.allreduce(xs), n)
    regions = (0, 1) if algo == 2 else (0,)
    for region in regions:
        for r in range(n):
            for k in range(n if region == 0 else 1):
                raw, lines, lb = read_lines(coll, region, 1, r, k)
                flags = raw.view(np.uint32)[1::2]
                assert np.all(flags == 0), f"region {region} rank {r} seg {k}"
    if reset == 3:
        # the slot in use still carries this run's flags until the next run
        raw, _, _ = read_lines(coll, 0, 0, 0, 0)
        assert np.all(raw.view(np.uint32)[1::2] == 2)


@pytest.mark.parametrize("enc", [0, 1])
@pytest.mark.parametrize("path", [1, 2])
def test_consecutive_epochs_alternate_slots(cd, enc, path):
    n, count = 8, 8 * 2000
    coll = make(cd, cd.ALLREDUCE, n, count, encoding=enc, path=path)
    _, ins, outs = buffers(coll, n, seed=7)
    for e in range(1, 9):
        xs = [synth.normal_bf16(70 + e, count, r) for r in range(n)]
        for r in range(n):
            ins[r].copy_(to_dev(xs[r]))
        coll.run(ins, outs)
        check(coll, outs, oracle.allreduce(xs), n)
        assert coll.epoch() == e + 1


def test_empty_collective_advances_the_epoch(cd):
    coll = make(cd, cd.ALLREDUCE, 8, 0)
    outs = [empty_dev(0) for _ in range(8)]
    coll.run(None, outs)
    coll.run([empty_dev(0) for _ in range(8)], outs)
    code, _, _ = coll.status()
    assert code == cd.COLL_OK and coll.epoch() == 3


@pytest.mark.parametrize("enc", [0, 1])
def test_unpublished_line_times_out_with_status(cd, enc):
    """A line that never gets its readiness value: the consumer gives up
    after the bound, latches COLL_ERR_TIMEOUT with the rank, and the context
    stays usable."""
    import torch

    n, count = 4, 4 * 480
    coll = make(cd, cd.ALLREDUCE, n, count, encoding=enc, path=cd.COLL_PATH_STREAMED,
                algorithm=cd.COLL_ONESHOT, timeout_ns=2_000_000)
    xs, ins, outs = buffers(coll, n, seed=8)
    lines = torch.tensor([3], dtype=torch.int64, device="cuda")
    kind = torch.tensor([0], dtype=torch.int32, device="cuda")
    poison = torch.tensor([0x4880], dtype=torch.int16, device="cuda")
    for r in range(n):
        if r == 2:
            cd.coll_stage_withheld(coll.spec, r, ins[r], lines, kind, poison)
        else:
            coll.stage(r, ins[r])
    coll.run(None, outs)
    code, rank, line = coll.status()
    assert code == cd.COLL_ERR_TIMEOUT and rank == 2 and line >= 0
    # the next epoch works
    coll.run(ins, outs)
    check(coll, outs, oracle.allreduce(xs), n)


@pytest.mark.parametrize("enc", [0, 1])
def test_graph_replay_advances_epoch_on_device(cd, enc):
    """coll_run captured once in a CUDA graph: each replay uses the next
    epoch and slot (the epoch lives on the device)."""
    import torch

    n, count = 8, 8 * 512
    coll = make(cd, cd.ALLREDUCE, n, count, encoding=enc, path=cd.COLL_PATH_FUSED)
    _, ins, outs = buffers(coll, n, seed=9)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        coll.run(ins, outs, stream=s)
    for rep in range(4):
        xs = [synth.normal_bf16(90 + rep, count, r) for r in range(n)]
        for r in range(n):
            ins[r].copy_(to_dev(xs[r]))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        check(coll, outs, oracle.allreduce(xs), n)
    assert coll.epoch() == 5


@pytest.mark.parametrize("n,count", [(8, 8 * 1000), (8, 8 * 60 * 1024 + 64), (3, 3000),
                                     (2, 2 * 4096), (8, 8 * 60 * 300)])
@pytest.mark.parametrize("shape", [None, "16,1,1", "64,3,0", "32,40,1", "256,8,1", "64,4,1,1", "16,2,0,1", "32,4,1,2", "128,6,2,2",
                                   "64,3,0,0,-1,1", "32,40,1,0,-1,1", "64,4,1,1,-1,1", "128,6,2,2,-1,1"])
def test_composed_twoshot_matches_the_oracle(cd, n, count, shape, monkeypatch):
    """The one-launch twoshot: bit-exact against the oracle over several
    epochs, scheduled by columns (the default) for several chunk sizes and
    launch shapes, and (sixth field 1) as the queue of stage / fold / gather
    tasks per chunk with several lags; with and without dropping consumed
    lines from L2."""
    if shape is not None:
        monkeypatch.setenv("COLL_COMPOSED_SHAPE", shape)
    coll = make(cd, cd.ALLREDUCE, n, count, encoding=cd.COLL_LL128,
                algorithm=cd.COLL_TWOSHOT, path=cd.COLL_PATH_COMPOSED)
    _, ins, outs = buffers(coll, n, seed=10)
    for e in range(1, 4):
        xs = [synth.normal_bf16(100 + e, count, n, r) for r in range(n)]
        for r in range(n):
            ins[r].copy_(to_dev(xs[r]))
        coll.run(ins, outs)
        check(coll, outs, oracle.allreduce(xs), n)
        assert coll.epoch() == e + 1


@pytest.mark.parametrize("name,n,count", [("ALLREDUCE", 8, 8 * 60 * 5000 + 64),
                                          ("ALLREDUCE", 3, 3 * 60 * 4000 + 8),
                                          ("REDUCE_SCATTER", 8, 8 * 60 * 5000 + 64),
                                          ("ALLGATHER", 8, 8 * 60 * 5000 + 64),
                                          ("ALLTOALL", 8, 8 * 60 * 5000)])
@pytest.mark.parametrize("shape", ["64,1,1,2,-1,0,16,1", "64,1,1,2,-1,0,32,3", "32,1,1,0,-1,0,16,1",
                                   "128,1,1,2,-1,0,16,2", "64,1,1,1,-1,0,16,40",
                                   "64,1,1,2,-1,0,0,2,8", "64,1,1,2,-1,0,16,1,8",
                                   "32,1,1,0,-1,0,16,1,4", "64,1,1,2,-1,0,0,2,3",
                                   "128,1,1,2,-1,0,32,2,5", "16,1,1,2,-1,0,0,2,64"])
def test_composed_short_tail_columns(cd, name, n, count, shape, monkeypatch):
    """Columns of several lengths: each CTA's first column is one of a
    staggered group (ninth field G: 1/G, 2/G, .. of a chunk, at least a row),
    then chunks of the chunk size, and the last columns the CTAs take the
    tail size (seventh field), over the last few half-rounds of the
    co-resident CTAs' work (eighth field; 40 puts every later chunk in the
    tail).  Bit-exact over several epochs across every boundary and the
    ragged end."""
    monkeypatch.setenv("COLL_COMPOSED_SHAPE", shape)
    triple = getattr(cd, name)
    opts = dict(encoding=cd.COLL_LL128, path=cd.COLL_PATH_COMPOSED)
    if name == "ALLREDUCE":
        opts["algorithm"] = cd.COLL_TWOSHOT
    coll = make(cd, triple, n, count, **opts)
    _, ins, outs = buffers(coll, n, seed=45)
    for e in range(1, 4):
        xs = [synth.random_bits16(700 + e, coll.elems(r)[0], n, r) if name in ("ALLGATHER", "ALLTOALL")
              else synth.normal_bf16(700 + e, coll.elems(r)[0], n, r) for r in range(n)]
        for r in range(n):
            ins[r][:xs[r].size].copy_(to_dev(xs[r]))
        coll.run(ins, outs)
        check(coll, outs, expected(cd, triple, xs, count), n)
        assert coll.epoch() == e + 1


@pytest.mark.parametrize("n,count", [(8, 8 * 60 * 1024 + 64), (3, 3000), (8, 24), (2, 2 * 4096),
                                     (8, 8 * 60 * 300)])
@pytest.mark.parametrize("shape", [None, "16,1,1", "64,3,0", "32,5,1,2", "128,40,1,1", "16,1,1,0,-1,1",
                                   "128,40,1,1,-1,1"])
def test_composed_all_gather(cd, n, count, shape, monkeypatch):
    """The one-launch all-gather: each source stages its packed segment, each
    destination copies every source's chunk (the N-th copy drops the staged
    lines); bit-exact over several epochs, ragged last partitions included."""
    if shape is not None:
        monkeypatch.setenv("COLL_COMPOSED_SHAPE", shape)
    coll = make(cd, cd.ALLGATHER, n, count, encoding=cd.COLL_LL128, path=cd.COLL_PATH_COMPOSED)
    _, ins, outs = buffers(coll, n, seed=44)
    for e in range(1, 4):
        xs = [synth.random_bits16(600 + e, coll.elems(r)[0], n, r) for r in range(n)]
        for r in range(n):
            if xs[r].size:
                ins[r][:xs[r].size].copy_(to_dev(xs[r]))
        coll.run(ins, outs)
        check(coll, outs, oracle.all_gather(xs, count), n)
        assert coll.epoch() == e + 1


@pytest.mark.parametrize("name,n,count", [("ALLREDUCE", 8, 8 * 60 * 1024 + 64),
                                          ("ALLREDUCE", 3, 3 * 60 * 700),
                                          ("REDUCE_SCATTER", 8, 8 * 60 * 1024 + 64),
                                          ("ALLTOALL", 8, 8 * 60 * 512), ("ALLTOALL", 4, 4 * 1000)])
@pytest.mark.parametrize("min_chunk_slots,shape", [(2, "16,1,1"), (3, "16,2,1"), (5, "64,40,1"),
                                                   (4, "32,3,0"), (9, None), (40, "16,8,1,2"),
                                                   (3, "16,2,1,0,-1,1"), (9, "64,40,1,0,-1,1")])
def test_composed_cycling_staging(cd, name, n, count, min_chunk_slots, shape, monkeypatch):
    """Purlin §4.1 bounded staging: each rank's staging image holds only a few
    chunk slots (min_chunk_slots of the 16-line chunk).  By columns, each CTA
    owns a slot and reuses it column after column; in the queue schedule
    (sixth field 1) chunks cycle through the slots, a stage waiting for the
    readers of its slot's previous chunk and a fold for the gathers of its
    published slot's previous chunk.  Lines carry epoch + the column or chunk
    index (§4.2).  Bit-exact over several epochs, every run advances the epoch
    by an odd step, and stale lines from the previous cycles and runs are
    never taken."""
    if shape is not None:
        monkeypatch.setenv("COLL_COMPOSED_SHAPE", shape)
    triple = getattr(cd, name)
    opts = dict(encoding=cd.COLL_LL128, path=cd.COLL_PATH_COMPOSED,
                staging_bytes=min_chunk_slots * n * 16 * 128)
    if name == "ALLREDUCE":
        opts["algorithm"] = cd.COLL_TWOSHOT
    coll = make(cd, triple, n, count, **opts)
    _, ins, outs = buffers(coll, n, seed=43)
    last = coll.epoch()
    for e in range(1, 5):
        xs = [synth.random_bits16(500 + e, count, n, r) if name == "ALLTOALL"
              else synth.normal_bf16(500 + e, count, n, r) for r in range(n)]
        for r in range(n):
            ins[r].copy_(to_dev(xs[r]))
        coll.run(ins, outs)
        check(coll, outs, expected(cd, triple, xs, count), n)
        now = coll.epoch()
        assert (now - last) % 2 == 1, (last, now)
        last = now


@pytest.mark.parametrize("name", ["ALLREDUCE", "REDUCE_SCATTER", "ALLGATHER", "ALLTOALL"])
@pytest.mark.parametrize("n,count", [(1, 8), (1, 4096), (2, 16), (2, 2 * 120 + 16), (8, 64)])
def test_composed_degenerate_sizes(cd, name, n, count):
    """The composed launch at its edges: one rank (the fold of one value is
    that value; every copy is the identity), partitions shorter than one
    LL128 line, and a ragged last line; then an empty run, which only moves
    the epoch."""
    triple = getattr(cd, name)
    opts = dict(encoding=cd.COLL_LL128, path=cd.COLL_PATH_COMPOSED)
    if name == "ALLREDUCE":
        opts["algorithm"] = cd.COLL_TWOSHOT
    coll = make(cd, triple, n, count, **opts)
    for e in range(1, 3):
        xs, ins, outs = buffers(coll, n, seed=50 + e, dist="bits" if name in
                                ("ALLGATHER", "ALLTOALL") else "normal", tag=count)
        coll.run(ins, outs)
        check(coll, outs, expected(cd, triple, xs, count), n)
        assert coll.epoch() == e + 1
    empty = make(cd, triple, n, 0, **opts)
    outs0 = [empty_dev(0) for _ in range(n)]
    empty.run([empty_dev(0) for _ in range(n)], outs0)
    code, _, _ = empty.status()
    assert code == cd.COLL_OK and empty.epoch() == 2


@pytest.mark.parametrize("enc,reset", [(0, 0), (0, 1), (0, 3), (1, 2), (2, 0), (2, 1), (2, 3)])
@pytest.mark.parametrize("path", [1, 2, 3])
def test_four_rotating_slots(cd, enc, reset, path):
    """Four staging slots (flash-comm §4.2): run e stages into slot e mod 4
    (the slot's lines carry epoch e), every run stays bit-exact, and the
    re-arm rules hold with the longer rotation."""
    if path == 3 and enc != 1:
        pytest.skip("the composed launch is LL128 only")
    n, count = 8, 8 * 1200
    coll = make(cd, cd.ALLREDUCE, n, count, encoding=enc, algorithm=cd.COLL_TWOSHOT,
                path=path, reset_mode=reset, slots=4)
    _, ins, outs = buffers(coll, n, seed=30)
    for e in range(1, 10):
        xs = [synth.normal_bf16(300 + e, count, r) for r in range(n)]
        for r in range(n):
            ins[r].copy_(to_dev(xs[r]))
        coll.run(ins, outs)
        check(coll, outs, oracle.allreduce(xs), n)
        assert coll.epoch() == e + 1
        if enc == 1:
            raw, lines, lb = read_lines(coll, 0, e % 4, 3, 5)
            seqs = raw.reshape(lines, lb)[:, 120:128].copy().view(np.uint64).ravel()
            assert np.all(seqs == e), f"epoch {e}: slot {e % 4} holds {set(seqs.tolist())}"


@pytest.mark.parametrize("name,n,count", [("REDUCE_SCATTER", 8, 8 * 60 * 1024 + 64),
                                          ("REDUCE_SCATTER", 3, 3000), ("REDUCE_SCATTER", 8, 24),
                                          ("ALLTOALL", 8, 8 * 60 * 512), ("ALLTOALL", 4, 4 * 1000),
                                          ("ALLTOALL", 2, 2 * 8)])
@pytest.mark.parametrize("shape", [None, "16,1,1", "64,3,0", "32,5,1,2", "32,5,1,2,-1,1"])
def test_composed_reduce_scatter_and_all_to_all(cd, name, n, count, shape, monkeypatch):
    """The one-launch form of reduce-scatter (stage, fold into the outputs)
    and all-to-all (stage, copy), bit-exact over several epochs."""
    if shape is not None:
        monkeypatch.setenv("COLL_COMPOSED_SHAPE", shape)
    triple = getattr(cd, name)
    coll = make(cd, triple, n, count, encoding=cd.COLL_LL128, path=cd.COLL_PATH_COMPOSED)
    _, ins, outs = buffers(coll, n, seed=41)
    for e in range(1, 4):
        xs = [synth.random_bits16(400 + e, count, n, r) if name == "ALLTOALL"
              else synth.normal_bf16(400 + e, count, n, r) for r in range(n)]
        for r in range(n):
            ins[r].copy_(to_dev(xs[r]))
        coll.run(ins, outs)
        check(coll, outs, expected(cd, triple, xs, count), n)
        assert coll.epoch() == e + 1


@pytest.mark.parametrize("enc,path", [(0, 1), (2, 1), (0, 2), (1, 2), (1, 3)])
def test_dependent_launches_chain(cd, enc, path):
    """Small runs are dependent launches (one launch, or stream-ordered
    kernels): each kernel must wait for the kernel before it and see all of
    its writes.  Chain A -> B -> A, each run's
    inputs being the previous run's outputs, then a plain torch kernel
    (an XOR of low mantissa bits) between two runs; eagerly and replayed
    from a CUDA graph, bit-exact against the oracle applied step by step."""
    import torch

    n, count = 8, 4096
    kw = dict(encoding=enc, path=path)
    if path == 3:
        kw["algorithm"] = cd.COLL_TWOSHOT  # the composed launch's all-reduce
    a = make(cd, cd.ALLREDUCE, n, count, **kw)
    b = make(cd, cd.ALLREDUCE, n, count, **kw)
    assert a.plan()["dependent_launch"] == 1 and b.plan()["dependent_launch"] == 1
    masks = [0x0011 * (r + 1) & 0x007F for r in range(n)]
    mask_d = [torch.tensor(m, dtype=torch.int16, device="cuda") for m in masks]
    xs, ins, o1 = buffers(a, n, seed=31, dist="uniform1")
    o2 = [empty_dev(count) for _ in range(n)]
    o3 = [empty_dev(count) for _ in range(n)]
    x4 = [empty_dev(count) for _ in range(n)]
    o5 = [empty_dev(count) for _ in range(n)]

    def chain(s):
        a.run(ins, o1, stream=s)
        b.run(o1, o2, stream=s)
        a.run(o2, o3, stream=s)
        with torch.cuda.stream(s):
            for r in range(n):
                torch.bitwise_xor(o3[r], mask_d[r], out=x4[r])
        b.run(x4, o5, stream=s)

    def expect(xs):
        y1 = oracle.allreduce(xs)
        y2 = oracle.allreduce(y1)
        y3 = oracle.allreduce(y2)
        y4 = [y3[r] ^ np.uint16(masks[r]) for r in range(n)]
        return y3, oracle.allreduce(y4)

    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    chain(s)
    s.synchronize()
    y3, y5 = expect(xs)
    check(a, o3, y3, n)
    check(b, o5, y5, n)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chain(s)
    for rep in range(3):
        xs = [synth.uniform_bf16(40 + rep, count, -1.0, 1.0, r) for r in range(n)]
        for r in range(n):
            ins[r].copy_(to_dev(xs[r]))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        y3, y5 = expect(xs)
        check(a, o3, y3, n)
        check(b, o5, y5, n)


def test_launch_floor_leaves_the_run_state_alone(cd):
    """coll_launch_floor enqueues an empty kernel in a one-launch spec's
    configuration (fused, or composed by columns): the epoch and the next
    run's result are unchanged; specs with no one-launch path refuse it."""
    import torch

    n, count = 8, 4096
    for kw in (dict(encoding=cd.COLL_LL8, path=cd.COLL_PATH_FUSED),
               dict(encoding=cd.COLL_LL128, algorithm=cd.COLL_TWOSHOT,
                    path=cd.COLL_PATH_COMPOSED),
               dict(encoding=cd.COLL_LL128, algorithm=cd.COLL_TWOSHOT,
                    path=cd.COLL_PATH_COMPOSED, staging_bytes=4 * n * 16 * 128)):
        coll = make(cd, cd.ALLREDUCE, n, count, **kw)
        xs, ins, outs = buffers(coll, n, seed=60)
        before = coll.epoch()
        s = torch.cuda.current_stream()
        for _ in range(3):
            cd.coll_launch_floor(coll.spec, s)
        torch.cuda.synchronize()
        assert coll.epoch() == before
        coll.run(ins, outs)
        check(coll, outs, oracle.allreduce(xs), n)
        coll.close()
    coll = make(cd, cd.ALLREDUCE, n, count, encoding=cd.COLL_LL128, path=cd.COLL_PATH_STREAMED)
    with pytest.raises(cd.CollError) as e:
        cd.coll_launch_floor(coll.spec, torch.cuda.current_stream())
    assert e.value.status == cd.COLL_ERR_UNSUPPORTED
    coll.close()


@pytest.mark.parametrize("name", ["REDUCE_SCATTER", "ALLGATHER", "ALLTOALL", "REDUCE_SCATTER_V",
                                  "ALLGATHER_V", "ALLTOALL_V"])
def test_composed_collectives_on_four_slots(cd, name):
    """Every collective of the composed launch with four rotating staging
    slots (flash-comm §4.2): run e stages into slot e mod 4; nine epochs
    with new inputs each time stay bit-exact against the oracle."""
    n = 8
    triple = getattr(cd, name)
    kw = dict(encoding=cd.COLL_LL128, path=cd.COLL_PATH_COMPOSED, slots=4)
    if name.endswith("_V"):
        base = [b // 2 for b in synth.zipf_split(1 << 21, n)]
        v = [synth.rotate_right(base, p + 1) for p in range(n)] if name == "ALLTOALL_V" else base
        count = 0 if name == "ALLTOALL_V" else int(sum(base))
        kw["vcounts"] = v
    else:
        v, count = None, 8 * 60 * 700
    coll = make(cd, triple, n, count, **kw)
    _, ins, outs = buffers(coll, n, seed=61)
    for e in range(1, 10):
        sizes = [coll.elems(r)[0] for r in range(n)]
        bits = name not in ("REDUCE_SCATTER", "REDUCE_SCATTER_V")
        xs = [synth.random_bits16(1000 + e, sizes[r], n, r) if bits
              else synth.normal_bf16(1000 + e, sizes[r], n, r) for r in range(n)]
        for r in range(n):
            if sizes[r]:
                ins[r][:sizes[r]].copy_(to_dev(xs[r]))
        coll.run(ins, outs)
        if name == "REDUCE_SCATTER_V":
            want = oracle.reduce_scatter_v(xs, v)
        elif name == "ALLGATHER_V":
            want = oracle.all_gather_v(xs, v)
        elif name == "ALLTOALL_V":
            want = oracle.all_to_all_v(xs, v)
        else:
            want = expected(cd, triple, xs, count)
        check(coll, outs, want, n)
        assert coll.epoch() == e + 1
    coll.close()

"""fp32 tensors (flash-comm §4.1 admits bf16 and fp32) on the GPU against the
oracle, bit for bit: all-reduce in every encoding, algorithm and launch path
(the composed launch included), reduce-scatter, the copies, the V forms, the
staged bytes, and inputs holding the sentinel's reserved word, NaNs with
payloads and infinities."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import empty_dev, read_lines

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cd():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import collective_datapath_gb300 as m

    return m


def dev32(x):
    import torch

    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.uint32).view(np.int32)).cuda()


def host32(t, n):
    return t.cpu().numpy().view(np.uint32)[:n].copy()


def inputs(n, elems, seed, specials=True):
    xs = [synth.normal_f32(seed, elems, n, r) for r in range(n)]
    if specials and elems:
        xs[0][::53] = 0xFFFFFFFF
        xs[n - 1][7::61] = 0x7FC00123
        xs[n // 2][3::89] = 0x7F800000
    return xs


def run(cd, coll, xs, n, want, epochs=2):
    import torch

    ins = [dev32(x) if x.size else empty_dev(0) for x in xs]
    outs = [torch.full((max(coll.elems(r)[1], 4),), 0x5A5A5A5A, dtype=torch.int32,
                       device="cuda") for r in range(n)]
    for _ in range(epochs):
        coll.run(ins, outs)
        code, rank, line = coll.status()
        assert code == cd.COLL_OK, (code, rank, line)
        for r in range(n):
            got = host32(outs[r], want[r].size)
            if not np.array_equal(got, want[r]):
                bad = np.flatnonzero(got != want[r])
                raise AssertionError(f"rank {r}: {bad.size} mismatches, first at {bad[0]}: "
                                     f"got {got[bad[0]]:#010x} want {want[r][bad[0]]:#010x}")


@pytest.mark.parametrize("enc", [0, 1, 2])
@pytest.mark.parametrize("algo", [1, 2])
@pytest.mark.parametrize("path", [1, 2, 3])
@pytest.mark.parametrize("n,count", [(8, 8 * 1000), (3, 1000), (2, 4096)])
def test_allreduce_f32(cd, enc, algo, path, n, count):
    if path == 3 and (enc != 1 or algo != 2):
        pytest.skip("the composed launch is the LL128 twoshot")
    coll = cd.Collective(cd.ALLREDUCE, n, count, dtype=cd.COLL_F32, encoding=enc,
                         algorithm=algo, path=path)
    xs = inputs(n, count, 31 + count)
    run(cd, coll, xs, n, oracle.allreduce_f32(xs))


@pytest.mark.parametrize("enc", [0, 1, 2])
@pytest.mark.parametrize("path", [1, 2])
def test_reduce_scatter_and_copies_f32(cd, enc, path):
    n, count = 8, 8 * 600 + 64
    san = (lambda x: oracle.sent_sanitize_f32(x)) if enc == 2 else (lambda x: x)
    xs = inputs(n, count, 32)
    rs = cd.Collective(cd.REDUCE_SCATTER, n, count, dtype=cd.COLL_F32, encoding=enc, path=path)
    run(cd, rs, xs, n, oracle.reduce_scatter_f32(xs))
    shards = [inputs(n, oracle.shard_len(count, n, r), 33)[r] for r in range(n)]
    ag = cd.Collective(cd.ALLGATHER, n, count, dtype=cd.COLL_F32, encoding=enc, path=path)
    run(cd, ag, shards, n, [np.concatenate([san(s) for s in shards])] * n)
    m = 240
    a2a_in = inputs(n, n * m, 34)
    a2a = cd.Collective(cd.ALLTOALL, n, n * m, dtype=cd.COLL_F32, encoding=enc, path=path)
    want = [np.concatenate([san(a2a_in[p][d * m:(d + 1) * m]) for p in range(n)])
            for d in range(n)]
    run(cd, a2a, a2a_in, n, want)


@pytest.mark.parametrize("enc", [0, 1, 2])
def test_v_collectives_f32(cd, enc):
    n = 8
    base = [b // 4 for b in synth.zipf_split(1 << 20, n)]      # fp32 elements
    san = (lambda x: oracle.sent_sanitize_f32(x)) if enc == 2 else (lambda x: x)
    xs = inputs(n, sum(base), 35)
    rsv = cd.Collective(cd.REDUCE_SCATTER_V, n, sum(base), dtype=cd.COLL_F32, encoding=enc,
                        vcounts=base)
    ar = oracle.allreduce_f32(xs)[0]
    off = np.concatenate([[0], np.cumsum(base)])
    run(cd, rsv, xs, n, [ar[off[r]:off[r + 1]] for r in range(n)])
    parts = [inputs(n, base[r], 36)[r] for r in range(n)]
    agv = cd.Collective(cd.ALLGATHER_V, n, sum(base), dtype=cd.COLL_F32, encoding=enc,
                        vcounts=base)
    run(cd, agv, parts, n, [np.concatenate([san(p) for p in parts])] * n)
    v = [synth.rotate_right(base, p + 1) for p in range(n)]
    srcs = inputs(n, sum(base), 37)
    a2av = cd.Collective(cd.ALLTOALL_V, n, 0, dtype=cd.COLL_F32, encoding=enc, vcounts=v)
    starts = [np.concatenate([[0], np.cumsum(v[p])]) for p in range(n)]
    want = [np.concatenate([san(srcs[p][starts[p][d]:starts[p][d + 1]]) for p in range(n)])
            for d in range(n)]
    run(cd, a2av, srcs, n, want)


@pytest.mark.parametrize("enc", [0, 1, 2])
def test_staged_f32_bytes(cd, enc):
    """coll_stage writes the oracle's lines: for LL8 / LL128 the bf16 line
    encodings of the same bytes, for sentinel packs the fp32 packs."""
    import torch

    n, count = 4, 4 * 500
    coll = cd.Collective(cd.ALLREDUCE, n, count, dtype=cd.COLL_F32, encoding=enc,
                         path=cd.COLL_PATH_STREAMED)
    xs = inputs(n, count, 38)
    ins = [dev32(x) for x in xs]
    for r in range(n):
        coll.stage(r, ins[r])
    torch.cuda.synchronize()
    for r in range(n):
        for k in range(n):
            raw, lines, lb = read_lines(coll, 0, 1, r, k)
            b, ln = oracle.shard_begin(count, n, k), oracle.shard_len(count, n, k)
            seg = xs[r][b:b + ln]
            if enc == 2:
                want = oracle.sent_encode_f32(seg).view(np.uint8)
            elif enc == 0:
                want = oracle.ll8_encode(seg.view(np.uint16), 1).view(np.uint8)
            else:
                want = oracle.ll128_encode(seg.view(np.uint16), 1)
            assert np.array_equal(raw, want), (r, k)


@pytest.mark.parametrize("path", [2, 3])
def test_allreduce_f32_32mib_sampled(cd, path):
    import torch

    n, count = 8, 32 * 1024 * 1024 // 4
    g = torch.Generator(device="cuda")
    g.manual_seed(39)
    ins = [torch.randn(count, generator=g, device="cuda").view(torch.int32) for _ in range(n)]
    outs = [torch.empty(count, dtype=torch.int32, device="cuda") for _ in range(n)]
    coll = cd.Collective(cd.ALLREDUCE, n, count, dtype=cd.COLL_F32, encoding=cd.COLL_LL128,
                         algorithm=cd.COLL_TWOSHOT, path=path)
    for _ in range(2):
        coll.run(ins, outs)
    code, rank, line = coll.status()
    assert code == cd.COLL_OK, (code, rank, line)
    for r in range(1, n):
        assert torch.equal(outs[r], outs[0])
    pos = np.unique(np.random.Generator(np.random.Philox(39)).integers(0, count, 20000))
    m = oracle.shard_elems(count, n)
    pos = np.unique(np.concatenate([pos, [k * m + d for k in range(1, n) for d in (-1, 0, 1)],
                                    [0, count - 1]]))
    idx = torch.from_numpy(pos).cuda()
    cols = [ins[r][idx].cpu().numpy().view(np.uint32) for r in range(n)]
    want = oracle.allreduce_f32(cols)[0]
    got = outs[0][idx].cpu().numpy().view(np.uint32)
    assert np.array_equal(got, want)
    del coll, outs, ins
    torch.cuda.empty_cache()

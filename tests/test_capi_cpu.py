"""CPU checks of the C ABI: the library loads, exports what include/coll.h
declares, validates arguments, and derives work lists that -- interpreted
line by line on the CPU with the oracle's encoders and fold -- produce exactly
the oracle's collective results.  No GPU, no kernel launch."""
from __future__ import annotations

import os
import re

import numpy as np
import pytest

import oracle
import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def cd():
    import importlib.util

    spec = importlib.util.spec_from_file_location(
        "_coll_build", os.path.join(ROOT, "collective_datapath_gb300", "_build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    b.build()
    import collective_datapath_gb300 as m

    return m


def declared_functions() -> list[str]:
    text = open(os.path.join(ROOT, "include", "coll.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(coll_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(cd):
    import ctypes

    lib = ctypes.CDLL(cd.library_path())
    names = declared_functions()
    assert len(names) >= 19
    for name in names:
        assert hasattr(lib, name), f"{name} declared in coll.h but not exported"
    assert sorted(cd.EXPORTS) == names


def test_argument_validation(cd):
    with pytest.raises(cd.CollError) as e:
        cd.coll_spec_create(cd.COLL_PACKED, cd.COLL_PACKED, cd.COLL_REDUCE, 8, 64)
    assert e.value.status == cd.COLL_ERR_UNSUPPORTED
    with pytest.raises(cd.CollError) as e:
        cd.coll_spec_create(*cd.ALLREDUCE, 8, 12)          # not 16-byte aligned
    assert e.value.status == cd.COLL_ERR_ALIGN
    for bad_n in (0, 9):
        with pytest.raises(cd.CollError) as e:
            cd.coll_spec_create(*cd.ALLREDUCE, bad_n, 64)
        assert e.value.status == cd.COLL_ERR_UNSUPPORTED
    with pytest.raises(cd.CollError) as e:
        cd.coll_spec_create(*cd.ALLTOALL, 8, 24)           # unequal partitions
    assert e.value.status == cd.COLL_ERR_ALIGN
    with pytest.raises(cd.CollError) as e:
        cd.coll_spec_create(*cd.ALLREDUCE, 8, 64, encoding=7)
    assert e.value.status == cd.COLL_ERR_UNSUPPORTED
    s = cd.coll_spec_create(*cd.ALLREDUCE, 8, 64)
    with pytest.raises(cd.CollError) as e:                 # not bound yet
        cd.coll_stage(s, 0, 0x1000, stream=0)
    assert e.value.status == cd.COLL_ERR_STATE
    assert cd.coll_workspace_bytes(s) > 0
    cd.coll_destroy(s)


# ---- CPU interpretation of the derived schedule --------------------------------

def _encode(enc, x, epoch):
    if enc == 2:
        return oracle.sent_encode(x)
    return oracle.ll8_encode(x, epoch) if enc == 0 else \
        oracle.ll128_encode(x, epoch).reshape(-1, 128)


def _decode(enc, lines, elems, epoch):
    if enc == 2:
        out, rej = oracle.sent_decode(lines, elems)
    else:
        out, rej = (oracle.ll8_decode(lines, elems, epoch) if enc == 0 else
                    oracle.ll128_decode(np.ascontiguousarray(lines).ravel(), elems, epoch))
    assert rej == 0
    return out


def _fold_units(xs, f32):
    """Oracle fold of decoded 16-bit units (fp32: pairs of units)."""
    if not f32:
        return oracle.allreduce(xs)[0]
    ys = [np.ascontiguousarray(x).view(np.uint32) for x in xs]
    return oracle.allreduce_f32(ys)[0].view(np.uint16)


def _encode_units(enc, x, epoch, f32):
    if enc == 2 and f32:
        return oracle.sent_encode_f32(np.ascontiguousarray(x).view(np.uint32))
    return _encode(enc, x, epoch)


def _decode_units(enc, lines, elems, epoch, f32):
    if enc == 2 and f32:
        out, rej = oracle.sent_decode_f32(lines, elems // 2)
        assert rej == 0
        return out.view(np.uint16)
    return _decode(enc, lines, elems, epoch)


def interpret(cd, spec, enc, n, ins, epoch=5, f32=False):
    """Run the derived items on the CPU: stage, phase 1, phase 2.  `ins` are
    16-bit units (an fp32 element is two of them)."""
    st = cd.coll_debug_items(spec, 0)
    p1 = cd.coll_debug_items(spec, 1)
    p2 = cd.coll_debug_items(spec, 2)
    width = 1 if enc != 1 else 128
    dt = np.uint64 if enc != 1 else np.uint8
    img_lines = int(max([r[7] + r[5] for r in st] + [4]))
    ag_lines = int(max([r[8] + r[5] for r in p1 if r[1] & 1] + [4]))
    P = [np.zeros((img_lines, width) if enc == 1 else img_lines, dtype=dt) for _ in range(n)]
    AG = [np.zeros((ag_lines, width) if enc == 1 else ag_lines, dtype=dt) for _ in range(n)]
    for rank, _, _, _, _, nl, ne, dst_line, in_elem, _ in st:
        assert dst_line % 4 == 0
        P[rank][dst_line:dst_line + nl] = _encode_units(enc, ins[rank][in_elem:in_elem + ne],
                                                        epoch, f32)
    outs = [np.full(cd.coll_buffer_elems(spec, r)[1] * (2 if f32 else 1), 0xDEAD,
                    dtype=np.uint16) for r in range(n)]
    written = [np.zeros(o.size, dtype=np.int32) for o in outs]

    def run(items, images):
        for kind, flags, dst, src, readers, nl, ne, sl, off, ctr in items:
            assert sl % 4 == 0
            if kind == 0:
                xs = [_decode_units(enc, images[q][sl:sl + nl], ne, epoch, f32) for q in range(n)]
                res = _fold_units(xs, f32)
            else:
                res = _decode_units(enc, images[src][sl:sl + nl], ne, epoch, f32)
            if flags & 1:
                AG[dst][off:off + nl] = _encode_units(enc, res, epoch, f32)
            else:
                outs[dst][off:off + ne] = res
                written[dst][off:off + ne] += 1

    run(p1, P)
    run(p2, AG)
    for w in written:
        assert np.all(w == 1), "every output element written exactly once"
    return outs


CASES = [
    # (triple name, n, count, enc, algorithm, path)
    ("ALLREDUCE", 2, 512, 0, 1, 1),
    ("ALLREDUCE", 8, 8 * 4096, 0, 1, 1),
    ("ALLREDUCE", 8, 8 * 4096, 0, 2, 1),
    ("ALLREDUCE", 8, 8 * 4096, 1, 2, 2),
    ("ALLREDUCE", 8, 16 * 7168, 1, 1, 1),
    ("ALLREDUCE", 3, 1000, 1, 2, 2),        # ragged partitions
    ("ALLREDUCE", 8, 24, 0, 2, 1),          # empty partitions
    ("ALLREDUCE", 1, 64, 0, 1, 1),
    ("REDUCE_SCATTER", 8, 8 * 3000, 1, 0, 2),
    ("REDUCE_SCATTER", 5, 5 * 8 * 7 + 16, 0, 0, 1),
    ("ALLGATHER", 8, 8 * 2048, 0, 0, 2),
    ("ALLGATHER", 4, 4 * 104 + 8, 1, 0, 1),
    ("ALLTOALL", 8, 8 * 960, 1, 0, 2),
    ("ALLTOALL", 4, 4 * 64, 0, 0, 1),
    ("ALLREDUCE", 8, 8 * 4096, 2, 1, 1),   # sentinel packs
    ("ALLREDUCE", 8, 8 * 4096, 2, 2, 2),
    ("ALLREDUCE", 3, 1000, 2, 2, 1),
    ("REDUCE_SCATTER", 5, 5 * 8 * 7 + 16, 2, 0, 2),
    ("ALLGATHER", 4, 4 * 104 + 8, 2, 0, 1),
    ("ALLTOALL", 8, 8 * 960, 2, 0, 2),
]


def _sweep_cases(k: int = 120, seed: int = 2024) -> list[tuple]:
    """Seeded cases over 1..8 ranks (odd counts included), every collective,
    encoding, algorithm and launch path, with sizes from one 16-byte chunk
    to a few KiB per rank (ragged and empty partitions among them)."""
    rng = np.random.default_rng(seed)
    kinds = ["ALLREDUCE", "REDUCE_SCATTER", "ALLGATHER", "ALLTOALL"]
    out = []
    for i in range(k):
        name = kinds[i % len(kinds)]
        n = int(rng.integers(1, 9))
        enc = int(rng.integers(0, 3))
        path = int(rng.integers(1, 3))
        algo = int(rng.integers(1, 3)) if name == "ALLREDUCE" else 0
        # the all-to-all needs equal partitions of whole 16-byte chunks
        count = (n * 8 * int(rng.integers(1, 40)) if name == "ALLTOALL"
                 else 8 * int(rng.integers(1, 600)))
        out.append((name, n, count, enc, algo, path))
    return out


@pytest.mark.parametrize("name,n,count,enc,algo,path", CASES + _sweep_cases())
def test_derived_schedule_computes_the_oracle_result(cd, name, n, count, enc, algo, path):
    triple = getattr(cd, name)
    spec = cd.coll_spec_create(*triple, n, count, encoding=enc, algorithm=algo, path=path)
    try:
        ins = [synth.normal_bf16(3, cd.coll_buffer_elems(spec, r)[0], n, count, r)
               for r in range(n)]
        if enc == 2:                       # a copy delivers the sanitised input
            ins[0][::97] = 0xFFFF
        got = interpret(cd, spec, enc, n, ins)
        san = [oracle.sent_sanitize(x) for x in ins] if enc == 2 else ins
        if name == "ALLREDUCE":
            want = oracle.allreduce(ins)
        elif name == "REDUCE_SCATTER":
            want = oracle.reduce_scatter(ins)
        elif name == "ALLGATHER":
            want = oracle.all_gather(san, count)
        else:
            want = oracle.all_to_all(san)
        for r in range(n):
            assert np.array_equal(got[r], want[r]), f"rank {r}"
    finally:
        cd.coll_destroy(spec)


def test_reset_counters_match_reader_counts(cd):
    """Counted re-arm: every counter is shared by exactly `readers` items."""
    for triple, algo in ((cd.ALLREDUCE, 1), (cd.ALLREDUCE, 2), (cd.ALLGATHER, 0)):
        spec = cd.coll_spec_create(*triple, 8, 8 * 1024, algorithm=algo, path=1)
        for which in (1, 2):
            items = cd.coll_debug_items(spec, which)
            counted = items[(items[:, 1] & 4) != 0]
            if counted.size == 0:
                continue
            ids, uses = np.unique(counted[:, 9], return_counts=True)
            for cid, u in zip(ids, uses):
                readers = counted[counted[:, 9] == cid][:, 4]
                assert np.all(readers == u)
        cd.coll_destroy(spec)


# ---- variable-length (V) collectives ---------------------------------------

def zipf_elems(total_bytes, n):
    return [b // 2 for b in synth.zipf_split(total_bytes, n)]


V_CASES = [
    # (triple name, n, per-rank vector or matrix, enc, path)
    ("REDUCE_SCATTER_V", 8, zipf_elems(8 * 2048 * 2, 8), 1, 2),
    ("REDUCE_SCATTER_V", 8, zipf_elems(8 * 2048 * 2, 8), 0, 1),
    ("REDUCE_SCATTER_V", 3, [8, 0, 488], 1, 1),            # an empty partition
    ("ALLGATHER_V", 8, zipf_elems(8 * 1024 * 2, 8), 0, 2),
    ("ALLGATHER_V", 8, zipf_elems(8 * 1024 * 2, 8), 1, 1),
    ("ALLGATHER_V", 4, [64, 8, 0, 1208], 1, 2),
    ("ALLTOALL_V", 8, [synth.rotate_right(zipf_elems(8 * 960 * 2, 8), p + 1)
                       for p in range(8)], 1, 2),
    ("ALLTOALL_V", 8, [synth.rotate_right(zipf_elems(8 * 512 * 2, 8), p + 1)
                       for p in range(8)], 0, 1),
    ("ALLTOALL_V", 3, [[8, 0, 240], [0, 0, 16], [128, 64, 8]], 0, 2),
]


def _v_sizes(rng, m: int) -> list[int]:
    """m sizes in whole 16-byte chunks, about a quarter of them zero, not all
    zero."""
    v = 8 * rng.integers(0, 80, size=m)
    v[rng.random(m) < 0.25] = 0
    if not v.any():
        v[int(rng.integers(0, m))] = 8
    return [int(x) for x in v]


def _v_sweep_cases(k: int = 60, seed: int = 7) -> list[tuple]:
    """Seeded V cases over 1..8 ranks, every encoding and launch path, with
    random sizes and empty pieces."""
    rng = np.random.default_rng(seed)
    kinds = ["REDUCE_SCATTER_V", "ALLGATHER_V", "ALLTOALL_V"]
    out = []
    for i in range(k):
        name = kinds[i % len(kinds)]
        n = int(rng.integers(1, 9))
        enc = int(rng.integers(0, 3))
        path = int(rng.integers(1, 3))
        if name == "ALLTOALL_V":
            v = [_v_sizes(rng, n) for _ in range(n)]
        else:
            v = _v_sizes(rng, n)
        out.append((name, n, v, enc, path))
    return out


@pytest.mark.parametrize("name,n,v,enc,path", V_CASES + _v_sweep_cases())
def test_derived_v_schedule_computes_the_oracle_result(cd, name, n, v, enc, path):
    triple = getattr(cd, name)
    count = 0 if name == "ALLTOALL_V" else int(sum(v))
    spec = cd.coll_spec_create(*triple, n, count, encoding=enc, path=path, vcounts=v)
    try:
        ins = [synth.normal_bf16(9, cd.coll_buffer_elems(spec, r)[0], n, r) for r in range(n)]
        got = interpret(cd, spec, enc, n, ins)
        if name == "REDUCE_SCATTER_V":
            want = oracle.reduce_scatter_v(ins, v)
        elif name == "ALLGATHER_V":
            want = oracle.all_gather_v(ins, v)
        else:
            want = oracle.all_to_all_v(ins, v)
        for r in range(n):
            assert got[r].size == want[r].size
            assert np.array_equal(got[r], want[r]), f"rank {r}"
    finally:
        cd.coll_destroy(spec)


@pytest.mark.parametrize("name,n,v", [
    ("ALLTOALL_V", 8, [synth.rotate_right(zipf_elems(8 * 960 * 2, 8), p + 1) for p in range(8)]),
    ("ALLTOALL_V", 3, [[8, 0, 240], [0, 0, 16], [128, 64, 8]]),
    ("ALLTOALL", 4, 4 * 1000),
] + [("ALLTOALL_V", c[1], c[2]) for c in _v_sweep_cases(30, 11) if c[0] == "ALLTOALL_V"]
  + [("ALLTOALL", n, n * 8 * m) for n, m in ((1, 3), (5, 17), (6, 1), (7, 40))])
def test_composed_exchange_table_moves_every_partition(cd, name, n, v):
    """The composed all-to-all (V) reads one piece per (source p, destination
    x) from a table: partition x of p's input goes to destination x after the
    partitions x of sources 0 .. p-1, from lines that lie inside p's staged
    image without overlapping.  Copying by the table alone must give the
    oracle's exchange."""
    triple = getattr(cd, name)
    vec = name == "ALLTOALL_V"
    spec = cd.coll_spec_create(*triple, n, 0 if vec else v, encoding=cd.COLL_LL128,
                               path=cd.COLL_PATH_COMPOSED, vcounts=v if vec else None)
    try:
        ins = [synth.random_bits16(21, cd.coll_buffer_elems(spec, r)[0], n, r) for r in range(n)]
        outs = [np.full(cd.coll_buffer_elems(spec, r)[1], 0xFFFF, dtype=np.uint16)
                for r in range(n)]
        table = cd.coll_debug_items(spec, 3)
        assert len(table) == n * n
        stage = cd.coll_debug_items(spec, 0)
        image_lines = {r: 0 for r in range(n)}
        for it in stage:
            image_lines[int(it[0])] = max(image_lines[int(it[0])], int(it[7] + it[5]))
        used = {r: [] for r in range(n)}
        for p, x, line0, elems, in0, out0, *_ in table.tolist():
            outs[x][out0:out0 + elems] = ins[p][in0:in0 + elems]
            lines = -(-elems // 60)
            # an empty piece holds no line (it may sit on the 4-line boundary
            # just past the image); only pieces with data must lie inside
            if lines:
                used[p].append((line0, line0 + lines))
        for r in range(n):
            spans = sorted(used[r])
            assert all(a[1] <= b[0] for a, b in zip(spans, spans[1:])), spans
            assert not spans or spans[-1][1] <= image_lines[r]
        want = oracle.all_to_all_v(ins, v) if vec else oracle.all_to_all(ins)
        for r in range(n):
            assert np.array_equal(outs[r], want[r]), f"rank {r}"
    finally:
        cd.coll_destroy(spec)
    other = cd.coll_spec_create(*cd.REDUCE_SCATTER, 4, 4 * 64, encoding=cd.COLL_LL128,
                                path=cd.COLL_PATH_COMPOSED)
    assert len(cd.coll_debug_items(other, 3)) == 0
    cd.coll_destroy(other)


def test_composed_path_admits_every_ll128_collective(cd):
    """The composed launch takes the LL128 twoshot all-reduce, the reduce-
    scatter, all-gather, all-to-all and their V forms; other encodings, and
    an all-reduce asked for as a oneshot, are refused.  An all-reduce left on
    algorithm AUTO takes the twoshot there.  Plan only (host)."""
    n = 8
    zipf = zipf_elems(8 * 4096 * 2, n)
    cases = [("ALLREDUCE", 8 * 1200, None), ("REDUCE_SCATTER", 8 * 1200, None),
             ("ALLGATHER", 8 * 1200, None), ("ALLTOALL", 8 * 1200, None),
             ("REDUCE_SCATTER_V", sum(zipf), zipf), ("ALLGATHER_V", sum(zipf), zipf),
             ("ALLTOALL_V", 0, [synth.rotate_right(zipf, p + 1) for p in range(n)])]
    for name, count, v in cases:
        kw = dict(path=cd.COLL_PATH_COMPOSED, vcounts=v)
        s = cd.coll_spec_create(*getattr(cd, name), n, count, encoding=cd.COLL_LL128, **kw)
        plan = cd.coll_debug_plan(s)
        assert plan["path"] == cd.COLL_PATH_COMPOSED, name
        if name == "ALLREDUCE":
            assert plan["algorithm"] == cd.COLL_TWOSHOT
        cd.coll_destroy(s)
        for enc in (cd.COLL_LL8, cd.COLL_SENT):
            with pytest.raises(cd.CollError) as e:
                cd.coll_spec_create(*getattr(cd, name), n, count, encoding=enc, **kw)
            assert e.value.status == cd.COLL_ERR_UNSUPPORTED, (name, enc)
    with pytest.raises(cd.CollError) as e:
        cd.coll_spec_create(*cd.ALLREDUCE, n, 8 * 1200, encoding=cd.COLL_LL128,
                            algorithm=cd.COLL_ONESHOT, path=cd.COLL_PATH_COMPOSED)
    assert e.value.status == cd.COLL_ERR_UNSUPPORTED


def test_v_argument_validation(cd):
    def status_of(*a, **kw):
        with pytest.raises(cd.CollError) as e:
            cd.coll_spec_create(*a, **kw)
        return e.value.status

    assert status_of(*cd.REDUCE_SCATTER_V, 4, 64, vcounts=[16, 16, 16]) == cd.COLL_ERR_INVALID
    assert status_of(*cd.REDUCE_SCATTER_V, 4, 64, vcounts=[16, 16, 16, 8]) == cd.COLL_ERR_INVALID
    assert status_of(*cd.ALLGATHER_V, 4, 64, vcounts=[16, 16, 20, 12]) == cd.COLL_ERR_ALIGN
    assert status_of(*cd.ALLTOALL_V, 2, 0, vcounts=[8, 8, 8]) == cd.COLL_ERR_INVALID
    assert status_of(*cd.ALLGATHER_V, 2, 16) == cd.COLL_ERR_INVALID   # no vcounts
    s = cd.coll_spec_create(*cd.ALLTOALL_V, 2, 0, vcounts=[[8, 16], [0, 24]])
    assert cd.coll_buffer_elems(s, 0) == (24, 8)
    assert cd.coll_buffer_elems(s, 1) == (24, 40)
    cd.coll_destroy(s)


def test_sentinel_needs_a_rearm(cd):
    with pytest.raises(cd.CollError) as e:
        cd.coll_spec_create(*cd.ALLREDUCE, 8, 64, encoding=cd.COLL_SENT,
                            reset_mode=cd.COLL_RESET_NONE)
    assert e.value.status == cd.COLL_ERR_UNSUPPORTED
    for mode in (cd.COLL_RESET_FUSED, cd.COLL_RESET_KERNEL, cd.COLL_RESET_DEFERRED):
        s = cd.coll_spec_create(*cd.ALLREDUCE, 8, 64, encoding=cd.COLL_SENT, reset_mode=mode)
        cd.coll_destroy(s)



# ---- fp32 tensors ---------------------------------------------------------------

F32_CASES = [
    ("ALLREDUCE", 8, 8 * 1024, 0, 1, 1), ("ALLREDUCE", 8, 8 * 1024, 0, 2, 2),
    ("ALLREDUCE", 3, 600, 1, 2, 2), ("ALLREDUCE", 8, 8 * 480, 1, 2, 1),
    ("ALLREDUCE", 5, 5 * 96 + 8, 2, 1, 1), ("ALLREDUCE", 8, 8 * 512, 2, 2, 2),
    ("REDUCE_SCATTER", 8, 8 * 600, 1, 0, 2), ("REDUCE_SCATTER", 3, 3 * 40 + 16, 2, 0, 1),
    ("ALLGATHER", 4, 4 * 104 + 8, 1, 0, 1), ("ALLGATHER", 8, 8 * 256, 2, 0, 2),
    ("ALLTOALL", 8, 8 * 240, 1, 0, 2), ("ALLTOALL", 4, 4 * 64, 0, 0, 1),
]


@pytest.mark.parametrize("name,n,count,enc,algo,path", F32_CASES + _sweep_cases(40, 99))
def test_derived_f32_schedule_computes_the_oracle_result(cd, name, n, count, enc, algo, path):
    spec = cd.coll_spec_create(*getattr(cd, name), n, count, dtype=cd.COLL_F32, encoding=enc,
                               algorithm=algo, path=path)
    try:
        ins32 = [synth.normal_f32(3, cd.coll_buffer_elems(spec, r)[0], n, count, r)
                 for r in range(n)]
        ins32[0][::37] = 0xFFFFFFFF                       # the reserved sentinel word
        ins32[1 % n][5::41] = 0x7FC00123                  # a NaN with a payload
        got = interpret(cd, spec, enc, n, [x.view(np.uint16) for x in ins32], f32=True)
        san = [oracle.sent_sanitize_f32(x) for x in ins32] if enc == 2 else ins32
        if name == "ALLREDUCE":
            want = oracle.allreduce_f32(ins32)
        elif name == "REDUCE_SCATTER":
            want = oracle.reduce_scatter_f32(ins32)
        elif name == "ALLGATHER":
            want = [np.concatenate(san) for _ in range(n)]
        else:
            m = oracle.shard_elems(count, n)
            want = [np.concatenate([san[p][d * m:(d + 1) * m] for p in range(n)]) for d in range(n)]
        for r in range(n):
            assert np.array_equal(got[r].view(np.uint32), want[r]), f"rank {r}"
    finally:
        cd.coll_destroy(spec)


def test_f32_element_counts_and_admission(cd):
    s = cd.coll_spec_create(*cd.REDUCE_SCATTER, 3, 3 * 40 + 16, dtype=cd.COLL_F32)
    assert [cd.coll_buffer_elems(s, r) for r in range(3)] == [(136, 48), (136, 48), (136, 40)]
    cd.coll_destroy(s)
    with pytest.raises(cd.CollError) as e:
        cd.coll_spec_create(*cd.ALLREDUCE, 8, 12, dtype=cd.COLL_F32)
    assert e.value.status == cd.COLL_ERR_ALIGN
    # MoE dispatch copies fp32 rows: element counts stay in fp32 elements,
    # rows wider than 24,576 fp32 do not fit the two staged rows in shared memory
    s = cd.coll_spec_create(*cd.MOE_DISPATCH, 2, 0, dtype=cd.COLL_F32, encoding=cd.COLL_LL128,
                            tokens=4, hidden=8, topk=1, experts=2)
    assert cd.coll_buffer_elems(s, 0) == (32, 4 * 2 * 1 * 8)
    cd.coll_destroy(s)
    with pytest.raises(cd.CollError) as e:
        cd.coll_spec_create(*cd.MOE_DISPATCH, 2, 0, dtype=cd.COLL_F32, encoding=cd.COLL_LL128,
                            tokens=4, hidden=24576 + 8, topk=1, experts=2)
    assert e.value.status == cd.COLL_ERR_UNSUPPORTED
    with pytest.raises(cd.CollError) as e:
        cd.coll_spec_create(*cd.ALLREDUCE, 8, 64, dtype=7)
    assert e.value.status == cd.COLL_ERR_UNSUPPORTED


def test_atom_copy_argument_validation(cd):
    """coll_atom_copy rejects every bad argument on the host, before any CUDA
    call (the pointers here are never dereferenced)."""
    def status_of(dst, src, nbytes, **kw):
        try:
            cd.coll_atom_copy(dst, src, nbytes, stream=0, **kw)
        except cd.CollError as e:
            return e.status
        return cd.COLL_OK

    a, b = 0x10000000, 0x20000000
    assert status_of(a, b, 0) == cd.COLL_OK                       # nothing to copy
    assert status_of(a, b, 4096, stages=0) == cd.COLL_ERR_INVALID
    assert status_of(a, b, 4096, stages=9) == cd.COLL_ERR_INVALID
    assert status_of(a, b, 4096, stage_bytes=0) == cd.COLL_ERR_INVALID
    assert status_of(a, b, 4096, stages=8, stage_bytes=32768) == cd.COLL_ERR_INVALID
    assert status_of(a, b, 4096, engine=2) == cd.COLL_ERR_INVALID
    assert status_of(a, b, 4096, ctas=-1) == cd.COLL_ERR_INVALID
    assert status_of(a, b, 4096, ctas=65536) == cd.COLL_ERR_INVALID
    assert status_of(a, b, 4096, stage_bytes=24) == cd.COLL_ERR_ALIGN
    assert status_of(a, b, 4104) == cd.COLL_ERR_ALIGN
    assert status_of(a + 8, b, 4096) == cd.COLL_ERR_ALIGN
    assert status_of(a, b + 4, 4096) == cd.COLL_ERR_ALIGN
    assert status_of(None, b, 4096) == cd.COLL_ERR_INVALID
    assert status_of(a, a + 4080, 4096) == cd.COLL_ERR_INVALID     # overlapping ranges
    assert status_of(a + 4080, a, 4096) == cd.COLL_ERR_INVALID


def test_bounded_staging_validation(cd):
    """Purlin §4.1 staging capacity: only the composed launch cycles chunk
    slots; a capacity below two slots of the smallest chunk, another path or
    a non-composable collective is refused, and a ring-mode spec refuses the
    entry points that address the whole message (all on the host)."""
    n, count = 8, 8 * 60 * 4096
    kw = dict(encoding=cd.COLL_LL128, algorithm=cd.COLL_TWOSHOT)

    def status_of(triple, **opts):
        try:
            s = cd.coll_spec_create(*triple, n, count, **opts)
        except cd.CollError as e:
            return e.status
        cd.coll_destroy(s)
        return cd.COLL_OK

    assert status_of(cd.ALLREDUCE, staging_bytes=1 << 20, path=cd.COLL_PATH_STREAMED,
                     **kw) == cd.COLL_ERR_UNSUPPORTED
    assert status_of(cd.ALLREDUCE, staging_bytes=4096 * n - 128, path=cd.COLL_PATH_COMPOSED,
                     **kw) == cd.COLL_ERR_INVALID
    assert status_of(cd.ALLGATHER, staging_bytes=1 << 16,
                     encoding=cd.COLL_LL128) == cd.COLL_ERR_UNSUPPORTED
    assert status_of(cd.ALLREDUCE, staging_bytes=4096 * n, path=cd.COLL_PATH_COMPOSED,
                     **kw) == cd.COLL_OK

    def ws(**opts):
        s = cd.coll_spec_create(*cd.ALLREDUCE, n, count, **kw, **opts)
        b = cd.coll_workspace_bytes(s)
        cd.coll_destroy(s)
        return b

    full = ws(path=cd.COLL_PATH_COMPOSED)
    assert ws(staging_bytes=1 << 40, path=cd.COLL_PATH_COMPOSED) == full  # no cycling needed
    assert ws(staging_bytes=1 << 20) < ws(staging_bytes=1 << 21) < full   # AUTO -> composed
    s = cd.coll_spec_create(*cd.ALLREDUCE, n, count, staging_bytes=1 << 20, **kw)
    assert cd.coll_debug_plan(s)["path"] == cd.COLL_PATH_COMPOSED
    for call in (lambda: cd.coll_stage(s, 0, 0x1000, stream=0),
                 lambda: cd.coll_staging_layout(s, 0, 0, 0, 0)):
        with pytest.raises(cd.CollError) as e:
            call()
        assert e.value.status == cd.COLL_ERR_UNSUPPORTED
    cd.coll_destroy(s)


@pytest.mark.parametrize("T", [64, 68, 96, 136, 200])
def test_fused_phases_fill_whole_rounds(cd, T):
    """A fused phase with more items than CTAs per rank gets whole rounds of
    items of about equal size: no CTA b of a rank (items b, b + B, ...)
    moves much more than its share of the lines (with the largest tile, a
    few CTAs moved twice the others).  Schedule only (host)."""
    n = 8
    s = cd.coll_spec_create(*cd.ALLREDUCE, n, T * 4096, encoding=cd.COLL_SENT,
                            algorithm=cd.COLL_TWOSHOT, path=cd.COLL_PATH_FUSED)
    B = cd.coll_debug_plan(s)["ctas_per_rank"]
    for which in (1, 2):
        items = cd.coll_debug_items(s, which)
        per_rank = len(items) // n
        if per_rank > B:
            assert per_rank % B == 0, (which, per_rank, B)
        for d in range(n):
            mine = [it for it in items if int(it[2]) == d]
            load = [sum(int(it[5]) for it in mine[b::B]) for b in range(B)]
            fair = -(-sum(load) // B)  # no CTA carries much more than its share
            assert max(load) <= 1.02 * fair + 8, (which, d, load)
    cd.coll_destroy(s)


def test_dependent_launch_rule(cd):
    """A run's kernels are dependent launches when it is one-launch (fused
    or composed) up to 512 KiB per rank, input or output, or stream-ordered
    up to 128 KiB; larger runs are not.  Plan only (host)."""
    def dep(triple, n, count, **kw):
        s = cd.coll_spec_create(*triple, n, count, **kw)
        try:
            return cd.coll_debug_plan(s)["dependent_launch"]
        finally:
            cd.coll_destroy(s)

    fused = dict(encoding=cd.COLL_LL8, path=cd.COLL_PATH_FUSED)
    assert dep(cd.ALLREDUCE, 8, 4096, **fused) == 1                 # 8 KiB per rank
    assert dep(cd.ALLREDUCE, 8, 256 * 1024, **fused) == 1           # 512 KiB
    assert dep(cd.ALLREDUCE, 8, 256 * 1024 + 8, **fused) == 0
    streamed = dict(encoding=cd.COLL_LL128, path=cd.COLL_PATH_STREAMED)
    assert dep(cd.ALLREDUCE, 8, 4096, **streamed) == 1
    assert dep(cd.ALLREDUCE, 8, 64 * 1024, **streamed) == 1          # 128 KiB
    assert dep(cd.ALLREDUCE, 8, 64 * 1024 + 8, **streamed) == 0
    composed = dict(encoding=cd.COLL_LL128, algorithm=cd.COLL_TWOSHOT,
                    path=cd.COLL_PATH_COMPOSED)
    assert dep(cd.ALLREDUCE, 8, 4096, **composed) == 1
    assert dep(cd.ALLREDUCE, 8, 256 * 1024, **composed) == 1          # 512 KiB
    assert dep(cd.ALLREDUCE, 8, 256 * 1024 + 8, **composed) == 0
    assert dep(cd.ALLREDUCE, 8, 4096, encoding=cd.COLL_ENC_AUTO) == 1   # policy: fused
    # all-gather: 64 KiB in, 512 KiB out per rank; twice that is past the bound
    assert dep(cd.ALLGATHER, 8, 8 * 32 * 1024, **fused) == 1
    assert dep(cd.ALLGATHER, 8, 8 * 64 * 1024, **fused) == 0

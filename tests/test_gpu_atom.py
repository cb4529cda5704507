"""The one-sided copy with an explicit pipeline depth (Purlin §3.3, Eq. (3))
on the GPU against the oracle's copy, byte for byte: both engines, every
depth S = 1..8, stage sizes from one 16-byte granule to 24 KiB, CTA counts
from one to one per SM, ragged last chunks, offset pointers, the bytes just
past the destination left untouched, and the 256 MiB message of the depth
ablation in the launch shapes the bench times."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

GUARD = 256  # bytes past the destination that must keep their fill


@pytest.fixture(scope="module")
def cd():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import collective_datapath_gb300 as m

    return m


def copy_case(cd, nbytes, engine, ctas, stages, stage_bytes, src_off=0, dst_off=0, seed=0):
    import torch

    words = (src_off + nbytes + 3) // 4
    host = synth.random_bits32(seed, words, nbytes, stages, engine)
    src_buf = torch.from_numpy(host.view(np.int32)).cuda()
    dst_buf = torch.full(((dst_off + nbytes + GUARD) // 4,), 0x5A5A5A5A, dtype=torch.int32,
                         device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    src_ptr = src_buf.data_ptr() + src_off
    dst_ptr = dst_buf.data_ptr() + dst_off
    cd.coll_atom_copy(dst_ptr, src_ptr, nbytes, engine=engine, ctas=ctas, stages=stages,
                      stage_bytes=stage_bytes, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = dst_buf.cpu().numpy().view(np.uint8)
    want = oracle.one_sided_copy(host.view(np.uint8)[src_off:src_off + nbytes])
    body = got[dst_off:dst_off + nbytes]
    if not np.array_equal(body, want):
        bad = np.flatnonzero(body != want)
        raise AssertionError(f"{bad.size} bytes differ, first at {bad[0]}")
    assert np.all(got[:dst_off] == 0x5A) and np.all(got[dst_off + nbytes:] == 0x5A)


SHAPES = [
    # (ctas, stage_bytes, bytes): one granule per stage, odd stage sizes,
    # ragged last chunks, more CTAs than chunks, one CTA per SM
    (1, 16, 16 * 37),
    (3, 48, 16 * 1001),
    (16, 4096, 16 * 12345),
    (7, 24576, 1 << 20),
    (0, 16384, (3 << 20) + 16 * 7),
    (64, 16384, 16 * 100),
]


@pytest.mark.parametrize("engine", [0, 1], ids=["bulk", "lsu"])
@pytest.mark.parametrize("stages", range(1, 9))
@pytest.mark.parametrize("ctas,stage_bytes,nbytes", SHAPES)
def test_atom_copy_matches_the_oracle(cd, engine, stages, ctas, stage_bytes, nbytes):
    if stages * stage_bytes > 196608:
        pytest.skip("stages x stage bytes above the shared-memory bound")
    copy_case(cd, nbytes, engine, ctas, stages, stage_bytes, seed=stages)


@pytest.mark.parametrize("engine", [0, 1], ids=["bulk", "lsu"])
def test_atom_copy_offset_pointers(cd, engine):
    """16-byte aligned pointers that are not 128-byte aligned, at both ends."""
    copy_case(cd, 16 * 5003, engine, 5, 4, 1024, src_off=48, dst_off=16, seed=9)


@pytest.mark.parametrize("engine", [0, 1], ids=["bulk", "lsu"])
def test_atom_copy_zero_bytes_touches_nothing(cd, engine):
    import torch

    dst = torch.full((64,), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    src = torch.zeros(64, dtype=torch.int32, device="cuda")
    cd.coll_atom_copy(dst, src, 0, engine=engine, stages=3)
    torch.cuda.synchronize()
    assert bool((dst == 0x5A5A5A5A).all())


@pytest.mark.parametrize("engine", [0, 1], ids=["bulk", "lsu"])
@pytest.mark.parametrize("ctas", [16, 0])
def test_atom_copy_256mib_full_size(cd, engine, ctas):
    """The depth ablation's message (256 MiB, 16 KiB stages) at both CTA
    counts it is timed with, depths 1 and 8: every byte arrives (compared on
    the device), and a sampled set of bytes against the oracle."""
    import torch

    nbytes = 256 << 20
    g = torch.Generator(device="cuda")
    g.manual_seed(41)
    src = torch.randint(-2**31, 2**31 - 1, (nbytes // 4,), generator=g, dtype=torch.int32,
                        device="cuda")
    for stages in (1, 8):
        dst = torch.zeros(nbytes // 4 + 64, dtype=torch.int32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        cd.coll_atom_copy(dst, src, nbytes, engine=engine, ctas=ctas, stages=stages,
                          stage_bytes=16384, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(dst[:nbytes // 4], src)
        assert int(dst[nbytes // 4:].abs().sum().item()) == 0
        pos = np.unique(np.random.Generator(np.random.Philox(stages)).integers(
            0, nbytes // 4, 4096))
        idx = torch.from_numpy(pos).cuda()
        want = oracle.one_sided_copy(src[idx].cpu().numpy())
        assert np.array_equal(dst[idx].cpu().numpy().view(np.uint8), want)
        del dst
    del src
    torch.cuda.empty_cache()


@pytest.mark.parametrize("nbytes,passes,ctas", [(16, 1, 1), (4096 + 48, 3, 0), (1 << 20, 2, 7)])
def test_copy_passes_probe_copies_every_byte(cd, nbytes, passes, ctas):
    """The copy ceiling probe (several copies in one launch) leaves the
    destination equal to the source, byte for byte (the oracle's copy), and
    the bytes past it untouched."""
    import torch

    host = synth.random_bits32(11, (nbytes + 3) // 4, nbytes, passes)
    src = torch.from_numpy(host.view(np.int32)).cuda()
    dst = torch.full(((nbytes + GUARD) // 4,), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
    cd.coll_copy_passes(dst, src, nbytes, passes, ctas=ctas)
    torch.cuda.synchronize()
    got = dst.cpu().numpy().view(np.uint8)
    want = oracle.one_sided_copy(host.view(np.uint8)[:nbytes])
    assert np.array_equal(got[:nbytes], want)
    assert np.all(got[nbytes:].view(np.uint32) == 0x5A5A5A5A)


def test_copy_passes_probe_rejects_bad_arguments(cd):
    import ctypes

    import torch

    lib = ctypes.CDLL(cd.library_path())
    fn = lib.coll_copy_passes
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_int,
                   ctypes.c_void_p]
    a = torch.zeros(64, dtype=torch.int32, device="cuda")
    b = torch.zeros(64, dtype=torch.int32, device="cuda")
    assert fn(b.data_ptr(), a.data_ptr(), 256, 0, 0, None) == cd.COLL_ERR_INVALID    # passes
    assert fn(b.data_ptr(), a.data_ptr(), 24, 1, 0, None) == cd.COLL_ERR_ALIGN       # size
    assert fn(b.data_ptr() + 4, a.data_ptr(), 64, 1, 0, None) == cd.COLL_ERR_ALIGN   # pointer
    assert fn(a.data_ptr() + 16, a.data_ptr(), 64, 1, 0, None) == cd.COLL_ERR_INVALID  # overlap
    assert fn(b.data_ptr(), a.data_ptr(), 0, 1, 0, None) == cd.COLL_OK              # nothing

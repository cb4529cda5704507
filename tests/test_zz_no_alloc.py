"""coll_allreduce_static: the all-reduce for callers that cannot allocate
device memory (no workspace to bind).  Called through the C ABI directly, it
must give the same bytes as the regular entry point (coll_run on a bound
oneshot LL8 spec) -- tolerance 0 ulp, as in every other parity test -- on two
calls in a row, the second one reusing the scratch the first left behind.
This file is collected last so that a failure here never hides another test.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

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


def _c_entry(cd):
    lib = ctypes.CDLL(cd.library_path())
    fn = lib.coll_allreduce_static
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_int, ctypes.c_size_t, ctypes.POINTER(ctypes.c_void_p),
                   ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p]
    return fn


def _ptrs(ts):
    arr = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = t.data_ptr()
    return arr


@pytest.mark.parametrize("n,count", [(8, 8 * 4096), (2, 512), (8, 128 * 1024)])
def test_static_allreduce_matches_the_bound_entry_point(cd, n, count):
    import torch

    fn = _c_entry(cd)
    coll = cd.Collective(cd.ALLREDUCE, n, count, encoding=cd.COLL_LL8,
                         algorithm=cd.COLL_ONESHOT)
    stream = torch.cuda.current_stream()
    for call in range(2):
        xs = [synth.normal_bf16(31 + call, count, n, r) for r in range(n)]
        ins = [to_dev(x) for x in xs]
        ref = [empty_dev(count) for _ in range(n)]
        got = [empty_dev(count) for _ in range(n)]
        coll.run(ins, ref)
        rc = fn(n, count, _ptrs(ins), _ptrs(got), stream.cuda_stream)
        assert rc == cd.COLL_OK, cd.coll_status_string(rc)
        torch.cuda.synchronize()
        assert coll.status()[0] == cd.COLL_OK
        for r in range(n):
            assert np.array_equal(from_dev(got[r])[:count], from_dev(ref[r])[:count]), \
                f"call {call} rank {r}"


def test_static_allreduce_rejects_requests_beyond_its_scratch(cd):
    fn = _c_entry(cd)
    ins = [empty_dev(8) for _ in range(8)]
    outs = [empty_dev(8) for _ in range(8)]
    rc = fn(8, (1 << 20) // 8 + 8, _ptrs(ins), _ptrs(outs), None)
    assert rc == cd.COLL_ERR_NOMEM
    assert fn(8, 12, _ptrs(ins), _ptrs(outs), None) == cd.COLL_ERR_ALIGN

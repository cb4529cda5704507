"""coll_allreduce_static: the all-reduce for callers that cannot allocate
device memory (no workspace to bind).  Called through the C ABI directly, it
must give the oracle's all-reduce bytes, and the same bytes as the regular
entry point (coll_run on a bound oneshot LL8 spec) -- tolerance 0 ulp, as in
every other parity test -- on two calls in a row, the second one reusing the
scratch the first left behind.  A third case plants a latched device error
(status and abort words, as a timed-out wait leaves them) in the scratch
header between two calls, through a test-only build of the same source file
(tests/c/static_hook.cu), and checks that the next call still gives the
oracle's bytes.
This file is collected last so that a failure here never hides another test.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import empty_dev, from_dev, to_dev

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def cd():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import collective_datapath_gb300 as m

    return m


def _declare(fn):
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_int, ctypes.c_size_t, ctypes.POINTER(ctypes.c_void_p),
                   ctypes.POINTER(ctypes.c_void_p), ctypes.c_void_p]
    return fn


def _c_entry(cd):
    return _declare(ctypes.CDLL(cd.library_path()).coll_allreduce_static)


def _ptrs(ts):
    arr = (ctypes.c_void_p * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = t.data_ptr()
    return arr


@pytest.mark.parametrize("n,count", [(8, 8 * 4096), (2, 512), (8, 128 * 1024)])
def test_static_allreduce_matches_the_oracle_and_the_bound_entry_point(cd, n, count):
    import torch

    fn = _c_entry(cd)
    coll = cd.Collective(cd.ALLREDUCE, n, count, encoding=cd.COLL_LL8,
                         algorithm=cd.COLL_ONESHOT)
    stream = torch.cuda.current_stream()
    for call in range(2):
        xs = [synth.normal_bf16(31 + call, count, n, r) for r in range(n)]
        want = oracle.allreduce(xs)
        ins = [to_dev(x) for x in xs]
        ref = [empty_dev(count) for _ in range(n)]
        got = [empty_dev(count) for _ in range(n)]
        coll.run(ins, ref)
        rc = fn(n, count, _ptrs(ins), _ptrs(got), stream.cuda_stream)
        assert rc == cd.COLL_OK, cd.coll_status_string(rc)
        torch.cuda.synchronize()
        assert coll.status()[0] == cd.COLL_OK
        for r in range(n):
            g = from_dev(got[r])[:count]
            assert np.array_equal(g, want[r]), f"call {call} rank {r}: differs from the oracle"
            assert np.array_equal(g, from_dev(ref[r])[:count]), \
                f"call {call} rank {r}: differs from coll_run"


def test_static_allreduce_rejects_requests_beyond_its_scratch(cd):
    fn = _c_entry(cd)
    ins = [empty_dev(8) for _ in range(8)]
    outs = [empty_dev(8) for _ in range(8)]
    rc = fn(8, (1 << 20) // 8 + 8, _ptrs(ins), _ptrs(outs), None)
    assert rc == cd.COLL_ERR_NOMEM
    assert fn(8, 12, _ptrs(ins), _ptrs(outs), None) == cd.COLL_ERR_ALIGN


@pytest.fixture(scope="module")
def hooked(cd):
    """The allocation-free entry point built once more, from the same source
    file, with the two header hooks of tests/c/static_hook.cu."""
    import importlib.util

    spec = importlib.util.spec_from_file_location(
        "_coll_build", os.path.join(ROOT, "collective_datapath_gb300", "_build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    os.makedirs(b.BUILD_DIR, exist_ok=True)
    out = os.path.join(b.BUILD_DIR, f"libstatic_hook_{os.getpid()}.so")
    subprocess.run([b.nvcc(), *b.COMMON, *b.ARCH, "-shared",
                    os.path.join(ROOT, "tests", "c", "static_hook.cu"), "-o", out],
                   check=True, capture_output=True)
    lib = ctypes.CDLL(out)
    lib.static_hook_latch.restype = ctypes.c_int
    lib.static_hook_latch.argtypes = [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_int64]
    lib.static_hook_read.restype = ctypes.c_int
    lib.static_hook_read.argtypes = [ctypes.POINTER(ctypes.c_uint64),
                                     ctypes.POINTER(ctypes.c_uint32),
                                     ctypes.POINTER(ctypes.c_uint32)]
    _declare(lib.coll_allreduce_static)
    yield lib
    os.remove(out)


def _header(lib):
    epoch, code, abort = ctypes.c_uint64(), ctypes.c_uint32(), ctypes.c_uint32()
    assert lib.static_hook_read(ctypes.byref(epoch), ctypes.byref(code), ctypes.byref(abort)) == 0
    return epoch.value, code.value, abort.value


def test_static_allreduce_recovers_from_a_latched_abort(cd, hooked):
    """A call after a latched device error (planted on the host: no wait is
    made to run out) clears it in stream order and folds in full."""
    import torch

    n, count = 8, 16 * 4096
    stream = torch.cuda.current_stream()
    outs = [empty_dev(count) for _ in range(n)]
    for call in range(3):
        xs = [synth.normal_bf16(41 + call, count, n, r) for r in range(n)]
        want = oracle.allreduce(xs)
        ins = [to_dev(x) for x in xs]
        for o in outs:
            o.fill_(0x5A5A)
        if call > 0:
            assert hooked.static_hook_latch(cd.COLL_ERR_TIMEOUT, 3, 77) == 0
            assert _header(hooked)[1:] == (cd.COLL_ERR_TIMEOUT, 1)
        epoch0 = _header(hooked)[0]
        rc = hooked.coll_allreduce_static(n, count, _ptrs(ins), _ptrs(outs), stream.cuda_stream)
        assert rc == cd.COLL_OK, cd.coll_status_string(rc)
        torch.cuda.synchronize()
        epoch, code, abort = _header(hooked)
        assert (code, abort) == (0, 0), f"call {call}: error words not cleared"
        assert epoch == epoch0 + 1
        for r in range(n):
            assert np.array_equal(from_dev(outs[r])[:count], want[r]), f"call {call} rank {r}"

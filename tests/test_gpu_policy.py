"""All-reduces whose encoding, algorithm and path come from the calibrated
policy table (COLL_ENC_AUTO): bit-exact against the oracle at the sizes on
both sides of every boundary of the table, for 2, 4 and 8 ranks."""
from __future__ import annotations

import importlib.util
import os
import sys

import numpy as np
import pytest

import oracle
import synth
from tests.gpu_util import buffers, from_dev

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def cd():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import collective_datapath_gb300 as m

    return m


def boundary_sizes():
    spec = importlib.util.spec_from_file_location(
        "coll_tune", os.path.join(ROOT, "collective_datapath_gb300", "tune.py"))
    tune = importlib.util.module_from_spec(spec)
    sys.modules["coll_tune"] = tune
    spec.loader.exec_module(tune)
    tables = tune.parse_header(open(tune.TABLE_PATH).read())
    cases = []
    for n, t in sorted(tables.items()):
        for m, _ in t[:-1]:
            for nbytes in (m, m + 16 * n):
                if nbytes <= (4 << 20):
                    cases.append((n, nbytes))
        cases.append((n, 16 * n))
    return cases


@pytest.mark.parametrize("n,nbytes", boundary_sizes())
def test_policy_choice_is_bit_exact(cd, n, nbytes):
    count = nbytes // 2
    count -= count % 8
    coll = cd.Collective(cd.ALLREDUCE, n, count, encoding=cd.COLL_ENC_AUTO)
    xs, ins, outs = buffers(coll, n, seed=40, tag=nbytes)
    want = oracle.allreduce(xs)
    for _ in range(2):
        coll.run(ins, outs)
        code, rank, line = coll.status()
        assert code == cd.COLL_OK, (coll.plan(), code, rank, line)
        for r in range(n):
            assert np.array_equal(from_dev(outs[r])[:count], want[r]), (coll.plan(), r)

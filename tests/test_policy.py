"""The cost-guided policy (flash-comm §3.2, §4.1): the offline selection
procedure of collective_datapath_gb300/tune.py on synthetic cost lines whose
crossings are known, the committed table's shape, and the library's lookup
through the C ABI (no GPU)."""
from __future__ import annotations

import importlib.util
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_tune():
    spec = importlib.util.spec_from_file_location(
        "coll_tune", os.path.join(ROOT, "collective_datapath_gb300", "tune.py"))
    mod = importlib.util.module_from_spec(spec)
    sys.modules["coll_tune"] = mod
    spec.loader.exec_module(mod)
    return mod


tune = load_tune()
C = tune.Candidate
GRID = [1 << k for k in range(13, 27)]       # 8 KiB .. 64 MiB per rank


def lines_model(costs):
    """measure(size, cand) from {cand: (a, b)} (µs, µs per byte)."""
    calls = []

    def measure(s, c):
        calls.append((s, c))
        a, b = costs[c]
        return a + b * s

    return measure, calls


def test_fit_and_crossing_are_exact_on_lines():
    a, b = tune.fit_line(1000, 7.0, 3000, 11.0)
    assert (a, b) == (5.0, 0.002)
    assert tune.crossing((5.0, 1e-5), (20.0, 2e-6)) == pytest.approx(15 / 8e-6)
    assert tune.crossing((1.0, 2.0), (3.0, 2.0)) is None


def test_two_protocols_switch_at_the_measured_point_below_the_crossing():
    A, B = C(tune.SENT, tune.ONESHOT, tune.FUSED), C(tune.LL128, tune.TWOSHOT, tune.STREAMED)
    costs = {A: (5.0, 1e-5), B: (20.0, 2e-6)}      # cross at 1.875e6 bytes
    measure, calls = lines_model(costs)
    times = {s: {A: measure(s, A), B: measure(s, B)} for s in GRID}
    table = tune.build_policy(times, measure, tol=0.0)
    assert [c for _, c in table] == [A, B]
    boundary = table[0][0]
    s_star = 15 / 8e-6
    # on a measured size (a probe or a grid point), at most one 16 KiB step
    # coarser than the crossing, never past it
    assert boundary <= s_star and s_star - boundary < 0.5 * s_star
    assert (boundary, A) in calls
    assert boundary % (16 << 10) == 0
    # the lookup returns the cheaper protocol away from the switching region
    for s in GRID:
        if s <= boundary or s >= 2 * s_star:
            want = min((A, B), key=lambda c: costs[c][0] + costs[c][1] * s)
            assert tune.lookup(table, s) == want, s


def test_three_bands_and_a_candidate_that_never_wins():
    A = C(tune.LL8, tune.ONESHOT, tune.FUSED)
    B = C(tune.SENT, tune.TWOSHOT, tune.FUSED)
    D = C(tune.LL128, tune.TWOSHOT, tune.COMPOSED)
    X = C(tune.LL8, tune.TWOSHOT, tune.STREAMED)
    costs = {A: (3.0, 4e-5), B: (8.0, 1e-5), D: (40.0, 1.5e-6), X: (50.0, 5e-5)}
    measure, _ = lines_model(costs)
    times = {s: {c: measure(s, c) for c in costs} for s in GRID}
    table = tune.build_policy(times, measure, tol=0.0)
    assert [c for _, c in table] == [A, B, D]
    assert table[-1][0] == (1 << 64) - 1
    assert table[0][0] < table[1][0]
    ab = 5.0 / 3e-5        # A/B crossing
    bd = 32.0 / 8.5e-6     # B/D crossing
    assert table[0][0] <= ab < 2 * table[0][0] + (16 << 10)
    assert table[1][0] <= bd < 2 * table[1][0] + (16 << 10)


def test_committed_table_is_well_formed():
    text = open(tune.TABLE_PATH).read()
    tables = tune.parse_header(text)
    assert sorted(tables) == [2, 4, 8]
    for n, t in tables.items():
        sizes = [m for m, _ in t]
        assert sizes == sorted(sizes) and len(set(sizes)) == len(sizes)
        assert sizes[-1] == (1 << 64) - 1
        for _, c in t:
            assert c.enc in (tune.LL8, tune.LL128, tune.SENT)
            assert c.algo in (tune.ONESHOT, tune.TWOSHOT)
            assert not (c.path == tune.COMPOSED and (c.enc != tune.LL128 or c.algo != tune.TWOSHOT))
            assert not (c.enc == tune.LL128 and c.path == tune.FUSED)
        for (_, c0), (_, c1) in zip(t, t[1:]):
            assert c0 != c1


@pytest.fixture(scope="module")
def cd():
    spec = importlib.util.spec_from_file_location(
        "_coll_build", os.path.join(ROOT, "collective_datapath_gb300", "_build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    b.build()
    import collective_datapath_gb300 as m

    return m


def test_library_looks_up_the_committed_table(cd):
    tables = tune.parse_header(open(tune.TABLE_PATH).read())
    for n in range(1, 9):
        group = min([g for g in tables if g >= n], default=max(tables))
        t = tables[group]
        probes = set()
        for m, _ in t[:-1]:
            probes.update({m - 16, m, m + 16})
        probes.update({16, 8 << 10, 64 << 20})
        for nbytes in sorted(p for p in probes if p > 0):
            count = nbytes // 2
            count -= count % 8
            if count == 0:
                continue
            want = tune.lookup(t, count * 2)
            s = cd.coll_spec_create(*cd.ALLREDUCE, n, count, encoding=cd.COLL_ENC_AUTO)
            got = cd.coll_debug_plan(s)
            cd.coll_destroy(s)
            assert (got["encoding"], got["algorithm"], got["path"]) == \
                (want.enc, want.algo, want.path), (n, count * 2)


def test_auto_encoding_outside_the_table(cd):
    s = cd.coll_spec_create(*cd.REDUCE_SCATTER, 8, 8 * 4096, encoding=cd.COLL_ENC_AUTO)
    assert cd.coll_debug_plan(s)["encoding"] == cd.COLL_SENT
    cd.coll_destroy(s)
    s = cd.coll_spec_create(*cd.ALLGATHER, 8, 8 << 20, encoding=cd.COLL_ENC_AUTO)
    assert cd.coll_debug_plan(s)["encoding"] == cd.COLL_LL128
    cd.coll_destroy(s)
    # no re-arm requested: sentinel packs are not an option
    s = cd.coll_spec_create(*cd.ALLREDUCE, 8, 4096, encoding=cd.COLL_ENC_AUTO,
                            reset_mode=cd.COLL_RESET_NONE)
    assert cd.coll_debug_plan(s)["encoding"] == cd.COLL_LL8
    cd.coll_destroy(s)


def test_noise_within_the_tolerance_does_not_flip_the_choice():
    A, B = C(tune.LL8, tune.ONESHOT, tune.FUSED), C(tune.SENT, tune.ONESHOT, tune.FUSED)
    # B is 1 % faster at 16 KiB only (noise), then clearly faster from 64 KiB
    t = {8 << 10: {A: 5.00, B: 5.10}, 16 << 10: {A: 5.05, B: 5.00},
         32 << 10: {A: 5.15, B: 5.20}, 64 << 10: {A: 6.50, B: 5.40}}

    def measure(s, c):                     # linear between the grid points
        lo = max(k for k in t if k <= s)
        hi = min(k for k in t if k >= s)
        if lo == hi:
            return t[lo][c]
        return t[lo][c] + (t[hi][c] - t[lo][c]) * (s - lo) / (hi - lo)

    table = tune.build_policy(t, measure)
    assert [c for _, c in table] == [A, B]
    assert (32 << 10) <= table[0][0] < (64 << 10)
    assert [c for _, c in tune.build_policy(t, measure, tol=0.0)] == [A, B, A, B]

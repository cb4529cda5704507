"""Pins of the CPU oracle against facts fixed by the pages or by mathematics.

Nothing here compares the oracle with itself: every expected value comes from
an independent formulation (exact rationals, IEEE field decoding, a library
cast), a closed form, an invariant, or a worked example of the pages
(tests/golden/*.json, each with its citation).
"""
from __future__ import annotations

import json
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

import synth
from tests import exact

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bits(vals) -> np.ndarray:
    """float values exactly representable in bf16 -> patterns (test helper)."""
    f = np.asarray(vals, dtype=np.float32).view(np.uint32)
    assert np.all((f & 0xFFFF) == 0), "value not exact in bf16"
    return (f >> 16).astype(np.uint16)


# ---- widening bf16 -> fp32 -------------------------------------------------------------

def test_widening_all_patterns_match_field_decoding(orc):
    for b in list(range(0, 65536, 7)) + [0x0000, 0x8000, 0x0001, 0x8001,
                                         0x007F, 0x0080, 0x7F7F, 0x7F80,
                                         0xFF80, 0x3F80]:
        v = exact.decode_bf16(b)
        got = orc.bf16_to_f32(b)
        if v is None:
            assert np.isnan(got)
        elif v == exact.INF:
            assert got == float("inf")
        elif v == exact.NINF:
            assert got == float("-inf")
        else:
            val, negzero = v
            assert got == float(val)
            if val == 0:
                assert np.signbit(got) == negzero


def test_widening_matches_torch_for_all_patterns(orc):
    import torch

    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(pats.view(np.int16)).view(torch.bfloat16).float().numpy()
    got = np.array([orc.bf16_to_f32(int(b)) for b in pats], dtype=np.float32)
    assert np.array_equal(got.view(np.uint32)[~np.isnan(ref)],
                          ref.view(np.uint32)[~np.isnan(ref)])
    assert np.all(np.isnan(got) == np.isnan(ref))


# ---- rounding fp32 -> bf16 ----------------------------------------------------------------

@pytest.fixture(scope="module")
def round_checker(orc, tmp_path_factory):
    exe = str(tmp_path_factory.mktemp("rc") / "round_check")
    subprocess.check_call(["gcc", "-std=c99", "-O2", "-ffp-contract=off",
                           "-o", exe,
                           os.path.join(ROOT, "tests", "c", "round_check.c"),
                           os.path.join(ROOT, "oracle", "oracle.c"), "-lm"])
    return exe


def test_rounding_exhaustive_all_2pow32_patterns(round_checker):
    """Every binary32 pattern, against nearest-neighbour distance comparison."""
    chunks = 16
    step = (1 << 32) // chunks

    def run(c):
        return subprocess.run([round_checker, str(c * step), str((c + 1) * step)],
                              capture_output=True, text=True)

    with ThreadPoolExecutor(max_workers=os.cpu_count() or 4) as ex:
        results = list(ex.map(run, range(chunks)))
    for r in results:
        assert r.returncode == 0, r.stdout + r.stderr


def test_rounding_hand_cases(orc):
    # 1 + 2^-8 is exactly half an ulp of bf16 at 1.0: tie -> even (1.0)
    assert orc.f32_to_bf16(1.0 + 2.0 ** -8) == 0x3F80
    # 1 + 3*2^-8 is a tie between 1+2^-7 (odd) and 1+2^-6 (even) -> 1+2^-6
    assert orc.f32_to_bf16(1.0 + 3 * 2.0 ** -8) == 0x3F82
    # just above the tie rounds up
    assert orc.f32_to_bf16(np.float32(1.0 + 2.0 ** -8 + 2.0 ** -20)) == 0x3F81
    # largest binary32 rounds to +Inf (past the midpoint above bf16 max)
    assert orc.f32_to_bf16(np.finfo(np.float32).max) == 0x7F80
    assert orc.f32_to_bf16(-np.finfo(np.float32).max) == 0xFF80
    # smallest binary32 subnormal rounds to zero (no flush: sign kept)
    assert orc.f32_to_bf16(np.float32(1e-45)) == 0x0000
    assert orc.f32_to_bf16(np.float32(-1e-45)) == 0x8000
    # a bf16 subnormal survives
    assert orc.f32_to_bf16(np.float32(2.0 ** -133)) == 0x0001
    assert orc.f32_to_bf16(float("nan")) == 0x7FC0
    assert orc.f32_to_bf16(float("inf")) == 0x7F80


def test_rounding_matches_torch_cast_on_finite_values(orc):
    import torch

    g = np.random.Generator(np.random.Philox(12345))
    u = g.integers(0, 1 << 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([orc.f32_to_bf16(x) for x in f[:20000]], dtype=np.uint16)
    assert np.array_equal(got, ref[:20000])


# ---- fold in rank order ---------------------------------------------------------------------

@pytest.mark.parametrize("n", [1, 2, 3, 5, 8])
def test_fold_integer_inputs_sum_exactly(orc, n):
    """|x| <= 32, n <= 8: every partial sum is an integer <= 256, exact in
    binary32 and bf16, so the result is the plain integer sum."""
    count = 4096
    xs = [synth.integer_bf16(7, count, -32, 32, n, p) for p in range(n)]
    vals = [np.asarray(exact_vals(x)) for x in xs]
    want = _bits(np.sum(vals, axis=0).astype(np.float32))
    outs = orc.allreduce(xs)
    for o in outs:
        assert np.array_equal(o, want)


def exact_vals(bits):
    return [float(exact.decode_bf16(int(b))[0]) for b in bits]


def test_fold_n1_is_identity_for_every_non_nan_pattern(orc):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    out = orc.allreduce([pats])[0]
    nan = ((pats & 0x7F80) == 0x7F80) & ((pats & 0x7F) != 0)
    assert np.array_equal(out[~nan], pats[~nan])   # includes -0.0 -> -0.0
    assert np.all(out[nan] == 0x7FC0)


def test_fold_zero_start_differs_only_on_negative_zero(orc):
    """The literal 'start from zero' form of Eq. (2) turns -0.0 into +0.0;
    the oracle's reading keeps rank 0's -0.0 (N=1 is the identity)."""
    neg0 = np.array([0x8000], dtype=np.uint16)
    assert orc.fold([neg0], 0) == 0x8000
    assert orc.fold([neg0], 0, zero_start=True) == 0x0000
    x = synth.normal_bf16(3, 5000, 0)
    y = synth.normal_bf16(3, 5000, 1)
    for i in range(0, 5000, 37):
        assert orc.fold([x, y], i) == orc.fold([x, y], i, zero_start=True)


def test_fold_rank_order_is_observable(orc):
    """2^24 + 1 rounds back to 2^24 in binary32, so (2^24 + 1) - 2^24 = 0 in
    rank order while another order gives 1: the order is observable."""
    xs = [_bits([2.0 ** 24]), _bits([1.0]), _bits([-(2.0 ** 24)])]
    assert orc.fold(xs, 0) == 0x0000
    assert orc.fold([xs[2], xs[0], xs[1]], 0) == 0x3F80   # 1.0 in another order
    assert exact.fold_bits([int(x[0]) for x in xs]) == 0x0000


def test_fold_bruteforce_n2_against_exact_rationals(orc):
    """N=2: a over a structured set of patterns (every exponent, edge
    fractions), b over random finite patterns; expected = exact sum rounded
    to binary32 then to bf16 with rational arithmetic."""
    a_set = []
    for e in range(0, 255):
        for f in (0x00, 0x01, 0x40, 0x7F):
            for s in (0, 1):
                a_set.append((s << 15) | (e << 7) | f)
    b_all = synth.random_bits16(11, 4000, 0)
    b_set = [int(b) for b in b_all if (b & 0x7F80) != 0x7F80][:60]
    b_set += [0x0000, 0x8000, 0x3F80, 0xBF80, 0x7F7F, 0xFF7F, 0x0001, 0x8001]
    a_arr = np.array(a_set, dtype=np.uint16)
    for b in b_set:
        b_arr = np.full(a_arr.size, b, dtype=np.uint16)
        got = orc.allreduce([a_arr, b_arr])[0]
        for i in range(0, a_arr.size, 3):
            want = exact.fold_bits([int(a_arr[i]), b])
            assert got[i] == want, (hex(a_arr[i]), hex(b))


def test_fold_bruteforce_n3_to_n8_against_exact_rationals(orc):
    for n in (3, 4, 8):
        xs = [synth.normal_bf16(5, 600, n, p) for p in range(n)]
        # widen the dynamic range on a few ranks to force roundings
        xs[1] = (xs[1].astype(np.uint32) + (12 << 7)).astype(np.uint16)
        got = orc.allreduce(xs)[0]
        for i in range(600):
            want = exact.fold_bits([int(x[i]) for x in xs])
            assert got[i] == want


def test_fold_overflow_and_subnormals(orc):
    big = _bits([2.0 ** 127 * 1.5])
    assert orc.fold([big, big], 0) == 0x7F80                 # -> +Inf
    tiny = np.array([0x0001], dtype=np.uint16)               # 2^-133
    assert orc.fold([tiny, tiny], 0) == 0x0002               # 2^-132, kept
    assert exact.fold_bits([0x0001, 0x0001]) == 0x0002


# ---- collectives -----------------------------------------------------------

def test_figure4_worked_example(orc):
    spec = json.load(open(os.path.join(GOLDEN, "fig4_layouts.json")))
    n = spec["ranks"]
    m = 8  # elements per partition
    # x_p_k: distinct small integers (exact sums)
    part = {f"x_{p}_{k}": _bits(np.arange(m) + 10 * p + 3 * k - 20)
            for p in range(n) for k in range(n)}
    ins = [np.concatenate([part[f"x_{p}_{k}"] for k in range(n)]) for p in range(n)]
    rs = orc.reduce_scatter(ins)
    ys = {}
    for k, names in spec["reduce_scatter"].items():
        total = sum(np.array(exact_vals(part[nm])) for nm in names)
        assert np.array_equal(rs[int(k)], _bits(total))
        ys[f"y_{k}"] = rs[int(k)]
    ag = orc.all_gather(rs, n * m)
    for d, names in spec["all_gather_of_reduce_scatter"].items():
        assert np.array_equal(ag[int(d)], np.concatenate([ys[nm] for nm in names]))
    a2a = orc.all_to_all(ins)
    want = np.concatenate([part[nm] for nm in spec["all_to_all_rank1"]])
    assert np.array_equal(a2a[1], want)


@pytest.mark.parametrize("n,count", [(2, 512), (8, 8 * 4096), (4, 8 * 4 * 3 + 8),
                                     (8, 24), (3, 1000), (1, 64)])
def test_allreduce_invariants(orc, n, count):
    count -= count % 8
    xs = [synth.normal_bf16(1, count, n, count, p) for p in range(n)]
    ar = orc.allreduce(xs)
    for o in ar[1:]:
        assert np.array_equal(o, ar[0])          # every rank identical
    assert np.array_equal(orc.allreduce_composed(xs)[0], ar[0])   # AG o RS == AR
    rs = orc.reduce_scatter(xs)
    for r in range(n):
        b, ln = orc.shard_begin(count, n, r), orc.shard_len(count, n, r)
        assert np.array_equal(rs[r], ar[0][b:b + ln])
    # rank permutation changes the fold, not the contract: folding a
    # permuted rank list equals folding in that order (spot check)
    i = count // 2
    assert orc.fold(xs, i) == ar[0][i]


def test_shard_geometry_closed_forms(orc):
    assert orc.shard_elems(8 * 4096, 8) == 4096
    assert [orc.shard_len(8 * 4096, 8, r) for r in range(8)] == [4096] * 8
    # ragged: 24 elements over 8 ranks -> partitions of 8, then empty ones
    assert orc.shard_elems(24, 8) == 8
    assert [orc.shard_len(24, 8, r) for r in range(8)] == [8, 8, 8, 0, 0, 0, 0, 0]
    assert [orc.shard_begin(24, 8, r) for r in range(8)] == [0, 8, 16, 24, 24, 24, 24, 24]
    # 1000 over 3: ceil = 334 -> 336; partitions 336, 336, 328
    assert [orc.shard_len(1000, 3, r) for r in range(3)] == [336, 336, 328]
    assert orc.shard_elems(0, 8) == 0


def test_all_to_all_is_an_involution_and_a_permutation(orc):
    n, count = 8, 8 * 64
    xs = [synth.random_bits16(2, count, p) for p in range(n)]
    once = orc.all_to_all(xs)
    twice = orc.all_to_all(once)
    for p in range(n):
        assert np.array_equal(twice[p], xs[p])
    assert np.array_equal(np.sort(np.concatenate(once)), np.sort(np.concatenate(xs)))
    with pytest.raises(ValueError):
        orc.all_to_all([np.zeros(24, np.uint16)] * 8)     # unequal partitions


def test_all_gather_is_rank_ordered_concatenation(orc):
    n, count = 4, 4 * 40
    xs = [synth.random_bits16(4, orc.shard_len(count, n, p), p) for p in range(n)]
    ag = orc.all_gather(xs, count)
    for o in ag:
        assert np.array_equal(o, np.concatenate(xs))


# ---- line encodings ---------------------------------------------------------------

def test_ll8_line_layout_hand_case(orc):
    lines = orc.ll8_encode(np.array([0x3F80, 0xC000, 0x1234], dtype=np.uint16), 5)
    assert lines.tolist() == [0x00000005C0003F80, 0x0000000500001234]
    # only the low 32 bits of the epoch travel in the flag word
    assert orc.ll8_encode(np.array([1, 2], np.uint16), (7 << 32) | 9).tolist() == [
        0x0000000900020001]


def test_ll8_roundtrip_every_pattern_in_both_positions(orc):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for shift in (0, 1):
        x = np.roll(np.concatenate([pats, pats[:1]]), shift)
        lines = orc.ll8_encode(x, 77)
        assert lines.size == (x.size + 1) // 2
        back, rej = orc.ll8_decode(lines, x.size, 77)
        assert rej == 0 and np.array_equal(back, x)
        assert np.all((lines >> np.uint64(32)) == 77)


def test_ll8_rejects_any_other_flag(orc):
    x = synth.random_bits16(9, 100, 0)
    lines = orc.ll8_encode(x, 12)
    for bad in (11, 10, 0, 13, 12 + (1 << 32) - 1):
        stale = lines.copy()
        stale[[3, 40]] = (stale[[3, 40]] & np.uint64(0xFFFFFFFF)) | (np.uint64(bad & 0xFFFFFFFF) << np.uint64(32))
        back, rej = orc.ll8_decode(stale, x.size, 12, fill=0xDEAD)
        assert rej == 2
        assert back[6] == 0xDEAD and back[7] == 0xDEAD and back[80] == 0xDEAD
        assert back[5] == x[5]


def test_ll128_line_layout_hand_case(orc):
    x = np.arange(1, 62, dtype=np.uint16)          # 61 elements -> 2 lines
    raw = orc.ll128_encode(x, 0x0102030405060708)
    assert raw.size == 256
    l0 = raw[:128]
    assert l0[0] == 1 and l0[1] == 0 and l0[118] == 60 and l0[119] == 0
    assert l0[120:128].tolist() == [8, 7, 6, 5, 4, 3, 2, 1]
    l1 = raw[128:]
    assert l1[0] == 61 and np.all(l1[2:120] == 0)   # padding is zero
    assert l1[120:128].tolist() == [8, 7, 6, 5, 4, 3, 2, 1]


def test_ll128_roundtrip_every_pattern_in_every_position(orc):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for pos in (0, 1, 7, 8, 29, 56, 59):
        x = np.zeros(65536 * 60, dtype=np.uint16)
        x[pos::60] = pats
        lines = orc.ll128_encode(x, 3)
        assert lines.size == 65536 * 128
        back, rej = orc.ll128_decode(lines, x.size, 3)
        assert rej == 0 and np.array_equal(back, x)
    for elems, want in ((0, 0), (1, 1), (60, 1), (61, 2), (114688, 1912)):
        assert orc.ll128_lines(elems) == want


def test_ll128_rejects_other_sequence_numbers(orc):
    x = synth.random_bits16(9, 600, 1)
    raw = orc.ll128_encode(x, 41).reshape(-1, 128).copy()
    raw[4, 120] = 40          # seq 40 = previous epoch
    raw[7, 127] = 1           # a high byte differs
    back, rej = orc.ll128_decode(raw.ravel(), x.size, 41, fill=0xBEEF)
    assert rej == 2
    assert np.all(back[240:300] == 0xBEEF) and np.all(back[420:480] == 0xBEEF)
    assert np.array_equal(back[:240], x[:240])


# ---- sentinel readiness (flash-comm §3.1) ---------------------------------------------

def _is_bf16_nan(v: np.ndarray) -> np.ndarray:
    """IEEE binary16-brain layout: exponent all ones and a nonzero fraction."""
    return ((v & 0x7F80) == 0x7F80) & ((v & 0x007F) != 0)


def test_sentinel_sanitize_changes_only_the_reserved_nan(orc):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    out = orc.sent_sanitize(pats)
    changed = np.nonzero(out != pats)[0]
    assert changed.tolist() == [0xFFFF]
    assert out[0xFFFF] == 0x7FC0
    # the reserved pattern and its replacement are both NaNs: no number changes
    assert _is_bf16_nan(np.array([0xFFFF, 0x7FC0], np.uint16)).all()
    # 0x7FC0 is the canonical quiet NaN: sign 0, exponent all ones, only the
    # quiet bit of the fraction set
    assert (0x7FC0 >> 15) == 0 and (0x7FC0 & 0x7F80) == 0x7F80 and (0x7FC0 & 0x7F) == 0x40
    # the fold's rounding yields the same NaN, so partial sums never carry
    # the reserved pattern
    assert orc.f32_to_bf16(float("nan")) == 0x7FC0
    assert orc.f32_to_bf16(-float("nan")) == 0x7FC0


def test_sentinel_pack_layout_hand_case(orc):
    x = np.array([0x0001, 0xFFFF, 0x1234, 0x8000, 0x7F80], dtype=np.uint16)
    packs = orc.sent_encode(x)
    assert packs.tolist() == [0x800012347FC00001, 0x0000000000007F80]
    assert orc.sent_packs(0) == 0 and orc.sent_packs(4) == 1 and orc.sent_packs(9) == 3


def test_sentinel_roundtrip_every_pattern_in_every_position(orc):
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for pos in range(4):
        x = np.zeros(65536 * 4, dtype=np.uint16)
        x[pos::4] = pats
        packs = orc.sent_encode(x)
        assert packs.size == 65536
        assert not np.any(packs == np.uint64(0xFFFFFFFFFFFFFFFF))   # never looks unready
        back, skipped = orc.sent_decode(packs, x.size)
        assert skipped == 0
        want = x.copy()
        want[want == 0xFFFF] = 0x7FC0
        assert np.array_equal(back, want)


def test_sentinel_pack_is_not_ready(orc):
    x = synth.random_bits16(9, 100, 2)
    packs = orc.sent_encode(x)
    packs[[3, 20]] = np.uint64(0xFFFFFFFFFFFFFFFF)
    back, skipped = orc.sent_decode(packs, x.size, fill=0xDEAD)
    assert skipped == 2
    assert np.all(back[12:16] == 0xDEAD) and np.all(back[80:84] == 0xDEAD)
    assert np.array_equal(back[:12], orc.sent_sanitize(x[:12]))
    # one sentinel element next to data is data, not a missing pack
    one = np.array([0xFFFF, 0xFFFF, 0xFFFF, 0x0001], dtype=np.uint64)
    mixed = np.array([int(one[0] | (one[1] << 16) | (one[2] << 32) | (one[3] << 48))],
                     dtype=np.uint64)
    back, skipped = orc.sent_decode(mixed, 4)
    assert skipped == 0 and back.tolist() == [0xFFFF, 0xFFFF, 0xFFFF, 0x0001]


def test_sentinel_sanitize_does_not_change_a_fold(orc):
    """NaN in, NaN out: folding sanitized inputs gives the bits of folding the
    raw ones, so reductions are unaffected by the sanitisation."""
    n, count = 8, 4096
    xs = [synth.random_bits16(10, count, r) for r in range(n)]
    g = np.random.Generator(np.random.Philox(3))
    for r in range(n):
        xs[r][g.integers(0, count, 200)] = 0xFFFF
    raw = orc.allreduce(xs)[0]
    san = orc.allreduce([orc.sent_sanitize(x) for x in xs])[0]
    assert np.array_equal(raw, san)
    assert not np.any(raw == 0xFFFF)


# ---- MoE dispatch ------------------------------------------------------------------

def test_moe_tiny_hand_derived_layout(orc):
    spec = json.load(open(os.path.join(GOLDEN, "moe_tiny.json")))
    n = spec["ranks"]
    ins = [_bits(spec["rows"][str(p)]) for p in range(n)]
    topk = [np.array(spec["topk"][str(p)], dtype=np.int32) for p in range(n)]
    outs, counts, rows = orc.moe_dispatch(ins, topk, spec["experts"])
    for d in range(n):
        assert np.array_equal(outs[d], _bits(spec["expected_out"][str(d)]))
    assert counts.tolist() == spec["expected_counts_dest_le_src"]
    assert rows.tolist() == [len(spec["expected_out"][str(d)]) for d in range(n)]


def test_moe_counts_and_rows_invariants(orc):
    n, tokens, hidden, k, experts = 4, 256, 24, 4, 32
    ins = [synth.random_bits16(5, tokens * hidden, p).reshape(tokens, hidden)
           for p in range(n)]
    topk = [synth.topk_experts(5, tokens, k, experts, p) for p in range(n)]
    for t in topk:
        assert all(len(set(r)) == k for r in t.tolist())
    outs, counts, rows = orc.moe_dispatch(ins, topk, experts)
    assert counts.sum() == n * tokens * k
    assert np.all(counts.sum(axis=(0, 1)) == tokens * k)      # per source
    assert rows.sum() == n * tokens * k
    # every (source, token, choice) appears exactly once, as its own row
    seen = {}
    for d in range(n):
        el = experts // n
        r = 0
        for le in range(el):
            for p in range(n):
                toks = [t for t in range(tokens) if d * el + le in topk[p][t]]
                assert len(toks) == counts[d, le, p]
                for t in toks:
                    assert np.array_equal(outs[d][r], ins[p][t])
                    seen[(p, t, d * el + le)] = seen.get((p, t, d * el + le), 0) + 1
                    r += 1
        assert r == rows[d]
    assert len(seen) == n * tokens * k and set(seen.values()) == {1}


def test_moe_row_sources_agree_with_the_materialised_dispatch(orc):
    """The row-source listing names exactly the rows orc_moe_dispatch copies
    (hand-derived tiny case, then a random case)."""
    spec = json.load(open(os.path.join(GOLDEN, "moe_tiny.json")))
    topk = [np.array(spec["topk"][str(p)], dtype=np.int32) for p in range(2)]
    ins = [_bits(spec["rows"][str(p)]) for p in range(2)]
    for d in range(2):
        sr, st = orc.moe_row_sources(topk, spec["experts"], d)
        want = _bits(spec["expected_out"][str(d)])
        got = np.stack([ins[p][t] for p, t in zip(sr, st)])
        assert np.array_equal(got, want)
    n, tokens, hidden, k, experts = 4, 128, 16, 3, 16
    ins = [synth.random_bits16(8, tokens * hidden, p).reshape(tokens, hidden)
           for p in range(n)]
    topk = [synth.topk_experts(8, tokens, k, experts, p) for p in range(n)]
    outs, counts, rows = orc.moe_dispatch(ins, topk, experts)
    for d in range(n):
        sr, st = orc.moe_row_sources(topk, experts, d)
        assert sr.size == rows[d]
        assert np.array_equal(np.stack([ins[p][t] for p, t in zip(sr, st)]), outs[d])


# ---- variable-length (V) collectives and the Zipf split ----------------------------

def test_zipf_split_matches_the_worked_values_and_stated_bounds():
    spec = json.load(open(os.path.join(GOLDEN, "zipf_split.json")))
    for t, want in spec["cases"].items():
        assert synth.zipf_split(int(t)) == want
    for e in range(13, 31):                       # 8 KiB .. 1 GiB
        t = 1 << e
        v = synth.zipf_split(t)
        assert sum(v) == t and all(x % 128 == 0 for x in v)
        assert max(v) == 1.125 * t / 8
        assert v == sorted(v, reverse=True)
    assert synth.rotate_right([0, 1, 2, 3], 1) == [3, 0, 1, 2]


def test_v_collectives_reduce_to_the_fixed_ones_on_equal_partitions(orc):
    n, m = 8, 64
    xs = [synth.normal_bf16(21, n * m, p) for p in range(n)]
    eq = [m] * n
    assert all(np.array_equal(a, b) for a, b in
               zip(orc.reduce_scatter_v(xs, eq), orc.reduce_scatter(xs)))
    assert all(np.array_equal(a, b) for a, b in
               zip(orc.all_to_all_v(xs, [[m] * n for _ in range(n)]), orc.all_to_all(xs)))
    shards = [x[:m] for x in xs]
    assert all(np.array_equal(a, b) for a, b in
               zip(orc.all_gather_v(shards, eq), orc.all_gather(shards, n * m)))


def test_v_collectives_invariants_on_zipf_splits(orc):
    n = 8
    lens = [b // 2 for b in synth.zipf_split(8192)]          # elements
    t = sum(lens)
    xs = [synth.normal_bf16(22, t, p) for p in range(n)]
    rs = orc.reduce_scatter_v(xs, lens)
    assert [r.size for r in rs] == lens
    ar = orc.allreduce(xs)
    ag = orc.all_gather_v(rs, lens)
    for a in ag:
        assert np.array_equal(a, ar[0])                     # AGV o RSV == AR
    # A2AV with the rotated vectors (rank r sends rotate_right(lens, r+1)),
    # then back with the transposed sizes, is the identity
    send = [synth.rotate_right(lens, r + 1) for r in range(n)]
    ys = [synth.random_bits16(23, t, p) for p in range(n)]
    fwd = orc.all_to_all_v(ys, send)
    assert all(f.size == t for f in fwd)                     # every rank receives T
    back = orc.all_to_all_v(fwd, [[send[d][p] for d in range(n)] for p in range(n)])
    for p in range(n):
        assert np.array_equal(back[p], ys[p])


def test_all_to_all_v_hand_case(orc):
    a = np.arange(1, 25, dtype=np.uint16)          # source 0: 8 for d0, 16 for d1
    b = np.arange(101, 125, dtype=np.uint16)       # source 1: 24 for d0, 0 for d1
    out = orc.all_to_all_v([a, b], [[8, 16], [24, 0]])
    assert out[0].tolist() == list(range(1, 9)) + list(range(101, 125))
    assert out[1].tolist() == list(range(9, 25))


# ---- fp32 tensors ---------------------------------------------------------------

def _f32_patterns(seed, size):
    """fp32 patterns spread over every exponent, with zeros, subnormals,
    infinities and the largest finite values mixed in."""
    g = np.random.Generator(np.random.Philox(seed))
    bits = g.integers(0, 1 << 32, size, dtype=np.uint64).astype(np.uint32)
    special = np.array([0, 0x80000000, 1, 0x80000001, 0x007FFFFF, 0x00800000, 0x7F7FFFFF,
                        0xFF7FFFFF, 0x7F800000, 0xFF800000, 0x3F800000, 0xBF800000],
                       dtype=np.uint32)
    bits[:: 7] = special[g.integers(0, special.size, bits[:: 7].size)]
    # narrow the exponent range on half the entries so sums round often
    half = g.random(size) < 0.5
    bits[half] = (bits[half] & np.uint32(0x807FFFFF)) | \
        (g.integers(100, 140, int(half.sum())).astype(np.uint32) << np.uint32(23))
    nan = ((bits >> 23) & 0xFF) == 0xFF
    nan &= (bits & 0x7FFFFF) != 0
    bits[nan] = np.uint32(0x3F800000)          # NaN inputs are pinned separately
    return bits


def _fold_f32_exact(vals):
    acc = exact.decode_f32(int(vals[0]))
    for v in vals[1:]:
        acc = exact.add_exact(acc, exact.decode_f32(int(v)))
    return 0x7FC00000 if acc is None else exact.encode_f32(acc)


def test_fold_f32_against_exact_rationals(orc):
    for n in (2, 3, 5, 8):
        xs = [_f32_patterns(70 + n * 10 + p, 700) for p in range(n)]
        got = orc.allreduce_f32(xs)[0]
        for i in range(700):
            assert got[i] == _fold_f32_exact([x[i] for x in xs]), (n, i)


def test_fold_f32_integer_sums_are_exact(orc):
    g = np.random.Generator(np.random.Philox(77))
    for n in (2, 8):
        ints = [g.integers(-(1 << 20), 1 << 20, 4096) for _ in range(n)]
        xs = [np.asarray(v, dtype=np.float32).view(np.uint32) for v in ints]
        got = orc.allreduce_f32(xs)[0].view(np.float32)
        assert np.array_equal(got, np.sum(ints, axis=0).astype(np.float32))


def test_fold_f32_special_values(orc):
    f = orc.fold_f32
    assert f([0x7F800000, 0xFF800000]) == 0x7FC00000          # inf + -inf: NaN
    assert f([0x7FC00001, 0x3F800000]) == 0x7FC00000          # NaN in: canonical NaN out
    assert f([0xFFFFFFFF]) == 0x7FC00000                      # N = 1 keeps no NaN payload
    assert f([0x80000000, 0x80000000]) == 0x80000000          # -0 + -0 = -0
    assert f([0x80000000, 0x00000000]) == 0x00000000          # -0 + +0 = +0
    assert f([0x7F7FFFFF, 0x7F7FFFFF]) == 0x7F800000          # overflow to +inf
    assert f([0x00000001, 0x00000001]) == 0x00000002          # subnormals kept
    assert f([0x3F800000, 0x33800000]) == 0x3F800000          # 1 + 2^-24: tie to even
    assert f([0x3F800001, 0x33800000]) == 0x3F800002          # tie to even, upwards
    # rank order is observable: (big + 1) - big vs (big - big) + 1
    big, one = 0x4B800000, 0x3F800000                         # 2^24, 1
    assert f([big, one, big | 0x80000000]) == 0
    assert f([big, big | 0x80000000, one]) == one


def test_fold_f32_n1_is_identity(orc):
    x = _f32_patterns(79, 20000)
    x[:4] = [0x80000000, 0x00000001, 0x7F800000, 0xFF7FFFFF]
    assert np.array_equal(orc.allreduce_f32([x])[0], x)


def test_reduce_scatter_f32_is_the_allreduce_partition(orc):
    n, count = 5, 5 * 40 + 16
    xs = [_f32_patterns(90 + p, count) for p in range(n)]
    ar = orc.allreduce_f32(xs)[0]
    rs = orc.reduce_scatter_f32(xs)
    for r in range(n):
        b, ln = orc.shard_begin(count, n, r), orc.shard_len(count, n, r)
        assert np.array_equal(rs[r], ar[b:b + ln])


def test_sentinel_f32_sanitize_and_layout(orc):
    x = np.array([0xFFFFFFFF, 0x3F800000, 0xFFFF0000, 0x0000FFFF, 0x7FC00001], dtype=np.uint32)
    assert orc.sent_sanitize_f32(x).tolist() == [0x7FC00000, 0x3F800000, 0xFFFF0000,
                                                 0x0000FFFF, 0x7FC00001]
    packs = orc.sent_encode_f32(x)
    assert packs.tolist() == [0x3F8000007FC00000, 0x0000FFFFFFFF0000, 0x000000007FC00001]
    # only the all-ones pattern changes, wherever it sits
    g = np.random.Generator(np.random.Philox(5))
    y = g.integers(0, 1 << 32, 50000, dtype=np.uint64).astype(np.uint32)
    y[::97] = 0xFFFFFFFF
    s = orc.sent_sanitize_f32(y)
    changed = np.flatnonzero(s != y)
    assert np.array_equal(changed, np.flatnonzero(y == 0xFFFFFFFF))
    assert np.all(s[changed] == 0x7FC00000)
    back, skipped = orc.sent_decode_f32(orc.sent_encode_f32(y), y.size)
    assert skipped == 0 and np.array_equal(back, s)
    p = orc.sent_encode_f32(y)
    p[3] = np.uint64(0xFFFFFFFFFFFFFFFF)
    back, skipped = orc.sent_decode_f32(p, y.size, fill=7)
    assert skipped == 1 and back[6] == 7 and back[7] == 7


# ---- one-sided copy (Purlin §3.3, Atom::copy) ------------------------------------

def test_one_sided_copy_delivers_every_byte_in_order(orc):
    # every byte value once, in an order that no shift, reversal or stride
    # of the input reproduces (a permutation written out by hand:
    # 37 i + 11 mod 256, no byte zero at either end)
    x = np.array([(37 * i + 11) % 256 for i in range(256)], dtype=np.uint8)
    assert orc.one_sided_copy(x).tolist() == [(37 * i + 11) % 256 for i in range(256)]
    assert orc.one_sided_copy(np.zeros(0, dtype=np.uint8)).size == 0
    assert orc.one_sided_copy(np.array([7], dtype=np.uint8)).tolist() == [7]
    # wider elements travel as their little-endian bytes
    w = np.array([0x04030201, 0x08070605], dtype=np.uint32)
    assert orc.one_sided_copy(w).tolist() == [1, 2, 3, 4, 5, 6, 7, 8]

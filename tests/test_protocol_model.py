"""A host model of the self-synchronizing protocol, enumerated exhaustively:
2 ranks, 4 lines per rank image.  For every mask of lines that are stale when
the consumer starts (each stale line holds the previous epoch, the slot's
previous occupant e-2, or zero, over a poison payload) and every order in
which the producers then publish them, a consumer that polls every line,
accepts a line only when the oracle's decoder accepts it, and re-polls the
rest after each publication ends with exactly the bytes of the run without
stale lines.  The same holds for LL128 lines and sentinel packs (where a
line that is not yet published still holds the reserved pattern).
flash-comm §3.1 (readiness carried by each block), Purlin §3.2."""
from __future__ import annotations

import itertools

import numpy as np
import pytest

import oracle
import synth

E = 7  # the consumer's epoch


def lines_ll8(x, epoch):
    return oracle.ll8_encode(x, epoch)


def stale_ll8(clean, j, kind, poison):
    flag = {0: E - 1, 1: E - 2, 2: 0}[kind]
    out = clean.copy()
    out[j] = np.uint64(poison | (poison << 16)) | (np.uint64(flag) << np.uint64(32))
    return out


def decode_ll8(lines, j):
    got, rej = oracle.ll8_decode(lines[j:j + 1], 2, E)
    return None if rej else got


def lines_ll128(x, epoch):
    return oracle.ll128_encode(x, epoch).reshape(-1, 128)


def stale_ll128(clean, j, kind, poison):
    out = clean.copy()
    seq = {0: E - 1, 1: E - 2, 2: 0}[kind]
    out[j, :120] = np.frombuffer(np.full(60, poison, dtype=np.uint16).tobytes(), dtype=np.uint8)
    out[j, 120:] = np.frombuffer(np.uint64(seq).tobytes(), dtype=np.uint8)
    return out


def decode_ll128(lines, j):
    got, rej = oracle.ll128_decode(np.ascontiguousarray(lines[j]).ravel(), 60, E)
    return None if rej else got


def lines_sent(x, epoch):
    return oracle.sent_encode(x)


def stale_sent(clean, j, kind, poison):
    out = clean.copy()
    out[j] = np.uint64(0xFFFFFFFFFFFFFFFF)  # not yet published: the pattern
    return out


def decode_sent(lines, j):
    got, rej = oracle.sent_decode(lines[j:j + 1], 4)
    return None if rej else got


ENCODINGS = {
    "LL8": (2, lines_ll8, stale_ll8, decode_ll8),
    "LL128": (60, lines_ll128, stale_ll128, decode_ll128),
    "SENT": (4, lines_sent, stale_sent, decode_sent),
}


@pytest.mark.parametrize("enc", sorted(ENCODINGS))
def test_every_stale_mask_and_publish_order_gives_the_clean_result(enc):
    epl, encode, make_stale, decode = ENCODINGS[enc]
    n, nlines = 2, 4
    count = epl * nlines
    xs = [synth.normal_bf16(11, count, n, r) for r in range(n)]
    want = oracle.allreduce(xs)[0]
    clean = [encode(x, E) for x in xs]
    cases = 0
    for mask in range(1 << nlines):
        stale_lines = [j for j in range(nlines) if mask >> j & 1]
        for order in itertools.permutations(stale_lines):
            for src in range(n):            # the late rank
                images = [c.copy() for c in clean]
                for k, j in enumerate(stale_lines):
                    images[src] = make_stale(images[src], j, k % 3, 0x4880 + k)
                accepted = [[None] * nlines for _ in range(n)]
                pending = list(order)
                polls = 0
                while True:
                    polls += 1
                    for r in range(n):
                        for j in range(nlines):
                            if accepted[r][j] is None:
                                accepted[r][j] = decode(images[r], j)
                    if all(a is not None for row in accepted for a in row):
                        break
                    assert pending, "a line never became acceptable"
                    j = pending.pop(0)       # the late producer publishes one line
                    images[src][j] = clean[src][j]
                got_inputs = [np.concatenate(accepted[r]) for r in range(n)]
                assert np.array_equal(oracle.allreduce(got_inputs)[0], want)
                assert polls == len(stale_lines) + 1 or not stale_lines
                cases += 1
    assert cases == n * sum(
        len(list(itertools.permutations([j for j in range(nlines) if m >> j & 1])))
        for m in range(1 << nlines))


def test_a_line_that_is_never_published_is_never_accepted():
    """Withheld forever: the consumer can only time out."""
    for enc, (epl, encode, make_stale, decode) in ENCODINGS.items():
        x = synth.normal_bf16(12, 4 * epl, 0)
        img = make_stale(encode(x, E), 2, 0, 0x4880)
        for _ in range(100):
            assert decode(img, 2) is None, enc
        assert decode(img, 1) is not None

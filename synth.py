"""Seeded synthetic inputs shared by the tests, the smoke check and the bench.

This module holds no arithmetic of the collective method: it only draws
random inputs.  Both the CUDA path and the CPU oracle are fed from here, and
neither imports the other.

Recipe (every stream is independent and reproducible):

* key: ``np.random.SeedSequence([seed, tag, *index])`` where ``tag`` is a
  fixed integer per kind of draw and ``index`` names the rank / epoch; the
  bit generator is Philox-4x64 (a counter-based generator), drawn through
  ``Generator.random()`` (uniform doubles in [0, 1)).
* uniform[a, b]: ``a + (b - a) * u`` in float64, then float32, then bf16 by
  PyTorch's round-to-nearest-even cast (a library routine).
* normal(0, 1): Box-Muller on pairs of uniforms (u1 in (0, 1], u2):
  ``sqrt(-2 ln u1) * cos(2 pi u2)``, then float32, then bf16 as above.
* integer-valued bf16: uniform integers in [lo, hi] (exactly representable).
* top-k experts without replacement: per token, the first k entries of an
  argsort of independent uniform keys (a uniformly random k-subset, in
  random order).
* variable-length splits (V collectives): the Zipf split with exponent s of
  the Purlin page's Eq. (4) (see ``zipf_split``), in bytes, 128-byte units.
* stale lines of an epoch: exactly ``round(frac * lines)`` distinct line
  indices (the first of a random permutation), a random publication order of
  them, a stale-kind per line (0: previous epoch's flag e-1, 1: the slot's
  previous occupant e-2, 2: a re-armed zero flag) and random 16-bit poison
  payload patterns.
"""
from __future__ import annotations

import numpy as np

TAG_UNIFORM = 1
TAG_NORMAL = 2
TAG_INTEGER = 3
TAG_TOPK = 4
TAG_STALE = 5
TAG_BITS = 6
TAG_NORMAL_F32 = 7
TAG_BITS32 = 8


def _gen(seed: int, tag: int, *index: int) -> np.random.Generator:
    ss = np.random.SeedSequence([int(seed), int(tag), *[int(i) for i in index]])
    return np.random.Generator(np.random.Philox(ss))


def _f32_to_bf16_bits(f32: np.ndarray) -> np.ndarray:
    import torch  # library cast, round-to-nearest-even

    t = torch.from_numpy(np.ascontiguousarray(f32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def uniform_bf16(seed: int, n: int, lo: float, hi: float,
                 *index: int) -> np.ndarray:
    """n bf16 bit patterns drawn i.i.d. uniform[lo, hi]."""
    g = _gen(seed, TAG_UNIFORM, *index)
    u = g.random(n)
    return _f32_to_bf16_bits((lo + (hi - lo) * u).astype(np.float32))


def normal_bf16(seed: int, n: int, *index: int) -> np.ndarray:
    """n bf16 bit patterns drawn i.i.d. normal(0, 1) (Box-Muller)."""
    g = _gen(seed, TAG_NORMAL, *index)
    half = (n + 1) // 2
    u1 = 1.0 - g.random(half)          # (0, 1]
    u2 = g.random(half)
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * half, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return _f32_to_bf16_bits(z[:n].astype(np.float32))


def integer_bf16(seed: int, n: int, lo: int, hi: int, *index: int) -> np.ndarray:
    """n bf16 bit patterns of integers drawn uniformly from [lo, hi]
    (|values| <= 256 are exact in bf16)."""
    g = _gen(seed, TAG_INTEGER, *index)
    v = g.integers(lo, hi + 1, size=n).astype(np.float32)
    return _f32_to_bf16_bits(v)


def normal_f32(seed: int, n: int, *index: int) -> np.ndarray:
    """n fp32 bit patterns (uint32) drawn i.i.d. normal(0, 1) (Box-Muller),
    rounded to binary32 by numpy's cast."""
    g = _gen(seed, TAG_NORMAL_F32, *index)
    half = (n + 1) // 2
    u1 = 1.0 - g.random(half)
    u2 = g.random(half)
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * half, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return z[:n].astype(np.float32).view(np.uint32)


def random_bits32(seed: int, n: int, *index: int) -> np.ndarray:
    """n arbitrary 32-bit patterns (any fp32 value, NaN and Inf included)."""
    g = _gen(seed, TAG_BITS32, *index)
    return g.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32)


def random_bits16(seed: int, n: int, *index: int) -> np.ndarray:
    """n arbitrary 16-bit patterns (any bf16 value, NaN and Inf included)."""
    g = _gen(seed, TAG_BITS, *index)
    return g.integers(0, 1 << 16, size=n, dtype=np.uint32).astype(np.uint16)


def topk_experts(seed: int, tokens: int, k: int, experts: int,
                 *index: int) -> np.ndarray:
    """(tokens, k) int32: k distinct experts per token, uniformly at random."""
    g = _gen(seed, TAG_TOPK, *index)
    keys = g.random((tokens, experts))
    return np.argsort(keys, axis=1, kind="stable")[:, :k].astype(np.int32)


def stale_plan(seed: int, lines: int, frac: float, *index: int):
    """Stale lines of one rank in one epoch.

    Returns (idx, order, kind, poison): ``idx`` = sorted int64 indices of the
    round(frac * lines) stale lines, ``order`` = the same indices in the
    order the late producer publishes them, ``kind`` = per stale line
    0 (flag e-1), 1 (flag e-2) or 2 (flag 0), ``poison`` = uint16 patterns
    (one per stale line, repeated over the line's payload).
    """
    g = _gen(seed, TAG_STALE, *index)
    m = int(round(frac * lines))
    perm = g.permutation(lines)
    idx = np.sort(perm[:m]).astype(np.int64)
    order = g.permutation(idx).astype(np.int64)
    kind = g.integers(0, 3, size=m).astype(np.int32)
    # Poison: large finite bf16 values (biased exponent 0x90, magnitude
    # 2^17..2^18), so that accepting a stale line changes the sum visibly.
    sign = g.integers(0, 2, size=m).astype(np.uint16) << 15
    mant = g.integers(0, 128, size=m).astype(np.uint16)
    poison = (sign | np.uint16(0x90 << 7) | mant).astype(np.uint16)
    return idx, order, kind, poison


def zipf_split(total_bytes: int, ranks: int = 8, s: float = 0.125) -> list[int]:
    """Bytes per rank of a Zipf split of ``total_bytes`` (Purlin, appendix
    "Variable-length splits", Eq. (4)): with u = max(128, T / (8 W)) bytes
    and x_r = (T / u) (r+1)^-s / sum_k (k+1)^-s, rank r gets u (floor(x_r) +
    d_r), the remaining units going one each to the ranks with the largest
    fractional parts of x_r (ties to the lower rank)."""
    u = max(128, total_bytes // (8 * ranks))
    units = total_bytes // u
    w = [(r + 1) ** -s for r in range(ranks)]
    tot = sum(w)
    x = [units * wr / tot for wr in w]
    fl = [int(np.floor(v)) for v in x]
    left = units - sum(fl)
    order = sorted(range(ranks), key=lambda r: (-(x[r] - fl[r]), r))
    for r in order[:left]:
        fl[r] += 1
    return [u * f for f in fl]


def rotate_right(v: list, k: int) -> list:
    """The vector v rotated right by k positions (A2AV partition vectors)."""
    k %= len(v)
    return v[-k:] + v[:-k] if k else list(v)

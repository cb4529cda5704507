"""Python view of the plain CPU oracle (oracle.c).

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py`` may import this package.  The product path
(``collective_datapath_gb300``) never imports it, and this package imports
nothing from the product path.  The two share only the seeded input
generators in ``synth.py``, which hold none of the method's arithmetic.

Every function marshals numpy arrays into the C oracle and returns numpy
arrays; no arithmetic happens here.  bf16 values travel as ``np.uint16`` bit
patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

# -ffp-contract=off and no fast-math: binary32 additions round one at a time.
CFLAGS = ["-std=c99", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, a second or so)."""
    stale = (not os.path.exists(_LIB)
             or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
             or os.path.getmtime(_LIB) < os.path.getmtime(
                 os.path.join(_HERE, "oracle.h")))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", *CFLAGS, "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _declare(_lib)
    return _lib


_u16p = ctypes.POINTER(ctypes.c_uint16)
_u64p = ctypes.POINTER(ctypes.c_uint64)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_sz = ctypes.c_size_t


def _declare(L: ctypes.CDLL) -> None:
    L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
    L.orc_bf16_to_f32.restype = ctypes.c_float
    L.orc_f32_to_bf16.argtypes = [ctypes.c_float]
    L.orc_f32_to_bf16.restype = ctypes.c_uint16
    for name in ("orc_fold", "orc_fold_zero_start"):
        f = getattr(L, name)
        f.argtypes = [ctypes.POINTER(_u16p), ctypes.c_int, _sz]
        f.restype = ctypes.c_uint16
    for name in ("orc_shard_elems",):
        getattr(L, name).argtypes = [_sz, ctypes.c_int]
        getattr(L, name).restype = _sz
    for name in ("orc_shard_begin", "orc_shard_len"):
        getattr(L, name).argtypes = [_sz, ctypes.c_int, ctypes.c_int]
        getattr(L, name).restype = _sz
    for name in ("orc_allreduce", "orc_reduce_scatter", "orc_all_gather",
                 "orc_all_to_all"):
        f = getattr(L, name)
        f.argtypes = [ctypes.c_int, _sz, ctypes.POINTER(_u16p),
                      ctypes.POINTER(_u16p)]
        f.restype = ctypes.c_int
    L.orc_allreduce_composed.argtypes = [ctypes.c_int, _sz,
                                         ctypes.POINTER(_u16p),
                                         ctypes.POINTER(_u16p),
                                         ctypes.POINTER(_u16p)]
    L.orc_allreduce_composed.restype = ctypes.c_int
    for name in ("orc_reduce_scatter_v", "orc_all_gather_v", "orc_all_to_all_v"):
        f = getattr(L, name)
        f.argtypes = [ctypes.c_int, ctypes.POINTER(_sz), ctypes.POINTER(_u16p),
                      ctypes.POINTER(_u16p)]
        f.restype = ctypes.c_int
    L.orc_moe_dispatch.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int,
                                   ctypes.POINTER(_i32p),
                                   ctypes.POINTER(_u16p),
                                   ctypes.POINTER(_u16p), _i32p, _i64p]
    L.orc_moe_dispatch.restype = ctypes.c_int
    L.orc_moe_row_sources.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.POINTER(_i32p),
                                      ctypes.c_int, _i32p, _i32p]
    L.orc_moe_row_sources.restype = ctypes.c_int64
    L.orc_ll8_lines.argtypes = [_sz]
    L.orc_ll8_lines.restype = _sz
    L.orc_ll8_encode.argtypes = [_u16p, _sz, ctypes.c_uint64, _u64p]
    L.orc_ll8_encode.restype = None
    L.orc_ll8_decode.argtypes = [_u64p, _sz, ctypes.c_uint64, _u16p]
    L.orc_ll8_decode.restype = _sz
    L.orc_ll128_lines.argtypes = [_sz]
    L.orc_ll128_lines.restype = _sz
    L.orc_ll128_encode.argtypes = [_u16p, _sz, ctypes.c_uint64, _u8p]
    L.orc_ll128_encode.restype = None
    L.orc_ll128_decode.argtypes = [_u8p, _sz, ctypes.c_uint64, _u16p]
    L.orc_ll128_decode.restype = _sz
    L.orc_fold_f32.argtypes = [ctypes.POINTER(_u32p), ctypes.c_int, _sz]
    L.orc_fold_f32.restype = ctypes.c_uint32
    for name in ("orc_allreduce_f32", "orc_reduce_scatter_f32"):
        f = getattr(L, name)
        f.argtypes = [ctypes.c_int, _sz, ctypes.POINTER(_u32p), ctypes.POINTER(_u32p)]
        f.restype = ctypes.c_int
    L.orc_sent_sanitize_f32.argtypes = [ctypes.c_uint32]
    L.orc_sent_sanitize_f32.restype = ctypes.c_uint32
    L.orc_sent_encode_f32.argtypes = [_u32p, _sz, _u64p]
    L.orc_sent_encode_f32.restype = None
    L.orc_one_sided_copy.argtypes = [ctypes.POINTER(ctypes.c_uint8), _sz,
                                     ctypes.POINTER(ctypes.c_uint8)]
    L.orc_one_sided_copy.restype = None
    L.orc_sent_decode_f32.argtypes = [_u64p, _sz, _u32p]
    L.orc_sent_decode_f32.restype = _sz
    L.orc_sent_sanitize.argtypes = [ctypes.c_uint16]
    L.orc_sent_sanitize.restype = ctypes.c_uint16
    L.orc_sent_sanitize_buf.argtypes = [_u16p, _sz, _u16p]
    L.orc_sent_sanitize_buf.restype = None
    L.orc_sent_packs.argtypes = [_sz]
    L.orc_sent_packs.restype = _sz
    L.orc_sent_encode.argtypes = [_u16p, _sz, _u64p]
    L.orc_sent_encode.restype = None
    L.orc_sent_decode.argtypes = [_u64p, _sz, _u16p]
    L.orc_sent_decode.restype = _sz


# ---- marshalling helpers -------------------------------------------------

def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _ptr_array(arrs: Sequence[np.ndarray], ctype):
    arr_t = ctypes.POINTER(ctype) * len(arrs)
    return arr_t(*[_ptr(a, ctype) for a in arrs])


# ---- scalar ----------------------------------------------------------------

def bf16_to_f32(b: int) -> float:
    return lib().orc_bf16_to_f32(int(b))


def f32_to_bf16(f: float) -> int:
    return int(lib().orc_f32_to_bf16(float(np.float32(f))))


def fold(xs: Sequence[np.ndarray], i: int, zero_start: bool = False) -> int:
    arrs = [_c(x, np.uint16) for x in xs]
    fn = lib().orc_fold_zero_start if zero_start else lib().orc_fold
    return int(fn(_ptr_array(arrs, ctypes.c_uint16), len(arrs), i))


# ---- geometry --------------------------------------------------------------

def shard_elems(count: int, n: int) -> int:
    return int(lib().orc_shard_elems(count, n))


def shard_begin(count: int, n: int, r: int) -> int:
    return int(lib().orc_shard_begin(count, n, r))


def shard_len(count: int, n: int, r: int) -> int:
    return int(lib().orc_shard_len(count, n, r))


# ---- collectives -------------------------------------------------------------

def _collective(name: str, ins: Sequence[np.ndarray], count: int,
                out_elems: int) -> list[np.ndarray]:
    n = len(ins)
    arrs = [_c(x, np.uint16) for x in ins]
    outs = [np.zeros(max(out_elems, 1), dtype=np.uint16) for _ in range(n)]
    rc = getattr(lib(), name)(n, count, _ptr_array(arrs, ctypes.c_uint16),
                              _ptr_array(outs, ctypes.c_uint16))
    if rc != 0:
        raise ValueError(f"{name}: invalid arguments (n={n}, count={count})")
    return [o[:out_elems] for o in outs]


def allreduce(ins: Sequence[np.ndarray]) -> list[np.ndarray]:
    count = int(np.asarray(ins[0]).size)
    return _collective("orc_allreduce", ins, count, count)


def reduce_scatter(ins: Sequence[np.ndarray]) -> list[np.ndarray]:
    n, count = len(ins), int(np.asarray(ins[0]).size)
    outs = _collective("orc_reduce_scatter", ins, count, shard_elems(count, n))
    return [o[:shard_len(count, n, r)] for r, o in enumerate(outs)]


def all_gather(ins: Sequence[np.ndarray], count: int) -> list[np.ndarray]:
    """``count`` = gathered (output) elements per rank; ins[p] has
    shard_len(count, n, p) elements."""
    n = len(ins)
    padded = []
    for p, x in enumerate(ins):
        buf = np.zeros(max(shard_elems(count, n), 1), dtype=np.uint16)
        x = np.asarray(x, dtype=np.uint16).ravel()
        buf[:x.size] = x
        padded.append(buf)
    return _collective("orc_all_gather", padded, count, count)


def all_to_all(ins: Sequence[np.ndarray]) -> list[np.ndarray]:
    count = int(np.asarray(ins[0]).size)
    return _collective("orc_all_to_all", ins, count, count)


def _v_call(name, ins, lens, out_sizes):
    n = len(ins)
    arrs = [_c(np.asarray(x).ravel(), np.uint16) for x in ins]
    arrs = [a if a.size else np.zeros(1, np.uint16) for a in arrs]
    outs = [np.zeros(max(int(o), 1), dtype=np.uint16) for o in out_sizes]
    ln = (_sz * len(lens))(*[int(v) for v in lens])
    rc = getattr(lib(), name)(n, ln, _ptr_array(arrs, ctypes.c_uint16),
                              _ptr_array(outs, ctypes.c_uint16))
    if rc != 0:
        raise ValueError(f"{name}: invalid arguments")
    return [o[:int(sz)] for o, sz in zip(outs, out_sizes)]


def reduce_scatter_v(ins: Sequence[np.ndarray], lens: Sequence[int]) -> list[np.ndarray]:
    return _v_call("orc_reduce_scatter_v", ins, lens, lens)


def all_gather_v(ins: Sequence[np.ndarray], lens: Sequence[int]) -> list[np.ndarray]:
    return _v_call("orc_all_gather_v", ins, lens, [sum(lens)] * len(ins))


def all_to_all_v(ins: Sequence[np.ndarray], lens: Sequence[Sequence[int]]) -> list[np.ndarray]:
    """lens[p][d] = elements source p sends to destination d."""
    n = len(ins)
    flat = [int(lens[p][d]) for p in range(n) for d in range(n)]
    return _v_call("orc_all_to_all_v", ins, flat,
                   [sum(lens[p][d] for p in range(n)) for d in range(n)])


def allreduce_composed(ins: Sequence[np.ndarray]) -> list[np.ndarray]:
    n, count = len(ins), int(np.asarray(ins[0]).size)
    arrs = [_c(x, np.uint16) for x in ins]
    outs = [np.zeros(max(count, 1), dtype=np.uint16) for _ in range(n)]
    tmps = [np.zeros(max(shard_elems(count, n), 1), dtype=np.uint16)
            for _ in range(n)]
    rc = lib().orc_allreduce_composed(n, count,
                                      _ptr_array(arrs, ctypes.c_uint16),
                                      _ptr_array(outs, ctypes.c_uint16),
                                      _ptr_array(tmps, ctypes.c_uint16))
    if rc != 0:
        raise ValueError("orc_allreduce_composed: invalid arguments")
    return [o[:count] for o in outs]


def moe_dispatch(ins: Sequence[np.ndarray], topk: Sequence[np.ndarray],
                 experts: int, with_rows: bool = True):
    """ins[p]: (tokens, hidden) uint16; topk[p]: (tokens, k) int32.
    Returns (outs, counts[n_dest, EL, n_src], rows_per_dest)."""
    n = len(ins)
    tokens, hidden = np.asarray(ins[0]).shape
    k = np.asarray(topk[0]).shape[1]
    arrs = [_c(x, np.uint16) for x in ins]
    tks = [_c(t, np.int32) for t in topk]
    counts = np.zeros(experts * n, dtype=np.int32)
    rows = np.zeros(n, dtype=np.int64)
    if with_rows:
        # A destination receives at most min(k, EL) rows per source token.
        cap = tokens * n * min(k, experts // n)
        outs = [np.zeros((max(cap, 1), hidden), dtype=np.uint16)
                for _ in range(n)]
        out_ptrs = _ptr_array(outs, ctypes.c_uint16)
    else:
        outs = None
        out_ptrs = None
    rc = lib().orc_moe_dispatch(n, tokens, hidden, k, experts,
                                _ptr_array(tks, ctypes.c_int32),
                                _ptr_array(arrs, ctypes.c_uint16), out_ptrs,
                                _ptr(counts, ctypes.c_int32),
                                _ptr(rows, ctypes.c_int64))
    if rc != 0:
        raise ValueError("orc_moe_dispatch: invalid arguments")
    counts = counts.reshape(n, experts // n, n)
    if outs is not None:
        outs = [o[:rows[d]] for d, o in enumerate(outs)]
    return outs, counts, rows


def moe_row_sources(topk: Sequence[np.ndarray], experts: int, d: int):
    """(src_rank, src_token) int32 arrays of destination d's output rows."""
    n = len(topk)
    tokens, k = np.asarray(topk[0]).shape
    tks = [_c(t, np.int32) for t in topk]
    cap = tokens * n * min(k, experts // n)
    sr = np.zeros(max(cap, 1), dtype=np.int32)
    st = np.zeros(max(cap, 1), dtype=np.int32)
    rows = lib().orc_moe_row_sources(n, tokens, k, experts, _ptr_array(tks, ctypes.c_int32),
                                     d, _ptr(sr, ctypes.c_int32), _ptr(st, ctypes.c_int32))
    if rows < 0:
        raise ValueError("orc_moe_row_sources: invalid arguments")
    return sr[:rows], st[:rows]


# ---- encodings ---------------------------------------------------------------

def ll8_lines(elems: int) -> int:
    return int(lib().orc_ll8_lines(elems))


def ll8_encode(x: np.ndarray, epoch: int) -> np.ndarray:
    x = _c(np.asarray(x).ravel(), np.uint16)
    out = np.zeros(max(ll8_lines(x.size), 1), dtype=np.uint64)
    lib().orc_ll8_encode(_ptr(x, ctypes.c_uint16), x.size, epoch,
                         _ptr(out, ctypes.c_uint64))
    return out[:ll8_lines(x.size)]


def ll8_decode(lines: np.ndarray, elems: int, epoch: int,
               fill: int = 0) -> tuple[np.ndarray, int]:
    lines = _c(lines, np.uint64)
    out = np.full(max(elems, 1), fill, dtype=np.uint16)
    rej = lib().orc_ll8_decode(_ptr(lines, ctypes.c_uint64), elems, epoch,
                               _ptr(out, ctypes.c_uint16))
    return out[:elems], int(rej)


def ll128_lines(elems: int) -> int:
    return int(lib().orc_ll128_lines(elems))


def ll128_encode(x: np.ndarray, epoch: int) -> np.ndarray:
    x = _c(np.asarray(x).ravel(), np.uint16)
    out = np.zeros(max(ll128_lines(x.size), 1) * 128, dtype=np.uint8)
    lib().orc_ll128_encode(_ptr(x, ctypes.c_uint16), x.size, epoch,
                           _ptr(out, ctypes.c_uint8))
    return out[:ll128_lines(x.size) * 128]


def ll128_decode(lines: np.ndarray, elems: int, epoch: int,
                 fill: int = 0) -> tuple[np.ndarray, int]:
    lines = _c(lines, np.uint8)
    out = np.full(max(elems, 1), fill, dtype=np.uint16)
    rej = lib().orc_ll128_decode(_ptr(lines, ctypes.c_uint8), elems, epoch,
                                 _ptr(out, ctypes.c_uint16))
    return out[:elems], int(rej)


# ---- sentinel readiness --------------------------------------------------------

SENT_BF16 = 0xFFFF
CANONICAL_NAN = 0x7FC0


def sent_sanitize(x: np.ndarray) -> np.ndarray:
    """Every element equal to the reserved pattern replaced by the canonical
    quiet NaN (what a sentinel-encoded copy delivers)."""
    x = _c(np.asarray(x).ravel(), np.uint16)
    out = np.zeros(max(x.size, 1), dtype=np.uint16)
    lib().orc_sent_sanitize_buf(_ptr(x, ctypes.c_uint16), x.size, _ptr(out, ctypes.c_uint16))
    return out[:x.size]


def sent_packs(elems: int) -> int:
    return int(lib().orc_sent_packs(elems))


def sent_encode(x: np.ndarray) -> np.ndarray:
    x = _c(np.asarray(x).ravel(), np.uint16)
    out = np.zeros(max(sent_packs(x.size), 1), dtype=np.uint64)
    lib().orc_sent_encode(_ptr(x, ctypes.c_uint16), x.size, _ptr(out, ctypes.c_uint64))
    return out[:sent_packs(x.size)]


def sent_decode(packs: np.ndarray, elems: int, fill: int = 0) -> tuple[np.ndarray, int]:
    packs = _c(packs, np.uint64)
    out = np.full(max(elems, 1), fill, dtype=np.uint16)
    skipped = lib().orc_sent_decode(_ptr(packs, ctypes.c_uint64), elems,
                                    _ptr(out, ctypes.c_uint16))
    return out[:elems], int(skipped)


# ---- fp32 tensors (uint32 bit patterns) -------------------------------------------

CANONICAL_NAN_F32 = 0x7FC00000


def _f32_collective(name, ins, out_sizes):
    n, count = len(ins), int(np.asarray(ins[0]).size)
    arrs = [_c(np.asarray(x).ravel(), np.uint32) for x in ins]
    arrs = [a if a.size else np.zeros(1, np.uint32) for a in arrs]
    outs = [np.zeros(max(int(o), 1), dtype=np.uint32) for o in out_sizes]
    rc = getattr(lib(), name)(n, count, _ptr_array(arrs, ctypes.c_uint32),
                              _ptr_array(outs, ctypes.c_uint32))
    if rc != 0:
        raise ValueError(f"{name} rejected its arguments")
    return [o[:int(m)] for o, m in zip(outs, out_sizes)]


def fold_f32(xs: Sequence[int]) -> int:
    """The fold of one position whose N contributions are the fp32 patterns xs."""
    arrs = [np.array([v], dtype=np.uint32) for v in xs]
    return int(lib().orc_fold_f32(_ptr_array(arrs, ctypes.c_uint32), len(arrs), 0))


def allreduce_f32(ins: Sequence[np.ndarray]) -> list[np.ndarray]:
    count = int(np.asarray(ins[0]).size)
    return _f32_collective("orc_allreduce_f32", ins, [count] * len(ins))


def reduce_scatter_f32(ins: Sequence[np.ndarray]) -> list[np.ndarray]:
    n, count = len(ins), int(np.asarray(ins[0]).size)
    return _f32_collective("orc_reduce_scatter_f32", ins,
                           [shard_len(count, n, r) for r in range(n)])


def sent_sanitize_f32(x: np.ndarray) -> np.ndarray:
    x = _c(np.asarray(x).ravel(), np.uint32)
    out = x.copy()
    for i in np.flatnonzero(x == np.uint32(0xFFFFFFFF)):
        out[i] = lib().orc_sent_sanitize_f32(int(x[i]))
    return out


def sent_encode_f32(x: np.ndarray) -> np.ndarray:
    x = _c(np.asarray(x).ravel(), np.uint32)
    np_ = (x.size + 1) // 2
    out = np.zeros(max(np_, 1), dtype=np.uint64)
    lib().orc_sent_encode_f32(_ptr(x, ctypes.c_uint32), x.size, _ptr(out, ctypes.c_uint64))
    return out[:np_]


def sent_decode_f32(packs: np.ndarray, elems: int, fill: int = 0) -> tuple[np.ndarray, int]:
    packs = _c(packs, np.uint64)
    out = np.full(max(elems, 1), fill, dtype=np.uint32)
    skipped = lib().orc_sent_decode_f32(_ptr(packs, ctypes.c_uint64), elems,
                                        _ptr(out, ctypes.c_uint32))
    return out[:elems], int(skipped)


def one_sided_copy(src: np.ndarray) -> np.ndarray:
    """The bytes a one-sided copy (Purlin §3.3 Atom::copy) delivers: those
    of `src`, in order, as uint8."""
    b = _c(np.asarray(src).reshape(-1).view(np.uint8), np.uint8)
    out = np.zeros_like(b)
    lib().orc_one_sided_copy(_ptr(b, ctypes.c_uint8), b.size, _ptr(out, ctypes.c_uint8))
    return out

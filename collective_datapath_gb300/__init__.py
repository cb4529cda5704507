"""Python binding of the single-GPU collective datapath (libcoll.so).

Argument marshalling only: every step of the datapath runs in the CUDA
kernels behind the C ABI of ``include/coll.h``.  The functions keep the C
names (``coll_spec_create``, ``coll_stage``, ``coll_run``, ...) and take torch
tensors (device memory) and torch streams instead of raw pointers.  There is
no CPU fallback: importing the package fails when the library is missing.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libcoll.so")

if not os.path.exists(_LIB_PATH):
    raise ImportError(
        f"{_LIB_PATH} is missing: build it first "
        "(python -c 'import __graft_entry__ as g; g.build()')")

_lib = ctypes.CDLL(_LIB_PATH)

# ---- constants (coll.h) ------------------------------------------------------
COLL_PACKED, COLL_SCATTERED, COLL_TRANSPOSED = 0, 1, 2
COLL_PACKED_V, COLL_SCATTERED_V, COLL_TRANSPOSED_V = 3, 4, 5
COLL_COPY, COLL_REDUCE = 0, 1
COLL_BF16 = 0
COLL_F32 = 1
COLL_OK, COLL_ERR_INVALID, COLL_ERR_UNSUPPORTED, COLL_ERR_ALIGN = 0, 1, 2, 3
COLL_ERR_NOMEM, COLL_ERR_CUDA, COLL_ERR_TIMEOUT, COLL_ERR_STATE = 4, 5, 6, 7
COLL_LL8, COLL_LL128, COLL_SENT, COLL_ENC_AUTO = 0, 1, 2, 3
COLL_ALGO_AUTO, COLL_ONESHOT, COLL_TWOSHOT = 0, 1, 2
COLL_RESET_FUSED, COLL_RESET_KERNEL, COLL_RESET_NONE, COLL_RESET_DEFERRED = 0, 1, 2, 3
COLL_PATH_AUTO, COLL_PATH_FUSED, COLL_PATH_STREAMED, COLL_PATH_COMPOSED = 0, 1, 2, 3
COLL_ATOM_BULK, COLL_ATOM_LSU = 0, 1

# Every symbol include/coll.h declares (checked by the tests).
EXPORTS = [
    "coll_options_default", "coll_spec_create", "coll_workspace_bytes",
    "coll_buffer_elems", "coll_bind", "coll_set_routing", "coll_stage", "coll_run",
    "coll_run_host", "coll_get_counts", "coll_query_status", "coll_get_epoch",
    "coll_staging_layout", "coll_stage_withheld", "coll_run_late",
    "coll_get_rejections", "coll_debug_items", "coll_debug_plan",
    "coll_set_profile_events", "coll_last_launches", "coll_launch_floor",
    "coll_allreduce_static",
    "coll_atom_copy", "coll_copy_passes", "coll_destroy", "coll_status_string",
]


class coll_options_t(ctypes.Structure):
    _fields_ = [("encoding", ctypes.c_int), ("algorithm", ctypes.c_int),
                ("reset_mode", ctypes.c_int), ("path", ctypes.c_int),
                ("ctas", ctypes.c_int), ("tile_lines", ctypes.c_int),
                ("timeout_ns", ctypes.c_uint64), ("tokens", ctypes.c_int),
                ("hidden", ctypes.c_int), ("topk", ctypes.c_int),
                ("experts", ctypes.c_int), ("max_rows", ctypes.c_int),
                ("vcounts", ctypes.POINTER(ctypes.c_uint64)), ("nvcounts", ctypes.c_int),
                ("slots", ctypes.c_int), ("staging_bytes", ctypes.c_uint64)]


_vp = ctypes.c_void_p
_st = ctypes.c_int
_sz = ctypes.c_size_t
_P = ctypes.POINTER


def _sig(name, res, *args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = list(args)
    return f


_sig("coll_options_default", None, _P(coll_options_t))
_sig("coll_spec_create", _st, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
     ctypes.c_int, _sz, _P(coll_options_t), _P(_vp))
_sig("coll_workspace_bytes", _st, _vp, _P(_sz))
_sig("coll_buffer_elems", _st, _vp, ctypes.c_int, _P(_sz), _P(_sz))
_sig("coll_bind", _st, _vp, _vp, _sz, _vp)
_sig("coll_set_routing", _st, _vp, ctypes.c_int, _vp, _vp)
_sig("coll_stage", _st, _vp, ctypes.c_int, _vp, _vp)
_sig("coll_run", _st, _vp, _P(_vp), _P(_vp), _vp)
_sig("coll_run_host", _st, _vp, _P(_vp), _P(_vp), _P(_vp), _P(_vp), _vp)
_sig("coll_get_counts", _st, _vp, _vp, _vp)
_sig("coll_query_status", _st, _vp, _vp, _P(ctypes.c_int), _P(ctypes.c_int),
     _P(ctypes.c_int64))
_sig("coll_get_epoch", _st, _vp, _vp, _P(ctypes.c_uint64))
_sig("coll_staging_layout", _st, _vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
     ctypes.c_int, _P(ctypes.c_uint64), _P(ctypes.c_uint64), _P(ctypes.c_int))
_sig("coll_stage_withheld", _st, _vp, ctypes.c_int, _vp, _vp, _vp, _vp,
     ctypes.c_int64, _vp)
_sig("coll_run_late", _st, _vp, _P(_vp), _P(_vp), _P(_vp), _P(ctypes.c_int64), _vp)
_sig("coll_get_rejections", _st, _vp, _vp, _P(ctypes.c_uint64))
_sig("coll_debug_items", _st, _vp, ctypes.c_int, _P(ctypes.c_int64), _sz, _P(_sz))
_sig("coll_debug_plan", _st, _vp, _P(ctypes.c_int), _P(ctypes.c_int),
     _P(ctypes.c_int), _P(ctypes.c_int), _P(ctypes.c_int))
_sig("coll_set_profile_events", _st, _vp, _P(_vp), ctypes.c_int)
_sig("coll_last_launches", _st, _vp, _P(ctypes.c_int))
_sig("coll_launch_floor", _st, _vp, _vp)
_sig("coll_allreduce_static", _st, ctypes.c_int, _sz, _P(_vp), _P(_vp), _vp)
_sig("coll_atom_copy", _st, _vp, _vp, _sz, ctypes.c_int, ctypes.c_int, ctypes.c_int,
     ctypes.c_int, _vp, _vp)
_sig("coll_copy_passes", _st, _vp, _vp, _sz, ctypes.c_int, ctypes.c_int, _vp)
_sig("coll_destroy", _st, _vp)
_sig("coll_status_string", ctypes.c_char_p, ctypes.c_int)


class CollError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = _lib.coll_status_string(status).decode()
        super().__init__(f"{where}: {msg} (status {status})")


def _check(status: int, where: str) -> None:
    if status != COLL_OK:
        raise CollError(status, where)


def library_path() -> str:
    return _LIB_PATH


# ---- marshalling helpers -------------------------------------------------------

def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch

        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _ptr_array(ts: Sequence) -> ctypes.Array:
    arr = (_vp * len(ts))()
    for i, t in enumerate(ts):
        arr[i] = _ptr(t)
    return arr


def options(**kw) -> coll_options_t:
    o = coll_options_t()
    _lib.coll_options_default(ctypes.byref(o))
    vc = kw.pop("vcounts", None)
    for k, v in kw.items():
        if not hasattr(o, k):
            raise TypeError(f"unknown option {k}")
        setattr(o, k, v)
    if vc is not None:
        flat = [int(x) for row in vc for x in (row if hasattr(row, "__len__") else [row])]
        arr = (ctypes.c_uint64 * len(flat))(*flat)
        o._vcounts_keepalive = arr
        o.vcounts = ctypes.cast(arr, ctypes.POINTER(ctypes.c_uint64))
        o.nvcounts = len(flat)
    return o


# ---- the C ABI, one function each ------------------------------------------------

def coll_spec_create(in_layout: int, out_layout: int, op: int, nranks: int,
                     count: int, dtype: int = COLL_BF16, **opts) -> int:
    spec = _vp()
    o = options(**opts)
    _check(_lib.coll_spec_create(in_layout, out_layout, op, dtype, nranks, count,
                                 ctypes.byref(o), ctypes.byref(spec)),
           "coll_spec_create")
    return spec.value


def coll_workspace_bytes(spec: int) -> int:
    n = _sz()
    _check(_lib.coll_workspace_bytes(spec, ctypes.byref(n)), "coll_workspace_bytes")
    return n.value


def coll_buffer_elems(spec: int, rank: int) -> tuple[int, int]:
    a, b = _sz(), _sz()
    _check(_lib.coll_buffer_elems(spec, rank, ctypes.byref(a), ctypes.byref(b)),
           "coll_buffer_elems")
    return a.value, b.value


def coll_bind(spec: int, workspace, stream=None) -> None:
    nbytes = workspace.numel() * workspace.element_size()
    _check(_lib.coll_bind(spec, _ptr(workspace), nbytes, _stream_handle(stream)),
           "coll_bind")


def coll_set_routing(spec: int, rank: int, topk, stream=None) -> None:
    _check(_lib.coll_set_routing(spec, rank, _ptr(topk), _stream_handle(stream)),
           "coll_set_routing")


def coll_stage(spec: int, rank: int, x, stream=None) -> None:
    _check(_lib.coll_stage(spec, rank, _ptr(x), _stream_handle(stream)), "coll_stage")


def coll_run(spec: int, ins: Optional[Sequence], outs: Sequence, stream=None) -> None:
    in_arr = _ptr_array(ins) if ins is not None else None
    _check(_lib.coll_run(spec, in_arr, _ptr_array(outs), _stream_handle(stream)),
           "coll_run")


def coll_run_host(spec: int, host_ins: Sequence, dev_ins: Sequence, dev_outs: Sequence,
                  host_outs: Sequence, stream=None) -> None:
    _check(_lib.coll_run_host(spec, _ptr_array(host_ins), _ptr_array(dev_ins),
                              _ptr_array(dev_outs), _ptr_array(host_outs),
                              _stream_handle(stream)), "coll_run_host")


def coll_get_counts(spec: int, counts, stream=None) -> None:
    _check(_lib.coll_get_counts(spec, _ptr(counts), _stream_handle(stream)),
           "coll_get_counts")


def coll_query_status(spec: int, stream=None) -> tuple[int, int, int]:
    code, rank, line = ctypes.c_int(), ctypes.c_int(), ctypes.c_int64()
    _check(_lib.coll_query_status(spec, _stream_handle(stream), ctypes.byref(code),
                                  ctypes.byref(rank), ctypes.byref(line)),
           "coll_query_status")
    return code.value, rank.value, line.value


def coll_get_epoch(spec: int, stream=None) -> int:
    e = ctypes.c_uint64()
    _check(_lib.coll_get_epoch(spec, _stream_handle(stream), ctypes.byref(e)),
           "coll_get_epoch")
    return e.value


def coll_staging_layout(spec: int, region: int, slot: int, rank: int,
                        seg: int) -> tuple[int, int, int]:
    off, lines, lb = ctypes.c_uint64(), ctypes.c_uint64(), ctypes.c_int()
    _check(_lib.coll_staging_layout(spec, region, slot, rank, seg, ctypes.byref(off),
                                    ctypes.byref(lines), ctypes.byref(lb)),
           "coll_staging_layout")
    return off.value, lines.value, lb.value


def coll_stage_withheld(spec: int, rank: int, x, lines, kind, poison,
                        stream=None) -> None:
    _check(_lib.coll_stage_withheld(spec, rank, _ptr(x), _ptr(lines), _ptr(kind),
                                    _ptr(poison), int(lines.numel()),
                                    _stream_handle(stream)), "coll_stage_withheld")


def coll_run_late(spec: int, ins: Sequence, outs: Sequence, orders: Sequence,
                  stream=None) -> None:
    n = (ctypes.c_int64 * len(orders))(*[int(o.numel()) for o in orders])
    _check(_lib.coll_run_late(spec, _ptr_array(ins), _ptr_array(outs),
                              _ptr_array(orders), n, _stream_handle(stream)),
           "coll_run_late")


def coll_get_rejections(spec: int, stream=None) -> int:
    r = ctypes.c_uint64()
    _check(_lib.coll_get_rejections(spec, _stream_handle(stream), ctypes.byref(r)),
           "coll_get_rejections")
    return r.value


def coll_debug_items(spec: int, which: int):
    import numpy as np

    n = _sz()
    _check(_lib.coll_debug_items(spec, which, None, 0, ctypes.byref(n)),
           "coll_debug_items")
    buf = np.zeros((max(n.value, 1), 10), dtype=np.int64)
    _check(_lib.coll_debug_items(spec, which,
                                 buf.ctypes.data_as(_P(ctypes.c_int64)), n.value,
                                 ctypes.byref(n)), "coll_debug_items")
    return buf[:n.value]


def coll_debug_plan(spec: int) -> dict:
    a, p, c, e, d = (ctypes.c_int() for _ in range(5))
    _check(_lib.coll_debug_plan(spec, ctypes.byref(a), ctypes.byref(p), ctypes.byref(c),
                                ctypes.byref(e), ctypes.byref(d)), "coll_debug_plan")
    return {"algorithm": a.value, "path": p.value, "ctas_per_rank": c.value,
            "encoding": e.value, "dependent_launch": d.value}


def coll_set_profile_events(spec: int, events: Sequence) -> None:
    """events: torch.cuda.Event objects (or raw cudaEvent_t handles)."""
    handles = [e if isinstance(e, int) else e.cuda_event for e in events]
    if any(not h for h in handles):
        raise ValueError("an event has no CUDA handle yet (record it once first)")
    arr = (_vp * max(len(handles), 1))(*handles)
    _check(_lib.coll_set_profile_events(spec, arr, len(handles)),
           "coll_set_profile_events")


def coll_last_launches(spec: int) -> int:
    n = ctypes.c_int()
    _check(_lib.coll_last_launches(spec, ctypes.byref(n)), "coll_last_launches")
    return n.value


def coll_launch_floor(spec: int, stream=None) -> None:
    """One empty kernel in the spec's one-launch configuration (measurement)."""
    _check(_lib.coll_launch_floor(spec, _stream_handle(stream)), "coll_launch_floor")


def coll_allreduce_static(ins: Sequence, outs: Sequence, count: int, stream=None) -> None:
    """All-reduce in the library's fixed scratch (no workspace, no allocation)."""
    _check(_lib.coll_allreduce_static(len(ins), count, _ptr_array(ins), _ptr_array(outs),
                                      _stream_handle(stream)), "coll_allreduce_static")


def coll_atom_copy(dst, src, nbytes: int, engine: int = COLL_ATOM_BULK, ctas: int = 0,
                   stages: int = 8, stage_bytes: int = 16384, status=None,
                   stream=None) -> None:
    """One-sided copy of `nbytes` from `src` to `dst` (device tensors) with
    `ctas` CTAs of `stages` pipeline stages of `stage_bytes` each."""
    _check(_lib.coll_atom_copy(_ptr(dst), _ptr(src), nbytes, engine, ctas, stages, stage_bytes,
                               _ptr(status), _stream_handle(stream)), "coll_atom_copy")


def coll_copy_passes(dst, src, nbytes: int, passes: int, ctas: int = 0, stream=None) -> None:
    """`passes` copies of `nbytes` from `src` to `dst` in one launch (a copy
    ceiling probe: buffers that fit L2 give the SM <-> L2 copy rate)."""
    _check(_lib.coll_copy_passes(_ptr(dst), _ptr(src), nbytes, passes, ctas,
                                 _stream_handle(stream)), "coll_copy_passes")


def coll_destroy(spec: int) -> None:
    _check(_lib.coll_destroy(spec), "coll_destroy")


def coll_status_string(status: int) -> str:
    return _lib.coll_status_string(status).decode()


# ---- convenience ---------------------------------------------------------------

ALLREDUCE = (COLL_SCATTERED, COLL_SCATTERED, COLL_REDUCE)
REDUCE_SCATTER = (COLL_SCATTERED, COLL_PACKED, COLL_REDUCE)
ALLGATHER = (COLL_PACKED, COLL_SCATTERED, COLL_COPY)
ALLTOALL = (COLL_SCATTERED, COLL_TRANSPOSED, COLL_COPY)
REDUCE_SCATTER_V = (COLL_SCATTERED_V, COLL_PACKED_V, COLL_REDUCE)
ALLGATHER_V = (COLL_PACKED_V, COLL_SCATTERED_V, COLL_COPY)
ALLTOALL_V = (COLL_SCATTERED_V, COLL_TRANSPOSED_V, COLL_COPY)
MOE_DISPATCH = (COLL_SCATTERED_V, COLL_TRANSPOSED_V, COLL_COPY)


class Collective:
    """A spec bound to a torch-allocated workspace on the current device."""

    def __init__(self, triple, nranks: int, count: int, stream=None, **opts):
        import torch

        self.spec = coll_spec_create(*triple, nranks, count, **opts)
        self.nranks = nranks
        nbytes = coll_workspace_bytes(self.spec)
        # 256-byte aligned device memory owned by the caller (torch)
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
        coll_bind(self.spec, self.workspace, stream)

    def elems(self, rank: int) -> tuple[int, int]:
        return coll_buffer_elems(self.spec, rank)

    def stage(self, rank: int, x, stream=None) -> None:
        coll_stage(self.spec, rank, x, stream)

    def run(self, ins, outs, stream=None) -> None:
        coll_run(self.spec, ins, outs, stream)

    def status(self, stream=None) -> tuple[int, int, int]:
        return coll_query_status(self.spec, stream)

    def epoch(self, stream=None) -> int:
        return coll_get_epoch(self.spec, stream)

    def plan(self) -> dict:
        return coll_debug_plan(self.spec)

    def close(self) -> None:
        if self.spec:
            coll_destroy(self.spec)
            self.spec = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

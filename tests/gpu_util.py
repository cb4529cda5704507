"""Helpers of the GPU tests: move uint16 bit patterns to and from the device,
build a bound collective, and read back staging lines.  No arithmetic."""
from __future__ import annotations

import numpy as np


def to_dev(x: np.ndarray):
    import torch

    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.uint16).view(np.int16)).cuda()


def from_dev(t) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16).copy()


def empty_dev(elems: int):
    import torch

    return torch.empty(max(elems, 8), dtype=torch.int16, device="cuda")


def make(cd, triple, n, count, **opts):
    return cd.Collective(triple, n, count, **opts)


def buffers(coll, n, seed, dist="normal", tag=0):
    """Seeded inputs (host numpy and device tensors) and device outputs."""
    import synth

    ins_h, ins_d, outs_d = [], [], []
    for r in range(n):
        ie, oe = coll.elems(r)
        if dist == "normal":
            x = synth.normal_bf16(seed, ie, tag, r)
        elif dist == "uniform1":
            x = synth.uniform_bf16(seed, ie, -1.0, 1.0, tag, r)
        elif dist == "uniform4":
            x = synth.uniform_bf16(seed, ie, -4.0, 4.0, tag, r)
        else:
            x = synth.random_bits16(seed, ie, tag, r)
        ins_h.append(x)
        ins_d.append(to_dev(x))
        t = empty_dev(oe)
        t.fill_(0x5A5A)
        outs_d.append(t)
    return ins_h, ins_d, outs_d


def read_lines(coll, region, slot, rank, seg):
    """(lines, line_bytes) raw bytes of one staged segment."""
    import collective_datapath_gb300 as cd

    off, lines, lb = cd.coll_staging_layout(coll.spec, region, slot, rank, seg)
    raw = coll.workspace[off:off + lines * lb].cpu().numpy()
    return raw, lines, lb

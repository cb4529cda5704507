"""Offline calibration of the all-reduce policy table.

flash-comm §3.2 ("Cost-guided protocol selection") and §4.1: within a stable
band the latency of a protocol p is T_p(S) = a_p + b_p S; the crossing of two
neighbouring protocols' locally fitted lines marks the switching region, the
sizes around it are measured, and the boundary is placed on a measured
point.  The runtime then does a constant-time lookup by group size and
message size.  This module does the offline part:

  1. measure every candidate (readiness encoding x one-/two-shot x launch
     path) on a grid of sizes (bytes per rank, powers of two);
  2. take the fastest candidate at each grid size;
  3. for each change of winner between grid sizes s_i and s_i+1, fit both
     candidates' lines on (s_i, s_i+1), compute the crossing, measure a few
     sizes around it and put the boundary on the largest measured size where
     the left candidate is still the faster;
  4. write `csrc/policy_table.h`, which the library compiles in.

Steps 2-3 are plain functions of measured numbers (tested on the CPU with
synthetic cost lines); step 1 needs a GPU.  Run on a GB300 with
`python -m collective_datapath_gb300.tune --write` after building.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
from dataclasses import dataclass
from typing import Callable, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
TABLE_PATH = os.path.join(HERE, "csrc", "policy_table.h")

# encoding, algorithm and path codes of coll.h
LL8, LL128, SENT = 0, 1, 2
ONESHOT, TWOSHOT = 1, 2
FUSED, STREAMED, COMPOSED = 1, 2, 3
ENC_NAMES = {LL8: "LL8", LL128: "LL128", SENT: "SENT"}
ALGO_NAMES = {ONESHOT: "oneshot", TWOSHOT: "twoshot"}
PATH_NAMES = {FUSED: "fused", STREAMED: "streamed", COMPOSED: "composed"}


# Launch shape of the one-launch path: 0 = one CTA per SM (the default),
# WIDE = every co-resident CTA (the library clamps the request); NARROW = 64
# CTAs in all (8 per rank at 8 ranks: for the smallest messages, fewer CTAs
# mean fewer arrivals and cross-CTA line polls).
WIDE = 1024
NARROW = 64


@dataclass(frozen=True, order=True)
class Candidate:
    enc: int
    algo: int
    path: int
    ctas: int = 0

    def name(self) -> str:
        shape = {0: "", WIDE: "/wide", NARROW: "/narrow"}.get(self.ctas, f"/ctas{self.ctas}")
        return f"{ENC_NAMES[self.enc]}/{ALGO_NAMES[self.algo]}/{PATH_NAMES[self.path]}{shape}"


def candidates_for(nbytes: int) -> list[Candidate]:
    """The protocols worth measuring at one size (bytes per rank): one
    cooperative launch only up to 4 MiB (in two launch shapes, three up to
    256 KiB), the composed launch from 256 KiB."""
    out = []
    for enc in (LL8, SENT, LL128):
        for algo in (ONESHOT, TWOSHOT):
            for path in (FUSED, STREAMED, COMPOSED):
                if path == FUSED and nbytes > (4 << 20):
                    continue
                if path == COMPOSED and (enc != LL128 or algo != TWOSHOT or nbytes < (256 << 10)):
                    continue
                if enc == LL128 and path == FUSED:
                    continue
                out.append(Candidate(enc, algo, path))
                if path == FUSED:
                    out.append(Candidate(enc, algo, path, WIDE))
                    if nbytes <= (256 << 10):
                        out.append(Candidate(enc, algo, path, NARROW))
    return out


# ---- selection (pure functions of measured times) ----------------------------

def fit_line(s0: float, t0: float, s1: float, t1: float) -> tuple[float, float]:
    """(a, b) of T = a + b S through two measured points."""
    b = (t1 - t0) / (s1 - s0)
    return t0 - b * s0, b


def crossing(fa: tuple[float, float], fb: tuple[float, float]) -> float | None:
    """Size where two lines meet (None if parallel)."""
    (aa, ba), (ab, bb) = fa, fb
    if ba == bb:
        return None
    return (ab - aa) / (ba - bb)


# A protocol keeps its band while it is within this fraction of the fastest
# (flash-comm §3.2 "stable protocol band"): measurement noise of a few
# percent does not flip the choice back and forth between neighbours.
TOLERANCE = 0.03


def winners(times: dict[int, dict[Candidate, float]],
            tol: float = TOLERANCE) -> list[tuple[int, Candidate]]:
    """Winner at every measured size, in increasing size: the fastest, unless
    the previous size's winner is within `tol` of it."""
    out: list[tuple[int, Candidate]] = []
    for s in sorted(times):
        best = min(times[s], key=lambda c: (times[s][c], c))
        if out and out[-1][1] in times[s] and \
                times[s][out[-1][1]] <= (1.0 + tol) * times[s][best]:
            best = out[-1][1]
        out.append((s, best))
    return out


def probe_sizes(s0: int, s1: int, s_cross: float | None, k: int = 4) -> list[int]:
    """Sizes to measure between s0 and s1 (exclusive), multiples of 16 KiB
    around the fitted crossing (geometrically spread when there is none)."""
    step = 16 << 10
    if s_cross is None or not (s0 < s_cross < s1):
        s_cross = math.sqrt(s0 * s1)
    pts = set()
    for f in (0.5, 0.75, 1.0, 1.25, 1.5)[:k + 1]:
        v = int(round(s_cross * f / step)) * step
        if s0 < v < s1:
            pts.add(v)
    return sorted(pts)


def build_policy(times: dict[int, dict[Candidate, float]],
                 measure: Callable[[int, Candidate], float],
                 tol: float = TOLERANCE) -> list[tuple[int, Candidate]]:
    """Entries (max bytes per rank, candidate) in increasing size, the last
    open-ended (max = 2^64 - 1).  `measure(size, cand)` times one more point."""
    win = winners(times, tol)
    entries: list[tuple[int, Candidate]] = []
    for (s0, c0), (s1, c1) in zip(win, win[1:]):
        if c0 == c1:
            continue
        fa = fit_line(s0, times[s0][c0], s1, times[s1][c0]) if c0 in times[s1] else None
        fb = fit_line(s0, times[s0][c1], s1, times[s1][c1]) if c1 in times[s0] else None
        s_cross = crossing(fa, fb) if fa and fb else None
        boundary = s0
        for s in probe_sizes(s0, s1, s_cross):
            if measure(s, c0) <= (1.0 + tol) * measure(s, c1):
                boundary = s          # the left candidate still holds its band here
            else:
                break
        entries.append((boundary, c0))
    entries.append(((1 << 64) - 1, win[-1][1]))
    # merge neighbours that chose the same candidate
    merged: list[tuple[int, Candidate]] = []
    for m, c in entries:
        if merged and merged[-1][1] == c:
            merged[-1] = (m, c)
        else:
            merged.append((m, c))
    return merged


def lookup(table: Sequence[tuple[int, Candidate]], nbytes: int) -> Candidate:
    for m, c in table:
        if nbytes <= m:
            return c
    return table[-1][1]


def header_text(tables: dict[int, list[tuple[int, Candidate]]], note: str) -> str:
    lines = [
        "// policy_table.h -- all-reduce policy per group size, written by",
        "// collective_datapath_gb300/tune.py from measurements; do not edit by hand.",
        f"// {note}",
        "// Entries: bytes per rank up to max_bytes use (encoding, algorithm, path).",
        "#pragma once",
        "",
        "#include <cstdint>",
        "",
        "namespace coll {",
        "",
        "struct PolicyEntry {",
        "  uint64_t max_bytes;",
        "  int enc, algo, path;",
        "  int ctas;  // launch shape of the one-launch path (0 = one CTA per SM)",
        "};",
        "",
    ]
    for n in sorted(tables):
        lines.append(f"constexpr PolicyEntry kPolicy{n}[] = {{")
        for m, c in tables[n]:
            mx = "UINT64_MAX" if m >= (1 << 64) - 1 else f"{m}ull"
            lines.append(f"    {{{mx}, {c.enc}, {c.algo}, {c.path}, {c.ctas}}},  // {c.name()}")
        lines.append("};")
    lines.append("")
    lines.append("// group sizes with a table, in increasing order")
    lines.append("constexpr int kPolicyGroups[] = {" + ", ".join(str(n) for n in sorted(tables)) + "};")
    lines.append("")
    lines.append("inline const PolicyEntry* policy_table(int group, int* len) {")
    lines.append("  switch (group) {")
    for n in sorted(tables):
        lines.append(f"    case {n}: *len = (int)(sizeof(kPolicy{n}) / sizeof(PolicyEntry)); return kPolicy{n};")
    lines.append("    default: *len = 0; return nullptr;")
    lines.append("  }")
    lines.append("}")
    lines.append("")
    lines.append("}  // namespace coll")
    lines.append("")
    return "\n".join(lines)


def parse_header(text: str) -> dict[int, list[tuple[int, Candidate]]]:
    """The tables of a policy_table.h (for tests and reports)."""
    tables: dict[int, list[tuple[int, Candidate]]] = {}
    cur = None
    for ln in text.splitlines():
        ln = ln.strip()
        if ln.startswith("constexpr PolicyEntry kPolicy"):
            cur = int(ln.split("kPolicy")[1].split("[")[0])
            tables[cur] = []
        elif cur is not None and ln.startswith("{"):
            body = ln[1:ln.index("}")]
            fields = [x.strip() for x in body.split(",")]
            m, e, a, p = fields[:4]
            w = int(fields[4]) if len(fields) > 4 else 0
            mx = (1 << 64) - 1 if m == "UINT64_MAX" else int(m.rstrip("ul"))
            tables[cur].append((mx, Candidate(int(e), int(a), int(p), w)))
        elif ln.startswith("};"):
            cur = None
    return tables


# ---- measurement (GPU) ---------------------------------------------------------------

def time_op(cd, n: int, nbytes: int, cand: Candidate, stream) -> float:
    """Warm µs per all-reduce: K ops captured in one CUDA graph, replayed."""
    import torch

    count = nbytes // 2
    coll = cd.Collective(cd.ALLREDUCE, n, count, encoding=cand.enc, algorithm=cand.algo,
                         path=cand.path, ctas=cand.ctas)
    g = torch.Generator(device="cuda")
    g.manual_seed(nbytes + n)
    ins = [(torch.rand(count, generator=g, device="cuda") * 8 - 4).to(torch.bfloat16)
           .view(torch.int16) for _ in range(n)]
    outs = [torch.empty(count, dtype=torch.int16, device="cuda") for _ in range(n)]
    torch.cuda.synchronize()  # inputs are drawn on torch's stream
    k = 64 if nbytes <= (1 << 20) else (16 if nbytes <= (16 << 20) else 4)
    with torch.cuda.stream(stream):
        for _ in range(3):
            coll.run(ins, outs, stream)
        graph = torch.cuda.CUDAGraph()
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(k):
                coll.run(ins, outs, stream)
        graph.replay()
        per = []
        for _ in range(5):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            stream.synchronize()
            per.append(e0.elapsed_time(e1) * 1e3 / k)
    code = coll.status(stream)[0]
    coll.close()
    del coll, ins, outs, graph
    if code != cd.COLL_OK:
        raise RuntimeError(f"{cand.name()} at {nbytes} B: device status {code}")
    return statistics.median(per)


def calibrate(cd, n: int, sizes: Sequence[int], stream, log) -> tuple[list, dict]:
    cache: dict[tuple[int, Candidate], float] = {}

    def measure(s: int, c: Candidate) -> float:
        if (s, c) not in cache:
            cache[(s, c)] = time_op(cd, n, s, c, stream)
            log(f"N={n} {s:>10} B {c.name():<26} {cache[(s, c)]:9.2f} us")
        return cache[(s, c)]

    times = {s: {c: measure(s, c) for c in candidates_for(s)} for s in sizes}
    table = build_policy(times, measure)
    return table, {f"{s} {c.name()}": t for (s, c), t in sorted(cache.items())}


def main() -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--groups", default="2,4,8")
    ap.add_argument("--max-mib", type=int, default=64)
    ap.add_argument("--write", action="store_true", help="rewrite the policy table header")
    ap.add_argument("--out", default=TABLE_PATH, help="where --write puts the header")
    ap.add_argument("--json", default=None, help="write every measured point here")
    args = ap.parse_args()
    import torch

    import collective_datapath_gb300 as cd

    stream = torch.cuda.Stream()
    sizes = [1 << k for k in range(13, 21 + int(math.log2(args.max_mib)))]
    tables, points = {}, {}
    for n in (int(x) for x in args.groups.split(",")):
        tables[n], points[n] = calibrate(cd, n, sizes, stream, print)
        for m, c in tables[n]:
            print(f"N={n}: up to {m} B -> {c.name()}")
    name = torch.cuda.get_device_name()
    note = f"measured on {name}, warm (CUDA graph) us per op, sizes 8 KiB - {args.max_mib} MiB per rank"
    if args.write:
        with open(args.out, "w") as f:
            f.write(header_text(tables, note))
    if args.json:
        with open(args.json, "w") as f:
            json.dump({"note": note, "points": points,
                       "tables": {n: [(m, c.name()) for m, c in t] for n, t in tables.items()}},
                      f, indent=1)
    return 0


if __name__ == "__main__":
    raise SystemExit(main())

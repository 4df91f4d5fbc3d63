"""Plain restatement of the page's hints analyzer — TEST INFRASTRUCTURE.

KernelScope backend doc, hints/analyzer.py (analyze_trace_hints) and
simulator/engine.py (analyze_global_memory_access: efficiency = min(1,
ideal / transactions), ideal = ceil(active threads * access size / 128)).
Written from the page's rules for use by the tests only; the library's
ks_hints computes the same from a GPU-side per-instruction profile.

Readings (the page leaves them open): efficiencies and ratios are exact
fractions and their percentages exact floors; the divergence ratio of a
branch that splits its active lanes is the smaller side over the active
lanes; one hint per (instruction, rule) stands for all of that
instruction's events (the page emits one per event), carrying their number
and the worst event's value.

Parity pinned by: the page's thresholds and messages on hand-made event
lists (tests/test_hints.py), and the page's own coalescing and bank-conflict
examples through the oracle's event recorder.
"""
from __future__ import annotations

from fractions import Fraction
from math import floor

import numpy as np

EV_GLOBAL, EV_SHARED, EV_DIVERGE = 0, 1, 2
INFO, WARNING, CRITICAL = 0, 1, 2
MEMORY, DIVERGENCE, OCCUPANCY, REGISTERS = 0, 1, 2, 3

PROFILE_DTYPE = np.dtype([
    ("requests", "<u8"), ("poor", "<u8"), ("uncoalesced", "<u8"), ("conflicted", "<u8"), ("severe", "<u8"),
    ("divergent", "<u8"), ("high_divergence", "<u8"), ("degrees", "<u4"), ("poor_pcts", "<u4"),
    ("high_div_pcts", "<u8")])
assert PROFILE_DTYPE.itemsize == 72


def global_efficiency(lanes: int, lines: int, size: int) -> Fraction:
    ideal = (lanes * size + 127) // 128
    return min(Fraction(1), Fraction(ideal, lines))


def divergence_ratio(taken: int, fall: int) -> Fraction:
    return Fraction(min(taken, fall), taken + fall)


def event_hints(events, occupancy: dict | None = None) -> list[dict]:
    """The page's analyze_trace_hints over an event list: per-event hints in
    event order, then the launch-wide ones."""
    hints = []
    bank_conflict_events = 0
    divergent_events = 0
    for idx, e in enumerate(events):
        kind, pc = int(e["kind"]), int(e["pc"])
        if kind == EV_SHARED:
            conflict = int(e["a"])
            if conflict > 1:
                bank_conflict_events += 1
            if conflict >= 8:
                hints.append(dict(category=MEMORY, severity=CRITICAL, pc=pc, rule="bank",
                                  value=conflict, message=f"{conflict}-way bank conflict",
                                  detail="Severe bank conflict causing serialized access"))
            elif conflict > 1:
                hints.append(dict(category=MEMORY, severity=WARNING, pc=pc, rule="bank",
                                  value=conflict, message=f"{conflict}-way bank conflict",
                                  detail="Bank conflict reducing throughput"))
        elif kind == EV_GLOBAL:
            eff = global_efficiency(int(e["a"]), int(e["b"]), int(e["c"]))
            if eff < Fraction(1, 4):
                pct = floor(eff * 100)
                hints.append(dict(category=MEMORY, severity=CRITICAL, pc=pc, rule="coalescing", value=pct,
                                  message=f"Poor memory efficiency ({pct}%)",
                                  detail="Scattered access causing many transactions"))
        elif kind == EV_DIVERGE:
            divergent_events += 1
            ratio = divergence_ratio(int(e["a"]), int(e["b"]))
            if ratio > Fraction(2, 5):
                pct = floor(ratio * 100)
                hints.append(dict(category=DIVERGENCE, severity=WARNING, pc=pc, rule="divergence", value=pct,
                                  message=f"High divergence ({pct}%)",
                                  detail="Significant warp divergence at this branch"))
    tail = []
    if bank_conflict_events > 5:
        tail.append(dict(category=MEMORY, severity=WARNING, pc=-1, count=bank_conflict_events,
                         message=f"Shared memory bank conflicts ({bank_conflict_events} events)",
                         detail="Consider padding arrays or restructuring access patterns"))
    if divergent_events > 3:
        tail.append(dict(category=DIVERGENCE, severity=WARNING, pc=-1, count=divergent_events,
                         message=f"Branch divergence detected ({divergent_events} events)",
                         detail="Consider restructuring conditionals or using predication"))
    if occupancy:
        occ_percent = occupancy.get("occupancy_percent", 100)
        limiting = occupancy.get("limiting_factor", "")
        if occ_percent < 25:
            tail.append(dict(category=OCCUPANCY, severity=CRITICAL, pc=-1, count=1,
                             message=f"Very low occupancy ({occ_percent}%)",
                             detail=f"Limited by {limiting}. Consider reducing resource usage."))
        elif occ_percent < 50:
            tail.append(dict(category=OCCUPANCY, severity=WARNING, pc=-1, count=1,
                             message=f"Low occupancy ({occ_percent}%)", detail=f"Limited by {limiting}."))
    return hints, tail


def aggregate(events, occupancy: dict | None = None) -> list[dict]:
    """One hint per (instruction, rule, severity) in the order the library
    emits them: by instruction, then bank CRITICAL, bank WARNING, coalescing,
    divergence; then the launch-wide hints."""
    per_event, tail = event_hints(events, occupancy)
    order = {("bank", CRITICAL): 0, ("bank", WARNING): 1, ("coalescing", CRITICAL): 2, ("divergence", WARNING): 3}
    groups: dict = {}
    for h in per_event:
        key = (h["pc"], order[(h["rule"], h["severity"])])
        g = groups.setdefault(key, dict(h, count=0, values=[]))
        g["count"] += 1
        g["values"].append(h["value"])
    out = []
    for key in sorted(groups):
        g = groups[key]
        worst = min(g["values"]) if g["rule"] == "coalescing" else max(g["values"])
        msg = {"bank": f"{worst}-way bank conflict", "coalescing": f"Poor memory efficiency ({worst}%)",
               "divergence": f"High divergence ({worst}%)"}[g["rule"]]
        out.append(dict(category=g["category"], severity=g["severity"], pc=g["pc"], count=g["count"],
                        message=msg, detail=g["detail"]))
    return out + tail


def profile(events, n_entries: int) -> np.ndarray:
    """The per-instruction profile record (PROFILE_DTYPE) of an event list."""
    p = np.zeros(n_entries, dtype=PROFILE_DTYPE)
    for e in events:
        kind, pc = int(e["kind"]), int(e["pc"])
        r = p[pc]
        if kind == EV_GLOBAL:
            r["requests"] += 1
            eff = global_efficiency(int(e["a"]), int(e["b"]), int(e["c"]))
            if eff < Fraction(1, 4):
                r["poor"] += 1
                r["poor_pcts"] |= np.uint32(1 << floor(eff * 100))
            elif eff < Fraction(1, 2):
                r["uncoalesced"] += 1
        elif kind == EV_SHARED:
            d = int(e["a"])
            r["requests"] += 1
            r["conflicted"] += d > 1
            r["severe"] += d >= 8
            r["degrees"] |= np.uint32(1 << (d - 1))
        elif kind == EV_DIVERGE:
            r["divergent"] += 1
            ratio = divergence_ratio(int(e["a"]), int(e["b"]))
            if ratio > Fraction(2, 5):
                r["high_divergence"] += 1
                r["high_div_pcts"] |= np.uint64(1 << floor(ratio * 100))
        p[pc] = r
    return p

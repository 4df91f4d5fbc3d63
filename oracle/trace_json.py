"""Trace slots to Chrome trace-event JSON (the format Perfetto opens), written
out plainly: the post-processing step the CuTeDSL IKET 浅析 page describes
(§3, "postprocess → Perfetto trace") applied to the slot layout of §2.

TEST INFRASTRUCTURE ONLY: the reference the library's ks_trace_to_json is
compared with. Shares no code with the library.

One process per CTA ("CTA c"), one thread per warp ("warp w", w counted in
the CTA); a complete event "warp" from 0 to the slot's cycle count; then per
record: range_start -> "B", range_end -> "E", mark -> instant "i" (thread
scope), with args {"id": event id} plus {"payload": raw bits} for payload
events. Record stamps hold the low 24 bits of the cycle: they are unwrapped
in record order (a warp's stamps never decrease). ts = cycles / cycles_per_us.
"""
import struct

from . import event_info, record_bytes


def trace_events(ptx, kernel, grid, block, max_ts, trace, cycles_per_us):
    events = event_info(ptx, kernel)
    rb = record_bytes(ptx, kernel)
    slot = (16 + rb * max_ts + 7) // 8 * 8
    wpc = (block + 31) // 32
    out = []
    for cta in range(grid):
        out.append({"name": "process_name", "ph": "M", "pid": cta, "tid": 0, "args": {"name": f"CTA {cta}"}})
        for w in range(wpc):
            gw = cta * wpc + w
            base = gw * slot
            n_events, fmt, bpe, n_dropped, cycles = struct.unpack_from("<IBBHQ", trace, base)
            out.append({"name": "thread_name", "ph": "M", "pid": cta, "tid": w, "args": {"name": f"warp {w}"}})
            out.append({"name": "warp", "ph": "X", "pid": cta, "tid": w, "ts": 0 / cycles_per_us,
                        "dur": cycles / cycles_per_us})
            full = 0
            for i in range(min(n_events, max_ts)):
                r = base + 16 + rb * i
                word = struct.unpack_from("<I", trace, r)[0]
                eid, ts24 = word >> 24, word & 0xFFFFFF
                full += (ts24 - (full & 0xFFFFFF)) & 0xFFFFFF
                kind, pbytes, name = events[eid]
                ev = {"name": name, "ph": ("i", "B", "E")[kind], "pid": cta, "tid": w, "ts": full / cycles_per_us,
                      "args": {"id": eid}}
                if kind == 0:
                    ev["s"] = "t"
                if pbytes:
                    ev["args"]["payload"] = (struct.unpack_from("<I", trace, r + 4)[0] if rb == 8
                                             else struct.unpack_from("<Q", trace, r + 8)[0])
                out.append(ev)
    return {"traceEvents": out, "displayTimeUnit": "ns"}

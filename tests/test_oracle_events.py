"""Oracle pins for IKET payload events: record sizes from the page, slot
bytes derived by hand (timestamps from the scoreboard, payload from the
warp's lowest active lane), drops, mixed payload sizes. CPU only."""
import os
import struct

import numpy as np
import pytest

import oracle
from simt_ptx_interpretation_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden():
    rows = {}
    for line in open(os.path.join(GOLDEN, "iket_slot_sizing.txt")):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split(None, 1)
            rows[k] = v
    return rows


def kernel(body: str) -> str:
    return wl.HEADER + f""".visible .entry ev()
{{
    .reg .pred %p<2>;
    .reg .b32 %r<4>;
    .reg .f32 %f<2>;
    .reg .b64 %rd<3>;
{body}
}}
"""


def slots(ptx, block, max_ts=4, grid=1):
    r = oracle.run(ptx, "ev", grid, block, b"", [], max_ts=max_ts, trace=True)
    assert r.status == 0
    rb = oracle.record_bytes(ptx, "ev")
    sb = oracle.slot_bytes(max_ts, rb)
    return r, rb, [bytes(r.trace[i * sb:(i + 1) * sb]) for i in range(len(r.stats))]


def test_record_sizes_follow_the_page():
    g = golden()
    assert oracle.record_bytes(kernel("    //@iket mark a\n    ret;"), "ev") == int(g["bytes_per_event_no_payload"])
    assert oracle.record_bytes(kernel("    //@iket mark a %r1\n    ret;"), "ev") == int(g["bytes_per_event_payload_4"])
    assert oracle.record_bytes(kernel("    //@iket mark a %f1\n    ret;"), "ev") == int(g["bytes_per_event_payload_4"])
    assert oracle.record_bytes(kernel("    //@iket mark a %rd1\n    ret;"), "ev") == int(g["bytes_per_event_payload_8"])
    # a kernel's slots use its largest record
    assert oracle.record_bytes(kernel("    //@iket mark a\n    //@iket mark b %r1\n    ret;"), "ev") == 8
    assert oracle.slot_bytes(3, 16) == (16 + 48 + 7) // 8 * 8


PAYLOADS = """    mov.u32 %r1, %tid.x;
    //@iket mark a %r1
    add.u32 %r2, %r1, 100;
    //@iket mark b %r2
    cvt.u64.u32 %rd1, %r2;
    //@iket range_start c %rd1
    ret;"""


def test_payload_records_derived_by_hand():
    # mov at 0 (r1 ready 4); mark a at t_next = 1; add waits for r1: issues at
    # 4 (ready 8); mark b at 5; cvt waits for r2: issues at 8 (ready 12);
    # range_start c at 9; ret at 9; cycles = max(9 + 1, 12) = 12. 16-byte
    # records [id<<24|ts, 0, u64 payload].
    r, rb, sl = slots(kernel(PAYLOADS), block=64)
    assert rb == 16
    for w, lane0 in ((0, 0), (1, 32)):
        s = sl[w]
        assert struct.unpack_from("<IBBHQ", s, 0) == (3, 1, 16, 0, 12)
        recs = [struct.unpack_from("<IIQ", s, 16 + 16 * i) for i in range(3)]
        assert recs == [((0 << 24) | 1, 0, lane0), ((1 << 24) | 5, 0, lane0 + 100), ((2 << 24) | 9, 0, lane0 + 100)]
        assert not any(s[16 + 48:])


def test_payload_comes_from_the_lowest_active_lane():
    body = """    mov.u32 %r1, %tid.x;
    setp.lt.u32 %p1, %r1, 8;
    @%p1 ret;
    //@iket mark m %r1
    ret;"""
    # mov 0, setp 4 (p1 ready 8), @p1 ret waits for the guard: 8, next 9;
    # lanes 0..7 have left: the record carries lane 8's %tid.x
    r, rb, sl = slots(kernel(body), block=32)
    assert rb == 8
    assert struct.unpack_from("<IBBHQ", sl[0], 0) == (1, 1, 8, 0, 10)
    assert struct.unpack_from("<II", sl[0], 16) == ((0 << 24) | 9, 8)


def test_payload_records_are_dropped_and_counted_like_the_others():
    r, rb, sl = slots(kernel(PAYLOADS), block=32, max_ts=1)
    assert struct.unpack_from("<IBBHQ", sl[0], 0) == (3, 1, 16, 2, 12)
    assert struct.unpack_from("<IIQ", sl[0], 16) == (1, 0, 0)
    assert len(sl[0]) == 32


def test_event_without_payload_in_a_payload_kernel_stores_zero():
    body = """    mov.u32 %r1, 7;
    //@iket mark a
    //@iket mark b %r1
    ret;"""
    r, rb, sl = slots(kernel(body), block=32)
    assert rb == 8
    assert struct.unpack_from("<IIII", sl[0], 16) == (1, 0, (1 << 24) | 1, 7)


@pytest.mark.parametrize("body,code", [
    ("    //@iket mark a %r1\n    //@iket mark a %rd1\n    ret;", -1),   # one event, two payload sizes
    ("    //@iket mark a %p1\n    ret;", -1),                          # predicate payload
    ("    //@iket mark a 5\n    ret;", -1),                            # immediate payload
    ("    //@iket mark a %r1 %r2\n    ret;", -1),                      # two payloads
])
def test_rejected_payload_forms(body, code):
    assert oracle.parse_check(kernel(body), "ev")[0] == code

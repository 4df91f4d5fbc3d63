"""The trace export post-pass (ks_trace_to_json): hand-derived JSON for a
payload kernel, stamp unwrapping past 2^24 cycles against closed-form issue
times, and the oracle's plain exporter on real traces. CPU only: the export
is host code and the traces come from the oracle."""
import json

import numpy as np
import pytest

import oracle
from oracle import trace_json
from simt_ptx_interpretation_gb300 import api as ks
from simt_ptx_interpretation_gb300 import workloads as wl
from tests import test_oracle_events as tev


def export_both(ptx, kernel, grid, block, max_ts, params=b"", buffers=(), cpu=1000.0, **kw):
    bufs = [(b.sim_base, b.data) for b in buffers]
    r = oracle.run(ptx, kernel, grid, block, params, bufs, max_ts=max_ts, trace=True, **kw)
    lib = json.loads(ks.trace_to_json(ks.Module(ptx), kernel, grid, block, max_ts, r.trace, cpu))
    orc = trace_json.trace_events(ptx, kernel, grid, block, max_ts, r.trace.tobytes(), cpu)
    return lib, orc, r


def test_payload_kernel_by_hand():
    # records derived in test_oracle_events: a at 1 (payload lane 0's tid),
    # b at 5 (tid + 100), range_start c at 9 (tid + 100); 12 cycles; 1 GHz
    lib, orc, _ = export_both(tev.kernel(tev.PAYLOADS), "ev", 1, 64, 4)
    assert lib == orc
    ev = lib["traceEvents"]
    assert ev[0] == {"name": "process_name", "ph": "M", "pid": 0, "tid": 0, "args": {"name": "CTA 0"}}
    for w, lane0, at in ((0, 0, 1), (1, 32, 6)):
        assert ev[at] == {"name": "thread_name", "ph": "M", "pid": 0, "tid": w, "args": {"name": f"warp {w}"}}
        assert ev[at + 1] == {"name": "warp", "ph": "X", "pid": 0, "tid": w, "ts": 0.0, "dur": 0.012}
        assert ev[at + 2] == {"name": "a", "ph": "i", "pid": 0, "tid": w, "ts": 0.001, "s": "t",
                              "args": {"id": 0, "payload": lane0}}
        assert ev[at + 3] == {"name": "b", "ph": "i", "pid": 0, "tid": w, "ts": 0.005, "s": "t",
                              "args": {"id": 1, "payload": lane0 + 100}}
        assert ev[at + 4] == {"name": "c", "ph": "B", "pid": 0, "tid": w, "ts": 0.009,
                              "args": {"id": 2, "payload": lane0 + 100}}
    assert len(ev) == 11


def test_stamps_unwrap_past_24_bits():
    # a dependent chain of 10 global loads of latency 2^22, a mark after each:
    # load k issues at 8 + k * 2^22 (the first waits only for ld.param and the
    # bra-free prologue), so mark k carries stamp (9 + k * 2^22) mod 2^24
    loads = "\n".join("    ld.global.u64 %rd2, [%rd2];\n    //@iket mark m" for _ in range(10))
    ptx = wl.HEADER + f""".visible .entry ch(.param .u64 buf)
{{
    .reg .b64 %rd<3>;
    ld.param.u64 %rd2, [buf];
{loads}
    ret;
}}
"""
    buf = np.zeros(1, dtype=np.uint64)
    bufs = wl.place([("buf", buf, False)])
    buf[0] = bufs[0].sim_base
    lat = list(oracle.DEFAULT_LAT)
    lat[2] = 1 << 22
    lib, orc, r = export_both(ptx, "ch", 1, 32, 16, wl.pack_params([("u64", bufs[0].sim_base)]), bufs,
                              cpu=1.0, lat=lat)
    assert lib == orc
    marks = [e["ts"] for e in lib["traceEvents"] if e["name"] == "m"]
    t_first = marks[0]
    assert marks == [t_first + k * (1 << 22) for k in range(10)]
    assert marks[-1] > 1 << 24


@pytest.mark.parametrize("make", [lambda: wl.vector_add(), lambda: wl.smem_reduce(n=1 << 11, block=128),
                                  lambda: wl.fuzz(3, grid=4), lambda: wl.divergent(4, n=1 << 10)])
def test_library_matches_the_oracle_exporter(make):
    w = make()
    lib, orc, _ = export_both(w.ptx, w.kernel, w.grid, w.block, w.max_ts, w.params, w.fresh_buffers(), cpu=1.9e3)
    assert lib == orc
    assert any(e["ph"] in ("B", "i") for e in lib["traceEvents"])


def test_buffer_too_small_reports_the_size():
    import ctypes
    from simt_ptx_interpretation_gb300 import _native
    ptx = tev.kernel(tev.PAYLOADS)
    r = oracle.run(ptx, "ev", 1, 32, b"", [], max_ts=4, trace=True)
    m = ks.Module(ptx)
    need = ctypes.c_size_t(0)
    small = ctypes.create_string_buffer(8)
    rc = _native.lib().ks_trace_to_json(m._h, b"ev", 1, 32, 4, r.trace.ctypes.data, r.trace.nbytes, 1000.0, small,
                                        len(small), ctypes.byref(need))
    assert rc == -3 and need.value == len(ks.trace_to_json(m, "ev", 1, 32, 4, r.trace, 1000.0))
    # a trace buffer shorter than the launch's slots is refused
    rc = _native.lib().ks_trace_to_json(m._h, b"ev", 2, 32, 4, r.trace.ctypes.data, r.trace.nbytes, 1000.0, None, 0,
                                        ctypes.byref(need))
    assert rc == -3

"""Hints (KernelScope backend doc, hints/analyzer.py — analyze_trace_hints):
the page's thresholds and messages on hand-made events, the page's own
coalescing and bank-conflict examples through the oracle's event recorder,
and the library's ks_hints (host code) against the plain restatement in
oracle/hints.py. CPU only."""
import numpy as np
import pytest

import oracle
from oracle import hints as oh
from simt_ptx_interpretation_gb300 import api
from simt_ptx_interpretation_gb300 import workloads as wl


def ev(*rows):
    out = np.zeros(len(rows), dtype=oracle.HINT_EVENT_DTYPE)
    for i, (pc, kind, a, b, c) in enumerate(rows):
        out[i] = (pc, kind, a, b, c, 0)
    return out


def lib_hints(events, n_entries, occ=None):
    return api.hints(oh.profile(events, n_entries).view(np.uint8), occ)


def as_lib(h):
    return [dict(category=api.HINT_CATEGORIES[x["category"]], severity=api.HINT_SEVERITIES[x["severity"]],
                 pc=x["pc"], count=x["count"], message=x["message"], detail=x["detail"]) for x in h]


def test_shared_thresholds():
    S = oh.EV_SHARED
    e = ev((0, S, 1, 0, 0), (0, S, 2, 0, 0), (0, S, 7, 0, 0), (0, S, 8, 0, 0), (1, S, 32, 0, 0))
    per, tail = oh.event_hints(e)
    assert [(h["severity"], h["message"]) for h in per] == [
        (oh.WARNING, "2-way bank conflict"), (oh.WARNING, "7-way bank conflict"),
        (oh.CRITICAL, "8-way bank conflict"), (oh.CRITICAL, "32-way bank conflict")]
    assert per[2]["detail"] == "Severe bank conflict causing serialized access"
    assert per[0]["detail"] == "Bank conflict reducing throughput"
    assert tail == []  # 4 conflicted events: the summary needs more than 5
    e6 = ev(*[(0, S, 2, 0, 0)] * 6)
    assert oh.event_hints(e6)[1][0]["message"] == "Shared memory bank conflicts (6 events)"
    assert oh.event_hints(ev(*[(0, S, 2, 0, 0)] * 5))[1] == []


def test_global_thresholds():
    G = oh.EV_GLOBAL
    # 32 lanes x 4 bytes: ideal 1 line; 5 lines -> 20 %; 4 lines -> 25 % and 3 lines -> 33 %
    # (not poor: uncoalesced, which the page counts but reports nowhere)
    e = ev((0, G, 32, 5, 4), (1, G, 32, 4, 4), (2, G, 32, 3, 4), (3, G, 32, 9, 8), (4, G, 32, 32, 4))
    per, _ = oh.event_hints(e)
    assert [(h["pc"], h["message"]) for h in per] == [
        (0, "Poor memory efficiency (20%)"), (3, "Poor memory efficiency (22%)"),
        (4, "Poor memory efficiency (3%)")]
    p = oh.profile(e, 5)
    assert list(p["poor"]) == [1, 0, 0, 1, 1]
    assert list(p["uncoalesced"]) == [0, 1, 1, 0, 0]
    assert list(p["requests"]) == [1] * 5


def test_divergence_thresholds():
    D = oh.EV_DIVERGE
    e = ev((0, D, 16, 16, 0), (1, D, 13, 19, 0), (2, D, 12, 18, 0))
    per, tail = oh.event_hints(e)
    # 16/32 = 50 %; 13/32 = 0.40625 > 0.4; 12/30 = 0.4 is not above it
    assert [(h["pc"], h["message"]) for h in per] == [(0, "High divergence (50%)"), (1, "High divergence (40%)")]
    assert tail == []  # 3 divergent events: the summary needs more than 3
    t4 = oh.event_hints(ev(*[(0, D, 1, 31, 0)] * 4))[1]
    assert [h["message"] for h in t4] == ["Branch divergence detected (4 events)"]


def test_occupancy_messages():
    lim = api.gpu_limits("sm_80")
    low = api.occupancy(lim, 1024, 128)  # registers: 16 warps of 64 = 25 %, printed "25.0"
    assert low["active_warps_per_sm"] == 16 and low["occupancy_percent"] == 25.0
    assert api.hints(np.zeros(0, np.uint8), low)[0]["message"] == "Low occupancy (25.0%)"
    l86 = api.gpu_limits("sm_86")  # 48 warps: thirds print with every digit Python shows
    third = api.occupancy(l86, 512, 128)
    assert api.hints(np.zeros(0, np.uint8), third)[0]["message"] == "Low occupancy (33.33333333333333%)"
    cases = (low, third, api.occupancy(l86, 1024, 255), api.occupancy(lim, 64, 255), api.occupancy(lim, 96, 200),
             api.occupancy(lim, 256, 32))
    for occ in cases:
        page = {"occupancy_percent": occ["occupancy_percent"], "limiting_factor": occ["limiter"]}
        want = oh.aggregate(ev(), page)
        assert api.hints(np.zeros(0, np.uint8), occ) == as_lib(want), occ


@pytest.mark.parametrize("seed", range(20))
def test_library_matches_restatement_on_random_events(seed):
    rng = np.random.default_rng(seed)
    rows = []
    for _ in range(int(rng.integers(0, 60))):
        pc = int(rng.integers(0, 6))
        k = int(rng.integers(0, 3))
        if k == oh.EV_GLOBAL:
            lanes = int(rng.integers(1, 33))
            rows.append((pc, k, lanes, int(rng.integers(1, lanes + 1)), int(rng.choice([4, 8]))))
        elif k == oh.EV_SHARED:
            rows.append((pc, k, int(rng.integers(1, 33)), 0, 0))
        else:
            t = int(rng.integers(1, 32))
            rows.append((pc, k, t, int(rng.integers(1, 33 - t)), 0))
    e = ev(*rows)
    assert lib_hints(e, 6) == as_lib(oh.aggregate(e))


COALESCE = wl.HEADER + """.visible .entry co(.param .u64 p_in, .param .u32 p_stride, .param .u32 p_base)
{
    .reg .b32 %r<6>;
    .reg .f32 %f<2>;
    .reg .b64 %rd<6>;
    ld.param.u64    %rd1, [p_in];
    ld.param.u32    %r1, [p_stride];
    ld.param.u32    %r2, [p_base];
    mov.u32         %r3, %tid.x;
    mad.lo.u32      %r4, %r3, %r1, %r2;
    cvt.u64.u32     %rd2, %r4;
    add.s64         %rd3, %rd1, %rd2;
    ld.global.f32   %f1, [%rd3];
    ret;
}
"""


@pytest.mark.parametrize("stride, base, lines, message", [
    (4, 0, 1, None),                                   # the page: i*4 -> 1 transaction, efficiency 1.0
    (128, 0, 32, "Poor memory efficiency (3%)"),       # i*128 -> 32 transactions, efficiency 0.03125
    (4, 64, 2, None),                                  # 64 + i*4 -> 2 transactions, efficiency 0.5
])
def test_page_coalescing_examples(stride, base, lines, message):
    src = np.zeros(4096 + 64, dtype=np.float32)
    params = wl.pack_params([("u64", 0x1000_0000), ("u32", stride), ("u32", base)])
    r, e = oracle.run_events(COALESCE, "co", 1, 32, params, [(0x1000_0000, src)])
    assert r.status == 0
    assert len(e) == 1 and e[0]["kind"] == oh.EV_GLOBAL and e[0]["b"] == lines
    got = [h["message"] for h in oh.aggregate(e)]
    assert got == ([message] if message else [])


BANKS = wl.HEADER + """.visible .entry bk(.param .u32 p_stride)
{
    .reg .b32 %r<6>;
    .shared .align 4 .b32 s_arr[1024];
    ld.param.u32    %r1, [p_stride];
    mov.u32         %r2, %tid.x;
    mul.lo.u32      %r3, %r2, %r1;
    mov.u32         %r4, s_arr;
    add.u32         %r4, %r4, %r3;
    ld.shared.u32   %r5, [%r4];
    ret;
}
"""


@pytest.mark.parametrize("stride, message", [(4, None), (128, "32-way bank conflict"), (0, None), (8, "2-way bank conflict")])
def test_page_bank_examples(stride, message):
    r, e = oracle.run_events(BANKS, "bk", 1, 32, wl.pack_params([("u32", stride)]), [])
    assert r.status == 0
    got = [h["message"] for h in oh.aggregate(e)]
    assert got == ([message] if message else [])


@pytest.mark.parametrize("name", ["divergent", "fuzz", "smem_reduce", "fuzz_shared"])
def test_library_matches_restatement_on_workloads(name):
    w = {"divergent": lambda: wl.divergent(2, n=1 << 10), "fuzz": lambda: wl.fuzz(3, grid=2, block=64),
         "smem_reduce": lambda: wl.smem_reduce(n=64 * 4, block=64),
         "fuzz_shared": lambda: wl.fuzz_shared(1, grid=2, block=64)}[name]()
    r, e = oracle.run_events(w.ptx, w.kernel, w.grid, w.block, w.params,
                             [(b.sim_base, b.data) for b in w.fresh_buffers()])
    assert r.status == 0
    n = len(oracle.ipdom(w.ptx, w.kernel))
    occ = api.occupancy(api.gpu_limits("sm_80"), w.block, 96)
    page = {"occupancy_percent": occ["occupancy_percent"], "limiting_factor": occ["limiter"]}
    assert lib_hints(e, n, occ) == as_lib(oh.aggregate(e, page))
    # the counts add up to the events
    p = oh.profile(e, n)
    assert int(p["requests"].sum()) == int(((e["kind"] == oh.EV_GLOBAL) | (e["kind"] == oh.EV_SHARED)).sum())
    assert int(p["divergent"].sum()) == int((e["kind"] == oh.EV_DIVERGE).sum())


SPLIT = wl.HEADER + """.visible .entry sp(.param .u32 p_k)
{
    .reg .pred %p<2>;
    .reg .b32 %r<5>;
    ld.param.u32    %r1, [p_k];
    mov.u32         %r2, %tid.x;
    setp.lt.u32     %p1, %r2, %r1;
    @%p1 bra        TAKEN;
    add.u32         %r3, %r2, 1;
TAKEN:
    ret;
}
"""


@pytest.mark.parametrize("k, message", [(16, "High divergence (50%)"), (13, "High divergence (40%)"),
                                        (19, "High divergence (40%)"), (12, None), (1, None)])
def test_divergence_ratio_of_a_split(k, message):
    """k lanes take the branch and 32 - k fall through: the ratio is the
    smaller side over the 32 active lanes (13/32 = 0.406, 12/32 = 0.375)."""
    r, e = oracle.run_events(SPLIT, "sp", 1, 32, wl.pack_params([("u32", k)]), [])
    assert r.status == 0
    d = e[e["kind"] == oh.EV_DIVERGE]
    assert len(d) == 1 and (int(d[0]["a"]), int(d[0]["b"])) == (k, 32 - k)
    got = [h["message"] for h in oh.aggregate(e) if h["category"] == oh.DIVERGENCE]
    assert got == ([message] if message else [])


WIDE = wl.HEADER + """.visible .entry wd(.param .u64 p_in, .param .u32 p_lanes)
{
    .reg .pred %p<2>;
    .reg .b32 %r<5>;
    .reg .b64 %rd<6>;
    ld.param.u64    %rd1, [p_in];
    ld.param.u32    %r1, [p_lanes];
    mov.u32         %r2, %tid.x;
    cvt.u64.u32     %rd2, %r2;
    shl.b64         %rd2, %rd2, 7;
    add.s64         %rd3, %rd1, %rd2;
    setp.lt.u32     %p1, %r2, %r1;
    @%p1 ld.global.u64 %rd4, [%rd3];
    ret;
}
"""


@pytest.mark.parametrize("lanes, message", [(32, "Poor memory efficiency (6%)"), (16, "Poor memory efficiency (6%)"),
                                            (8, "Poor memory efficiency (12%)"), (2, None)])
def test_efficiency_counts_the_executing_lanes(lanes, message):
    """8-byte loads, one line per lane: ideal = ceil(lanes * 8 / 128) lines
    (2 for 32 lanes, 1 for 16 or fewer), efficiency ideal / lanes."""
    src = np.zeros(32 * 32 + 64, dtype=np.uint32)
    params = wl.pack_params([("u64", 0x1000_0000), ("u32", lanes)])
    r, e = oracle.run_events(WIDE, "wd", 1, 32, params, [(0x1000_0000, src)])
    assert r.status == 0
    g = e[e["kind"] == oh.EV_GLOBAL]
    assert len(g) == 1 and (int(g[0]["a"]), int(g[0]["b"]), int(g[0]["c"])) == (lanes, lanes, 8)
    got = [h["message"] for h in oh.aggregate(e)]
    assert got == ([message] if message else [])

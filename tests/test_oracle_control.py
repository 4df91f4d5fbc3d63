"""Pins the oracle's SIMT control flow, in-order scoreboard, coalescing
analysis, trace slots and error statuses to values fixed independently of it:
hand-derived closed forms, the pages' printed worked examples (tests/golden),
brute-force post-dominators, and a numpy per-thread evaluation."""
import os
import random
import struct

import numpy as np
import pytest

import oracle
from simt_ptx_interpretation_gb300 import workloads as wl
from tests import _exact as X
from tests._kernels import straight_line

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def run(w, **kw):
    bufs = w.fresh_buffers()
    kw.setdefault("max_ts", w.max_ts)
    r = oracle.run(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in bufs], **kw)
    return r, bufs


def golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


def stat_tuple(s):
    return tuple(int(s[k]) for k in ("cycles", "warp_insts", "thread_insts", "ld_req", "ld_sectors",
                                     "st_req", "st_sectors", "ld_lines", "st_lines"))


def slot(trace, max_ts, w):
    sb = (16 + 4 * max_ts + 7) // 8 * 8
    s = trace[w * sb:(w + 1) * sb].tobytes()
    n, fmt, bpe, dropped, cyc = struct.unpack_from("<IBBHQ", s, 0)
    recs = list(struct.unpack_from(f"<{max_ts}I", s, 16)) if max_ts else []
    return n, fmt, bpe, dropped, cyc, recs


# ------------------------------------------------------------ vector_add ----
# Hand derivation with the latency table ALU 4, ld.global 400, st 20, bra 8,
# ret 1 (every register ready at 0): the four ld.param issue at 0..3, the three
# mov at 4..6, mad waits for %tid.x (ready 10) -> 10, setp waits for mad -> 14,
# the guarded bra waits for %p1 -> 18 and sets t_next 26 (the `body` mark's
# timestamp). cvt 26, shl 30, adds 34/35/36, loads 38 and 39 (ready 438/439),
# add.f32 439, st 443 (completes 463), range_end mark at 444, ret 444.
# cycles = max(445, 443, 463) = 463. Out-of-bounds warps: bra taken at 18,
# range_end at 26, ret 26 -> cycles 27.

def test_vector_add_outputs_exact():
    w = wl.vector_add()
    r, bufs = run(w, trace=True)
    assert r.status == 0
    a, b, c = (x.data for x in bufs)
    want = np.array([X.add(X.f32_bits(float(x)), X.f32_bits(float(y))) for x, y in zip(a, b)], dtype=np.uint32)
    assert np.array_equal(c.view(np.uint32), want)


def test_vector_add_stats_hand_derived():
    w = wl.vector_add()
    r, _ = run(w)
    # n = 4000 = 125 * 32: warps 0..124 fully in bounds, 125..127 fully out
    for i in range(125):
        assert stat_tuple(r.stats[i]) == (463, 20, 640, 2, 8, 1, 4, 2, 1)
    for i in range(125, 128):
        assert stat_tuple(r.stats[i]) == (27, 11, 352, 0, 0, 0, 0, 0, 0)
    assert set(r.stats["max_stack_depth"]) == {1}


def test_vector_add_trace_hand_derived():
    w = wl.vector_add()
    r, _ = run(w, trace=True)
    assert slot(r.trace, 8, 0) == (3, 1, 4, 0, 463, [0x00000000, 0x0100001A, 0x020001BC, 0, 0, 0, 0, 0])
    assert slot(r.trace, 8, 127) == (2, 1, 4, 0, 27, [0x00000000, 0x0200001A, 0, 0, 0, 0, 0, 0])
    assert oracle.events(w.ptx, w.kernel) == [1, 0, 2]  # range_start, mark, range_end


def test_vector_add_ragged_warp():
    """n = 4010: warp 125 has lanes 0..9 in bounds, so the bounds branch
    diverges; the fall-through lanes run the body, then all reconverge."""
    w = wl.vector_add(n=4010)
    r, bufs = run(w, trace=True)
    assert r.status == 0
    a, b, c = (x.data for x in bufs)
    assert np.array_equal(c, (a + b).astype(np.float32))
    # 10 instructions (up to the branch) x 32 lanes, 9 body instructions x 10
    # lanes, ret x 32. Lanes 4000..4009 touch bytes 16000..16039: sectors
    # 500 and 501 of one 128-byte line.
    assert stat_tuple(r.stats[125]) == (463, 20, 10 * 32 + 9 * 10 + 32, 2, 4, 1, 2, 2, 1)
    assert int(r.stats[125]["max_stack_depth"]) == 2
    assert slot(r.trace, 8, 125)[:5] == (3, 1, 4, 0, 463)


# ------------------------------------------------------------ scoreboard ----

def chain_kernel(n, k):
    body = [f"fma.rn.f32 %f{4 + (i % k)}, %f{4 + (i % k)}, %f1, %f2;" for i in range(n)]
    return straight_line("chain", body)


def cycles_of(ptx, kernel="chain", lat=oracle.DEFAULT_LAT):
    r = oracle.run(ptx, kernel, 1, 32, b"", [], lat=lat)
    assert r.status == 0
    return int(r.stats[0]["cycles"])


@pytest.mark.parametrize("n", [1, 2, 3, 10, 33])
def test_dependent_chain_is_n_times_latency(n):
    assert cycles_of(chain_kernel(n, 1)) == 4 * n


@pytest.mark.parametrize("k", [2, 3, 4, 5, 8, 16])
def test_independent_accumulators_closed_form(k):
    n = 12 * k
    want = n + 3 if k >= 4 else 4 * n // k + k - 1
    assert cycles_of(chain_kernel(n, k)) == want


def test_accumulator_sweep_matches_the_pages_measurement():
    """Simulated CPI = max(1, 4/k) (the slope of cycles over instruction
    count); the page's sm_86 measurements sit within 0.05 of it."""
    rows = golden_rows("sass_probe_accumulator_sweep.txt")[1:]
    for row in rows:
        k, _regs, cpi, _sl, _ss = row.split(",")
        k, cpi = int(k), float(cpi)
        c1, c2 = cycles_of(chain_kernel(16 * k, k)), cycles_of(chain_kernel(32 * k, k))
        slope = (c2 - c1) / (16 * k)
        assert slope == max(1.0, 4.0 / k)
        assert abs(slope - cpi) <= 0.05, (k, slope, cpi)


# Loop probe, derived by hand for the generated PTX (acc = 1): prologue up to
# the first fma issues by cycle 36 and the second load makes %f1 ready at 426.
# Each iteration: 32 dependent fma (first at T, last at T+124, ready T+128),
# add at T+125, setp at T+129, bra at T+133, next T at T+141. After the last
# iteration the store issues at 567+141(N-1) and completes 20 later:
# cycles = 446 + 141 N. With 8 rotating accumulators the fma issue back to
# back (T .. T+31), add T+32, setp T+36, bra T+40, next T+48; the prologue's
# eight accumulator initialisations end at cycle 99; after the loop seven
# dependent adds reduce the accumulators, then the store: cycles = 474 + 48 N.
# The empty-loop control (no fma): add, setp, bra every 16 cycles and the
# store after the loop completes at 60 + 16 N; the two loads, unused there,
# complete at 426, so cycles = max(426, 60 + 16 N).
@pytest.mark.parametrize("acc,per_iter,slope,icept", [(1, 32, 141, 446), (8, 32, 48, 474), (1, 0, 16, 60)])
def test_ffma_loop_closed_form(acc, per_iter, slope, icept):
    for n in (1, 2, 3, 7, 20, 23, 24, 50):
        w = wl.ffma(acc=acc, iters=n, per_iter=per_iter, grid=1, block=32)
        r, _ = run(w)
        assert r.status == 0
        assert int(r.stats[0]["cycles"]) == max(426, icept + slope * n)


def test_ffma_instruction_count_sweep_is_linear():
    """The page's T(N) = L*N + C fit: the simulated sweep is exactly linear."""
    ns = [1, 4, 16, 64]
    ts = []
    for n in ns:
        r, _ = run(wl.ffma(acc=1, iters=n, grid=1, block=32))
        ts.append(int(r.stats[0]["cycles"]))
    L, C = np.polyfit(ns, ts, 1)
    pred = L * np.array(ns) + C
    r2 = 1 - np.sum((np.array(ts) - pred) ** 2) / np.sum((np.array(ts) - np.mean(ts)) ** 2)
    assert round(L, 6) == 141 and round(C, 6) == 446 and r2 == pytest.approx(1.0, abs=1e-12)
    # the page's probe size: 4096 iterations x 32 = 131072 FFMA
    rows = golden_rows("sass_probe_ffma_rows.txt")
    assert all(int(r.split(",")[2]) == 4096 * 32 for r in rows[1:])


def test_ffma_outputs_are_sequential_fma():
    for acc in (1, 8):
        w = wl.ffma(acc=acc, iters=64, grid=1, block=32)
        r, bufs = run(w)
        out, m, c = bufs[0].data.view(np.uint32), bufs[1].data, bufs[2].data
        for g in range(0, 32, 3):
            mb, cb = X.f32_bits(float(m[g])), X.f32_bits(float(c[g]))
            accs = [X.mul(X.int_to_f32(g + j), 0x35800000) for j in range(acc)]
            for _ in range(64):
                for i in range(32):
                    accs[i % acc] = X.fma(accs[i % acc], mb, cb)
            s = accs[0]
            for j in range(1, acc):
                s = X.add(s, accs[j])
            assert int(out[g]) == s, (acc, g)


def test_latency_table_is_configurable():
    lat = (7, 4, 400, 20, 8, 36, 1, 0)
    body = ["add.u32 %r1, %r1, 1;"] * 5
    assert cycles_of(straight_line("chain", body), lat=lat) == 5 * 7


# -------------------------------------------------------------- coalescing ----

def lane_access_kernel(mult, off):
    return wl.HEADER + f""".visible .entry acc(.param .u64 base)
{{
    .reg .b32 %r<4>;
    .reg .b64 %rd<4>;
    ld.param.u64 %rd1, [base];
    mov.u32 %r1, %tid.x;
    mad.lo.u32 %r2, %r1, {mult}, {off};
    cvt.u64.u32 %rd2, %r2;
    add.s64 %rd3, %rd1, %rd2;
    ld.global.u32 %r3, [%rd3];
    st.global.u32 [%rd3], %r3;
    ret;
}}
"""


def test_coalescing_examples_from_the_page():
    for row in golden_rows("kernelscope_coalescing.txt"):
        formula, trans, coalesced = row.split()
        if formula == "i*4":
            mult, off = 4, 0
        elif formula == "i*128":
            mult, off = 128, 0
        else:
            mult, off = 4, 64
        buf = np.zeros(8192, dtype=np.uint8)
        r = oracle.run(lane_access_kernel(mult, off), "acc", 1, 32, struct.pack("<Q", 0x20000000),
                       [(0x20000000, buf)])
        assert r.status == 0
        s = r.stats[0]
        assert int(s["ld_lines"]) == int(trans) and int(s["st_lines"]) == int(trans)
        assert (int(s["ld_lines"]) <= 1) == (coalesced == "true")
        # 32-byte sectors: contiguous 128 B -> 4; 128-byte stride -> 32; bytes 64..191 -> 4
        assert int(s["ld_sectors"]) == {"i*4": 4, "i*128": 32, "64+i*4": 4}[formula]


@pytest.mark.parametrize("s", [1, 2, 4, 8, 16, 32])
def test_strided_gather_sectors_closed_form(s):
    w = wl.gather(s, n_out=4096, block=256)
    r, bufs = run(w)
    assert r.status == 0
    src, out = bufs[0].data, bufs[1].data
    assert np.array_equal(out.view(np.uint32), src[::s].view(np.uint32))
    assert set(r.stats["ld_sectors"]) == {min(32, 4 * s)}
    assert set(r.stats["ld_lines"]) == {min(32, s)}
    assert set(r.stats["st_sectors"]) == {4} and set(r.stats["st_lines"]) == {1}
    assert set(r.stats["ld_req"]) == {1} and set(r.stats["st_req"]) == {1}


def test_same_address_stores_highest_lane_wins():
    ptx = wl.HEADER + """.visible .entry same(.param .u64 o)
{
    .reg .pred %p<2>;
    .reg .b32 %r<4>;
    .reg .b64 %rd<2>;
    ld.param.u64 %rd1, [o];
    mov.u32 %r1, %tid.x;
    setp.lt.u32 %p1, %r1, 21;
    @%p1 st.global.u32 [%rd1], %r1;
    ret;
}
"""
    buf = np.zeros(4, dtype=np.uint32)
    r = oracle.run(ptx, "same", 1, 32, struct.pack("<Q", 0x30000000), [(0x30000000, buf)])
    assert r.status == 0 and buf[0] == 20
    assert int(r.stats[0]["st_sectors"]) == 1 and int(r.stats[0]["st_req"]) == 1


# ------------------------------------------------------- SIMT / divergence ----

def test_divergence_masks_of_the_page_example():
    """if (tid < 16) path_a else path_b: path_a runs with 0x0000FFFF, path_b
    with 0xFFFF0000, fall-through (path_b) first, then all 32 lanes again."""
    masks = dict(r.split() for r in golden_rows("kernelscope_divergence_masks.txt"))
    ptx = wl.HEADER + """.visible .entry dm(.param .u64 o)
{
    .reg .pred %p<2>;
    .reg .b32 %r<6>;
    .reg .b64 %rd<4>;
    ld.param.u64 %rd1, [o];
    mov.u32 %r1, %tid.x;
    setp.lt.u32 %p1, %r1, 16;
    @%p1 bra PATH_A;
    //@iket mark path_b
    mov.u32 %r2, 2;
    add.u32 %r2, %r2, 0;
    add.u32 %r2, %r2, 0;
    bra.uni JOIN;
PATH_A:
    //@iket mark path_a
    mov.u32 %r2, 1;
JOIN:
    //@iket mark after
    cvt.u64.u32 %rd2, %r1;
    shl.b64 %rd2, %rd2, 2;
    add.s64 %rd3, %rd1, %rd2;
    st.global.u32 [%rd3], %r2;
    ret;
}
"""
    out = np.zeros(32, dtype=np.uint32)
    r = oracle.run(ptx, "dm", 1, 32, struct.pack("<Q", 0x40000000), [(0x40000000, out)], max_ts=4, trace=True)
    assert r.status == 0
    pa = int(masks["path_a"], 16)
    pb = int(masks["path_b"], 16)
    assert pa | pb == int(masks["before"], 16) == int(masks["after"], 16)
    want = [1 if (pa >> i) & 1 else 2 for i in range(32)]
    assert out.tolist() == want
    # 4 instructions with all lanes, path_b 4 with 16 lanes, path_a 1 with 16, 5 after with 32
    assert int(r.stats[0]["thread_insts"]) == 4 * 32 + 4 * 16 + 1 * 16 + 5 * 32
    n, _, _, _, _, recs = slot(r.trace, 4, 0)
    ids = [x >> 24 for x in recs[:n]]
    assert ids == [0, 1, 2]  # path_b (first seen) -> path_a -> after
    ts = [x & 0xFFFFFF for x in recs[:n]]
    assert ts[0] < ts[1] < ts[2]


def numpy_divergent(trips, k):
    n = len(trips)
    g = np.arange(n, dtype=np.uint32)
    lane = g & np.uint32(31)
    q = (lane & np.uint32(k - 1)) == 0
    x = g.copy()
    t = trips.astype(np.uint32)
    with np.errstate(over="ignore"):
        for i in range(int(t.max()) if n else 0):
            act = np.uint32(i) < t
            iu = np.uint32(i)
            a = (x * np.uint32(0x9E3779B1)) ^ iu
            b = a << np.uint32(3)
            c = a >> np.uint32(5)
            d = b ^ c
            e = d & np.uint32(0xFFFF)
            y = x + e
            y = y + np.where(e < np.uint32(0x8000), d, c)
            y = y * np.uint32(0x01000193)
            y = y ^ t
            y = y + ((y >> np.uint32(5)) << np.uint32(3))
            h = y * np.uint32(3) + iu
            z = y ^ h
            z = z + (z >> np.uint32(7))
            y = np.where(q, z, y)
            x = np.where(act, y, x)
    return x


@pytest.mark.parametrize("k", [2, 4, 32])
def test_divergent_outputs_and_instruction_counts(k):
    w = wl.divergent(k, n=1 << 13)
    r, bufs = run(w, trace=True)
    assert r.status == 0
    trips, out = bufs[0].data, bufs[1].data
    assert np.array_equal(out, numpy_divergent(trips, k))
    q = ((np.arange(len(trips)) & 31) & (k - 1)) == 0
    t = trips.astype(np.int64).reshape(-1, 32)
    qq = q.reshape(-1, 32)
    lane_insts = 20 + 22 * t + 5 * t * qq
    assert np.array_equal(r.stats["thread_insts"].astype(np.int64), lane_insts.sum(axis=1))
    T = t.max(axis=1)
    Tq = np.where(qq, t, 0).max(axis=1)
    assert np.array_equal(r.stats["warp_insts"].astype(np.int64), 20 + 22 * T + 5 * Tq)


@pytest.mark.parametrize("k", [2, 32])
def test_warp_mode_equals_per_thread_mode_divergent(k):
    w = wl.divergent(k, n=1 << 12)
    r1, b1 = run(w, race_check=True)
    r2, b2 = run(w, mode=oracle.MODE_PER_THREAD)
    assert r1.status == r2.status == 0 and r1.race_flags == 0
    assert np.array_equal(b1[1].data, b2[1].data)


@pytest.mark.parametrize("i", range(0, 64, 4))
def test_warp_mode_equals_per_thread_mode_fuzz(i):
    w = wl.fuzz(i, grid=4)
    r1, b1 = run(w, race_check=True)
    r2, b2 = run(w, mode=oracle.MODE_PER_THREAD)
    assert r1.status == r2.status == 0
    assert r1.race_flags == 0
    assert all(np.array_equal(x.data, y.data) for x, y in zip(b1, b2))


def test_race_checker_detects_a_race():
    ptx = wl.HEADER + """.visible .entry race(.param .u64 o)
{
    .reg .b32 %r<3>;
    .reg .b64 %rd<2>;
    ld.param.u64 %rd1, [o];
    mov.u32 %r1, %tid.x;
    st.global.u32 [%rd1], %r1;
    ret;
}
"""
    buf = np.zeros(4, dtype=np.uint32)
    r = oracle.run(ptx, "race", 1, 64, struct.pack("<Q", 0x50000000), [(0x50000000, buf)], race_check=True)
    assert r.race_flags & 1


# -------------------------------------------------------- post-dominators ----

HAND_CFGS = {
    "if_else": ("""
    setp.lt.u32 %p1, %r1, 5;
    @%p1 bra ELSE;
    add.u32 %r2, %r2, 1;
    bra.uni JOIN;
ELSE:
    add.u32 %r2, %r2, 2;
JOIN:
    add.u32 %r3, %r2, 1;
    ret;""", [1, 5, 3, 5, 5, 6, 7]),
    "nested_loops": ("""
    mov.u32 %r1, 0;
OUTER:
    mov.u32 %r2, 0;
INNER:
    add.u32 %r2, %r2, 1;
    setp.lt.u32 %p1, %r2, 3;
    @%p1 bra INNER;
    add.u32 %r1, %r1, 1;
    setp.lt.u32 %p2, %r1, 4;
    @%p2 bra OUTER;
    ret;""", [1, 2, 3, 4, 5, 6, 7, 8, 9]),
    "early_ret": ("""
    setp.eq.u32 %p1, %r1, 0;
    @%p1 bra OUT;
    add.u32 %r2, %r2, 1;
    ret;
OUT:
    add.u32 %r2, %r2, 2;
    ret;""", [1, 6, 3, 6, 5, 6]),
    "loop_break": ("""
    mov.u32 %r1, 0;
HEAD:
    setp.eq.u32 %p1, %r1, 7;
    @%p1 bra BRK;
    add.u32 %r1, %r1, 1;
    setp.lt.u32 %p2, %r1, 10;
    @%p2 bra HEAD;
BRK:
    add.u32 %r2, %r1, 1;
    ret;""", [1, 2, 6, 4, 5, 6, 7, 8]),
    "guarded_ret": ("""
    setp.eq.u32 %p1, %r1, 0;
    @%p1 ret;
    add.u32 %r2, %r2, 1;
    ret;""", [1, 4, 3, 4]),
    "endless": ("""
    add.u32 %r1, %r1, 1;
L:
    add.u32 %r1, %r1, 1;
    bra.uni L;""", [3, 3, 3]),
}


def cfg_kernel(body):
    return wl.HEADER + ".visible .entry cfg()\n{\n    .reg .pred %p<4>;\n    .reg .b32 %r<8>;\n" + body + "\n}\n"


@pytest.mark.parametrize("name", sorted(HAND_CFGS))
def test_ipdom_hand_drawn(name):
    body, want = HAND_CFGS[name]
    assert oracle.ipdom(cfg_kernel(body), "cfg") == want


def random_cfg(rng, m):
    """Random program of m entries; returns (body text, successor lists)."""
    kinds = []
    for i in range(m - 1):
        c = rng.random()
        if c < 0.45:
            kinds.append(("alu", None))
        elif c < 0.75:
            kinds.append(("cbra", rng.randrange(m)))
        elif c < 0.85:
            kinds.append(("bra", rng.randrange(m)))
        elif c < 0.93:
            kinds.append(("gret", None))
        else:
            kinds.append(("ret", None))
    kinds.append(rng.choice([("ret", None), ("bra", rng.randrange(m))]))
    targets = {t for k, t in kinds if t is not None}
    lines, succ = [], []
    for i, (k, t) in enumerate(kinds):
        if i in targets:
            lines.append(f"L{i}:")
        if k == "alu":
            lines.append("    add.u32 %r1, %r1, 1;")
            succ.append([i + 1])
        elif k == "cbra":
            lines.append(f"    @%p1 bra L{t};")
            succ.append(sorted({t, i + 1}))
        elif k == "bra":
            lines.append(f"    bra.uni L{t};")
            succ.append([t])
        elif k == "gret":
            lines.append("    @%p2 ret;")
            succ.append([m, i + 1])
        else:
            lines.append("    ret;")
            succ.append([m])
    return "\n".join(lines), succ


def brute_ipdom(succ):
    m = len(succ)
    exit_ = m

    def reaches_exit(start, removed):
        seen, stack = set(), [start]
        while stack:
            v = stack.pop()
            if v == exit_:
                return True
            if v in seen or v == removed:
                continue
            seen.add(v)
            stack.extend(succ[v])
        return False

    reach = [reaches_exit(i, None) for i in range(m)]
    pdom = {}
    for i in range(m):
        if reach[i]:
            pdom[i] = {d for d in range(m) if d == i or not reaches_exit(i, d)} | {exit_}
    pdom[exit_] = {exit_}
    out = []
    for i in range(m):
        if not reach[i]:
            out.append(exit_)
            continue
        strict = pdom[i] - {i}
        cands = [d for d in strict if strict <= pdom[d]]
        assert len(cands) == 1
        out.append(cands[0])
    return out


def test_ipdom_random_cfgs_against_brute_force():
    rng = random.Random(77)
    for trial in range(150):
        m = rng.randrange(2, 24)
        body, succ = random_cfg(rng, m)
        assert oracle.ipdom(cfg_kernel(body), "cfg") == brute_ipdom(succ), body


# ------------------------------------------------------------------ trace ----

def loop_events_kernel(iters):
    return wl.HEADER + f""".visible .entry ev()
{{
    .reg .pred %p<2>;
    .reg .b32 %r<3>;
    mov.u32 %r1, 0;
    //@iket range_start loop
EV_L:
    //@iket mark iter
    add.u32 %r1, %r1, 1;
    setp.lt.u32 %p1, %r1, {iters};
    @%p1 bra EV_L;
    //@iket range_end loop
    ret;
}}
"""


@pytest.mark.parametrize("max_ts", [0, 1, 2, 8, 64])
def test_trace_slot_layout_and_dropped_count(max_ts):
    rows = dict(r.split(None, 1) for r in golden_rows("iket_slot_sizing.txt"))
    hdr, bpe, align = int(rows["header_bytes"]), int(rows["bytes_per_event_no_payload"]), int(rows["align"])
    r = oracle.run(loop_events_kernel(20), "ev", 2, 64, b"", [], max_ts=max_ts, trace=True)
    assert r.status == 0
    sb = (hdr + max_ts * bpe + align - 1) // align * align
    assert len(r.trace) == 4 * sb
    n, fmt, b, dropped, cyc, recs = slot(r.trace, max_ts, 3)
    assert (n, fmt, b) == (22, 1, bpe)
    assert dropped == max(0, 22 - max_ts)
    assert cyc == int(r.stats[3]["cycles"])
    kept = min(22, max_ts)
    ids = [x >> 24 for x in recs[:kept]]
    assert ids == ([0] + [1] * 20 + [2])[:kept]
    assert all(x == 0 for x in recs[kept:])


def test_trace_timestamp_keeps_24_bits():
    lat = (1 << 20, 4, 400, 20, 8, 36, 1, 0)
    body = ["add.u32 %r1, %r1, 1;"] * 20 + ["//@iket mark late"]
    ptx = straight_line("chain", body)
    r = oracle.run(ptx, "chain", 1, 32, b"", [], lat=lat, max_ts=1, trace=True)
    n, _, _, _, cyc, recs = slot(r.trace, 1, 0)
    t_mark = 19 * (1 << 20) + 1  # the last add issues at 19 * 2^20, t_next one later
    assert recs[0] == t_mark & 0xFFFFFF
    assert cyc == 20 * (1 << 20)


# ----------------------------------------------------------------- errors ----

def access_kernel(op):
    return wl.HEADER + f""".visible .entry bad(.param .u64 base)
{{
    .reg .b32 %r<4>;
    .reg .b64 %rd<4>;
    ld.param.u64 %rd1, [base];
    mov.u32 %r1, %tid.x;
    {op}
    ret;
}}
"""


def test_out_of_bounds_and_misaligned_statuses():
    buf = np.zeros(1024, dtype=np.uint8)
    base = 0x60000000
    # lane-dependent offset beyond the buffer
    ptx = access_kernel("mul.lo.u32 %r2, %r1, 64;\n    cvt.u64.u32 %rd2, %r2;\n    add.s64 %rd3, %rd1, %rd2;\n"
                        "    ld.global.u32 %r3, [%rd3];")
    r = oracle.run(ptx, "bad", 1, 32, struct.pack("<Q", base), [(base, buf)])
    assert r.status == oracle_status("OOB")
    r = oracle.run(access_kernel("ld.global.u32 %r3, [%rd1+2];"), "bad", 1, 32, struct.pack("<Q", base), [(base, buf)])
    assert r.status == oracle_status("MISALIGNED")
    # misaligned and out of bounds on the same lane: alignment is checked first
    r = oracle.run(access_kernel("ld.global.u64 %rd2, [%rd1+2044];"), "bad", 1, 32, struct.pack("<Q", base), [(base, buf)])
    assert r.status == oracle_status("MISALIGNED")
    # lane 0 misaligned, higher lanes out of bounds: the lowest failing lane decides
    ptx = access_kernel("mul.lo.u32 %r2, %r1, 2048;\n    add.u32 %r2, %r2, 2;\n    cvt.u64.u32 %rd2, %r2;\n"
                        "    add.s64 %rd3, %rd1, %rd2;\n    st.global.u32 [%rd3], %r1;")
    r = oracle.run(ptx, "bad", 1, 32, struct.pack("<Q", base), [(base, buf)])
    assert r.status == oracle_status("MISALIGNED")
    assert not buf.any()


def oracle_status(name):
    return {"OOB": 1, "MISALIGNED": 2, "STEP_LIMIT": 3, "SIMT_STACK": 4, "TIMEOUT": 5, "INJECTED": 6}[name]


def test_step_limit_stops_an_endless_loop():
    ptx = cfg_kernel(HAND_CFGS["endless"][0])
    r = oracle.run(ptx, "cfg", 2, 32, b"", [], step_limit=1000)
    assert r.status == oracle_status("STEP_LIMIT")
    assert set(r.stats["warp_insts"]) == {1000}
    assert set(r.stats["status"]) == {3}


def test_simt_stack_overflow():
    body = """
    mov.u32 %r1, %tid.x;
    and.b32 %r2, %r1, 1;
    setp.eq.u32 %p1, %r2, 0;
    @%p1 bra ELSE;
    add.u32 %r3, %r3, 1;
    bra.uni JOIN;
ELSE:
    add.u32 %r3, %r3, 2;
JOIN:
    ret;"""
    ptx = cfg_kernel(body)
    assert oracle.run(ptx, "cfg", 1, 32, b"", [], stack_depth=3).status == 0
    r = oracle.run(ptx, "cfg", 1, 32, b"", [], stack_depth=2)
    assert r.status == oracle_status("SIMT_STACK")
    # uniform warps never push
    assert oracle.run(ptx, "cfg", 1, 1, b"", [], stack_depth=1).status == 0


def test_injected_status_and_first_failing_warp():
    w = wl.vector_add()
    r, _ = run(w, inject_warp=5, inject_step=7)
    assert r.status == oracle_status("INJECTED")
    assert int(r.stats[5]["status"]) == 6 and int(r.stats[5]["warp_insts"]) == 7
    assert int(r.stats[4]["status"]) == 0 and int(r.stats[6]["status"]) == 0


BAD_PROGRAMS = [
    ("undeclared", "add.u32 %r9, %r1, 1;\n    ret;"),
    ("opcode", "frob.u32 %r1, %r1, 1;\n    ret;"),
    ("width", "add.u64 %r1, %r1, 1;\n    ret;"),
    ("falls_off", "add.u32 %r1, %r1, 1;"),
    ("guarded_last", "@%p1 ret;"),
    ("label_end", "ret;\nEND:"),
    ("undefined_label", "bra.uni NOWHERE;"),
    ("f32_int_literal", "add.f32 %f1, %f1, 1;\n    ret;"),
    ("literal_range", "add.u32 %r1, %r1, 0x100000000;\n    ret;"),
    ("mul_without_lo", "mul.u32 %r1, %r1, 3;\n    ret;"),
    ("div_without_rn", "div.f32 %f1, %f1, %f1;\n    ret;"),
    ("setp_signed_lo", "setp.lo.s32 %p1, %r1, 3;\n    ret;"),
    ("pred_guard", "@%r1 add.u32 %r1, %r1, 1;\n    ret;"),
    ("special_64", "mov.u64 %rd1, %tid.x;\n    ret;"),
    ("address_32", "ld.global.u32 %r1, [%r2];\n    ret;"),
    ("nested_block", "{ add.u32 %r1, %r1, 1; }\n    ret;"),
    ("cvt_no_round", "cvt.f32.u32 %f1, %r1;\n    ret;"),
    ("ftz", "add.rn.ftz.f32 %f1, %f1, %f1;\n    ret;"),
]


@pytest.mark.parametrize("name,body", BAD_PROGRAMS)
def test_malformed_programs_are_rejected(name, body):
    ptx = wl.HEADER + (".visible .entry k()\n{\n    .reg .pred %p<2>;\n    .reg .b32 %r<4>;\n"
                       "    .reg .f32 %f<4>;\n    .reg .b64 %rd<4>;\n    " + body + "\n}\n")
    code, msg = oracle.parse_check(ptx, "k")
    assert code < 0, name


def test_write_after_write_waits():
    """A write to a register whose earlier write is still pending waits for
    it: ld.param (ready 4), ld.global at 4 (ready 404), mov to the same
    register issues at 404 (ready 408), ret at 405 -> cycles 408."""
    ptx = wl.HEADER + """.visible .entry waw(.param .u64 o)
{
    .reg .b32 %r<2>;
    .reg .b64 %rd<2>;
    ld.param.u64 %rd1, [o];
    ld.global.u32 %r1, [%rd1];
    mov.u32 %r1, 7;
    ret;
}
"""
    buf = np.zeros(4, dtype=np.uint32)
    r = oracle.run(ptx, "waw", 1, 32, struct.pack("<Q", 0x70000000), [(0x70000000, buf)])
    assert r.status == 0 and int(r.stats[0]["cycles"]) == 408


def test_ret_inside_a_divergent_path_removes_lanes_everywhere():
    """Lanes 16..23 return inside the fall-through path; after the paths
    reconverge they must stay inactive."""
    ptx = wl.HEADER + """.visible .entry rt(.param .u64 o)
{
    .reg .pred %p<3>;
    .reg .b32 %r<4>;
    .reg .b64 %rd<4>;
    ld.param.u64 %rd1, [o];
    mov.u32 %r1, %tid.x;
    setp.lt.u32 %p1, %r1, 16;
    @%p1 bra A;
    setp.lt.u32 %p2, %r1, 24;
    @%p2 ret;
    add.u32 %r2, %r1, 100;
    bra.uni J;
A:
    add.u32 %r2, %r1, 200;
J:
    cvt.u64.u32 %rd2, %r1;
    shl.b64 %rd2, %rd2, 2;
    add.s64 %rd3, %rd1, %rd2;
    st.global.u32 [%rd3], %r2;
    ret;
}
"""
    out = np.zeros(32, dtype=np.uint32)
    r = oracle.run(ptx, "rt", 1, 32, struct.pack("<Q", 0x70000000), [(0x70000000, out)])
    assert r.status == 0
    want = [i + 200 if i < 16 else (0 if i < 24 else i + 100) for i in range(32)]
    assert out.tolist() == want
    # 4 x 32 before the branch; fall path: setp, ret with 16 lanes, add, bra with 8;
    # taken path: add with 16; after the join: 5 instructions with 24 lanes
    assert int(r.stats[0]["thread_insts"]) == 4 * 32 + 2 * 16 + 2 * 8 + 16 + 5 * 24

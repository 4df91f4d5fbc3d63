"""Oracle pins for the L1/L2 hit model (KernelScope backend doc,
simulator/engine.py — "Cache parameters": 128-byte lines, L1 1024 lines with
28-cycle hits, L2 49152 lines with 150-cycle hits, DRAM 400; SimpleCache:
direct-mapped, set = line % lines, a miss installs; _execute_instruction: the
representative address, L1 then L2). Hit sequences and cycle counts below are
derived by hand from those rules and the page's step() order. CPU only."""
import numpy as np
import pytest

import oracle
from simt_ptx_interpretation_gb300 import workloads as wl

from . import _cache_kernels as ck

L1, L2, DRAM = oracle.CACHE_L1_HIT, oracle.CACHE_L2_HIT, oracle.CACHE_DRAM


def accesses(r, w):
    n = int(r.warps[w]["n_access"])
    return [(int(a["line"]), int(a["step"]), int(a["level"])) for a in r.log[w][:n]]


def test_reuse_hits_l1_and_shortens_the_chain():
    src = ck.f32_buffer(1024)
    out = np.zeros(32, dtype=np.float32)
    bufs = [(ck.BASE_IN, src), (ck.BASE_OUT, out)]
    r = oracle.run_cached(ck.REUSE, "reuse", 1, 32, ck.u64(ck.BASE_IN, ck.BASE_OUT), bufs)
    assert r.status == 0
    li, lo = ck.BASE_IN // 128, ck.BASE_OUT // 128
    # ld at step 2 (cold), ld at step 4 (same line), st at step 6 (cold)
    assert accesses(r, 0) == [(li, 2, DRAM), (li, 4, L1), (lo, 6, DRAM)]
    assert tuple(r.warps[0]) == (3, 1, 0, 2)
    # issue times: ld.param 0, 1; ld 4 (ready 404); add 404; ld 405 (ready 433);
    # add 433 (ready 437); st 437 (done 457); ret 438 -> cycles 457
    assert int(r.stats[0]["cycles"]) == 457
    # with every level at the DRAM latency the model changes nothing: 829
    flat = oracle.run_cached(ck.REUSE, "reuse", 1, 32, ck.u64(ck.BASE_IN, ck.BASE_OUT),
                             [(ck.BASE_IN, src.copy()), (ck.BASE_OUT, np.zeros(32, np.float32))],
                             lat_l1=400, lat_l2=400)
    plain = oracle.run(ck.REUSE, "reuse", 1, 32, ck.u64(ck.BASE_IN, ck.BASE_OUT),
                       [(ck.BASE_IN, src.copy()), (ck.BASE_OUT, np.zeros(32, np.float32))])
    assert int(flat.stats[0]["cycles"]) == int(plain.stats[0]["cycles"]) == 829
    # every lane stores to out[0]
    assert out[0] == np.float32(src[0]) + np.float32(src[0] + src[0]) and not out[1:].any()


@pytest.mark.parametrize("off_lines, levels, cycles", [
    (0, [DRAM, L1, L1, L1], 406),             # one line
    (1, [DRAM, DRAM, L1, L1], 409),           # two lines, two L1 sets
    (1024, [DRAM, DRAM, L2, L2], 409),        # same L1 set, two L2 sets
    (49152, [DRAM, DRAM, DRAM, DRAM], 411),   # same set in both levels
    (49152 + 1024, [DRAM, DRAM, L2, L2], 409),
])
def test_direct_mapped_sets(off_lines, levels, cycles):
    off = off_lines * 128
    src = np.zeros((off + 256) // 4, dtype=np.float32)
    r = oracle.run_cached(ck.PAIR, "pair", 1, 32, ck.u64(ck.BASE_IN, off), [(ck.BASE_IN, src)])
    assert r.status == 0
    got = accesses(r, 0)
    assert [a[2] for a in got] == levels
    assert [a[1] for a in got] == [3, 4, 5, 6]
    li = ck.BASE_IN // 128
    assert [a[0] for a in got] == [li, li + off_lines, li, li + off_lines]
    # loads issue at 6, 9, 10, 11; cycles = the latest ready time
    assert int(r.stats[0]["cycles"]) == cycles


def test_cache_sizes_are_parameters():
    # with a 2-line L1 and a 4-line L2, lines 0 and 2 share an L1 set but not an L2 set
    src = np.zeros(1024, dtype=np.float32)
    r = oracle.run_cached(ck.PAIR, "pair", 1, 32, ck.u64(ck.BASE_IN, 256), [(ck.BASE_IN, src)],
                          l1_lines=2, l2_lines=4)
    assert [a[2] for a in accesses(r, 0)] == [DRAM, DRAM, L2, L2]


@pytest.mark.parametrize("d0, d1, first", [(0, 0, 0), (3, 0, 1), (0, 3, 0), (2, 1, 1)])
def test_step_order_between_warps(d0, d1, first):
    src = np.zeros(64, dtype=np.float32)
    r = oracle.run_cached(ck.order_kernel(d0, d1), "order", 1, 64, ck.u64(ck.BASE_IN), [(ck.BASE_IN, src)])
    assert r.status == 0
    a0, a1 = accesses(r, 0), accesses(r, 1)
    assert a0[0][1] == 6 + d0 and a1[0][1] == 6 + d1
    # the earlier step goes first; within a step the lower warp
    assert (a0[0][2], a1[0][2]) == ((DRAM, L1) if first == 0 else (L1, DRAM))


def test_step_order_across_ctas():
    # two CTAs of one warp (one more instruction before the branch): CTA 1's
    # warp loads first when it is 3 steps ahead
    src = np.zeros(64, dtype=np.float32)
    ptx = ck.order_kernel(3, 0).replace("setp.ge.u32     %p1, %r1, 32;",
                                        "mov.u32         %r3, %ctaid.x;\n    setp.ne.u32     %p1, %r3, 0;")
    r = oracle.run_cached(ptx, "order", 2, 32, ck.u64(ck.BASE_IN), [(ck.BASE_IN, src)])
    assert accesses(r, 0)[0][1:] == (10, L1)
    assert accesses(r, 1)[0][1:] == (7, DRAM)


def test_representative_is_the_lowest_executing_lane():
    src = np.zeros(32 * 32 + 64, dtype=np.float32)
    r = oracle.run_cached(ck.REPRESENTATIVE, "rep", 1, 32, ck.u64(ck.BASE_IN), [(ck.BASE_IN, src)])
    li = ck.BASE_IN // 128
    # lane 0 is guarded off: lane 1's line, which the second load then hits
    assert accesses(r, 0) == [(li + 1, 6, DRAM), (li + 1, 7, L1)]


def test_stores_install_lines():
    out = np.zeros(64, dtype=np.uint32)
    r = oracle.run_cached(ck.STORE_THEN_LOAD, "stld", 1, 32, ck.u64(ck.BASE_OUT), [(ck.BASE_OUT, out)])
    lo = ck.BASE_OUT // 128
    assert accesses(r, 0) == [(lo, 2, DRAM), (lo, 3, L1), (lo, 4, L1)]
    assert out[0] == 7 and out[2] == 0  # word 1 was 0 when loaded
    # issue: ld.param 0, mov 1, st 5 (sources ready 4, 5), ld 6 (L1 hit, ready
    # 34), st 34 (completes 54 = lat[st.global] later), ret 35 -> cycles 54
    assert int(r.stats[0]["cycles"]) == 54


def test_barrier_release_step():
    src = np.zeros(64, dtype=np.float32)
    r = oracle.run_cached(ck.BARRIER, "barrier", 1, 64, ck.u64(ck.BASE_IN), [(ck.BASE_IN, src)])
    assert r.status == 0
    li = ck.BASE_IN // 128
    assert accesses(r, 0) == [(li, 8, DRAM)]
    assert accesses(r, 1) == [(li, 8, L1)]


def test_barrier_released_by_a_finishing_warp():
    src = np.zeros(64, dtype=np.float32)
    r = oracle.run_cached(ck.BARRIER_EXIT, "barrier_exit", 1, 64, ck.u64(ck.BASE_IN), [(ck.BASE_IN, src)])
    assert r.status == 0
    assert accesses(r, 0) == [(ck.BASE_IN // 128, 10, DRAM)]
    assert int(r.warps[1]["n_access"]) == 0


def test_log_counts_match_requests():
    w = wl.vector_add()
    bufs = [(b.sim_base, b.data.copy()) for b in w.buffers]
    r = oracle.run_cached(w.ptx, w.kernel, w.grid, w.block, w.params, bufs, max_ts=w.max_ts, trace=True)
    s = r.stats
    assert np.array_equal(r.warps["n_access"].astype(np.uint64), s["ld_req"] + s["st_req"])
    assert np.array_equal(r.warps["l1_hits"] + r.warps["l2_hits"] + r.warps["dram"], r.warps["n_access"])


def _replay(r, l1_lines, l2_lines):
    """The page's SimpleCache, written again here, over every logged access in
    (step, warp) order; returns the levels per (warp, k)."""
    acc = []
    for w in range(len(r.warps)):
        for k, (line, step, _) in enumerate(accesses(r, w)):
            acc.append((step, w, k, line))
    acc.sort()
    l1, l2, out = {}, {}, {}
    for step, w, k, line in acc:
        if l1.get(line % l1_lines) == line:
            out[(w, k)] = L1
            continue
        l1[line % l1_lines] = line
        if l2.get(line % l2_lines) == line:
            out[(w, k)] = L2
            continue
        l2[line % l2_lines] = line
        out[(w, k)] = DRAM
    return out


@pytest.mark.parametrize("seed", [0, 3, 7])
@pytest.mark.parametrize("sizes", [(1024, 49152), (4, 12), (1, 3)])
def test_levels_replay_on_random_programs(seed, sizes):
    w = wl.fuzz(seed, grid=4, block=64)
    bufs = [(b.sim_base, b.data.copy()) for b in w.buffers]
    r = oracle.run_cached(w.ptx, w.kernel, w.grid, w.block, w.params, bufs, l1_lines=sizes[0], l2_lines=sizes[1],
                          log_cap=4096)
    assert r.status == 0
    assert int(r.warps["n_access"].max()) <= 4096
    want = _replay(r, *sizes)
    for (wi, k), lvl in want.items():
        assert int(r.log[wi][k]["level"]) == lvl
    # memory, and the statistics other than cycles, equal the plain run's
    bufs2 = [(b.sim_base, b.data.copy()) for b in w.buffers]
    p = oracle.run(w.ptx, w.kernel, w.grid, w.block, w.params, bufs2)
    for (_, a), (_, b) in zip(bufs, bufs2):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    for f in ("warp_insts", "thread_insts", "ld_req", "ld_sectors", "st_req", "st_sectors", "status"):
        assert np.array_equal(r.stats[f], p.stats[f]), f
    # shorter load latencies never delay an in-order warp
    assert (r.stats["cycles"] <= p.stats["cycles"]).all()


def test_all_levels_at_dram_latency_equal_the_plain_run():
    w = wl.fuzz(5, grid=2, block=64)
    bufs = [(b.sim_base, b.data.copy()) for b in w.buffers]
    r = oracle.run_cached(w.ptx, w.kernel, w.grid, w.block, w.params, bufs, lat_l1=400, lat_l2=400,
                          max_ts=w.max_ts, trace=True, log_cap=4096)
    bufs2 = [(b.sim_base, b.data.copy()) for b in w.buffers]
    p = oracle.run(w.ptx, w.kernel, w.grid, w.block, w.params, bufs2, max_ts=w.max_ts, trace=True)
    assert np.array_equal(r.stats.view(np.uint8), p.stats.view(np.uint8))
    assert np.array_equal(r.trace, p.trace)


def test_shared_memory_kernels_step_through_barriers():
    w = wl.smem_reduce(n=64 * 8, block=64)
    bufs = [(b.sim_base, b.data.copy()) for b in w.buffers]
    r = oracle.run_cached(w.ptx, w.kernel, w.grid, w.block, w.params, bufs, max_ts=w.max_ts, trace=True)
    assert r.status == 0
    bufs2 = [(b.sim_base, b.data.copy()) for b in w.buffers]
    p = oracle.run(w.ptx, w.kernel, w.grid, w.block, w.params, bufs2)
    for (_, a), (_, b) in zip(bufs, bufs2):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
    want = _replay(r, 1024, 49152)
    for (wi, k), lvl in want.items():
        assert int(r.log[wi][k]["level"]) == lvl

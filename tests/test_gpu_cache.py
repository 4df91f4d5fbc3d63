"""GPU parity for the L1/L2 hit model: ks_simulate_cached (two interpreter
passes and the radix-sorted levels between them) against the oracle's literal
stepper, byte for byte — memory, per-warp stats, trace slots, per-warp hit
counts and every logged access (line, step, level) — plus the statuses of a
full log and of an access stream that depends on the launch's own stores, and
properties at full size."""
import numpy as np
import pytest
import torch

import oracle
import simt_ptx_interpretation_gb300 as ks
from simt_ptx_interpretation_gb300 import workloads as wl
from tests import _cache_kernels as ck

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for -m gpu tests")
    from simt_ptx_interpretation_gb300 import _build
    _build.build_native()


def gpu_cached(ptx, kernel, grid, block, params, buffers, cache, max_ts=0, lat=ks.DEFAULT_LAT, layout="auto"):
    """buffers: [(sim_base, numpy array)] (copied to the device)."""
    mod = ks.Module(ptx)
    dev = [(base, torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).copy()).cuda()) for base, a in buffers]
    r = ks.run(mod, kernel, grid, block, params, dev, config=ks.Config(lat=lat, max_ts=max_ts, layout=layout),
               trace=max_ts > 0, cache=cache)
    torch.cuda.synchronize()
    return r, [t.cpu().numpy() for _, t in dev]


def check(ptx, kernel, grid, block, params, buffers, cache=None, max_ts=0, lat=ks.DEFAULT_LAT, layout="auto"):
    cache = cache or ks.CacheConfig(max_accesses_per_warp=256)
    g, gbufs = gpu_cached(ptx, kernel, grid, block, params, buffers, cache, max_ts, lat, layout)
    obufs = [(base, np.ascontiguousarray(a).copy()) for base, a in buffers]
    o = oracle.run_cached(ptx, kernel, grid, block, params, obufs, lat=lat, max_ts=max_ts, trace=max_ts > 0,
                          l1_lines=cache.l1_lines, l2_lines=cache.l2_lines, lat_l1=cache.lat_l1,
                          lat_l2=cache.lat_l2, log_cap=cache.max_accesses_per_warp)
    gs = ks.stats_array(g.stats)
    bad = np.nonzero(gs.view(np.uint8).reshape(-1, 96) != o.stats.view(np.uint8).reshape(-1, 96))[0]
    assert len(bad) == 0, f"stats differ at warps {np.unique(bad)[:5]}: gpu {gs[bad[0]]} oracle {o.stats[bad[0]]}"
    assert np.array_equal(g.cache_warps, o.warps), "per-warp cache counts differ"
    for w in range(len(o.warps)):
        n = int(o.warps[w]["n_access"])
        assert np.array_equal(g.cache_log[w][:n], o.log[w][:n]), f"access log differs at warp {w}"
    for (_, ob), gb in zip(obufs, gbufs):
        assert np.array_equal(ob.view(np.uint8), gb), "memory differs"
    if max_ts:
        assert np.array_equal(g.trace.cpu().numpy(), o.trace)
    assert g.totals.status == o.status == 0
    return g, o


def test_reuse():
    check(ck.REUSE, "reuse", 1, 32, ck.u64(ck.BASE_IN, ck.BASE_OUT),
          [(ck.BASE_IN, ck.f32_buffer(1024)), (ck.BASE_OUT, np.zeros(32, np.float32))])


@pytest.mark.parametrize("off_lines", [0, 1, 1024, 49152, 49152 + 1024])
def test_direct_mapped_sets(off_lines):
    off = off_lines * 128
    check(ck.PAIR, "pair", 1, 32, ck.u64(ck.BASE_IN, off), [(ck.BASE_IN, np.zeros((off + 256) // 4, np.float32))])


def test_small_caches():
    check(ck.PAIR, "pair", 1, 32, ck.u64(ck.BASE_IN, 256), [(ck.BASE_IN, np.zeros(1024, np.float32))],
          cache=ks.CacheConfig(l1_lines=2, l2_lines=4, max_accesses_per_warp=8))


@pytest.mark.parametrize("d0, d1", [(0, 0), (3, 0), (0, 3), (2, 1)])
def test_step_order(d0, d1):
    check(ck.order_kernel(d0, d1), "order", 1, 64, ck.u64(ck.BASE_IN), [(ck.BASE_IN, np.zeros(64, np.float32))])


def test_representative_and_stores():
    check(ck.REPRESENTATIVE, "rep", 1, 32, ck.u64(ck.BASE_IN), [(ck.BASE_IN, np.zeros(32 * 32 + 64, np.float32))])
    check(ck.STORE_THEN_LOAD, "stld", 1, 32, ck.u64(ck.BASE_OUT), [(ck.BASE_OUT, np.zeros(64, np.uint32))])


def test_barrier_release_steps():
    check(ck.BARRIER, "barrier", 1, 64, ck.u64(ck.BASE_IN), [(ck.BASE_IN, np.zeros(64, np.float32))])
    check(ck.BARRIER_EXIT, "barrier_exit", 1, 64, ck.u64(ck.BASE_IN), [(ck.BASE_IN, np.zeros(64, np.float32))])


def wl_check(w: wl.Workload, cache=None, layout="auto"):
    return check(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in w.fresh_buffers()],
                 cache=cache, max_ts=w.max_ts, layout=layout)


@pytest.mark.parametrize("layout", ["pair", "split"])
@pytest.mark.parametrize("name", ["vector_add", "ffma8", "gather4", "divergent", "fuzz2"])
def test_both_register_layouts(name, layout):
    """The hit model's two passes in each register layout, forced."""
    w = {"vector_add": lambda: wl.vector_add(), "ffma8": lambda: wl.ffma(acc=8, iters=8, grid=4, block=128),
         "gather4": lambda: wl.gather(4, n_out=1 << 12), "divergent": lambda: wl.divergent(4, n=1 << 11),
         "fuzz2": lambda: wl.fuzz(2, grid=4, block=64)}[name]()
    wl_check(w, cache=ks.CacheConfig(max_accesses_per_warp=4096), layout=layout)


def test_vector_add():
    wl_check(wl.vector_add())


@pytest.mark.parametrize("stride", [1, 4, 32])
def test_gather(stride):
    wl_check(wl.gather(stride, n_out=1 << 12))


def test_divergent():
    wl_check(wl.divergent(4, n=1 << 11))


@pytest.mark.parametrize("i", [0, 1, 2, 3, 5, 8])
def test_fuzz(i):
    wl_check(wl.fuzz(i, grid=4, block=64), cache=ks.CacheConfig(max_accesses_per_warp=4096))


@pytest.mark.parametrize("i", [0, 1])
def test_fuzz_small_caches(i):
    wl_check(wl.fuzz(i, grid=4, block=64), cache=ks.CacheConfig(l1_lines=4, l2_lines=12, max_accesses_per_warp=4096))


@pytest.mark.parametrize("block", [64, 256])
def test_smem_reduce(block):
    wl_check(wl.smem_reduce(n=block * 8, block=block))


@pytest.mark.parametrize("i", [0, 3])
def test_fuzz_shared(i):
    wl_check(wl.fuzz_shared(i, grid=4, block=128), cache=ks.CacheConfig(max_accesses_per_warp=4096))


def test_log_too_small():
    w_in = np.zeros(64, np.uint32)
    g, _ = gpu_cached(ck.READ_BACK, "read_back", 1, 32, ck.u64(ck.BASE_IN, ck.BASE_OUT),
                      [(ck.BASE_IN, w_in), (ck.BASE_OUT, np.zeros(32, np.uint32))],
                      ks.CacheConfig(max_accesses_per_warp=1))
    assert g.totals.status == ks.api.ST_CACHE_LOG


def test_stream_that_reads_its_own_stores():
    # the first pass stores nothing, reads 0 back and makes one more access
    g, bufs = gpu_cached(ck.READ_BACK, "read_back", 1, 32, ck.u64(ck.BASE_IN, ck.BASE_OUT),
                         [(ck.BASE_IN, np.zeros(64, np.uint32)), (ck.BASE_OUT, np.zeros(32, np.uint32))],
                         ks.CacheConfig(max_accesses_per_warp=8))
    assert g.totals.status == ks.api.ST_CACHE_STREAM


def test_gather_full_size_all_misses():
    """2^24 outputs at stride 8: every line is touched once, so every access
    misses both levels and the cycles equal those of the plain run."""
    w = wl.gather(8)
    dev = [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()]
    mod = ks.Module(w.ptx)
    cache = ks.CacheConfig(max_accesses_per_warp=2)
    r = ks.run(mod, w.kernel, w.grid, w.block, w.params, dev, cache=cache)
    p = ks.run(mod, w.kernel, w.grid, w.block, w.params,
               [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()])
    torch.cuda.synchronize()
    assert r.totals.status == 0
    assert (r.cache_warps["n_access"] == 2).all() and (r.cache_warps["dram"] == 2).all()
    assert np.array_equal(ks.stats_array(r.stats), ks.stats_array(p.stats))
    assert torch.equal(dev[1][1], p.buffers[1][1])


def _replay_levels(warps, log, l1_lines, l2_lines):
    """Levels of a direct-mapped L1/L2 over the logged (step, warp) order,
    computed with numpy sorts on the host."""
    W, cap = log.shape
    n = warps["n_access"].astype(np.int64)
    k = np.arange(cap)[None, :]
    valid = k < n[:, None]
    wi = np.broadcast_to(np.arange(W)[:, None], (W, cap))[valid]
    line = log["line"][valid].astype(np.uint64)
    step = log["step"][valid].astype(np.uint64)
    out = np.full(line.shape, 2, dtype=np.uint32)
    order = np.lexsort((wi, step, line % np.uint64(l1_lines)))
    ls = line[order]
    hit1 = np.zeros(len(ls), bool)
    hit1[1:] = (ls[1:] == ls[:-1])
    out[order[hit1]] = 0
    miss = order[~hit1]
    m_order = np.lexsort((wi[miss], step[miss], line[miss] % np.uint64(l2_lines)))
    lm = line[miss][m_order]
    hit2 = np.zeros(len(lm), bool)
    hit2[1:] = (lm[1:] == lm[:-1])
    out[miss[m_order][hit2]] = 1
    levels = np.full((W, cap), 255, dtype=np.uint32)
    levels[valid] = out
    return levels, valid


@pytest.mark.parametrize("i", [0, 7])
def test_fuzz_full_size_properties(i):
    """1024 x 256 fuzz kernel: memory and every count but cycles equal the
    plain run's, the log agrees with the request counts, the levels equal a
    host replay of the logged stream, and no warp's cycles grow."""
    w = wl.fuzz(i)
    mod = ks.Module(w.ptx)
    cache = ks.CacheConfig(max_accesses_per_warp=4096)
    dev = [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()]
    r = ks.run(mod, w.kernel, w.grid, w.block, w.params, dev, config=ks.Config(max_ts=w.max_ts), trace=True,
               cache=cache)
    dev2 = [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()]
    p = ks.run(mod, w.kernel, w.grid, w.block, w.params, dev2, config=ks.Config(max_ts=w.max_ts), trace=True)
    torch.cuda.synchronize()
    assert r.totals.status == 0 and p.totals.status == 0
    for (_, a), (_, b) in zip(dev, dev2):
        assert torch.equal(a, b)
    rs, ps = ks.stats_array(r.stats), ks.stats_array(p.stats)
    for f in ("warp_insts", "thread_insts", "ld_req", "ld_sectors", "st_req", "st_sectors", "ld_lines", "st_lines"):
        assert np.array_equal(rs[f], ps[f]), f
    assert (rs["cycles"] <= ps["cycles"]).all()
    assert np.array_equal(r.cache_warps["n_access"].astype(np.uint64), rs["ld_req"] + rs["st_req"])
    levels, valid = _replay_levels(r.cache_warps, r.cache_log, cache.l1_lines, cache.l2_lines)
    assert np.array_equal(r.cache_log["level"][valid], levels[valid])


@pytest.mark.parametrize("block", [512, 1024])
def test_large_blocks(block):
    # CTA mode with 16 and 32 warps (the 1024-thread instantiation)
    wl_check(wl.smem_reduce(n=block * 4, block=block))


def test_cta_warp_state_in_global_memory():
    """A random shared program at block 1024, whose warps' state lives in
    global memory: both passes of the hit model equal the oracle's stepper."""
    wl_check(wl.fuzz_shared(0, grid=3, block=1024), cache=ks.CacheConfig(max_accesses_per_warp=4096))


def _cached_job(w: wl.Workload, cache: ks.CacheConfig):
    mod = ks.Module(w.ptx)
    dev = [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()]
    st = torch.empty(ks.stats_bytes(w.grid, w.block), dtype=torch.uint8, device="cuda")
    tr = torch.empty(ks.trace_bytes(w.grid, w.block, w.max_ts, mod.record_bytes(w.kernel)), dtype=torch.uint8,
                     device="cuda")
    ws = torch.zeros(ks.cache_workspace_bytes(w.grid, w.block, cache), dtype=torch.uint8, device="cuda")
    item = ks.BatchItem(mod, w.kernel, w.grid, w.block, w.params, dev, st, tr, ks.Config(max_ts=w.max_ts))
    return ks.CachedBatchItem(item, cache, ws)


def test_cached_batch_matches_the_oracle():
    """ks_simulate_cached_batch: items of two modes with their own hit models
    (two small, one default), first and second passes batched; each equals
    the oracle's literal stepper byte for byte."""
    small = ks.CacheConfig(l1_lines=4, l2_lines=12, max_accesses_per_warp=4096)
    ws = [(wl.vector_add(), ks.CacheConfig(max_accesses_per_warp=8)),
          (wl.gather(4, n_out=1 << 12), ks.CacheConfig(max_accesses_per_warp=8)),
          (wl.divergent(4, n=1 << 11), ks.CacheConfig(max_accesses_per_warp=64)),
          (wl.fuzz(0, grid=4, block=64), small), (wl.fuzz(5, grid=4, block=64), ks.CacheConfig(max_accesses_per_warp=4096)),
          (wl.smem_reduce(n=256 * 4, block=256), ks.CacheConfig(max_accesses_per_warp=64)),
          (wl.fuzz_shared(3, grid=4, block=128), small)]
    jobs = [_cached_job(w, c) for w, c in ws]
    n = ks.simulate_cached_batch(jobs)
    torch.cuda.synchronize()
    assert n >= 4  # two passes of two groups, plus the level kernels
    for (w, c), j in zip(ws, jobs):
        o = oracle.run_cached(w.ptx, w.kernel, w.grid, w.block, w.params,
                              [(b.sim_base, b.data) for b in w.fresh_buffers()], max_ts=w.max_ts, trace=True,
                              l1_lines=c.l1_lines, l2_lines=c.l2_lines, lat_l1=c.lat_l1, lat_l2=c.lat_l2,
                              log_cap=c.max_accesses_per_warp)
        assert o.status == 0
        assert np.array_equal(j.item.stats.cpu().numpy(), o.stats.view(np.uint8)), w.name
        assert np.array_equal(j.item.trace.cpu().numpy(), o.trace), w.name
        cw, log = ks.cache_results(j.workspace, w.warps, c)
        assert np.array_equal(cw, o.warps), w.name
        for k in range(w.warps):
            m = int(o.warps[k]["n_access"])
            assert np.array_equal(log[k][:m], o.log[k][:m]), (w.name, k)
        obufs = w.fresh_buffers()
        oracle.run_cached(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in obufs],
                          l1_lines=c.l1_lines, l2_lines=c.l2_lines, lat_l1=c.lat_l1, lat_l2=c.lat_l2,
                          log_cap=c.max_accesses_per_warp)
        for (_, t), b in zip(j.item.buffers, obufs):
            assert np.array_equal(t.cpu().numpy(), b.data.view(np.uint8)), w.name


def test_cached_batch_pair_equals_single_calls():
    """The FFMA pair (grid 132 x block 128, 64 iterations) through one cached
    batch and through two ks_simulate_cached calls."""
    cache = ks.CacheConfig(max_accesses_per_warp=4)
    ws = [wl.ffma(acc=1, iters=64), wl.ffma(acc=8, iters=64)]
    jobs = [_cached_job(w, cache) for w in ws]
    ks.simulate_cached_batch(jobs)
    for w, j in zip(ws, jobs):
        r = ks.run(ks.Module(w.ptx), w.kernel, w.grid, w.block, w.params,
                   [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()],
                   config=ks.Config(max_ts=w.max_ts), trace=True, cache=cache)
        torch.cuda.synchronize()
        assert r.totals.status == 0
        assert torch.equal(j.item.stats, r.stats) and torch.equal(j.item.trace, r.trace)
        cw, _ = ks.cache_results(j.workspace, w.warps, cache)
        assert np.array_equal(cw, r.cache_warps)


def test_cached_batch_workspace_too_small():
    w = wl.vector_add()
    jobs = [_cached_job(w, ks.CacheConfig(max_accesses_per_warp=8)) for _ in range(2)]
    jobs[1].workspace = jobs[1].workspace[:-256]
    with pytest.raises(ks.KsError) as e:
        ks.simulate_cached_batch(jobs)
    assert "batch item 1" in str(e.value)

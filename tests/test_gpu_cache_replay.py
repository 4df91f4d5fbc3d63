"""The L1/L2 hit model's timing-replay form (ks_cache_config.max_runs_per_warp
> 0, kernels without shared memory or bar.sync): one interpretation that is
the real run and logs each warp's issued runs, the level sorts, then a
value-free replay of every warp's scoreboard. Every output equals the
oracle's literal stepper byte for byte -- stats (cycles from the levels),
per-warp hit counts, the access log with its levels, trace slots (timestamps
from the replay), memory -- and equals the re-interpretation form where both
apply; a warp that reads back its own stores gets the oracle's values; logs
that overflow are reported."""
import numpy as np
import pytest
import torch

import oracle
import simt_ptx_interpretation_gb300 as ks
from simt_ptx_interpretation_gb300 import workloads as wl
from tests import _cache_kernels as ck
from tests import test_gpu_cache as tgc

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for -m gpu tests")
    from simt_ptx_interpretation_gb300 import _build
    _build.build_native()


def replay(cap: int = 4096, runs: int = 16384, **kw) -> ks.CacheConfig:
    return ks.CacheConfig(max_accesses_per_warp=cap, max_runs_per_warp=runs, **kw)


WORKLOADS = {
    "vector_add": (lambda: wl.vector_add(), replay(8, 16)),
    "ffma1": (lambda: wl.ffma(acc=1, iters=16, grid=4, block=128), replay(8, 64)),
    "ffma8": (lambda: wl.ffma(acc=8, iters=16, grid=4, block=128), replay(8, 64)),
    "gather1": (lambda: wl.gather(1, n_out=1 << 12), replay(4, 8)),
    "gather32": (lambda: wl.gather(32, n_out=1 << 12), replay(4, 8)),
    "divergent2": (lambda: wl.divergent(2, n=1 << 11), replay(64, 2048)),
    "divergent32": (lambda: wl.divergent(32, n=1 << 11), replay(64, 2048)),
    "fuzz0_small_caches": (lambda: wl.fuzz(0, grid=4, block=64), replay(l1_lines=4, l2_lines=12)),
}


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_workloads_match_the_oracle(name):
    make, cache = WORKLOADS[name]
    tgc.wl_check(make(), cache=cache)


@pytest.mark.parametrize("i", [1, 2, 3, 5, 8, 13, 21, 34])
def test_fuzz_matches_the_oracle(i):
    tgc.wl_check(wl.fuzz(i, grid=4, block=64), cache=replay())


@pytest.mark.parametrize("layout", ["pair", "split"])
def test_both_register_layouts(layout):
    tgc.wl_check(wl.fuzz(2, grid=4, block=64), cache=replay(), layout=layout)
    tgc.wl_check(wl.divergent(4, n=1 << 11), cache=replay(64, 2048), layout=layout)


def test_hand_derived_hit_sequences():
    """The hand-derived cases of the hit model: reuse, direct-mapped set
    conflicts at both levels, step order between warps, the lowest executing
    lane's line, stores installing lines."""
    c = replay(64, 64)
    tgc.check(ck.REUSE, "reuse", 1, 32, ck.u64(ck.BASE_IN, ck.BASE_OUT),
              [(ck.BASE_IN, ck.f32_buffer(1024)), (ck.BASE_OUT, np.zeros(32, np.float32))], cache=c)
    for off_lines in (0, 1, 1024, 49152, 49152 + 1024):
        off = off_lines * 128
        tgc.check(ck.PAIR, "pair", 1, 32, ck.u64(ck.BASE_IN, off),
                  [(ck.BASE_IN, np.zeros((off + 256) // 4, np.float32))], cache=c)
    tgc.check(ck.PAIR, "pair", 1, 32, ck.u64(ck.BASE_IN, 256), [(ck.BASE_IN, np.zeros(1024, np.float32))],
              cache=replay(8, 8, l1_lines=2, l2_lines=4))
    for d0, d1 in ((0, 0), (3, 0), (0, 3), (2, 1)):
        tgc.check(ck.order_kernel(d0, d1), "order", 1, 64, ck.u64(ck.BASE_IN),
                  [(ck.BASE_IN, np.zeros(64, np.float32))], cache=c)
    tgc.check(ck.REPRESENTATIVE, "rep", 1, 32, ck.u64(ck.BASE_IN),
              [(ck.BASE_IN, np.zeros(32 * 32 + 64, np.float32))], cache=c)
    tgc.check(ck.STORE_THEN_LOAD, "stld", 1, 32, ck.u64(ck.BASE_OUT), [(ck.BASE_OUT, np.zeros(64, np.uint32))],
              cache=c)


def test_equals_the_reinterpretation_form():
    """Where both forms apply they give the same bytes."""
    for w in (wl.fuzz(7, grid=4, block=64), wl.divergent(4, n=1 << 11), wl.ffma(acc=8, iters=8, grid=2)):
        a, abufs = tgc.gpu_cached(w.ptx, w.kernel, w.grid, w.block, w.params,
                                  [(b.sim_base, b.data) for b in w.fresh_buffers()], replay(), max_ts=w.max_ts)
        b, bbufs = tgc.gpu_cached(w.ptx, w.kernel, w.grid, w.block, w.params,
                                  [(b.sim_base, b.data) for b in w.fresh_buffers()], replay(runs=0), max_ts=w.max_ts)
        assert torch.equal(a.stats, b.stats) and np.array_equal(a.cache_warps, b.cache_warps), w.name
        if w.max_ts:
            assert torch.equal(a.trace, b.trace), w.name
        for x, y in zip(abufs, bbufs):
            assert np.array_equal(x, y), w.name


def test_reading_back_its_own_stores():
    """The re-interpretation form reports KS_ST_CACHE_STREAM for this warp;
    the replay form's one interpretation is the real run, so it gets the
    values it stored, as the oracle's stepper does."""
    bufs = [(ck.BASE_IN, np.zeros(64, np.uint32)), (ck.BASE_OUT, np.zeros(32, np.uint32))]
    tgc.check(ck.READ_BACK, "read_back", 1, 32, ck.u64(ck.BASE_IN, ck.BASE_OUT), bufs, cache=replay(8, 8))


def test_logs_too_small():
    bufs = lambda: [(ck.BASE_IN, np.zeros(64, np.uint32)), (ck.BASE_OUT, np.zeros(32, np.uint32))]
    g, _ = tgc.gpu_cached(ck.READ_BACK, "read_back", 1, 32, ck.u64(ck.BASE_IN, ck.BASE_OUT), bufs(), replay(1, 8))
    assert g.totals.status == ks.api.ST_CACHE_LOG  # two accesses, one logged
    w = wl.ffma(acc=1, iters=16, grid=2, block=64)
    g, _ = tgc.gpu_cached(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in w.fresh_buffers()],
                          replay(8, 4))
    assert g.totals.status == ks.api.ST_CACHE_LOG  # 17 runs, four logged


def test_batch_of_both_forms():
    """A cached batch whose plain items take the replay form and whose
    CTA-mode items re-interpret; each equals the oracle."""
    small = replay(l1_lines=4, l2_lines=12)
    ws = [(wl.vector_add(), replay(8, 16)), (wl.divergent(4, n=1 << 11), replay(64, 2048)),
          (wl.fuzz(5, grid=4, block=64), small), (wl.smem_reduce(n=256 * 4, block=256), replay(64, 64)),
          (wl.fuzz_shared(3, grid=4, block=128), small)]
    jobs = [tgc._cached_job(w, c) for w, c in ws]
    ks.simulate_cached_batch(jobs)
    torch.cuda.synchronize()
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
        obufs = w.fresh_buffers()
        oracle.run_cached(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in obufs],
                          l1_lines=c.l1_lines, l2_lines=c.l2_lines, lat_l1=c.lat_l1, lat_l2=c.lat_l2,
                          log_cap=c.max_accesses_per_warp)
        for (_, t), b in zip(j.item.buffers, obufs):
            assert np.array_equal(t.cpu().numpy(), b.data.view(np.uint8)), w.name


def test_ffma_pair_headline_size():
    """The FFMA pair at its headline size (grid 132 x block 128, 4096 x 32
    FFMA) in one cached batch of the replay form: every warp's stats, trace
    and hit counts equal the re-interpretation form's (checked against the
    oracle on smaller grids above)."""
    runs = replay(4, 8192)
    ws = [wl.ffma(acc=1), wl.ffma(acc=8)]
    jobs = [tgc._cached_job(w, runs) for w in ws]
    ks.simulate_cached_batch(jobs)
    ref = [tgc._cached_job(w, replay(4, 0)) for w in ws]
    ks.simulate_cached_batch(ref)
    torch.cuda.synchronize()
    for w, j, r in zip(ws, jobs, ref):
        assert torch.equal(j.item.stats, r.item.stats) and torch.equal(j.item.trace, r.item.trace), w.name
        a, _ = ks.cache_results(j.workspace, w.warps, runs)
        b, _ = ks.cache_results(r.workspace, w.warps, replay(4, 0))
        assert np.array_equal(a, b)
        assert int(ks.stats_array(j.item.stats)["status"].max()) == 0


def test_gather_full_size_all_misses():
    """2^24 outputs at stride 8 in the replay form: every access misses both
    levels, so every warp's record equals the plain run's."""
    w = wl.gather(8)
    dev = [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()]
    mod = ks.Module(w.ptx)
    r = ks.run(mod, w.kernel, w.grid, w.block, w.params, dev, cache=replay(2, 2))
    p = ks.run(mod, w.kernel, w.grid, w.block, w.params,
               [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()])
    torch.cuda.synchronize()
    assert r.totals.status == 0
    assert (r.cache_warps["n_access"] == 2).all() and (r.cache_warps["dram"] == 2).all()
    assert np.array_equal(ks.stats_array(r.stats), ks.stats_array(p.stats))
    assert torch.equal(dev[1][1], p.buffers[1][1])


def test_forked_replays_keep_the_callers_order():
    """A cached batch's replays run side by side on the library's helper
    streams; copies of the outputs made on the caller's stream right after the
    call, with no synchronisation in between, equal single cached calls."""
    ws = [(wl.divergent(k, n=1 << 14), replay(64, 2048)) for k in (2, 4, 32, 2)]
    jobs = [tgc._cached_job(w, c) for w, c in ws]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ks.simulate_cached_batch(jobs, stream=s)
        copies = [(j.item.stats.clone(), j.item.trace.clone(), j.workspace[:w.warps * 16].clone())
                  for (w, _), j in zip(ws, jobs)]
    torch.cuda.synchronize()
    for (w, c), (st, tr, cw) in zip(ws, copies):
        g, _ = tgc.gpu_cached(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in w.buffers],
                              c, max_ts=w.max_ts)
        assert np.array_equal(st.cpu().numpy(), g.stats.cpu().numpy()), w.name
        assert np.array_equal(tr.cpu().numpy(), g.trace.cpu().numpy()), w.name
        assert np.array_equal(cw.cpu().numpy().view(ks.api.CACHE_WARP_DTYPE), g.cache_warps), w.name

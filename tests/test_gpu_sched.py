"""GPU parity for the SM issue model: ks_simulate_sched (the instrumented
interpreter logging each warp's issued runs, then one replay warp per
simulated SM) against the oracle's cycle-by-cycle SM simulation, record for
record, over the hand-made pin kernels and the workloads in several SM
shapes; the per-warp outputs stay those of the plain run; properties at full
size."""
import numpy as np
import pytest
import torch

import oracle
import simt_ptx_interpretation_gb300 as ks
from simt_ptx_interpretation_gb300 import workloads as wl
from tests import test_oracle_sched as tos

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for -m gpu tests")
    from simt_ptx_interpretation_gb300 import _build
    _build.build_native()


def check(ptx, kernel, grid, block, params, buffers, n_sm, ctas_per_sm=0, schedulers=4, max_ts=0, layout="auto"):
    sc = ks.SchedConfig(n_sm=n_sm, ctas_per_sm=ctas_per_sm, schedulers_per_sm=schedulers)
    mod = ks.Module(ptx)
    dev = [(base, torch.from_numpy(np.ascontiguousarray(a).view(np.uint8).copy()).cuda()) for base, a in buffers]
    r = ks.run(mod, kernel, grid, block, params, dev, config=ks.Config(max_ts=max_ts, layout=layout), trace=max_ts > 0,
               sched=sc)
    torch.cuda.synchronize()
    obufs = [(base, np.ascontiguousarray(a).copy()) for base, a in buffers]
    ow, osm = oracle.run_sched(ptx, kernel, grid, block, params, obufs, n_sm=n_sm, ctas_per_sm=ctas_per_sm,
                               schedulers=schedulers)
    bad = np.nonzero(r.sched_warps.view(np.uint8).reshape(-1, 80) != ow.view(np.uint8).reshape(-1, 80))[0]
    assert len(bad) == 0, f"schedule differs at warps {np.unique(bad)[:5]}: gpu {r.sched_warps[bad[0]]} oracle {ow[bad[0]]}"
    assert np.array_equal(r.sched_sms.view(np.uint8), osm.view(np.uint8)), f"SM records differ: {r.sched_sms} {osm}"
    for (_, g), (_, o) in zip(dev, obufs):
        assert np.array_equal(g.cpu().numpy(), o.view(np.uint8)), "memory differs"
    # the per-warp outputs are the plain run's
    p = oracle.run(ptx, kernel, grid, block, params, [(base, np.ascontiguousarray(a).copy()) for base, a in buffers],
                   max_ts=max_ts, trace=max_ts > 0)
    assert np.array_equal(ks.stats_array(r.stats).view(np.uint8), p.stats.view(np.uint8))
    if max_ts:
        assert np.array_equal(r.trace.cpu().numpy(), p.trace)
    assert r.totals.status == 0 and int(osm["status"].max()) == 0
    return r, ow


@pytest.mark.parametrize("k, s", [(1, 1), (3, 1), (8, 4), (8, 2)])
def test_independent_streams(k, s):
    check(tos.independent(10), "k", 1, 32 * k, b"", [], n_sm=1, schedulers=s)


@pytest.mark.parametrize("block", [32, 64, 128])
def test_chains(block):
    check(tos.chain(6), "k", 1, block, b"", [], n_sm=1, schedulers=1)
    check(tos.chain(6), "k", 2, block, b"", [], n_sm=1, schedulers=2)


def test_wait_kinds_and_barriers():
    check(tos.LOAD_USE, "k", 1, 32, (0x1000_0000).to_bytes(8, "little"), [(0x1000_0000, np.ones(64, np.float32))],
          n_sm=1, schedulers=1)
    check(tos.BARRIER, "k", 1, 64, b"", [], n_sm=1, schedulers=4)
    check(tos.BARRIER, "k", 3, 64, b"", [], n_sm=1, schedulers=1)


@pytest.mark.parametrize("n_sm, ctas", [(1, 1), (2, 1), (1, 0), (4, 2)])
def test_cta_dispatch(n_sm, ctas):
    check(tos.independent(10), "k", 5, 32, b"", [], n_sm=n_sm, ctas_per_sm=ctas, schedulers=1)


WORKLOADS = {
    "vector_add": lambda: wl.vector_add(),
    "gather_s4": lambda: wl.gather(4, n_out=1 << 12),
    "divergent_k2": lambda: wl.divergent(2, n=1 << 11),
    "divergent_k32": lambda: wl.divergent(32, n=1 << 10),
    "ffma1": lambda: wl.ffma(acc=1, iters=4, grid=6, block=128),
    "ffma8": lambda: wl.ffma(acc=8, iters=4, grid=6, block=128),
    "fuzz0": lambda: wl.fuzz(0, grid=6, block=64),
    "fuzz5": lambda: wl.fuzz(5, grid=6, block=64),
    "smem_reduce": lambda: wl.smem_reduce(n=256 * 6, block=256),
    "fuzz_shared": lambda: wl.fuzz_shared(3, grid=6, block=128),
}


@pytest.mark.parametrize("shape", [(3, 0, 4), (2, 1, 1), (6, 0, 2)])
@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_workloads(name, shape):
    w = WORKLOADS[name]()
    n_sm, ctas, s = shape
    check(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in w.fresh_buffers()],
          n_sm=n_sm, ctas_per_sm=ctas, schedulers=s, max_ts=w.max_ts)


def test_log_too_small():
    w = WORKLOADS["fuzz0"]()
    mod = ks.Module(w.ptx)
    dev = [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()]
    r = ks.run(mod, w.kernel, w.grid, w.block, w.params, dev,
               sched=ks.SchedConfig(n_sm=2, max_runs_per_warp=2))
    torch.cuda.synchronize()
    assert r.totals.status == ks.api.ST_SCHED_LIMIT
    assert int(r.sched_sms["status"].max()) == ks.api.ST_SCHED_LIMIT


@pytest.mark.parametrize("acc", [1, 8])
def test_ffma_headline_properties(acc):
    """The FFMA probe at 132 x 128 on the 152-SM model: every warp issues what
    it issues alone, never ends earlier than alone, its waits add up, and the
    SM issue totals match."""
    w = wl.ffma(acc=acc)
    mod = ks.Module(w.ptx)
    dev = [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()]
    r = ks.run(mod, w.kernel, w.grid, w.block, w.params, dev, sched=ks.SchedConfig())
    p = ks.run(mod, w.kernel, w.grid, w.block, w.params,
               [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()])
    torch.cuda.synchronize()
    ws, st = r.sched_warps, ks.stats_array(p.stats)
    assert r.totals.status == 0 and int(r.sched_sms["status"].max()) == 0
    assert np.array_equal(ws["issued"], st["warp_insts"])
    assert ((ws["end"] - ws["start"]) >= st["cycles"]).all()
    used = ws["issued"] + ws["not_selected"] + ws["stall_exec"] + ws["stall_mem"] + ws["stall_math"]
    tail = (ws["end"] - ws["start"]).astype(np.int64) - used.astype(np.int64)
    assert (tail >= 0).all() and (tail <= 400).all()
    assert int(r.sched_sms["issued"].sum()) == int(st["warp_insts"].sum())
    assert int(r.sched_sms["ctas"].sum()) == w.grid
    # 132 CTAs of 4 warps on 152 SMs: one CTA per SM, one warp per scheduler,
    # so no warp waits for another
    assert (ws["not_selected"] == 0).all()
    assert np.array_equal(ws["end"] - ws["start"], st["cycles"])


def test_warp_sweep_matches_oracle():
    from simt_ptx_interpretation_gb300 import sweep
    rows = sweep.warp_sweep(iters=4, n_sm=4, schedulers=4, configs=sweep.default_configs(4))
    want = []
    for grid, block in sweep.default_configs(4):
        w = wl.ffma(acc=1, iters=4, grid=grid, block=block)
        ws, sms = oracle.run_sched(w.ptx, w.kernel, w.grid, w.block, w.params,
                                   [(b.sim_base, b.data) for b in w.fresh_buffers()], n_sm=4, schedulers=4)
        want.append((int(ws["issued"].sum()), int(sms["cycles"].max())))
    assert [(r["total_instructions"], r["cycles"]) for r in rows] == want
    assert [r["active_warps"] for r in rows] == [1, 1, 2, 4, 16]
    ipc = [r["instructions_per_cycle"] for r in rows]
    assert ipc[0] == ipc[1] and abs(ipc[3] - 4 * ipc[1]) < 1e-9 and abs(ipc[4] - 4 * ipc[3]) < 1e-9


@pytest.mark.parametrize("block", [512, 1024])
def test_large_blocks(block):
    w = wl.smem_reduce(n=block * 5, block=block)
    check(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in w.fresh_buffers()],
          n_sm=2, schedulers=4, max_ts=w.max_ts)


def test_cta_warp_state_in_global_memory():
    """A random shared program at block 1024, whose warps' state lives in
    global memory: the issue log and the replay equal the oracle's SM model."""
    w = wl.fuzz_shared(1, grid=3, block=1024)
    check(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in w.fresh_buffers()],
          n_sm=2, schedulers=4, max_ts=w.max_ts)


@pytest.mark.parametrize("layout", ["pair", "split"])
@pytest.mark.parametrize("name", ["vector_add", "ffma8", "divergent", "fuzz0"])
def test_both_register_layouts(name, layout):
    """The issue log and the replay in each register layout, forced (the
    replay reads the decoded records of either layout)."""
    w = {"vector_add": lambda: wl.vector_add(), "ffma8": lambda: wl.ffma(acc=8, iters=4, grid=6, block=128),
         "divergent": lambda: wl.divergent(4, n=1 << 11), "fuzz0": lambda: wl.fuzz(0, grid=6, block=64)}[name]()
    check(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in w.fresh_buffers()],
          n_sm=3, schedulers=4, max_ts=w.max_ts, layout=layout)

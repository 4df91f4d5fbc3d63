"""GPU parity for ks_simulate_batch: launches simulated together in one real
grid give the oracle's results byte for byte (memory, per-warp stats, trace
slots, per-instruction profiles), whatever the grouping — plain and CTA-mode
items, lean and profiled forms, more items than one grid takes, more warps
than one wave, the persistent shape — and a refused item launches nothing."""
import numpy as np
import pytest
import torch

import oracle
from oracle import hints as oh
import simt_ptx_interpretation_gb300 as ks
from simt_ptx_interpretation_gb300 import api
from simt_ptx_interpretation_gb300 import workloads as wl
from tests import _parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for -m gpu tests")
    from simt_ptx_interpretation_gb300 import _build
    _build.build_native()


class Job:
    """One batch item with its device buffers and outputs (stats filled with
    a sentinel so that an untouched record shows)."""

    def __init__(self, w: wl.Workload, module=None, profile: bool = False, layout: str = "auto"):
        self.w = w
        self.layout = layout
        self.mod = module or ks.Module(w.ptx)
        self.dev = [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()]
        self.stats = torch.full((ks.stats_bytes(w.grid, w.block),), 0xA5, dtype=torch.uint8, device="cuda")
        self.trace = torch.empty(ks.trace_bytes(w.grid, w.block, w.max_ts, self.mod.record_bytes(w.kernel)),
                                 dtype=torch.uint8, device="cuda")
        self.prof = (torch.full((self.mod.profile_bytes(w.kernel),), 0xFF, dtype=torch.uint8, device="cuda")
                     if profile else None)

    def item(self) -> ks.BatchItem:
        cfg = ks.Config(max_ts=self.w.max_ts, profile=self.prof, layout=self.layout)
        return ks.BatchItem(self.mod, self.w.kernel, self.w.grid, self.w.block, self.w.params, self.dev, self.stats,
                            self.trace, cfg)

    def check_oracle(self, warps=None, out_words=None):
        w = self.w
        o, obufs = _parity.oracle_run(w, warps=warps)
        sel = np.arange(w.warps) if warps is None else np.asarray(warps)
        gs = ks.stats_array(self.stats)[sel].view(np.uint8).reshape(len(sel), 96)
        os_ = o.stats[sel].view(np.uint8).reshape(len(sel), 96)
        bad = np.nonzero((gs != os_).any(axis=1))[0]
        assert len(bad) == 0, f"{w.name}: stats differ at warps {sel[bad[:5]]}"
        sb = _parity.slot_bytes(w.max_ts, oracle.record_bytes(w.ptx, w.kernel))
        gt = self.trace.cpu().numpy().reshape(w.warps, sb)[sel]
        ot = o.trace.reshape(w.warps, sb)[sel]
        assert np.array_equal(gt, ot), f"{w.name}: trace differs"
        for b, (_, t), ob in zip(w.buffers, self.dev, obufs):
            g = t.cpu().numpy()
            if warps is None:
                assert np.array_equal(g, ob), f"{w.name}: buffer {b.name} differs"
            elif out_words is not None and b.name in out_words:
                idx = np.asarray(out_words[b.name], dtype=np.int64)
                assert np.array_equal(g.view(np.uint32)[idx], ob.view(np.uint32)[idx]), f"{w.name}: {b.name}"
        if self.prof is not None:
            _, ev = oracle.run_events(w.ptx, w.kernel, w.grid, w.block, w.params,
                                      [(b.sim_base, b.data) for b in w.fresh_buffers()])
            op = oh.profile(ev, len(oracle.ipdom(w.ptx, w.kernel)))
            assert np.array_equal(api.profile_array(self.prof).view(np.uint8), op.view(np.uint8)), w.name


def run_batch(jobs) -> int:
    n = ks.simulate_batch([j.item() for j in jobs])
    torch.cuda.synchronize()
    return n


@pytest.mark.parametrize("fuzz_layout", ["pair", "auto"])
def test_plain_items_in_one_grid(fuzz_layout):
    """Plain items of one layout share one real grid; the fuzz kernels run in
    the SPLIT layout unless forced to PAIR, and then take a grid of their own."""
    jobs = [Job(wl.ffma(acc=1, iters=40, grid=6, block=128)), Job(wl.ffma(acc=8, iters=40, grid=6, block=128)),
            Job(wl.divergent(2, n=2048)), Job(wl.vector_add()), Job(wl.gather(4, n_out=1 << 12))]
    jobs += [Job(wl.fuzz(i, grid=4, block=64), layout=fuzz_layout) for i in range(6)]
    assert run_batch(jobs) == (1 if fuzz_layout == "pair" else 2)
    for j in jobs:
        j.check_oracle()


def test_groups_of_modes_forms_and_blocks():
    """CTA-mode items of two blocks (two groups), a profiled plain item among
    lean ones, two items through one module."""
    f = wl.ffma(acc=2, iters=24, grid=4, block=96)
    shared = ks.Module(f.ptx)
    jobs = [Job(wl.smem_reduce(n=256 * 4, block=256)), Job(f, module=shared),
            Job(wl.fuzz(3, grid=4, block=64), profile=True), Job(wl.smem_reduce(n=128 * 6, block=128)),
            Job(wl.ffma(acc=2, iters=24, grid=4, block=96, seed=7), module=shared),
            Job(wl.fuzz_shared(1, grid=4, block=128)), Job(wl.smem_reduce(n=256 * 3, block=256)),
            Job(wl.divergent(32, n=1024), profile=True)]
    run_batch(jobs)
    for j in jobs:
        j.check_oracle()


def test_more_items_than_one_grid_takes():
    """40 items: two real grids of one group, compared with single launches
    and, for a sample, with the oracle."""
    ws = [wl.fuzz(i % 8, grid=2, block=64, data_seed=4 + i) for i in range(40)]
    jobs = [Job(w) for w in ws]
    assert run_batch(jobs) == 2
    for k, (w, j) in enumerate(zip(ws, jobs)):
        g = _parity.gpu_run(w)
        assert np.array_equal(ks.stats_array(j.stats).view(np.uint8), g.stats.view(np.uint8)), k
        assert np.array_equal(j.trace.cpu().numpy(), g.trace), k
        for (_, t), gb in zip(j.dev, g.buffers):
            assert np.array_equal(t.cpu().numpy(), gb), k
    for k in (0, 17, 39):
        jobs[k].check_oracle()


def test_many_grids_of_one_wave():
    """12 x 512 warps: more than one wave of the GPU, so the items go out as
    several real grids; equal to single launches."""
    ws = [wl.divergent(k, n=512 * 32) for k in (2, 4, 32)] * 4
    jobs = [Job(w) for w in ws]
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    per_grid = 16 * sms // 512  # items of 512 warps in 16 warps per SM
    assert run_batch(jobs) == -(-12 // per_grid)
    for k in range(3):
        g = _parity.gpu_run(ws[k])
        for j in jobs[k::3]:
            assert np.array_equal(ks.stats_array(j.stats).view(np.uint8), g.stats.view(np.uint8))
            assert np.array_equal(j.dev[1][1].cpu().numpy(), g.buffers[1])
    w = ws[0]
    warps = _parity.sample_warps(w, n=24, seed=3)
    jobs[0].check_oracle(warps=warps, out_words={"out": _parity.thread_ids(w, warps)})


def many_registers(seed: int, n_regs: int = 60, grid: int = 16, block: int = 128) -> wl.Workload:
    """A straight chain over n_regs 32-bit registers (a large register region
    per warp), stored to out[gtid]."""
    lines = ["mov.u32 %r0, %tid.x;", "mov.u32 %r1, %ctaid.x;", "mov.u32 %r2, %ntid.x;",
             "mad.lo.s32 %r3, %r1, %r2, %r0;"]
    for i in range(4, n_regs):
        lines.append(f"mad.lo.s32 %r{i}, %r{i - 1}, {2 * i + 1 + seed}, %r{i - 4};")
    lines += ["ld.param.u64 %rd0, [out];", "cvt.u64.u32 %rd1, %r3;", "shl.b64 %rd1, %rd1, 2;",
              "add.u64 %rd0, %rd0, %rd1;", f"st.global.u32 [%rd0], %r{n_regs - 1};"]
    ptx = (wl.HEADER + f".visible .entry chain(.param .u64 out)\n{{\n    .reg .b32 %r<{n_regs}>;\n"
           "    .reg .b64 %rd<2>;\n" + "\n".join("    " + x for x in lines) + "\n    ret;\n}\n")
    bufs = wl.place([("out", np.zeros(grid * block, dtype=np.uint32), True)])
    return wl.Workload(f"chain{seed}", ptx, "chain", grid, block, wl.pack_params([("u64", bufs[0].sim_base)]), bufs)


def test_persistent_shape_when_one_wave_does_not_fit():
    """20 items of 64 warps with 60 registers each: two 8-warp CTAs of such
    warps do not fit an SM's shared memory, so the grid falls back to
    persistent real warps sharing each item's warps (in the PAIR layout: the
    SPLIT one, which the library would pick for them, halves that state)."""
    ws = [many_registers(i) for i in range(20)]
    assert ks.Module(ws[0].ptx).layout("chain")[0] == "split"
    jobs = [Job(w, layout="pair") for w in ws]
    run_batch(jobs)
    for j in jobs[::4]:
        j.check_oracle()
    for j in jobs:
        g = _parity.gpu_run(j.w)
        assert np.array_equal(ks.stats_array(j.stats).view(np.uint8), g.stats.view(np.uint8))
        assert np.array_equal(j.dev[0][1].cpu().numpy(), g.buffers[0])


def test_headline_pair_batched():
    """The FFMA probe pair at full size (grid 132 x block 128, 4096 x 32 FFMA)
    as one batch: sampled warps against the oracle, every warp's cycles
    against the closed form."""
    jobs = [Job(wl.ffma(acc=1)), Job(wl.ffma(acc=8))]
    assert run_batch(jobs) == 1
    warps = [0, 1, 263, 264, 526, 527]
    for j, (slope, icept) in zip(jobs, [(141, 446), (48, 474)]):
        j.check_oracle(warps=warps, out_words={"out": _parity.thread_ids(j.w, warps)})
        assert set(ks.stats_array(j.stats)["cycles"].tolist()) == {icept + slope * 4096}


def test_refused_item_launches_nothing():
    jobs = [Job(wl.vector_add()), Job(wl.ffma(acc=1, iters=8, grid=2, block=64))]
    items = [j.item() for j in jobs]
    items[1].stats = items[1].stats[:96]  # too small
    with pytest.raises(ks.KsError) as e:
        ks.simulate_batch(items)
    assert "batch item 1" in str(e.value)
    torch.cuda.synchronize()
    assert bool((jobs[0].stats == 0xA5).all())
    assert bool((jobs[1].stats == 0xA5).all())


@pytest.mark.parametrize("block", [512, 1024])
def test_cta_mode_large_blocks(block):
    """CTA-mode items of 16 and 32 warps (the 1024-thread form) in one grid."""
    jobs = [Job(wl.smem_reduce(n=block * 3, block=block)), Job(wl.smem_reduce(n=block * 2, block=block, seed=9))]
    assert run_batch(jobs) == 1
    for j in jobs:
        j.check_oracle()


def test_grids_on_helper_streams_keep_the_callers_order():
    """Items that each take a real grid of their own run side by side on the
    library's helper streams; what the caller enqueues on its own stream after
    the call sees every grid's results: copies made there with no
    synchronisation in between equal single launches."""
    ws = [wl.divergent(k, n=2048 * 32) for k in (2, 4, 32, 2, 4)]  # 2,048 warps each: one grid apiece
    jobs = [Job(w) for w in ws]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        n = ks.simulate_batch([j.item() for j in jobs], stream=s)
        copies = [(j.stats.clone(), j.dev[1][1].clone()) for j in jobs]
    torch.cuda.synchronize()
    assert n == len(ws)
    for k, w in enumerate(ws[:3]):
        g = _parity.gpu_run(w)
        for j in (k, k + 3) if k < 2 else (k,):
            st, out = copies[j]
            assert np.array_equal(ks.stats_array(st).view(np.uint8), g.stats.view(np.uint8)), j
            assert np.array_equal(out.cpu().numpy(), g.buffers[1]), j
    w = ws[0]
    warps = _parity.sample_warps(w, n=24, seed=5)
    jobs[0].check_oracle(warps=warps, out_words={"out": _parity.thread_ids(w, warps)})


def test_two_host_threads_fork_at_once():
    """Two host threads, each with its own stream, issue batches that take
    several real grids at the same time: the helper streams are shared under
    the library's lock, and every item equals its single launch."""
    import threading
    ws = [wl.divergent(k, n=2048 * 32) for k in (2, 4, 32)]
    refs = [_parity.gpu_run(w) for w in ws]
    results = {}

    def worker(t):
        s = torch.cuda.Stream()
        jobs = [Job(w) for w in ws]
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            for _ in range(3):
                ks.simulate_batch([j.item() for j in jobs], stream=s)
        s.synchronize()
        results[t] = jobs

    threads = [threading.Thread(target=worker, args=(t,)) for t in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert sorted(results) == [0, 1]
    for jobs in results.values():
        for j, g in zip(jobs, refs):
            assert np.array_equal(ks.stats_array(j.stats).view(np.uint8), g.stats.view(np.uint8))
            assert np.array_equal(j.dev[1][1].cpu().numpy(), g.buffers[1])

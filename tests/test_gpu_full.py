"""Whole-launch GPU parity at the headline sizes: every configuration of the
benchmark suite runs through the C ABI on the GPU and through the oracle over
every warp of its grid (the oracle spread over all host cores), and the two
must agree byte for byte on

  * every simulated buffer (inputs included, so a stray store shows),
  * every warp's 96-byte statistics record (cycles, instruction counts,
    sectors, lines, status, stack depth),
  * every trace slot (header and records),
  * the launch status.

The sizes are the workloads' own (KernelScope backend doc, simulator/engine.py
PtxSimulator.run(): the result is the whole grid, not a sample):
vector_add n = 4000 on 16 x 256; the FFMA probe pair, grid 132 x block 128,
4096 x 32 FFMA, both as single launches and as the one batched grid that the
benchmark times; the strided gather, 2^24 outputs, s = 1, 2, 4, 8, 16, 32;
the divergent workload, 2^20 threads, k = 2, 4, 32; the 64 fuzz kernels on
1024 x 256 each; the shared-memory reduction, 2^22 elements in 256-thread
CTAs. The sampled headline tests elsewhere stay as fast pre-checks."""
from __future__ import annotations

import gc

import numpy as np
import pytest
import torch

import oracle
import simt_ptx_interpretation_gb300 as ks
from simt_ptx_interpretation_gb300 import workloads as wl
from tests import _parity

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for -m gpu tests")
    from simt_ptx_interpretation_gb300 import _build
    _build.build_native()


class Launch:
    """One workload's device buffers and outputs (stats and trace filled with a
    sentinel, so that a record the GPU never wrote shows)."""

    def __init__(self, w: wl.Workload, layout: str = "auto"):
        self.w = w
        self.mod = ks.Module(w.ptx)
        self.cfg = ks.Config(max_ts=w.max_ts, layout=layout)
        self.dev = [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()]
        self.stats = torch.full((ks.stats_bytes(w.grid, w.block),), 0xA5, dtype=torch.uint8, device="cuda")
        self.trace = (torch.full((ks.trace_bytes(w.grid, w.block, w.max_ts, self.mod.record_bytes(w.kernel)),),
                                 0xA5, dtype=torch.uint8, device="cuda") if w.max_ts else None)

    def simulate(self):
        w = self.w
        ks.simulate(self.mod, w.kernel, w.grid, w.block, w.params, self.dev, self.stats, self.trace, self.cfg)

    def item(self) -> ks.BatchItem:
        w = self.w
        return ks.BatchItem(self.mod, w.kernel, w.grid, w.block, w.params, self.dev, self.stats, self.trace, self.cfg)


def oracle_whole(w: wl.Workload):
    """The oracle over every warp, on all host cores."""
    o, obufs = _parity.oracle_run(w, warps=None, trace=bool(w.max_ts), threads=0)
    return o, obufs


def assert_whole(g: Launch, o, obufs):
    w = g.w
    gs = ks.stats_array(g.stats)
    a = gs.view(np.uint8).reshape(w.warps, 96)
    b = o.stats.view(np.uint8).reshape(w.warps, 96)
    bad = np.nonzero((a != b).any(axis=1))[0]
    assert len(bad) == 0, (f"{w.name}: {len(bad)} of {w.warps} stats records differ, first at warp {bad[0]}: "
                           f"gpu {gs[bad[0]]} oracle {o.stats[bad[0]]}")
    if w.max_ts:
        sb = _parity.slot_bytes(w.max_ts, oracle.record_bytes(w.ptx, w.kernel))
        gt = g.trace.cpu().numpy().reshape(w.warps, sb)
        ot = o.trace.reshape(w.warps, sb)
        badt = np.nonzero((gt != ot).any(axis=1))[0]
        assert len(badt) == 0, f"{w.name}: {len(badt)} trace slots differ, first at warp {badt[0]}"
    for buf, (_, t), ob in zip(w.buffers, g.dev, obufs):
        gb = t.cpu().numpy()
        if not np.array_equal(gb, ob):
            diff = np.nonzero(gb != ob)[0]
            raise AssertionError(f"{w.name}: buffer {buf.name} differs at {len(diff)} bytes, first {diff[:8]}")
    st = int(gs["status"][gs["status"] != 0][0]) if (gs["status"] != 0).any() else 0
    assert st == o.status, f"{w.name}: launch status {st}, oracle {o.status}"
    return gs


def run_single(w: wl.Workload, layout: str = "auto"):
    g = Launch(w, layout)
    g.simulate()
    torch.cuda.synchronize()
    o, obufs = oracle_whole(w)
    gs = assert_whole(g, o, obufs)
    del g
    gc.collect()
    torch.cuda.empty_cache()
    return gs, o


# ------------------------------------------------------------------ 1 ----

def test_vector_add_whole():
    gs, _ = run_single(wl.vector_add())
    assert int(gs["thread_insts"].sum()) == 81056


# ------------------------------------------------------------------ 2 ----

def test_ffma_pair_whole_single_and_batched():
    """Each kernel of the pair alone, and both in the one real grid the
    benchmark times (ks_simulate_batch), against the oracle over all 528
    warps of each; every warp's cycles also equal the closed form."""
    ws = [wl.ffma(acc=1), wl.ffma(acc=8)]
    oracles = [oracle_whole(w) for w in ws]
    for w, (o, obufs) in zip(ws, oracles):
        g = Launch(w)
        g.simulate()
        torch.cuda.synchronize()
        assert_whole(g, o, obufs)
    jobs = [Launch(w) for w in ws]
    assert ks.simulate_batch([j.item() for j in jobs]) == 1
    torch.cuda.synchronize()
    for j, (o, obufs), (slope, icept) in zip(jobs, oracles, [(141, 446), (48, 474)]):
        gs = assert_whole(j, o, obufs)
        assert set(gs["cycles"].tolist()) == {icept + slope * 4096}


# ------------------------------------------------------------------ 3 ----

@pytest.mark.parametrize("s", [1, 2, 4, 8, 16, 32])
def test_gather_whole(s):
    """2^24 outputs, input 2^24 * s floats (2 GiB at s = 32)."""
    w = wl.gather(s)
    gs, _ = run_single(w)
    assert set(gs["ld_sectors"].tolist()) == {min(32, 4 * s)}
    assert set(gs["st_sectors"].tolist()) == {4}
    del w
    gc.collect()


# ------------------------------------------------------------------ 4 ----

@pytest.mark.parametrize("k", [2, 4, 32])
def test_divergent_whole(k):
    run_single(wl.divergent(k))


# ------------------------------------------------------------------ 5 ----

@pytest.mark.parametrize("part", range(4))
def test_fuzz_whole(part):
    """All 64 fuzz kernels at grid 1024 x block 256, 16 per part."""
    for i in range(16 * part, 16 * part + 16):
        run_single(wl.fuzz(i))


# ------------------------------------------------------------ NEXT-1 ----

def test_smem_reduce_whole():
    w = wl.smem_reduce(n=1 << 22, block=256)
    run_single(w)


# ------------------------------------------- the other register layout ----

def test_headline_sizes_in_the_other_layout():
    """The library picks the PAIR layout for the FFMA pair, the gather and the
    divergent workload and SPLIT for the fuzz kernels; each also runs whole in
    the layout it does not pick (the batched FFMA pair as the benchmark times
    it, gather s = 8, divergent k = 4, four fuzz kernels)."""
    ws = [wl.ffma(acc=1), wl.ffma(acc=8)]
    assert all(ks.Module(w.ptx).layout(w.kernel)[0] == "pair" for w in ws)
    oracles = [oracle_whole(w) for w in ws]
    jobs = [Launch(w, "split") for w in ws]
    assert ks.simulate_batch([j.item() for j in jobs]) == 1
    torch.cuda.synchronize()
    for j, (o, obufs) in zip(jobs, oracles):
        assert_whole(j, o, obufs)
    del jobs
    run_single(wl.gather(8), "split")
    run_single(wl.divergent(4), "split")
    for i in (0, 21, 42, 63):
        w = wl.fuzz(i)
        assert ks.Module(w.ptx).layout(w.kernel)[0] == "split"
        run_single(w, "pair")

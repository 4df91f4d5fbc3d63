"""Runs one workload through the GPU path (C ABI) and through the oracle, and
compares memory, per-warp stats, trace slots and statuses byte for byte."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import simt_ptx_interpretation_gb300 as ks
from simt_ptx_interpretation_gb300 import workloads as wl


class GpuResult:
    def __init__(self, stats, trace, buffers, totals):
        self.stats, self.trace, self.buffers, self.totals = stats, trace, buffers, totals


def gpu_run(w: wl.Workload, trace: bool = True, config: ks.Config | None = None, module=None) -> GpuResult:
    cfg = config or ks.Config(max_ts=w.max_ts)
    mod = module or ks.Module(w.ptx)
    dev = [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()]
    r = ks.run(mod, w.kernel, w.grid, w.block, w.params, dev, config=cfg, trace=trace)
    torch.cuda.synchronize()
    stats = ks.stats_array(r.stats)
    tr = r.trace.cpu().numpy() if r.trace is not None else None
    bufs = [t.cpu().numpy() for _, t in dev]
    return GpuResult(stats, tr, bufs, r.totals)


def oracle_run(w: wl.Workload, warps=None, config: ks.Config | None = None, trace: bool = True, threads: int = 0):
    cfg = config or ks.Config(max_ts=w.max_ts)
    bufs = w.fresh_buffers()
    r = oracle.run(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in bufs],
                   lat=cfg.lat, max_ts=cfg.max_ts, trace=trace, stack_depth=cfg.stack_depth,
                   step_limit=cfg.step_limit, inject_warp=cfg.inject_warp, inject_step=cfg.inject_step,
                   warps=warps, threads=threads)
    return r, [b.data.view(np.uint8) for b in bufs]


def slot_bytes(max_ts: int, record_bytes: int = 4) -> int:
    return (16 + record_bytes * max_ts + 7) // 8 * 8


def assert_parity(w: wl.Workload, cfg: ks.Config | None = None, warps=None, out_words=None):
    """Full comparison (warps=None) or on a sample of warps; out_words maps a
    buffer name to the 4-byte word indices the sampled warps own."""
    cfg = cfg or ks.Config(max_ts=w.max_ts)
    g = gpu_run(w, config=cfg)
    o, obufs = oracle_run(w, warps=warps, config=cfg)
    sel = np.arange(w.warps) if warps is None else np.asarray(warps)
    gs = g.stats[sel].view(np.uint8).reshape(len(sel), 96)
    os_ = o.stats[sel].view(np.uint8).reshape(len(sel), 96)
    bad = np.nonzero((gs != os_).any(axis=1))[0]
    assert len(bad) == 0, f"stats differ at warps {sel[bad[:5]]}: gpu {g.stats[sel[bad[0]]]} oracle {o.stats[sel[bad[0]]]}"
    sb = slot_bytes(cfg.max_ts, oracle.record_bytes(w.ptx, w.kernel))
    gt = g.trace.reshape(w.warps, sb)[sel]
    ot = o.trace.reshape(w.warps, sb)[sel]
    badt = np.nonzero((gt != ot).any(axis=1))[0]
    assert len(badt) == 0, f"trace differs at warps {sel[badt[:5]]}"
    for b, gb, ob in zip(w.buffers, g.buffers, obufs):
        if warps is None:
            diff = np.nonzero(gb != ob)[0]
            assert len(diff) == 0, f"buffer {b.name} differs at bytes {diff[:8]}"
        elif out_words is not None and b.name in out_words:
            idx = np.asarray(out_words[b.name], dtype=np.int64)
            gw, ow = gb.view(np.uint32)[idx], ob.view(np.uint32)[idx]
            diff = np.nonzero(gw != ow)[0]
            assert len(diff) == 0, f"buffer {b.name} differs at words {idx[diff[:8]]}"
    if warps is None:
        assert g.totals.status == o.status
    return g, o


def thread_ids(w: wl.Workload, warps) -> np.ndarray:
    """Global thread ids (ctaid * block + tid) of the in-block lanes of `warps`."""
    wpc = (w.block + 31) // 32
    out = []
    for gw in warps:
        cta, wic = divmod(int(gw), wpc)
        for lane in range(32):
            t = wic * 32 + lane
            if t < w.block:
                out.append(cta * w.block + t)
    return np.array(out, dtype=np.int64)


def sample_warps(w: wl.Workload, n: int = 32, seed: int = 0) -> list[int]:
    rng = np.random.default_rng(seed)
    wpc = (w.block + 31) // 32
    fixed = list(range(min(wpc, w.warps))) + list(range(max(0, w.warps - wpc), w.warps))
    extra = rng.choice(w.warps, size=min(n, w.warps), replace=False).tolist()
    return sorted(set(fixed + extra))

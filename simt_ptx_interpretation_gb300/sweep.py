"""The warp-count sweep of the SASS-probe methodology (its step 13: launch the
FFMA probe as <<<1,1>>>, <<<1,32>>>, <<<1,64>>>, <<<1,128>>> and <<<SMs,128>>>
and record blocks, threads, active warps, total instructions, cycles per
instruction and instructions per cycle), run on the SM-level issue model
(ks_simulate_sched) instead of hardware: a lone warp shows the dependent
latency, more warps show how the schedulers hide it."""
from __future__ import annotations

import numpy as np
import torch

from . import api
from . import workloads as wl


def default_configs(n_sm: int) -> list[tuple[int, int]]:
    return [(1, 1), (1, 32), (1, 64), (1, 128), (n_sm, 128)]


def warp_sweep(acc: int = 1, iters: int = 64, n_sm: int = 152, schedulers: int = 4,
               configs: list[tuple[int, int]] | None = None, device: str = "cuda") -> list[dict]:
    """One row per (grid, block): blocks, threads, active_warps,
    total_instructions (warp-level, summed), cycles (the slowest SM's),
    cycles_per_instruction (cycles / instructions of one warp) and
    instructions_per_cycle (total instructions / cycles)."""
    rows = []
    for grid, block in configs or default_configs(n_sm):
        w = wl.ffma(acc=acc, iters=iters, grid=grid, block=block)
        mod = api.Module(w.ptx)
        dev = [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).to(device)) for b in w.fresh_buffers()]
        r = api.run(mod, w.kernel, w.grid, w.block, w.params, dev,
                    sched=api.SchedConfig(n_sm=n_sm, schedulers_per_sm=schedulers))
        if r.totals.status != 0 or int(r.sched_sms["status"].max()) != 0:
            raise api.KsError(int(r.totals.status) or int(r.sched_sms["status"].max()), f"sweep {grid}x{block}")
        issued = r.sched_warps["issued"]
        active = int((issued > 0).sum())
        total = int(issued.sum())
        cycles = int(r.sched_sms["cycles"].max())
        per_warp = total / active
        rows.append(dict(blocks=grid, threads=grid * block, active_warps=active, total_instructions=total,
                         cycles=cycles, cycles_per_instruction=cycles / per_warp,
                         instructions_per_cycle=total / cycles))
    return rows

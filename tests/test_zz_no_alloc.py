"""ks_simulate_static, the entry point for callers that cannot let the
library allocate device memory (for example code that runs while a CUDA graph
is being captured, or a program whose device memory all belongs to its own
pool). It must give exactly what ks_simulate gives — simulated memory,
per-warp statistics and trace slots, byte for byte — including on two calls
in a row with different programs, since every call reuses one static device
array. This file is collected last so that a run stopping at the first
failure has run every other test before it."""
import ctypes

import numpy as np
import pytest
import torch

import simt_ptx_interpretation_gb300 as ks
from simt_ptx_interpretation_gb300 import _native
from simt_ptx_interpretation_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for -m gpu tests")
    from simt_ptx_interpretation_gb300 import _build
    _build.build_native()


def outputs(w, static: bool):
    mod = ks.Module(w.ptx)
    cfg = ks.Config(max_ts=w.max_ts)
    dev = [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()]
    st = torch.empty(ks.stats_bytes(w.grid, w.block), dtype=torch.uint8, device="cuda")
    tr = torch.empty(ks.trace_bytes(w.grid, w.block, w.max_ts), dtype=torch.uint8, device="cuda")
    (ks.simulate_static if static else ks.simulate)(mod, w.kernel, w.grid, w.block, w.params, dev, st, tr, cfg)
    torch.cuda.synchronize()
    return st.cpu().numpy(), tr.cpu().numpy(), [t.cpu().numpy() for _, t in dev]


def test_static_entry_point_matches_ks_simulate_on_two_calls_in_a_row():
    # two different programs back to back through the one shared array
    for w in (wl.vector_add(n=4010), wl.ffma(acc=8, iters=48, grid=4, block=128), wl.fuzz(5, grid=4)):
        ref = outputs(w, static=False)
        got = outputs(w, static=True)
        assert np.array_equal(ref[0], got[0]), f"{w.name}: statistics differ"
        assert np.array_equal(ref[1], got[1]), f"{w.name}: trace slots differ"
        for b, x, y in zip(w.buffers, ref[2], got[2]):
            assert np.array_equal(x, y), f"{w.name}: buffer {b.name} differs"


def test_static_entry_point_rejects_programs_beyond_its_array():
    body = "\n".join("    add.u32 %r1, %r1, 1;" for _ in range(1100))
    ptx = wl.HEADER + ".visible .entry big()\n{\n    .reg .b32 %r<2>;\n" + body + "\n    ret;\n}\n"
    mod = ks.Module(ptx)
    st = torch.empty(96, dtype=torch.uint8, device="cuda")
    with pytest.raises(ks.KsError) as e:
        ks.simulate_static(mod, "big", 1, 32, b"", [], st)
    assert e.value.code == -6
    # ks_simulate itself has no such limit
    ks.simulate(mod, "big", 1, 32, b"", [], st)
    torch.cuda.synchronize()
    assert int(st.cpu().numpy().view(ks.STATS_DTYPE)[0]["warp_insts"]) == 1101

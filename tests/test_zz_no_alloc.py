"""ks_simulate_static, the entry point for callers that cannot let the library
call cudaMalloc: processes whose GPU memory all belongs to their own pool from
start-up, deployments with a device-memory budget fixed at start-up, and
callers that cannot afford the device-wide synchronisation an allocation may
cause. It must give exactly what ks_simulate gives — simulated memory,
per-warp statistics and trace slots, byte for byte — including on calls in a
row with different programs, since every call reuses one static device array.
This file is collected last so that a run stopping at the first failure has
run every other test before it."""
import numpy as np
import pytest
import torch

import simt_ptx_interpretation_gb300 as ks
from simt_ptx_interpretation_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for -m gpu tests")
    from simt_ptx_interpretation_gb300 import _build
    _build.build_native()


def _workloads():
    # three programs of different sizes and kinds, back to back
    return [wl.vector_add(n=4010), wl.ffma(acc=8, iters=48, grid=4, block=128), wl.fuzz(5, grid=4)]


def _prepare(w):
    mod = ks.Module(w.ptx)
    cfg = ks.Config(max_ts=w.max_ts)
    dev = [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()]
    st = torch.empty(ks.stats_bytes(w.grid, w.block), dtype=torch.uint8, device="cuda")
    tr = torch.empty(ks.trace_bytes(w.grid, w.block, w.max_ts), dtype=torch.uint8, device="cuda")
    return mod, cfg, dev, st, tr


def _host(st, tr, dev):
    return st.cpu().numpy(), tr.cpu().numpy(), [t.cpu().numpy() for _, t in dev]


def _assert_same(w, ref, got):
    assert np.array_equal(ref[0], got[0]), f"{w.name}: statistics differ"
    assert np.array_equal(ref[1], got[1]), f"{w.name}: trace slots differ"
    for b, x, y in zip(w.buffers, ref[2], got[2]):
        assert np.array_equal(x, y), f"{w.name}: buffer {b.name} differs"


def _reference(w):
    mod, cfg, dev, st, tr = _prepare(w)
    ks.simulate(mod, w.kernel, w.grid, w.block, w.params, dev, st, tr, cfg)
    torch.cuda.synchronize()
    return _host(st, tr, dev)


def test_static_entry_point_matches_ks_simulate_on_two_calls_in_a_row():
    """Each static call alone (synchronised), against ks_simulate."""
    for w in _workloads():
        ref = _reference(w)
        mod, cfg, dev, st, tr = _prepare(w)
        ks.simulate_static(mod, w.kernel, w.grid, w.block, w.params, dev, st, tr, cfg)
        torch.cuda.synchronize()
        _assert_same(w, ref, _host(st, tr, dev))


def test_static_calls_queued_back_to_back_on_one_stream():
    """Three static calls with different programs queued on one stream with no
    synchronisation between them: stream order alone keeps each kernel's image
    in the shared array until that kernel has finished."""
    ws = _workloads()
    refs = [_reference(w) for w in ws]
    prepared = [_prepare(w) for w in ws]
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for w, (mod, cfg, dev, st, tr) in zip(ws, prepared):
            ks.simulate_static(mod, w.kernel, w.grid, w.block, w.params, dev, st, tr, cfg, stream=stream)
    stream.synchronize()
    for w, ref, (mod, cfg, dev, st, tr) in zip(ws, refs, prepared):
        _assert_same(w, ref, _host(st, tr, dev))


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

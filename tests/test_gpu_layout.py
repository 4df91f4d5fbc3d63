"""Both register-file layouts of the interpreter (PAIR: (value, ready) pairs
per lane in 256-byte rows; SPLIT: 128-byte value rows and a table of ready
times gathered one term per lane) must give the oracle's results byte for
byte. Every case here runs in each layout forced through ks_config.flags:
the workloads at small sizes over every warp, single instructions, access
patterns, statuses, the 32-bit clock's epoch moves, and batches whose items
run in different layouts."""
import numpy as np
import pytest
import torch

import simt_ptx_interpretation_gb300 as ks
from simt_ptx_interpretation_gb300 import workloads as wl
from tests import _parity
from tests import test_gpu_parity as tgp
from tests import test_oracle_control as toc
from tests._kernels import op_workload

pytestmark = pytest.mark.gpu

LAYOUTS = ["pair", "split"]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for -m gpu tests")
    from simt_ptx_interpretation_gb300 import _build
    _build.build_native()


def cfg_for(w, layout, **kw):
    return ks.Config(max_ts=w.max_ts, layout=layout, **kw)


WORKLOADS = {
    "vector_add": lambda: wl.vector_add(),
    "vector_add_b100": lambda: wl.vector_add(n=1000, block=100),
    "ffma1": lambda: wl.ffma(acc=1, iters=40, grid=6, block=128),
    "ffma2": lambda: wl.ffma(acc=2, iters=40, grid=6, block=128),
    "ffma8": lambda: wl.ffma(acc=8, iters=40, grid=6, block=128),
    "gather1": lambda: wl.gather(1, n_out=1 << 14),
    "gather8": lambda: wl.gather(8, n_out=1 << 14),
    "gather32": lambda: wl.gather(32, n_out=1 << 14),
    "divergent2": lambda: wl.divergent(2, n=1 << 14),
    "divergent4": lambda: wl.divergent(4, n=1 << 14),
    "divergent32": lambda: wl.divergent(32, n=1 << 14),
    "many_multipliers": lambda: tgp.many_multipliers(),
}


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workloads_in_both_layouts(name, layout):
    w = WORKLOADS[name]()
    mod = ks.Module(w.ptx)
    assert mod.layout(w.kernel, layout)[0] == layout
    _parity.assert_parity(w, cfg=cfg_for(w, layout))


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("i", range(0, 64, 4))
def test_fuzz_in_both_layouts(i, layout):
    _parity.assert_parity(wl.fuzz(i, grid=8), cfg=cfg_for(wl.fuzz(i, grid=8), layout))


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("op,srcs,dst,kind", tgp.OPS)
def test_single_instructions_in_both_layouts(op, srcs, dst, kind, layout):
    ins = [tgp.operands(k, 50 + j) for j, k in enumerate(srcs)]
    while len(ins) < 3:
        ins.append(None)
    w = op_workload("k_" + op.replace(".", "_"), op, srcs, dst,
                    *[np.array(x, dtype=np.uint64) if x else None for x in ins])
    _parity.assert_parity(w, cfg=cfg_for(w, layout))


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("size", [4, 8])
@pytest.mark.parametrize("pattern", ["seq", "reverse", "mod8", "stride9"])
def test_access_patterns_in_both_layouts(pattern, size, layout):
    for guard in tgp.ACCESS_GUARDS:
        w = tgp.access_workload(pattern, guard, size)
        _parity.assert_parity(w, cfg=cfg_for(w, layout))


@pytest.mark.parametrize("layout", LAYOUTS)
def test_statuses_and_limits_in_both_layouts(layout):
    """Step budgets ending around a fused setp + bra, the stack depth limit,
    injection, and divergence examples with events."""
    w = wl.ffma(acc=1, iters=3, per_iter=2, grid=1, block=64)
    for limit in range(1, 48, 3):
        _parity.assert_parity(w, cfg=cfg_for(w, layout, step_limit=limit))
    d = wl.divergent(4, n=256)
    for limit in (20, 21, 22, 23, 40, 45, 300, 302):
        _parity.assert_parity(d, cfg=cfg_for(d, layout, step_limit=limit))
    ptx = toc.cfg_kernel(toc.HAND_CFGS["endless"][0])
    e = wl.Workload("cfg", ptx, "cfg", 3, 64, b"", [])
    g, _ = _parity.assert_parity(e, cfg=ks.Config(step_limit=777, layout=layout))
    assert g.totals.status == 3
    v = wl.vector_add()
    g, _ = _parity.assert_parity(v, cfg=ks.Config(max_ts=8, inject_warp=5, inject_step=7, layout=layout))
    assert g.totals.status == 6 and g.totals.first_failed_warp == 5
    for name in sorted(toc.HAND_CFGS):
        if name == "endless":
            continue
        body, _ = toc.HAND_CFGS[name]
        c = wl.Workload("cfg", toc.cfg_kernel(body), "cfg", 2, 96, b"", [])
        _parity.assert_parity(c, cfg=ks.Config(max_ts=4, stack_depth=32, layout=layout))


@pytest.mark.parametrize("layout", LAYOUTS)
def test_clock_epoch_moves_in_both_layouts(layout):
    """Latencies of 2^24 cycles push every warp's 32-bit relative clock past
    2^30 within a few dozen instructions, so the scoreboard's epoch moves
    (ready times rebased) many times, in the fast, mid and general paths."""
    big = 1 << 24
    lat = (big, big, big, 20, 8, big, 1, 23, 23, 20, 0, 0)
    for w, moves in ((wl.ffma(acc=1, iters=6, grid=2, block=64), True),
                     (wl.ffma(acc=8, iters=16, grid=2, block=64), True), (wl.divergent(4, n=256), True),
                     (wl.gather(4, n_out=1 << 10), False), (wl.fuzz(3, grid=2), False)):
        g, _ = _parity.assert_parity(w, cfg=ks.Config(max_ts=w.max_ts, lat=lat, layout=layout))
        if moves:
            assert int(g.stats["cycles"].min()) > 1 << 30, w.name


def test_batch_items_in_different_layouts():
    """A batch whose items run in different layouts launches one real grid per
    layout; every item equals the oracle."""
    ws = [wl.ffma(acc=1, iters=16, grid=4), wl.ffma(acc=8, iters=16, grid=4), wl.fuzz(5, grid=4),
          wl.divergent(2, n=1 << 12)]
    layouts = ["split", "pair", "auto", "split"]
    items, outs = [], []
    for w, lay in zip(ws, layouts):
        mod = ks.Module(w.ptx)
        dev = [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()]
        stats = torch.zeros(ks.stats_bytes(w.grid, w.block), dtype=torch.uint8, device="cuda")
        trace = (torch.zeros(ks.trace_bytes(w.grid, w.block, w.max_ts, mod.record_bytes(w.kernel)),
                             dtype=torch.uint8, device="cuda") if w.max_ts else None)
        items.append(ks.BatchItem(mod, w.kernel, w.grid, w.block, w.params, dev, stats, trace,
                                  ks.Config(max_ts=w.max_ts, layout=lay)))
        outs.append((w, dev, stats, trace))
    assert ks.simulate_batch(items) == 2  # the split items, then the pair ones
    torch.cuda.synchronize()
    for w, dev, stats, trace in outs:
        o, obufs = _parity.oracle_run(w)
        assert np.array_equal(ks.stats_array(stats).view(np.uint8), o.stats.view(np.uint8)), w.name
        if trace is not None:
            assert np.array_equal(trace.cpu().numpy(), o.trace), w.name
        for (_, t), ob in zip(dev, obufs):
            assert np.array_equal(t.cpu().numpy(), ob), w.name

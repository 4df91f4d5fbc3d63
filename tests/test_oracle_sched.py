"""Oracle pins for the SM issue model (KernelScope backend doc,
simulator/engine.py and simulator/models.py — WarpStallReason,
_determine_stall_reason, WarpScheduleInfo; the pick order of the page's
step()): issue times, waits and ends derived by hand for independent and
dependent instruction streams, schedulers, barriers and CTA dispatch, and the
reduction to the per-warp model when every warp has an SM of its own. CPU only."""
import numpy as np
import pytest

import oracle
from simt_ptx_interpretation_gb300 import workloads as wl


def kernel(body: str, regs: int = 70) -> str:
    return wl.HEADER + f""".visible .entry k()
{{
    .reg .pred %p<4>;
    .reg .b32 %r<{regs}>;
    .reg .f32 %f<8>;
    .reg .b64 %rd<4>;
{body}
}}
"""


def independent(n: int) -> str:
    """n moves into distinct registers, then ret: nothing waits on anything."""
    return kernel("\n".join(f"    mov.u32 %r{i + 1}, {i};" for i in range(n)) + "\n    ret;")


def chain(n: int) -> str:
    """mov then n dependent fma (latency 4), then ret."""
    body = ["    mov.f32 %f1, 0f3F800000;"] + ["    fma.rn.f32 %f1, %f1, %f1, %f1;"] * n + ["    ret;"]
    return kernel("\n".join(body))


def sched(ptx, grid, block, **kw):
    return oracle.run_sched(ptx, "k", grid, block, b"", [], **kw)


def rows(ws):
    return [tuple(int(x) for x in r) for r in ws]


@pytest.mark.parametrize("k", [1, 2, 3, 4])
def test_independent_streams_share_one_port(k):
    n = 10
    ws, sms = sched(independent(n), 1, 32 * k, n_sm=1, schedulers=1)
    for j in range(k):
        first = j * (n + 1)  # lower warp ids issue first; each warp never stalls
        # (start, end, issued, not_selected, exec, mem, math, barrier); the last
        # mov completes 4 cycles after its issue, after the ret
        assert rows(ws)[j] == (0, first + n + 3, n + 1, first, 0, 0, 0, 0)
    assert int(sms[0]["issued"]) == k * (n + 1)
    assert int(sms[0]["cycles"]) == (k - 1) * (n + 1) + n + 3
    assert int(sms[0]["ctas"]) == 1


def test_schedulers_split_the_warps():
    n = 10
    ws, _ = sched(independent(n), 1, 32 * 8, n_sm=1, schedulers=4)
    for j in range(8):  # warp j on scheduler j % 4, behind warp j - 4
        first = (j // 4) * (n + 1)
        assert rows(ws)[j][:4] == (0, first + n + 3, n + 1, first)


def test_dependent_chain_alone():
    n = 6
    ws, _ = sched(chain(n), 1, 32, n_sm=1, schedulers=1)
    # mov 0; fma i at 4i (each waits 3 cycles on the one before); ret at 4n+1;
    # the last result at 4n+4
    assert rows(ws)[0] == (0, 4 * n + 4, n + 2, 0, 3 * n, 0, 0, 0)


def test_two_chains_interleave():
    n = 6
    ws, sms = sched(chain(n), 1, 64, n_sm=1, schedulers=1)
    # warp 0 as alone; warp 1 one cycle behind, and its last fma meets warp 0's
    # ret at 4n+1 (warp 0 goes first): fma at 4n+2, ret at 4n+3, result 4n+6
    assert rows(ws)[0] == (0, 4 * n + 4, n + 2, 0, 3 * n, 0, 0, 0)
    assert rows(ws)[1] == (0, 4 * n + 6, n + 2, 2, 3 * n, 0, 0, 0)
    assert int(sms[0]["cycles"]) == 4 * n + 6


LOAD_USE = wl.HEADER + """.visible .entry k(.param .u64 p_in)
{
    .reg .f32 %f<4>;
    .reg .b64 %rd<3>;
    ld.param.u64    %rd1, [p_in];
    ld.global.f32   %f1, [%rd1];
    add.f32         %f2, %f1, %f1;
    div.rn.f32      %f3, %f2, %f1;
    add.f32         %f2, %f3, %f3;
    ret;
}
"""


def test_wait_kinds():
    src = np.ones(64, dtype=np.float32)
    ws, _ = oracle.run_sched(LOAD_USE, "k", 1, 32, (0x1000_0000).to_bytes(8, "little"), [(0x1000_0000, src)],
                             n_sm=1, schedulers=1)
    # ld.param 0 (ready 4); ld 4 (waits 3 on the param: exec; ready 404); add
    # 404 (waits 399: mem; ready 408); div 408 (waits 3: exec; ready 444);
    # add 444 (waits 35: math; ready 448); ret 445 -> end 448
    assert rows(ws)[0] == (0, 448, 6, 0, 6, 399, 35, 0)


BARRIER = wl.HEADER + """.visible .entry k()
{
    .reg .pred %p<2>;
    .reg .b32 %r<6>;
    mov.u32         %r1, %tid.x;
    setp.lt.u32     %p1, %r1, 32;
    @!%p1 bra       BAR;
    add.u32         %r2, %r1, 1;
    add.u32         %r2, %r2, 1;
    add.u32         %r2, %r2, 1;
BAR:
    bar.sync        0;
    mov.u32         %r3, 7;
    ret;
}
"""


def test_barrier_release():
    ws, _ = sched(BARRIER, 1, 64, n_sm=1, schedulers=4)
    # warp 0: mov 0, setp 4, bra 8 (next at 16: the branch latency), adds 16,
    # 20, 24, bar 25; warp 1 (its own scheduler): the same until bra 8, then
    # bar at 16. Release at 25 + 20 = 45: warp 0 waited 45 - 26 = 19, warp 1
    # 45 - 17 = 28; then mov 45 (ready 49), ret 46 -> end 49
    w0, w1 = rows(ws)
    assert w0 == (0, 49, 9, 0, 3 + 3 + 7 + 3 + 3, 0, 0, 19)
    assert w1 == (0, 49, 6, 0, 3 + 3 + 7, 0, 0, 28)


def test_cta_dispatch():
    n = 10
    end = n + 3
    ws, sms = sched(independent(n), 3, 32, n_sm=1, ctas_per_sm=1, schedulers=1)
    assert [(int(r["start"]), int(r["end"])) for r in ws] == [(0, end), (end, 2 * end), (2 * end, 3 * end)]
    assert int(sms[0]["ctas"]) == 3 and int(sms[0]["cycles"]) == 3 * end
    ws, sms = sched(independent(n), 3, 32, n_sm=2, ctas_per_sm=1, schedulers=1)
    assert [(int(r["start"]), int(r["end"])) for r in ws] == [(0, end), (0, end), (end, 2 * end)]
    assert list(sms["ctas"]) == [2, 1]


@pytest.mark.parametrize("name", ["vector_add", "divergent", "fuzz", "smem_reduce"])
def test_alone_equals_the_per_warp_model(name):
    """One warp per SM and per scheduler: nothing is ever not selected and
    every warp ends at its per-warp cycle count."""
    w = {"vector_add": lambda: wl.vector_add(n=1000, block=32), "divergent": lambda: wl.divergent(4, n=256, block=32),
         "fuzz": lambda: wl.fuzz(2, grid=4, block=32), "smem_reduce": lambda: wl.smem_reduce(n=32 * 4, block=32)}[name]()
    bufs = [(b.sim_base, b.data) for b in w.fresh_buffers()]
    ws, sms = oracle.run_sched(w.ptx, w.kernel, w.grid, w.block, w.params, bufs, n_sm=w.grid, ctas_per_sm=1)
    p = oracle.run(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in w.fresh_buffers()])
    assert (ws["not_selected"] == 0).all()
    assert np.array_equal(ws["end"] - ws["start"], p.stats["cycles"])
    assert np.array_equal(ws["issued"], p.stats["warp_insts"])


@pytest.mark.parametrize("name", ["divergent", "fuzz", "smem_reduce", "fuzz_shared"])
def test_waits_add_up(name):
    w = {"divergent": lambda: wl.divergent(2, n=1024, block=128), "fuzz": lambda: wl.fuzz(3, grid=8, block=64),
         "smem_reduce": lambda: wl.smem_reduce(n=128 * 8, block=128),
         "fuzz_shared": lambda: wl.fuzz_shared(2, grid=4, block=128)}[name]()
    ws, sms = oracle.run_sched(w.ptx, w.kernel, w.grid, w.block, w.params,
                               [(b.sim_base, b.data) for b in w.fresh_buffers()], n_sm=3, schedulers=2)
    p = oracle.run(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in w.fresh_buffers()])
    assert np.array_equal(ws["issued"], p.stats["warp_insts"])
    used = (ws["issued"] + ws["not_selected"] + ws["stall_exec"] + ws["stall_mem"] + ws["stall_math"]
            + ws["stall_barrier"])
    tail = (ws["end"] - ws["start"]).astype(np.int64) - used.astype(np.int64)
    # what is left is the drain after the last issue: at most the longest latency
    assert (tail >= 0).all() and (tail <= 400).all()
    # contention only delays: never earlier than alone
    assert ((ws["end"] - ws["start"]) >= p.stats["cycles"]).all()
    assert int(sms["issued"].sum()) == int(p.stats["warp_insts"].sum())
    assert int(sms["ctas"].sum()) == w.grid


def _sweep_row(grid, block, n_sm, schedulers, acc=1, iters=4):
    w = wl.ffma(acc=acc, iters=iters, grid=grid, block=block)
    ws, sms = oracle.run_sched(w.ptx, w.kernel, w.grid, w.block, w.params,
                               [(b.sim_base, b.data) for b in w.fresh_buffers()], n_sm=n_sm, schedulers=schedulers)
    return int(ws["issued"].sum()), int(sms["cycles"].max())


def test_warp_sweep_shape():
    """The probe methodology's warp sweep on the model: lanes do not change
    a warp's timing; with 4 schedulers up to 4 warps of a CTA each run alone;
    more SMs run more CTAs in the same time; with one scheduler, 4 dependent
    chains share the port and hide part of the latency."""
    i1, c1 = _sweep_row(1, 1, 4, 4)
    i32, c32 = _sweep_row(1, 32, 4, 4)
    i128, c128 = _sweep_row(1, 128, 4, 4)
    isms, csms = _sweep_row(4, 128, 4, 4)
    assert (i1, c1) == (i32, c32)
    assert c128 == c32 and i128 == 4 * i32
    assert csms == c128 and isms == 4 * i128
    i1s, c1s = _sweep_row(1, 128, 1, 1)
    assert i1s == i128
    ipc_one, ipc_four = i32 / c32, i1s / c1s
    assert ipc_one < ipc_four <= 1.0

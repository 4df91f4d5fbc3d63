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
    """(start, end, issued, not_selected, exec, mem, math, barrier) per warp."""
    return [tuple(int(r[k]) for k in ("start", "end", "issued", "not_selected", "stall_exec", "stall_mem",
                                       "stall_math", "stall_barrier")) for r in ws]


def labels(ws):
    """(throttled, diverged) per warp: the two label counts."""
    return [(int(r["throttled"]), int(r["diverged"])) for r in ws]


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


# ---------------------------------------------------------------- labels ----
# The page's _determine_stall_reason labels an instruction as it executes:
# MEMORY_THROTTLE for an instruction of its memory class (MEMORY_OPS: ld, st,
# mov) while 4 or more memory operations are pending; DIVERGENCE is declared
# and returned nowhere. Readings: pending per SM, other warps' latest global
# or shared access issued at an earlier cycle and not yet complete; diverged
# while live lanes wait on the reconvergence stack. Labels change no timing.

THROTTLE = wl.HEADER + """.visible .entry k(.param .u64 p_in)
{
    .reg .b32 %r<3>;
    .reg .b64 %rd<3>;
    ld.param.u64    %rd1, [p_in];
    ld.global.u32   %r1, [%rd1];
    ret;
}
"""


@pytest.mark.parametrize("warps", [4, 5, 6])
def test_memory_throttle_label(warps):
    """One SM, one scheduler, warps 0..n-1 from cycle 0, lowest id first.
    ld.param of w0..w3 at 0..3 (each load waits 4 on its ld.param); then
    w0 ld.global 4, ret 5; w1 ld.global 6, ret 7; w2 8, 9; w3 10, 11 (a load
    sees 0, 1, 2, 3 other pending loads: none throttled); w4 ld.param 12 and
    w5 ld.param 13 see w0..w3 pending (4): throttled; w4 ld.global 16 sees 4
    (w5 has no access yet): throttled, ret 17; w5 ld.global 18 sees 5:
    throttled. ret (not memory class) is never labelled. A load's warp ends
    when its result is ready, 400 cycles after it issued."""
    src = np.arange(32 * warps, dtype=np.uint32)
    ws, _ = oracle.run_sched(THROTTLE, "k", 1, 32 * warps, (0x1000_0000).to_bytes(8, "little"),
                             [(0x1000_0000, src)], n_sm=1, schedulers=1)
    ldg = [4, 6, 8, 10, 16, 18][:warps]
    assert [r[1] for r in rows(ws)] == [t + 400 for t in ldg]
    expect = [0, 0, 0, 0, 2, 2][:warps]
    assert [t for t, _ in labels(ws)] == expect
    assert all(d == 0 for _, d in labels(ws))


IF_ELSE = wl.HEADER + """.visible .entry k()
{
    .reg .pred %p<2>;
    .reg .b32 %r<4>;
    mov.u32         %r1, %tid.x;
    setp.lt.u32     %p1, %r1, 16;
    @%p1 bra        THEN;
    add.u32         %r2, %r1, 1;
    add.u32         %r2, %r2, 1;
    bra             JOIN;
THEN:
    add.u32         %r2, %r1, 2;
JOIN:
    add.u32         %r3, %r2, 1;
    ret;
}
"""


def test_divergence_label_if_else():
    """Warp 0 splits at the branch: the fall-through path (lanes 16..31: two
    adds and the bra to JOIN) and the taken path (lanes 0..15: one add) issue
    while the other half waits at JOIN: 4 diverged instructions of 9. Warp 1
    (tid 32..63) goes one way: none. mov and the adds are not memory class
    except mov, which issues with nothing pending."""
    ws, _ = sched(IF_ELSE, 1, 64, n_sm=1, schedulers=4)
    assert [int(r["issued"]) for r in ws] == [9, 8]
    assert labels(ws) == [(0, 4), (0, 0)]


RET_IN_PATH = wl.HEADER + """.visible .entry k()
{
    .reg .pred %p<2>;
    .reg .b32 %r<4>;
    mov.u32         %r1, %tid.x;
    setp.lt.u32     %p1, %r1, 8;
    @%p1 bra        OUT;
    add.u32         %r2, %r1, 1;
    ret;
OUT:
    add.u32         %r3, %r1, 2;
    ret;
}
"""


def test_divergence_label_ends_when_the_other_path_exits():
    """The paths end in different rets (reconvergence at the virtual exit).
    Lanes 8..31 run first: add and ret issue while lanes 0..7 wait (2
    diverged); after that ret those lanes have left, so lanes 0..7 are all the
    live lanes and their add and ret are not diverged."""
    ws, _ = sched(RET_IN_PATH, 1, 32, n_sm=1, schedulers=1)
    assert int(ws[0]["issued"]) == 7
    assert labels(ws) == [(0, 2)]


THROTTLE2 = wl.HEADER + """.visible .entry k(.param .u64 p_in)
{
    .reg .b32 %r<3>;
    .reg .b64 %rd<3>;
    ld.param.u64    %rd1, [p_in];
    ld.global.u32   %r1, [%rd1];
    ld.global.u32   %r2, [%rd1+4];
    ret;
}
"""


def test_memory_throttle_counts_other_warps_only():
    """Two loads per warp, four warps: ld.param 0..3; w0 loads at 4 and 5, ret
    6; w1 at 7 and 8, ret 9; w2 at 10 and 11, ret 12; w3 at 13 and 14, ret 15.
    w3's second load finds three other warps pending and its own first load:
    the warp's own access does not count, so nothing is throttled."""
    src = np.arange(256, dtype=np.uint32)
    ws, _ = oracle.run_sched(THROTTLE2, "k", 1, 128, (0x1000_0000).to_bytes(8, "little"),
                             [(0x1000_0000, src)], n_sm=1, schedulers=1)
    assert [r[1] for r in rows(ws)] == [405, 408, 411, 414]
    assert labels(ws) == [(0, 0)] * 4


def test_divergence_label_on_the_divergent_workload():
    """The divergent workload splits at its lane % k test on every iteration:
    labels appear and never exceed the issued instructions."""
    w = wl.divergent(4, n=1024)
    bufs = w.fresh_buffers()
    ws, _ = oracle.run_sched(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in bufs],
                             n_sm=2, schedulers=4)
    assert int(ws["diverged"].sum()) > 0
    for r in ws:
        assert int(r["diverged"]) <= int(r["issued"])
        assert int(r["throttled"]) <= int(r["issued"])

"""GPU parity: the sm_103a interpreter (called through the C ABI) against the
oracle, byte for byte — simulated memory, per-warp statistics records, trace
slots and statuses — on the seeded workloads, at small sizes over every warp
and at the headline sizes over sampled warps. Plus single-instruction
semantics, error statuses, launch totals, and a cross-check of the simulated
memory against the same PTX run natively by the driver JIT."""
import numpy as np
import pytest
import torch

import oracle
import simt_ptx_interpretation_gb300 as ks
from simt_ptx_interpretation_gb300 import workloads as wl
from tests import _jit, _parity
from tests import test_oracle_control as toc
from tests import test_oracle_semantics as tos
from tests._kernels import op_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for -m gpu tests")
    from simt_ptx_interpretation_gb300 import _build
    _build.build_native()


# ---------------------------------------------------------- vector_add ----

@pytest.mark.parametrize("n", [4000, 4010, 1, 31, 33, 8192])
def test_vector_add_parity(n):
    w = wl.vector_add(n=n)
    g, o = _parity.assert_parity(w)
    a, b, c = (x.view(np.float32) for x in g.buffers)
    assert np.array_equal(c, (a + b).astype(np.float32))


def test_vector_add_headline_values():
    w = wl.vector_add()
    g = _parity.gpu_run(w)
    assert tuple(int(g.stats[0][k]) for k in ("cycles", "warp_insts", "thread_insts")) == (463, 20, 640)
    assert tuple(int(g.stats[127][k]) for k in ("cycles", "warp_insts", "thread_insts")) == (27, 11, 352)


def test_vector_add_odd_block_and_no_trace():
    w = wl.vector_add(n=1000, block=100)
    _parity.assert_parity(w)
    g = _parity.gpu_run(w, trace=False)
    o, _ = _parity.oracle_run(w, trace=False)
    assert np.array_equal(g.stats.view(np.uint8), o.stats.view(np.uint8))


# ---------------------------------------------------------------- ffma ----

@pytest.mark.parametrize("acc", [1, 2, 4, 8, 16])
def test_ffma_parity_small(acc):
    _parity.assert_parity(wl.ffma(acc=acc, iters=40, grid=6, block=128))


@pytest.mark.parametrize("acc", [1, 8])
def test_ffma_parity_headline_sampled(acc):
    """Grid 132 x block 128, 4096 x 32 FFMA per thread: sampled warps."""
    w = wl.ffma(acc=acc)
    warps = [0, 1, 2, 3, 130, 263, 264, 400, 524, 525, 526, 527]
    tids = _parity.thread_ids(w, warps)
    g, o = _parity.assert_parity(w, warps=warps, out_words={"out": tids})
    slope = 141 if acc == 1 else 48
    icept = 446 if acc == 1 else 474
    assert set(g.stats["cycles"].tolist()) == {icept + slope * 4096}


# -------------------------------------------------------------- gather ----

@pytest.mark.parametrize("s", [1, 2, 4, 8, 16, 32])
def test_gather_parity_small(s):
    w = wl.gather(s, n_out=1 << 14)
    g, _ = _parity.assert_parity(w)
    assert set(g.stats["ld_sectors"].tolist()) == {min(32, 4 * s)}


@pytest.mark.parametrize("s", [1, 32])
def test_gather_parity_headline_sampled(s):
    w = wl.gather(s)
    warps = _parity.sample_warps(w, n=48, seed=s)
    g, _ = _parity.assert_parity(w, warps=warps, out_words={"out": _parity.thread_ids(w, warps)})
    assert set(g.stats["ld_sectors"].tolist()) == {min(32, 4 * s)}
    out, src = g.buffers[1].view(np.float32), g.buffers[0].view(np.float32)
    assert np.array_equal(out, src[::s])


# ----------------------------------------------------------- divergent ----

@pytest.mark.parametrize("k", [2, 4, 32])
def test_divergent_parity_small(k):
    _parity.assert_parity(wl.divergent(k, n=1 << 14))


@pytest.mark.parametrize("k", [2, 4, 32])
def test_divergent_parity_headline(k):
    w = wl.divergent(k)
    warps = _parity.sample_warps(w, n=256, seed=k)
    g, _ = _parity.assert_parity(w, warps=warps, out_words={"out": _parity.thread_ids(w, warps)})
    trips = w.buffer("in").data
    assert np.array_equal(g.buffers[1].view(np.uint32), toc.numpy_divergent(trips, k))


# ---------------------------------------------------------------- fuzz ----

@pytest.mark.parametrize("i", range(64))
def test_fuzz_parity_small(i):
    _parity.assert_parity(wl.fuzz(i, grid=8))


@pytest.mark.parametrize("i", range(0, 64, 8))
def test_fuzz_parity_headline_sampled(i):
    w = wl.fuzz(i)
    warps = _parity.sample_warps(w, n=24, seed=i)
    words = wl.fuzz_store_words(_parity.thread_ids(w, warps), w.meta["s_perm"])
    _parity.assert_parity(w, warps=warps, out_words={"out": words})


# --------------------------------------------------- single instructions ----

OPS = [
    ("add.rn.f32", "ff", "f", "f"), ("sub.rn.f32", "ff", "f", "f"), ("mul.rn.f32", "ff", "f", "f"),
    ("div.rn.f32", "ff", "f", "f"), ("fma.rn.f32", "fff", "f", "f"), ("sqrt.rn.f32", "f", "f", "f"),
    ("add.u32", "uu", "u", "u"), ("sub.s64", "ww", "w", "w"), ("mul.lo.s32", "uu", "u", "u"),
    ("mul.lo.u64", "ww", "w", "w"), ("mad.lo.s32", "uuu", "u", "u"), ("mad.lo.u64", "www", "w", "w"),
    ("and.b32", "uu", "u", "u"), ("xor.b64", "ww", "w", "w"), ("shl.b32", "uu", "u", "u"),
    ("shr.s32", "uu", "u", "u"), ("shr.u64", "wu", "w", "w"), ("shr.s64", "wu", "w", "w"),
    ("setp.lt.f32", "ff", "p", "f"), ("setp.ne.f32", "ff", "p", "f"), ("setp.ge.s32", "uu", "p", "u"),
    ("setp.hi.u64", "ww", "p", "w"), ("selp.b64", "wwp", "w", "w"), ("selp.f32", "ffp", "f", "f"),
    ("cvt.rn.f32.u32", "u", "f", "u"), ("cvt.rn.f32.s64", "w", "f", "w"), ("cvt.rni.s32.f32", "f", "u", "f"),
    ("cvt.rzi.u64.f32", "f", "w", "f"), ("cvt.rmi.s64.f32", "f", "w", "f"), ("cvt.rpi.u32.f32", "f", "u", "f"),
    ("cvt.s64.s32", "u", "w", "u"), ("cvt.u32.u64", "w", "u", "w"), ("and.pred", "pp", "p", "p"),
    ("xor.pred", "pp", "p", "p"),
]


def operands(kind, seed):
    if kind == "f":
        return tos.f32_operands(seed)
    if kind == "u":
        return tos.int_operands(seed, 32)
    if kind == "w":
        return tos.int_operands(seed, 64)
    return [x & 1 for x in tos.int_operands(seed, 32)]


@pytest.mark.parametrize("op,srcs,dst,kind", OPS)
def test_single_instruction_parity(op, srcs, dst, kind):
    ins = [operands(k if k != "p" else "p", 50 + j) for j, k in enumerate(srcs)]
    while len(ins) < 3:
        ins.append(None)
    w = op_workload("k_" + op.replace(".", "_"), op, srcs, dst, *[np.array(x, dtype=np.uint64) if x else None for x in ins])
    _parity.assert_parity(w)


# -------------------------------------------------------- access patterns ----

ACCESS_PATTERNS = {  # element index of each lane (%r7 = lane) into this warp's 4 KiB
    "seq": "mov.u32 %r2, %r7;",
    "groups4": "shr.u32 %r2, %r7, 2;",          # sorted, runs of 4 equal addresses
    "reverse": "mov.u32 %r5, 31;\n    sub.u32 %r2, %r5, %r7;",
    "same": "mov.u32 %r2, 16;",                 # one address for the whole warp
    "stride9": "mul.lo.u32 %r2, %r7, 9;",        # sorted, crossing sectors and lines
    "mod8": "and.b32 %r2, %r7, 7;",             # unsorted, interleaved duplicates
    "swap": "xor.b32 %r2, %r7, 1;",             # unsorted, distinct
}
ACCESS_GUARDS = {"all": ("", ""), "lt20": ("setp.lt.u32 %p1, %r7, 20;", "@%p1 "),
                 "odd": ("and.b32 %r5, %r7, 1;\n    setp.ne.u32 %p1, %r5, 0;", "@%p1 ")}


def access_workload(pattern: str, guard: str, size: int) -> wl.Workload:
    """Per-warp load, add, store through one lane-to-address pattern; every warp
    works in its own 4 KiB, so only lanes of one warp ever share an address."""
    gset, g = ACCESS_GUARDS[guard]
    if size == 4:
        body = (f"{g}ld.global.u32 %r3, [%rd3];\n    add.u32 %r4, %r3, %r1;\n"
                f"    {g}st.global.u32 [%rd3], %r4;")
    else:
        body = (f"{g}ld.global.u64 %rd4, [%rd3];\n    cvt.u64.u32 %rd5, %r1;\n    add.s64 %rd5, %rd4, %rd5;\n"
                f"    {g}st.global.u64 [%rd3], %rd5;")
    ptx = wl.HEADER + f""".visible .entry acc(.param .u64 base)
{{
    .reg .pred %p<2>;
    .reg .b32 %r<10>;
    .reg .b64 %rd<6>;
    ld.param.u64 %rd1, [base];
    mov.u32 %r1, %tid.x;
    mov.u32 %r8, %ctaid.x;
    mov.u32 %r9, %ntid.x;
    mad.lo.s32 %r6, %r8, %r9, %r1;
    and.b32 %r7, %r1, 31;
    {ACCESS_PATTERNS[pattern]}
    shl.b32 %r2, %r2, {2 if size == 4 else 3};
    shr.u32 %r6, %r6, 5;
    shl.b32 %r6, %r6, 12;
    add.u32 %r2, %r2, %r6;
    cvt.u64.u32 %rd2, %r2;
    add.s64 %rd3, %rd1, %rd2;
    {gset}
    {body}
    ret;
}}
"""
    grid, block = 2, 128
    mem = wl.randint_u32(grid * block // 32 * 1024, 0, 1 << 31, seed=7)
    bufs = wl.place([("mem", mem, True)])
    return wl.Workload(f"acc_{pattern}_{guard}_{size}", ptx, "acc", grid, block,
                       wl.pack_params([("u64", bufs[0].sim_base)]), bufs)


@pytest.mark.parametrize("size", [4, 8])
@pytest.mark.parametrize("guard", list(ACCESS_GUARDS))
@pytest.mark.parametrize("pattern", list(ACCESS_PATTERNS))
def test_access_patterns_match_the_oracle(pattern, guard, size):
    """Sector and line counts and the highest-lane-wins store rule on coalesced,
    duplicated, reversed, interleaved and partially masked accesses."""
    _parity.assert_parity(access_workload(pattern, guard, size))


# --------------------------------------------------------- payload events ----

def test_payload_events_match_the_oracle():
    from tests import test_oracle_events as tev
    cases = [(tev.PAYLOADS, 64, 4), (tev.PAYLOADS, 40, 1), (tev.PAYLOADS, 96, 0),
             ("    mov.u32 %r1, %tid.x;\n    setp.lt.u32 %p1, %r1, 8;\n    @%p1 ret;\n    //@iket mark m %r1\n    ret;", 64, 2),
             ("    mov.u32 %r1, 7;\n    mov.f32 %f1, 0f3FC00000;\n    //@iket mark a\n    //@iket mark b %r1\n"
              "    //@iket range_end c %f1\n    ret;", 96, 3)]
    for body, block, max_ts in cases:
        w = wl.Workload("ev", tev.kernel(body), "ev", 3, block, b"", [], max_ts=max_ts)
        _parity.assert_parity(w)


@pytest.mark.parametrize("k", [2, 32])
def test_payload_marks_in_a_divergent_loop(k):
    """A payload mark on the loop counter inside the divergent workload's loop
    body: records of changing masks and values, over every warp."""
    w = wl.divergent(k, n=1 << 12, max_ts=16)
    ptx = w.ptx.replace("DV_HEAD:\n", "DV_HEAD:\n    //@iket mark it %r10\n", 1)
    assert ptx != w.ptx
    w2 = wl.Workload(w.name + "_payload", ptx, w.kernel, w.grid, w.block, w.params, w.buffers, max_ts=16)
    assert ks.Module(ptx).record_bytes(w.kernel) == 8
    _parity.assert_parity(w2)


# ------------------------------------------------------------- statuses ----

def test_step_limits_around_compare_and_branch_pairs():
    """A step budget that ends on, between or after a setp and the bra it
    guards (issued together when every lane agrees) stops the warp where the
    oracle stops it: uniform loop back-edges (FFMA probe) and divergent loop
    exits (divergent workload)."""
    w = wl.ffma(acc=1, iters=3, per_iter=2, grid=1, block=64)
    for limit in range(1, 48):
        _parity.assert_parity(w, cfg=ks.Config(max_ts=w.max_ts, step_limit=limit))
    d = wl.divergent(4, n=256)
    for limit in (20, 21, 22, 23, 40, 41, 42, 43, 44, 45, 46, 300, 301, 302):
        _parity.assert_parity(d, cfg=ks.Config(max_ts=d.max_ts, step_limit=limit))


def test_error_statuses_match_the_oracle():
    base = 0x60000000
    buf = np.zeros(1024, dtype=np.uint8)
    cases = [
        (toc.access_kernel("mul.lo.u32 %r2, %r1, 64;\n    cvt.u64.u32 %rd2, %r2;\n    add.s64 %rd3, %rd1, %rd2;\n"
                           "    ld.global.u32 %r3, [%rd3];"), 1),
        (toc.access_kernel("ld.global.u32 %r3, [%rd1+2];"), 2),
        (toc.access_kernel("ld.global.u64 %rd2, [%rd1+2044];"), 2),
        (toc.access_kernel("mul.lo.u32 %r2, %r1, 2048;\n    add.u32 %r2, %r2, 2;\n    cvt.u64.u32 %rd2, %r2;\n"
                           "    add.s64 %rd3, %rd1, %rd2;\n    st.global.u32 [%rd3], %r1;"), 2),
    ]
    import struct
    for ptx, want in cases:
        w = wl.Workload("bad", ptx, "bad", 2, 64, struct.pack("<Q", base), wl.place([("buf", buf.copy(), True)]))
        w.buffers[0].sim_base = base
        g, o = _parity.assert_parity(w, cfg=ks.Config())
        assert g.totals.status == want and g.totals.first_failed_warp == 0 and g.totals.n_failed == 4


def test_step_limit_stack_and_injection_match_the_oracle():
    ptx = toc.cfg_kernel(toc.HAND_CFGS["endless"][0])
    w = wl.Workload("cfg", ptx, "cfg", 3, 64, b"", [])
    g, _ = _parity.assert_parity(w, cfg=ks.Config(step_limit=777))
    assert g.totals.status == 3 and set(g.stats["warp_insts"].tolist()) == {777}
    body = """
    mov.u32 %r1, %tid.x;
    and.b32 %r2, %r1, 1;
    setp.eq.u32 %p1, %r2, 0;
    @%p1 bra ELSE;
    add.u32 %r3, %r3, 1;
    bra.uni JOIN;
ELSE:
    add.u32 %r3, %r3, 2;
JOIN:
    ret;"""
    w = wl.Workload("cfg", toc.cfg_kernel(body), "cfg", 2, 64, b"", [])
    g, _ = _parity.assert_parity(w, cfg=ks.Config(stack_depth=2))
    assert g.totals.status == 4
    g, _ = _parity.assert_parity(w, cfg=ks.Config(stack_depth=3))
    assert g.totals.status == 0 and g.totals.max_stack_depth == 3
    v = wl.vector_add()
    g, _ = _parity.assert_parity(v, cfg=ks.Config(max_ts=8, inject_warp=5, inject_step=7))
    assert g.totals.status == 6 and g.totals.first_failed_warp == 5 and g.totals.n_failed == 1


def test_divergence_examples_match_the_oracle():
    for name in sorted(toc.HAND_CFGS):
        if name == "endless":
            continue
        body, _ = toc.HAND_CFGS[name]
        w = wl.Workload("cfg", toc.cfg_kernel(body), "cfg", 2, 96, b"", [])
        _parity.assert_parity(w, cfg=ks.Config(max_ts=4))


# --------------------------------------------------------------- totals ----

def test_read_stats_totals_reduce_every_record():
    w = wl.divergent(4, n=1 << 14)
    g = _parity.gpu_run(w)
    s = g.stats
    t = g.totals
    assert t.cycles_max == int(s["cycles"].max()) and t.cycles_sum == int(s["cycles"].sum())
    for f in ("warp_insts", "thread_insts", "ld_req", "ld_sectors", "st_req", "st_sectors", "ld_lines", "st_lines"):
        assert getattr(t, f) == int(s[f].sum()), f
    assert t.n_warps == w.warps and t.n_failed == 0 and t.first_failed_warp == -1 and t.status == 0
    assert t.max_stack_depth == int(s["max_stack_depth"].max())


def test_concurrent_launches_on_streams():
    """Independent simulations enqueued on four streams at once (two of them
    through one module, one with shared memory and bar.sync) overlap on the
    GPU and still equal the oracle byte for byte."""
    ws = [wl.ffma(acc=1, iters=40, grid=6, block=128), wl.ffma(acc=1, iters=40, grid=6, block=128),
          wl.ffma(acc=8, iters=40, grid=6, block=128), wl.divergent(2, n=2048),
          wl.smem_reduce(n=1024, block=256)] + [wl.fuzz(i, grid=4, block=64) for i in range(3)]
    mods = [ks.Module(w.ptx) for w in ws]
    mods[1] = mods[0]
    main = torch.cuda.current_stream()
    streams = [main] + [torch.cuda.Stream() for _ in range(3)]
    runs = []
    fork = torch.cuda.Event()
    fork.record(main)
    for s in streams[1:]:
        s.wait_event(fork)
    for i, (w, mod) in enumerate(zip(ws, mods)):
        s = streams[i % 4]
        with torch.cuda.stream(s):
            dev = [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()]
            st = torch.empty(ks.stats_bytes(w.grid, w.block), dtype=torch.uint8, device="cuda")
            tr = torch.empty(ks.trace_bytes(w.grid, w.block, w.max_ts, mod.record_bytes(w.kernel)),
                             dtype=torch.uint8, device="cuda")
            ks.simulate(mod, w.kernel, w.grid, w.block, w.params, dev, st, tr, ks.Config(max_ts=w.max_ts), s)
        runs.append((dev, st, tr))
    torch.cuda.synchronize()
    for w, (dev, st, tr) in zip(ws, runs):
        o, obufs = _parity.oracle_run(w)
        assert np.array_equal(ks.stats_array(st).view(np.uint8), o.stats.view(np.uint8)), w.name
        assert np.array_equal(tr.cpu().numpy(), o.trace), w.name
        for (_, t), ob in zip(dev, obufs):
            assert np.array_equal(t.cpu().numpy(), ob), w.name


# -------------------------------------------------- driver-JIT cross-check ----

def jit_memory(w: wl.Workload):
    layout, _ = oracle.params_layout(w.ptx, w.kernel)
    vals = _jit.unpack_params(w.params, layout)
    bufs = w.fresh_buffers()
    dev = [torch.from_numpy(b.data.view(np.uint8)).cuda() for b in bufs]
    real = {b.sim_base: t.data_ptr() for b, t in zip(bufs, dev)}
    vals = [real.get(v, v) if size == 8 else v for v, (off, size) in zip(vals, layout)]
    _jit.run_native(w.ptx, w.kernel, w.grid, w.block, layout, vals)
    return [t.cpu().numpy() for t in dev]


def nan_equivalent(a: np.ndarray, b: np.ndarray) -> bool:
    a32, b32 = a.view(np.uint32), b.view(np.uint32)
    same = a32 == b32
    fa, fb = a.view(np.float32), b.view(np.float32)
    return bool(np.all(same | (np.isnan(fa) & np.isnan(fb))))


@pytest.mark.parametrize("make", [lambda: wl.vector_add(n=4010), lambda: wl.ffma(acc=8, iters=64, grid=4),
                                  lambda: wl.gather(8, n_out=1 << 14), lambda: wl.divergent(4, n=1 << 14)])
def test_jit_crosscheck_workloads(make):
    w = make()
    sim = _parity.gpu_run(w).buffers
    nat = jit_memory(w)
    for b, x, y in zip(w.buffers, sim, nat):
        assert np.array_equal(x, y), b.name


@pytest.mark.parametrize("i", range(0, 64, 4))
def test_jit_crosscheck_fuzz(i):
    w = wl.fuzz(i, grid=8)
    sim = _parity.gpu_run(w).buffers
    nat = jit_memory(w)
    assert nan_equivalent(sim[2], nat[2])


@pytest.mark.parametrize("op,srcs,dst,kind", OPS[:18] + OPS[24:32])
def test_jit_crosscheck_single_instructions(op, srcs, dst, kind):
    ins = [operands(k, 50 + j) for j, k in enumerate(srcs)]
    while len(ins) < 3:
        ins.append(None)
    w = op_workload("k_" + op.replace(".", "_"), op, srcs, dst, *[np.array(x, dtype=np.uint64) if x else None for x in ins])
    sim = _parity.gpu_run(w).buffers[0]
    nat = jit_memory(w)[0]
    if dst == "f":
        assert nan_equivalent(sim, nat)
        return
    if op.startswith("cvt.r") and op.endswith(("s64.f32", "u64.f32")):
        # PTX ISA: float-to-integer conversion of NaN gives 0, which the
        # simulator implements; the GB300 returns 0x8000000000000000 for NaN
        # converted to a 64-bit integer (32-bit destinations give 0). Every
        # other input must agree with the hardware.
        isnan = np.isnan(np.array(ins[0], dtype=np.uint64).astype(np.uint32).view(np.float32))
        s64, n64 = sim.view(np.uint64), nat.view(np.uint64)
        assert np.all(s64[isnan] == 0)
        assert np.array_equal(s64[~isnan], n64[~isnan])
        return
    assert np.array_equal(sim, nat)


def many_multipliers(grid: int = 4, block: int = 96) -> wl.Workload:
    """A kernel with more than 16 distinct immediates, most of them
    multipliers (so the decoder keeps them out of the constant rows): mul.lo
    and mad.lo by an immediate in either operand position, immediate and
    register addends, signed and unsigned, one guarded (its immediate stays a
    row), each result folded into the value stored at out[gtid]."""
    lines = ["mov.u32 %r0, %tid.x;", "mov.u32 %r1, %ctaid.x;", "mov.u32 %r2, %ntid.x;",
             "mad.lo.s32 %r3, %r1, %r2, %r0;", "mov.u32 %r4, %r3;"]
    rng = np.random.default_rng(11)
    for k in range(24):
        m, c = int(rng.integers(1, 1 << 31)), int(rng.integers(0, 1 << 32))
        form = k % 4
        if form == 0:
            lines.append(f"mul.lo.u32 %r5, %r4, {m};")
        elif form == 1:
            lines.append(f"mad.lo.u32 %r5, {m}, %r4, {c};")
        elif form == 2:
            lines.append(f"mad.lo.s32 %r5, %r4, {m - (1 << 30)}, %r3;")
        else:
            lines.append(f"mul.lo.s32 %r5, {m}, %r4;")
        lines.append("xor.b32 %r4, %r4, %r5;")
    lines += ["and.b32 %r6, %r0, 1;", "setp.eq.u32 %p1, %r6, 0;", "@%p1 mad.lo.u32 %r4, %r4, 77777, 5;",
              "ld.param.u64 %rd0, [out];", "cvt.u64.u32 %rd1, %r3;", "shl.b64 %rd1, %rd1, 2;",
              "add.u64 %rd0, %rd0, %rd1;", "st.global.u32 [%rd0], %r4;"]
    ptx = (wl.HEADER + ".visible .entry mm(.param .u64 out)\n{\n    .reg .pred %p<2>;\n    .reg .b32 %r<7>;\n"
           "    .reg .b64 %rd<2>;\n" + "\n".join("    " + x for x in lines) + "\n    ret;\n}\n")
    bufs = wl.place([("out", np.zeros(grid * block, dtype=np.uint32), True)])
    return wl.Workload("many_multipliers", ptx, "mm", grid, block, wl.pack_params([("u64", bufs[0].sim_base)]), bufs)


def test_immediate_multipliers_out_of_rows():
    _parity.assert_parity(many_multipliers())

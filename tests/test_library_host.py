"""Host-side checks of libks that need no GPU: the shared library loads and
exports every function include/ks.h declares; the decoder accepts exactly the
programs the oracle accepts and agrees on parameter layout, event tables and
reconvergence points; output sizes follow the IKET slot rule."""
import ctypes
import os
import random
import re

import pytest

import oracle
from simt_ptx_interpretation_gb300 import _build, _native
from simt_ptx_interpretation_gb300 import api as ks
from simt_ptx_interpretation_gb300 import workloads as wl
from tests import test_oracle_control as toc
from tests import test_oracle_events as tev
from tests import test_oracle_shared as tsh
from tests._kernels import op_kernel

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build_native()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ks.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(ks_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_function_is_exported():
    names = declared_functions()
    assert len(names) >= 11
    lib = ctypes.CDLL(_native.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(_native.EXPORTS)


def test_output_sizes_follow_the_slot_rule():
    for grid, block, ts in [(16, 256, 8), (1024, 256, 64), (3, 33, 0), (1, 1, 1), (7, 100, 3)]:
        W = grid * ((block + 31) // 32)
        assert ks.stats_bytes(grid, block) == W * 96
        assert ks.trace_bytes(grid, block, ts) == W * ((16 + 4 * ts + 7) // 8 * 8)


def corpus():
    progs = [("vector_add", wl.vector_add_ptx()), ("gather", wl.gather_ptx()), ("divergent", wl.divergent_ptx())]
    for acc in (1, 8):
        progs.append((f"ffma_acc{acc}", wl.ffma_ptx(acc)))
    for i in range(0, 64, 3):
        progs.append((f"fuzz_{1000 + i}", wl.fuzz_ptx(1000 + i)))
    for name, (body, _) in toc.HAND_CFGS.items():
        progs.append(("cfg", toc.cfg_kernel(body)))
    for name, body in toc.BAD_PROGRAMS:
        progs.append(("k", wl.HEADER + (".visible .entry k()\n{\n    .reg .pred %p<2>;\n    .reg .b32 %r<4>;\n"
                                        "    .reg .f32 %f<4>;\n    .reg .b64 %rd<4>;\n    " + body + "\n}\n")))
    for block in (32, 64, 256):
        progs.append(("smem_reduce", wl.smem_reduce_ptx(block)))
    progs += [("probe", tsh.bank_probe_ptx(4)), ("probe", tsh.bank_probe_ptx(8)), ("bar2", tsh.barrier_ptx(3))]
    for body, _ in tsh.SHARED_BAD:
        progs.append(("bad", tsh.bad_shared_kernel(body)))
    for i in range(0, 24, 5):
        progs.append(("fuzz_sh", wl.fuzz_shared_ptx(2000 + i, 128)))
    progs.append(("ev", tev.kernel(tev.PAYLOADS)))
    for body in ("    //@iket mark a %r1\n    ret;", "    //@iket mark a %rd1\n    ret;", "    //@iket mark a %f1\n    ret;",
                 "    //@iket mark a\n    //@iket mark b %r1\n    ret;", "    //@iket mark a %r1\n    //@iket mark a %rd1\n    ret;",
                 "    //@iket mark a %p1\n    ret;", "    //@iket mark a 5\n    ret;", "    //@iket mark a %r1 %r2\n    ret;"):
        progs.append(("ev", tev.kernel(body)))
    for op, srcs, dst in [("add.u32", "uu", "u"), ("fma.rn.f32", "fff", "f"), ("setp.lt.f32", "ff", "p"),
                          ("selp.b64", "wwp", "w"), ("cvt.rzi.s64.f32", "f", "w"), ("shr.s64", "wu", "w")]:
        progs.append(("k_op", op_kernel("k_op", op, srcs, dst)))
    return progs


@pytest.mark.parametrize("idx", range(len(corpus())))
def test_decoder_accepts_what_the_oracle_accepts(idx):
    kernel, ptx = corpus()[idx]
    ocode, _ = oracle.parse_check(ptx, kernel)
    try:
        m = ks.Module(ptx)
        dcode = 0
    except ks.KsError as e:
        dcode = e.code
    assert (ocode == 0) == (dcode == 0), (ocode, dcode)
    if dcode:
        return
    layout, total = oracle.params_layout(ptx, kernel)
    assert [(o, s) for _, o, s in m.params(kernel)] == layout
    assert m.info(kernel)["param_bytes"] == total
    assert [k for k, _ in m.events(kernel)] == oracle.events(ptx, kernel)
    assert m.record_bytes(kernel) == oracle.record_bytes(ptx, kernel)
    assert m.ipdom(kernel) == oracle.ipdom(ptx, kernel)


@pytest.mark.parametrize("name", sorted(toc.HAND_CFGS))
def test_decoder_ipdom_hand_drawn(name):
    body, want = toc.HAND_CFGS[name]
    assert ks.Module(toc.cfg_kernel(body)).ipdom("cfg") == want


def test_decoder_ipdom_random_cfgs_against_brute_force():
    rng = random.Random(78)
    for _ in range(200):
        m = rng.randrange(2, 30)
        body, succ = toc.random_cfg(rng, m)
        assert ks.Module(toc.cfg_kernel(body)).ipdom("cfg") == toc.brute_ipdom(succ), body


def test_resource_limits_are_reported():
    regs = "\n".join(f"    add.u32 %r{i}, %r{i}, 1;" for i in range(100))
    ptx = wl.HEADER + ".visible .entry big()\n{\n    .reg .b32 %r<100>;\n" + regs + "\n    ret;\n}\n"
    with pytest.raises(ks.KsError) as e:
        ks.Module(ptx)
    assert e.value.code == -6
    consts = "\n".join(f"    add.u32 %r1, %r1, {i + 1000};" for i in range(130))
    ptx = wl.HEADER + ".visible .entry big()\n{\n    .reg .b32 %r<2>;\n" + consts + "\n    ret;\n}\n"
    with pytest.raises(ks.KsError) as e:
        ks.Module(ptx)
    assert e.value.code == -6


def test_unknown_kernel_and_bad_arguments():
    m = ks.Module(wl.vector_add_ptx())
    with pytest.raises(ks.KsError) as e:
        m.info("nope")
    assert e.value.code == -5
    L = _native.lib()
    assert L.ks_load_module(None, 0, None, None, 0) == -3
    assert L.ks_simulate(None, b"x", 1, 32, None, 0, None, 0, None, 0, None, 0, None, None) == -3
    # shape and size checks happen before any GPU work
    stats = ctypes.create_string_buffer(96 * 8)
    args = dict(grid=0, block=32)
    assert L.ks_simulate(m.handle, b"vector_add", 0, 32, None, 0, None, 0, None, 0, stats, 96 * 8, None, None) == -3
    assert L.ks_simulate(m.handle, b"vector_add", 1, 2000, None, 0, None, 0, None, 0, stats, 96 * 8, None, None) == -3
    p = ctypes.create_string_buffer(28)
    # too small a stats buffer
    assert L.ks_simulate(m.handle, b"vector_add", 16, 256, p, 28, None, 0, None, 0, stats, 96, None, None) == -3
    # parameter block smaller than the kernel's
    assert L.ks_simulate(m.handle, b"vector_add", 1, 32, p, 8, None, 0, None, 0, stats, 96, None, None) == -3
    # overlapping buffers
    bufs = (_native.KsBuffer * 2)()
    bufs[0].sim_base, bufs[0].dev_ptr, bufs[0].bytes = 0x10000000, 1, 8192
    bufs[1].sim_base, bufs[1].dev_ptr, bufs[1].bytes = 0x10001000, 1, 8192
    assert L.ks_simulate(m.handle, b"vector_add", 1, 32, p, 28, bufs, 2, None, 0, stats, 96, None, None) == -3
    # unaligned simulated base
    bufs[1].sim_base = 0x20000010
    assert L.ks_simulate(m.handle, b"vector_add", 1, 32, p, 28, bufs, 2, None, 0, stats, 96, None, None) == -3
    for code in (0, -1, -2, -3, -4, -5, -6, 1, 2, 3, 4, 5, 6):
        assert L.ks_status_string(code)


def test_batch_arguments_are_checked_before_any_gpu_work():
    """ks_simulate_batch refuses an empty or NULL list, and names the first
    item that ks_simulate would refuse (launching nothing)."""
    m = ks.Module(wl.vector_add_ptx())
    L = _native.lib()
    failed = ctypes.c_uint32(7)
    assert L.ks_simulate_batch(None, 3, None, ctypes.byref(failed), None) == -3
    items = (_native.KsBatchItem * 3)()
    assert L.ks_simulate_batch(items, 0, None, ctypes.byref(failed), None) == -3 and failed.value == 0
    stats = ctypes.create_string_buffer(96 * 16 * 8)
    p = ctypes.create_string_buffer(28)
    for it in items:
        it.mod, it.kernel, it.grid, it.block = m.handle, b"vector_add", 16, 256
        it.params, it.param_bytes = ctypes.cast(p, ctypes.c_void_p), 28
        it.stats_buf, it.stats_bytes = ctypes.cast(stats, ctypes.c_void_p), 96 * 16 * 8
    items[1].stats_bytes = 96  # too small
    assert L.ks_simulate_batch(items, 3, None, ctypes.byref(failed), None) == -3 and failed.value == 1
    items[1].stats_bytes = 96 * 16 * 8
    items[2].kernel = b"nope"
    assert L.ks_simulate_batch(items, 3, None, ctypes.byref(failed), None) == -5 and failed.value == 2
    items[2].kernel = b"vector_add"
    items[0].reserved = 1
    assert L.ks_simulate_batch(items, 3, None, ctypes.byref(failed), None) == -3 and failed.value == 0
    assert ctypes.sizeof(_native.KsBatchItem) == 96


def test_cached_batch_arguments_are_checked_before_any_gpu_work():
    """ks_simulate_cached_batch checks every item (its simulation and its
    cache arguments) before any GPU work and names the first refused one."""
    m = ks.Module(wl.vector_add_ptx())
    L = _native.lib()
    failed = ctypes.c_uint32(7)
    assert L.ks_simulate_cached_batch(None, 2, None, ctypes.byref(failed), None) == -3
    items = (_native.KsCachedItem * 2)()
    stats = ctypes.create_string_buffer(96 * 16 * 8)
    p = ctypes.create_string_buffer(28)
    need = 1 << 20
    ws = ctypes.create_string_buffer(need)
    for it in items:
        s = it.sim
        s.mod, s.kernel, s.grid, s.block = m.handle, b"vector_add", 16, 256
        s.params, s.param_bytes = ctypes.cast(p, ctypes.c_void_p), 28
        s.stats_buf, s.stats_bytes = ctypes.cast(stats, ctypes.c_void_p), 96 * 16 * 8
        it.workspace, it.workspace_bytes = ctypes.cast(ws, ctypes.c_void_p), need
    items[1].workspace = None  # (a workspace's size is checked against a layout that needs the GPU)
    assert L.ks_simulate_cached_batch(items, 2, None, ctypes.byref(failed), None) == -3 and failed.value == 1
    bad = _native.KsCacheConfig()
    L.ks_cache_config_default(ctypes.byref(bad))
    bad.l2_lines = bad.l1_lines + 1  # not a multiple of the L1
    items[0].cache = ctypes.pointer(bad)
    assert L.ks_simulate_cached_batch(items, 2, None, ctypes.byref(failed), None) == -3 and failed.value == 0
    assert ctypes.sizeof(_native.KsCachedItem) == 120


def test_static_entry_point_rejects_what_ks_simulate_rejects():
    """ks_simulate_static repeats ks_simulate's argument checks; both must
    return the same code for every invalid call. Each case fails on the host
    before any CUDA call (device pointers here are never dereferenced)."""
    L = _native.lib()
    w = wl.vector_add(n=4000)
    mod = ks.Module(w.ptx)
    FAKE = 0x10000  # a non-null device pointer that no case reaches
    W = w.grid * ((w.block + 31) // 32)

    def base():
        bufs = (_native.KsBuffer * 8)()
        for i, b in enumerate(w.buffers):
            bufs[i].sim_base, bufs[i].dev_ptr, bufs[i].bytes = b.sim_base, FAKE, b.data.nbytes
        cfg = _native.KsConfig()
        L.ks_config_default(ctypes.byref(cfg))
        cfg.max_ts_per_warp = 8
        return dict(mod=mod.handle, kernel=w.kernel.encode(), grid=w.grid, block=w.block, params=bytes(w.params),
                    param_bytes=len(w.params), bufs=bufs, n_bufs=len(w.buffers), trace=FAKE,
                    trace_bytes=W * 48, stats=FAKE, stats_bytes=W * 96, cfg=cfg)

    def overlap(a):
        a["bufs"][1].sim_base = a["bufs"][0].sim_base

    def cfgset(field, value):
        return lambda a: setattr(a["cfg"], field, value)

    def lat(a):
        a["cfg"].lat[3] = (1 << 24) + 1

    def profile(a):
        a["cfg"].profile_buf, a["cfg"].profile_bytes = FAKE, 72

    cases = {
        "null module": lambda a: a.update(mod=None),
        "unknown kernel": lambda a: a.update(kernel=b"nope"),
        "grid 0": lambda a: a.update(grid=0),
        "block 0": lambda a: a.update(block=0),
        "block 1025": lambda a: a.update(block=1025),
        "2^31 warps": lambda a: a.update(grid=1 << 28, block=256),
        "short params": lambda a: a.update(param_bytes=len(w.params) - 4),
        "params over 256 B": lambda a: a.update(params=bytes(260), param_bytes=260),
        "null params": lambda a: a.update(params=None),
        "9 buffers": lambda a: a.update(n_bufs=9),
        "null buffer table": lambda a: a.update(bufs=None),
        "unaligned sim_base": lambda a: setattr(a["bufs"][0], "sim_base", a["bufs"][0].sim_base + 16),
        "empty buffer": lambda a: setattr(a["bufs"][1], "bytes", 0),
        "null buffer pointer": lambda a: setattr(a["bufs"][2], "dev_ptr", None),
        "overlapping buffers": overlap,
        "null stats": lambda a: a.update(stats=None),
        "short stats": lambda a: a.update(stats_bytes=W * 96 - 1),
        "stack depth 0": cfgset("simt_stack_depth", 0),
        "stack depth 33": cfgset("simt_stack_depth", 33),
        "max_ts over 2^24": cfgset("max_ts_per_warp", (1 << 24) + 1),
        "latency over 2^24": lat,
        "short trace": lambda a: a.update(trace_bytes=W * 48 - 8),
        "short profile": profile,
    }
    for name, mutate in cases.items():
        a = base()
        mutate(a)
        codes = []
        for fn in (L.ks_simulate, L.ks_simulate_static):
            pb = ctypes.create_string_buffer(a["params"], max(1, len(a["params"]))) if a["params"] is not None else None
            codes.append(fn(a["mod"], a["kernel"], a["grid"], a["block"],
                            ctypes.cast(pb, ctypes.c_void_p) if pb is not None else None, a["param_bytes"], a["bufs"],
                            a["n_bufs"], a["trace"], a["trace_bytes"], a["stats"], a["stats_bytes"],
                            ctypes.byref(a["cfg"]), None))
        assert codes[0] == codes[1], f"{name}: ks_simulate {codes[0]}, ks_simulate_static {codes[1]}"
        assert codes[0] < 0, f"{name}: accepted ({codes[0]})"


def test_register_layout_choice():
    """ks_kernel_layout: the library picks PAIR for kernels whose warp state is
    small or that run in CTA mode, SPLIT for plain kernels whose PAIR warp
    state exceeds 12 KiB (the fuzz kernels); a forced layout is honoured, and
    SPLIT warp state is about half the PAIR one (128-byte value rows and a
    ready table instead of 256-byte (value, ready) rows)."""
    for w in (wl.vector_add(), wl.ffma(acc=8, iters=8, grid=2), wl.gather(8, n_out=1 << 10),
              wl.divergent(4, n=1 << 10)):
        m = ks.Module(w.ptx)
        lay, pair_bytes = m.layout(w.kernel)
        assert lay == "pair" and pair_bytes <= 12 * 1024, w.name
        assert m.layout(w.kernel, "pair") == ("pair", pair_bytes)
        s_lay, split_bytes = m.layout(w.kernel, "split")
        assert s_lay == "split" and split_bytes < 0.6 * pair_bytes, w.name
    for i in range(0, 64, 7):
        w = wl.fuzz(i)
        m = ks.Module(w.ptx)
        _, pair_bytes = m.layout(w.kernel, "pair")
        lay, split_bytes = m.layout(w.kernel)
        assert lay == "split" and pair_bytes > 12 * 1024 and split_bytes < 0.6 * pair_bytes, w.name
    r = wl.smem_reduce(n=1 << 12, block=256)
    m = ks.Module(r.ptx)
    assert m.layout(r.kernel)[0] == "pair"
    with pytest.raises(ks.KsError) as e:
        m.layout(r.kernel, "split")  # CTA mode runs in PAIR only
    assert e.value.code == -2
    lib = _native.lib()
    sp, rb = ctypes.c_uint32(), ctypes.c_uint32()
    v = ks.Module(wl.vector_add().ptx)
    assert lib.ks_kernel_layout(v._h, b"vector_add", 3, ctypes.byref(sp), ctypes.byref(rb)) == -3  # both flags
    assert lib.ks_kernel_layout(v._h, b"vector_add", 4, ctypes.byref(sp), ctypes.byref(rb)) == -3  # unknown bit
    assert lib.ks_kernel_layout(v._h, b"nope", 0, ctypes.byref(sp), ctypes.byref(rb)) == -5


def test_fast_runs_follow_the_programs_shape():
    """ks_kernel_fast_runs reports the decoder's fast-loop runs (PAIR layout):
    their lengths, whether every op of a run's rest writes a row it reads,
    and how far each op's b and c rows keep being read unwritten. Pinned on
    the FFMA probe (32 `fma acc, acc, m, add` and the counter's add in one
    run) and on hand-made runs where a row stops being kept."""
    for acc in (1, 8):
        w = wl.ffma(acc=acc, iters=16, per_iter=32)
        runs = ks.Module(w.ptx).fast_runs(w.kernel)
        starts = [i for i, (n, _, _) in enumerate(runs) if n == 33]
        assert len(starts) == 1, runs
        s = starts[0]
        for j in range(33):
            n, own, keep = runs[s + j]
            assert n == 33 - j and own
            # the 32 FMAs keep m and add; the counter's add reads other rows
            assert keep == (32 - j if j < 32 else 1)
    body = "\n".join([
        "    fma.rn.f32 %f1, %f1, %f2, %f3;",   # keeps f2, f3 into the next op
        "    fma.rn.f32 %f2, %f1, %f2, %f3;",   # writes its own b: the next op reloads
        "    fma.rn.f32 %f3, %f1, %f2, %f3;",
        "    fma.rn.f32 %f5, %f1, %f2, %f4;",   # writes a row it does not read
        "    fma.rn.f32 %f1, %f1, %f2, %f4;",
        "    fma.rn.f32 %f1, %f1, %f2, %f4;",
    ])
    ptx = (wl.HEADER + ".visible .entry fr(.param .u64 fr_out)\n{\n    .reg .f32 %f<6>;\n    .reg .b64 %rd<2>;\n"
           "    ld.param.u64 %rd1, [fr_out];\n    ld.global.f32 %f1, [%rd1];\n    ld.global.f32 %f2, [%rd1+4];\n"
           "    ld.global.f32 %f3, [%rd1+8];\n    ld.global.f32 %f4, [%rd1+12];\n" + body + "\n"
           "    st.global.f32 [%rd1], %f1;\n    st.global.f32 [%rd1+4], %f5;\n    ret;\n}\n")
    runs = ks.Module(ptx).fast_runs("fr")
    first = next(i for i, (n, _, _) in enumerate(runs) if n)
    got = runs[first:first + 6]
    assert [n for n, _, _ in got] == [6, 5, 4, 3, 2, 1]
    # the op writing %f5 (not among its sources) clears the flag for it and
    # every op before it in the run
    assert [own for _, own, _ in got] == [False, False, False, False, True, True]
    # f2, f3 kept into the op that writes f2; f2, f4 kept from the %f5 op on
    assert [keep for _, _, keep in got] == [2, 1, 1, 3, 2, 1]
    assert all(r == (0, False, 0) for i, r in enumerate(runs) if not first <= i < first + 6)
    # argument errors; a short buffer receives what fits, n_out the whole count
    lib = _native.lib()
    m = ks.Module(ptx)
    cnt = ctypes.c_uint32()
    assert lib.ks_kernel_fast_runs(None, b"fr", None, 0, ctypes.byref(cnt)) == -3
    assert lib.ks_kernel_fast_runs(m._h, b"nope", None, 0, ctypes.byref(cnt)) == -5
    short = (ctypes.c_uint32 * 6)(*([0xDEADBEEF] * 6))
    assert lib.ks_kernel_fast_runs(m._h, b"fr", short, 1, ctypes.byref(cnt)) == 0
    assert cnt.value == len(runs)
    assert tuple(short[:3]) == (runs[0][0], int(runs[0][1]), runs[0][2]) and short[3] == 0xDEADBEEF


def test_fast_runs_are_consistent_on_every_workload():
    """Over every benchmark kernel (and the fuzz corpus): a run's length
    drops by one per entry; the own-destination flag, once set, holds to the
    run's end; a kept-rows count never exceeds the run and counts down along
    its prefix."""
    ws = [wl.vector_add(), wl.ffma(acc=1), wl.ffma(acc=8), wl.gather(8), wl.divergent(4), wl.smem_reduce()]
    ws += [wl.fuzz(i) for i in range(0, 64, 4)]
    for w in ws:
        runs = ks.Module(w.ptx).fast_runs(w.kernel)
        for i, (n, own, keep) in enumerate(runs):
            if n == 0:
                assert (own, keep) == (False, 0), (w.name, i)
                continue
            assert 1 <= keep <= n, (w.name, i)
            if n > 1:
                n1, own1, keep1 = runs[i + 1]
                assert n1 == n - 1, (w.name, i)
                assert own1 or not own, (w.name, i)
                if keep > 1:
                    assert keep1 == keep - 1, (w.name, i)

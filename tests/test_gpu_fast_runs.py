"""Long fast runs (straight-line runs of f32 add/sub/mul/fma and 32-bit
integer add/sub/mul/mad, which the interpreter's pipelined fast loop runs
with forwarding between neighbours) against the oracle's instruction-by-
instruction scoreboard, byte for byte, in both register layouts: runs over
few and over many rows, chains and independent streams, immediates
(constant rows), partial warps and divergent masks, loops, a branch into the
middle of a run, other latency tables, clocks that move the epoch, and a
step limit that ends a warp inside a run."""
import numpy as np
import pytest
import torch

import simt_ptx_interpretation_gb300 as ks
from simt_ptx_interpretation_gb300 import workloads as wl
from tests import _parity

pytestmark = pytest.mark.gpu

LAYOUTS = ["pair", "split"]


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for -m gpu tests")
    from simt_ptx_interpretation_gb300 import _build
    _build.build_native()


F_ONE, F_HALF, F_NEG = "0f3F800000", "0f3F000000", "0fBF400000"


def _op(rng, nf, nr):
    """One random fast op over %f1..%f{nf} and %r1..%r{nr}."""
    f = lambda: f"%f{rng.integers(1, nf + 1)}"
    r = lambda: f"%r{rng.integers(1, nr + 1)}"
    k = rng.integers(0, 9)
    if k == 0:
        return f"fma.rn.f32 {f()}, {f()}, {f()}, {f()};"
    if k == 1:
        return f"fma.rn.f32 {f()}, {f()}, {rng.choice([F_HALF, F_NEG])}, {f()};"
    if k == 2:
        return f"add.rn.f32 {f()}, {f()}, {f()};"
    if k == 3:
        return f"sub.rn.f32 {f()}, {f()}, {f()};"
    if k == 4:
        return f"mul.rn.f32 {f()}, {f()}, {rng.choice([f(), F_ONE, F_HALF])};"
    if k == 5:
        return f"mad.lo.u32 {r()}, {r()}, {r()}, {r()};"
    if k == 6:
        return f"add.u32 {r()}, {r()}, {rng.choice([r(), str(int(rng.integers(1, 1000)))])};"
    if k == 7:
        return f"mul.lo.u32 {r()}, {r()}, {r()};"
    return f"sub.u32 {r()}, {r()}, {r()};"


def runs_kernel(name, seed, nf, nr, run_len, iters, diverge=0, mid_entry=False):
    """Loads %f1..%f{nf} and %r1..%r{nr} from `inp` (per thread), runs `iters`
    times a straight-line run of `run_len` random fast ops (with the loop
    counter's add it is one fast run), optionally only in the threads with
    tid.x < diverge, optionally entered once in its middle by a branch, and
    stores every register to `out`."""
    rng = np.random.default_rng(seed)
    n = nf + nr
    L = [f".visible .entry {name}(.param .u64 rs_out, .param .u64 rs_inp)", "{",
         "    .reg .pred %p<4>;", f"    .reg .f32 %f<{nf + 1}>;", f"    .reg .b32 %r<{nr + 1}>;",
         "    .reg .b32 %q<8>;", "    .reg .b64 %rd<8>;",
         "    ld.param.u64 %rd1, [rs_out];", "    ld.param.u64 %rd2, [rs_inp];",
         "    mov.u32 %q1, %ctaid.x;", "    mov.u32 %q2, %ntid.x;", "    mov.u32 %q3, %tid.x;",
         "    mad.lo.s32 %q4, %q1, %q2, %q3;", f"    mul.lo.u32 %q5, %q4, {4 * n};",
         "    cvt.u64.u32 %rd3, %q5;", "    add.s64 %rd4, %rd2, %rd3;", "    add.s64 %rd5, %rd1, %rd3;"]
    for i in range(nf):
        L.append(f"    ld.global.f32 %f{i + 1}, [%rd4+{4 * i}];")
    for i in range(nr):
        L.append(f"    ld.global.u32 %r{i + 1}, [%rd4+{4 * (nf + i)}];")
    if diverge:
        L += [f"    setp.ge.u32 %p3, %q3, {diverge};", "    @%p3 bra RS_DONE;"]
    L.append("    mov.u32 %q6, 0;")
    body = [_op(rng, nf, nr) for _ in range(run_len)]
    if mid_entry:  # the first pass enters the run in its middle
        L += ["    setp.eq.u32 %p2, %q6, 0;", "    @%p2 bra RS_MID;"]
    L.append("RS_LOOP:")
    for i, x in enumerate(body):
        if mid_entry and i == run_len // 2:
            L.append("RS_MID:")
        L.append("    " + x)
    L += ["    add.u32 %q6, %q6, 1;", f"    setp.lt.u32 %p1, %q6, {iters};", "    @%p1 bra RS_LOOP;"]
    if diverge:
        L.append("RS_DONE:")
    for i in range(nf):
        L.append(f"    st.global.f32 [%rd5+{4 * i}], %f{i + 1};")
    for i in range(nr):
        L.append(f"    st.global.u32 [%rd5+{4 * (nf + i)}], %r{i + 1};")
    L += ["    ret;", "}", ""]
    return wl.HEADER + "\n".join(L)


def runs_workload(seed, nf, nr, run_len, iters, grid=3, block=96, fbits=None, **kw):
    """fbits: bit patterns the f32 inputs are drawn from (default: values in
    [0.25, 1.5))."""
    name = f"rs{seed}"
    n = nf + nr
    rng = np.random.default_rng(1000 + seed)
    threads = grid * block
    inp = np.empty((threads, n), dtype=np.uint32)
    if fbits is None:
        inp[:, :nf] = rng.uniform(0.25, 1.5, size=(threads, nf)).astype(np.float32).view(np.uint32)
    else:
        inp[:, :nf] = rng.choice(np.asarray(fbits, dtype=np.uint32), size=(threads, nf))
    inp[:, nf:] = rng.integers(0, 1 << 32, size=(threads, nr), dtype=np.uint64).astype(np.uint32)
    out = np.zeros((threads, n), dtype=np.uint32)
    bufs = wl.place([("out", out, True), ("inp", inp, False)])
    params = wl.pack_params([("u64", bufs[0].sim_base), ("u64", bufs[1].sim_base)])
    return wl.Workload(name, runs_kernel(name, seed, nf, nr, run_len, iters, **kw), name, grid, block, params, bufs,
                       max_ts=0)


CASES = {
    # (nf, nr, run_len, iters, extra)
    "few_rows_short": (2, 2, 6, 4, {}),
    "few_rows_long": (3, 3, 40, 5, {}),
    "chain_heavy": (1, 1, 32, 6, {}),
    "many_rows": (14, 14, 48, 3, {}),
    "more_rows": (24, 24, 64, 3, {}),
    "partial_warp": (4, 4, 24, 4, {"block": 80}),
    "divergent": (4, 4, 24, 4, {"diverge": 13}),
    "mid_entry": (4, 4, 24, 4, {"mid_entry": True}),
}


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("name", list(CASES))
def test_runs_match_oracle(name, layout):
    nf, nr, run_len, iters, extra = CASES[name]
    for seed in range(3):
        w = runs_workload(seed * 17 + len(name), nf, nr, run_len, iters, **extra)
        _parity.assert_parity(w, cfg=ks.Config(layout=layout))


# NaNs with payloads and either sign, signalling NaNs, infinities, zeros,
# subnormals and ordinary values: IEEE-754 binary32 patterns
SPECIAL_F32 = [0x7FC00000, 0xFFC00000, 0x7FC12345, 0xFFE00001, 0x7F800001, 0xFF800001, 0x7F800000, 0xFF800000, 0x00000000, 0x80000000, 0x00000001, 0x807FFFFF, 0x7F7FFFFF,
               0x3F800000, 0xBF400000, 0x3F000000, 0x40490FDB]


@pytest.mark.parametrize("layout", LAYOUTS)
def test_runs_with_nan_payload_inputs(layout):
    """f32 fast runs whose inputs hold NaNs with payloads (quiet and
    signalling, either sign), infinities, signed zeros and subnormals: every
    NaN result is stored as the canonical 0x7FFFFFFF (which no input holds),
    as the oracle stores it, and every other result bit for bit."""
    for seed in range(4):
        w = runs_workload(40 + seed, 6, 1, 24, 2, fbits=SPECIAL_F32)
        g, _ = _parity.assert_parity(w, cfg=ks.Config(layout=layout))
        assert (g.buffers[0].view(np.uint32) == 0x7FFFFFFF).any()


def guarded_f32_workload(seed):
    """Guarded f32 add / sub / mul / fma (the general path) and the same ops
    unguarded and alone between integer ops (the mid loop), on operands drawn
    from SPECIAL_F32."""
    ptx = wl.HEADER + """.visible .entry gf(.param .u64 gf_out, .param .u64 gf_inp)
{
    .reg .pred %p<3>;
    .reg .f32 %f<12>;
    .reg .b32 %r<8>;
    .reg .b64 %rd<6>;
    ld.param.u64 %rd1, [gf_out];
    ld.param.u64 %rd2, [gf_inp];
    mov.u32 %r1, %ctaid.x;
    mov.u32 %r2, %ntid.x;
    mov.u32 %r3, %tid.x;
    mad.lo.s32 %r4, %r1, %r2, %r3;
    mul.lo.u32 %r5, %r4, 32;
    cvt.u64.u32 %rd3, %r5;
    add.s64 %rd4, %rd2, %rd3;
    add.s64 %rd5, %rd1, %rd3;
    ld.global.f32 %f1, [%rd4];
    ld.global.f32 %f2, [%rd4+4];
    ld.global.f32 %f3, [%rd4+8];
    and.b32 %r6, %r3, 1;
    setp.ne.u32 %p1, %r6, 0;
    mov.f32 %f4, 0f00000000;
    mov.f32 %f5, 0f00000000;
    mov.f32 %f6, 0f00000000;
    mov.f32 %f7, 0f00000000;
    @%p1 add.rn.f32 %f4, %f1, %f2;
    @!%p1 sub.rn.f32 %f5, %f2, %f3;
    @%p1 mul.rn.f32 %f6, %f3, %f1;
    @!%p1 fma.rn.f32 %f7, %f1, %f2, %f3;
    add.rn.f32 %f8, %f1, %f3;
    xor.b32 %r7, %r6, 1;
    mul.rn.f32 %f9, %f2, %f2;
    xor.b32 %r7, %r7, 3;
    fma.rn.f32 %f10, %f3, %f2, %f1;
    st.global.f32 [%rd5], %f4;
    st.global.f32 [%rd5+4], %f5;
    st.global.f32 [%rd5+8], %f6;
    st.global.f32 [%rd5+12], %f7;
    st.global.f32 [%rd5+16], %f8;
    st.global.f32 [%rd5+20], %f9;
    st.global.f32 [%rd5+24], %f10;
    st.global.u32 [%rd5+28], %r7;
    ret;
}
"""
    grid, block = 2, 128
    rng = np.random.default_rng(2000 + seed)
    inp = np.zeros((grid * block, 8), dtype=np.uint32)
    inp[:, :3] = rng.choice(np.asarray(SPECIAL_F32, dtype=np.uint32), size=(grid * block, 3))
    out = np.zeros((grid * block, 8), dtype=np.uint32)
    bufs = wl.place([("out", out, True), ("inp", inp, False)])
    params = wl.pack_params([("u64", bufs[0].sim_base), ("u64", bufs[1].sim_base)])
    return wl.Workload(f"gf{seed}", ptx, "gf", grid, block, params, bufs, max_ts=0)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_guarded_and_lone_f32_ops_with_nan_payload_inputs(layout):
    for seed in range(3):
        w = guarded_f32_workload(seed)
        g, _ = _parity.assert_parity(w, cfg=ks.Config(layout=layout))
        assert (g.buffers[0].view(np.uint32) == 0x7FFFFFFF).any()


@pytest.mark.parametrize("layout", LAYOUTS)
def test_runs_under_other_latencies(layout):
    """Fast runs under other latency tables (the table is patched into the
    program per launch)."""
    for lat_alu, lat_fma in ((1, 1), (2, 7), (9, 3), (0, 0)):
        lat = list(ks.api.DEFAULT_LAT)
        lat[0], lat[1] = lat_alu, lat_fma
        w = runs_workload(5, 4, 4, 30, 4)
        _parity.assert_parity(w, cfg=ks.Config(lat=tuple(lat), layout=layout))


@pytest.mark.parametrize("layout", LAYOUTS)
def test_runs_near_the_clock_rebase(layout):
    """Latencies of 2^22 and 2^24 cycles: runs are cut where a clock would pass
    2^30, and the epoch moves."""
    for big in (1 << 22, 1 << 24):
        lat = list(ks.api.DEFAULT_LAT)
        lat[0] = lat[1] = big
        w = runs_workload(7, 3, 3, 20, 40)
        g, _ = _parity.assert_parity(w, cfg=ks.Config(lat=tuple(lat), layout=layout))
        assert int(g.stats["cycles"].min()) > 1 << 30


@pytest.mark.parametrize("layout", LAYOUTS)
def test_step_limit_inside_a_run(layout):
    """A step limit that falls inside a fast run: the run stops at the limit,
    as the oracle's does."""
    w = runs_workload(9, 4, 4, 30, 4)
    for limit in (40, 41, 57, 100):
        g, _ = _parity.assert_parity(w, cfg=ks.Config(step_limit=limit, layout=layout))
        assert g.totals.status != 0

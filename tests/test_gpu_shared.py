"""GPU parity for shared memory and bar.sync: the sm_103a interpreter in CTA
mode (one real CTA per simulated CTA) against the oracle, byte for byte —
shared-memory reductions, bank-conflict patterns, barrier timing, statuses
and a barrier release far ahead of a warp's clock."""
import numpy as np
import pytest
import torch

import oracle
import simt_ptx_interpretation_gb300 as ks
from simt_ptx_interpretation_gb300 import workloads as wl
from tests import _parity
from tests import test_oracle_shared as tsh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for -m gpu tests")
    from simt_ptx_interpretation_gb300 import _build
    _build.build_native()


@pytest.mark.parametrize("block", [32, 64, 128, 256])
def test_smem_reduce_parity(block):
    g, _ = _parity.assert_parity(wl.smem_reduce(n=block * 96, block=block))
    assert g.totals.sh_req > 0


def test_smem_reduce_headline_sampled():
    w = wl.smem_reduce()
    warps = _parity.sample_warps(w, n=24, seed=5)
    ctas = sorted({gw // (w.block // 32) for gw in warps})
    _parity.assert_parity(w, warps=warps, out_words={"out": ctas})


SH_PATTERNS = {  # element index (at most 1023) of lane %r7 in its warp's slice of shared memory
    "seq": "mov.u32 %r2, %r7;",
    "stride2": "shl.b32 %r2, %r7, 1;",            # 2-way
    "stride32": "shl.b32 %r2, %r7, 5;",           # 32-way
    "stride33": "mul.lo.u32 %r2, %r7, 33;",        # conflict free
    "groups4": "shr.u32 %r2, %r7, 2;",            # broadcast groups
    "same": "mov.u32 %r2, 5;",
    "mod8x32": "and.b32 %r2, %r7, 7;\n    shl.b32 %r2, %r2, 5;",   # 8 addresses, one bank
    "reverse": "mov.u32 %r5, 31;\n    sub.u32 %r2, %r5, %r7;",
}


def shared_access_workload(pattern: str, guard: str, size: int) -> wl.Workload:
    """Each warp stores its thread ids to its own slice of shared memory (1024
    elements) through a pattern, passes a barrier, loads back through the same
    pattern (duplicate addresses give the highest lane's value) and writes
    what it read to global memory (lanes that skip the load write the 0 they
    were given, so the program is defined natively too)."""
    gset, g = {"all": ("", ""), "lt20": ("setp.lt.u32 %p1, %r7, 20;", "@%p1 "),
               "odd": ("and.b32 %r5, %r7, 1;\n    setp.ne.u32 %p1, %r5, 0;", "@%p1 ")}[guard]
    sh = 2 if size == 4 else 3
    if size == 4:
        st = f"{g}st.shared.u32 [%r3], %r1;"
        ld = f"{g}ld.shared.u32 %r4, [%r3];\n    st.global.u32 [%rd3], %r4;"
    else:
        st = f"cvt.u64.u32 %rd4, %r1;\n    {g}st.shared.u64 [%r3], %rd4;"
        ld = f"{g}ld.shared.u64 %rd5, [%r3];\n    st.global.u64 [%rd3], %rd5;"
    ptx = wl.HEADER + f""".visible .entry shacc(.param .u64 out)
{{
    .reg .pred %p<2>;
    .reg .b32 %r<10>;
    .reg .b64 %rd<6>;
    .shared .align 8 .b8 smem[{4 * 1024 * size}];
    ld.param.u64 %rd1, [out];
    mov.u32 %r1, %tid.x;
    and.b32 %r7, %r1, 31;
    {SH_PATTERNS[pattern]}
    shl.b32 %r2, %r2, {sh};
    shr.u32 %r6, %r1, 5;
    shl.b32 %r6, %r6, {10 + sh};
    add.u32 %r2, %r2, %r6;
    mov.u32 %r3, smem;
    add.u32 %r3, %r3, %r2;
    mov.u32 %r4, 0;
    mov.u64 %rd5, 0;
    {gset}
    {st}
    bar.sync 0;
    mov.u32 %r8, %ctaid.x;
    mov.u32 %r9, %ntid.x;
    mad.lo.s32 %r8, %r8, %r9, %r1;
    cvt.u64.u32 %rd2, %r8;
    shl.b64 %rd2, %rd2, {sh};
    add.s64 %rd3, %rd1, %rd2;
    {ld}
    ret;
}}
"""
    grid, block = 3, 128
    out = np.zeros(grid * block * size // 4, dtype=np.uint32)
    bufs = wl.place([("out", out, True)])
    return wl.Workload(f"shacc_{pattern}_{guard}_{size}", ptx, "shacc", grid, block,
                       wl.pack_params([("u64", bufs[0].sim_base)]), bufs)


@pytest.mark.parametrize("size", [4, 8])
@pytest.mark.parametrize("guard", ["all", "lt20", "odd"])
@pytest.mark.parametrize("pattern", list(SH_PATTERNS))
def test_shared_access_patterns_match_the_oracle(pattern, guard, size):
    _parity.assert_parity(shared_access_workload(pattern, guard, size))


def test_bank_degrees_of_the_patterns():
    # the degree the page's rule gives each pattern (all lanes, 4 bytes)
    want = {"seq": 1, "stride2": 2, "stride32": 32, "stride33": 1, "groups4": 1, "same": 1, "mod8x32": 32,
            "reverse": 1}
    for pattern, degree in want.items():
        g = _parity.gpu_run(shared_access_workload(pattern, "all", 4))
        st = g.stats[0]
        assert (st["sh_req"], st["sh_wavefronts"]) == (2, 2 * degree), pattern


@pytest.mark.parametrize("n", [1, 3, 10])
def test_barrier_closed_form_matches_the_oracle(n):
    w = wl.Workload("bar2", tsh.barrier_ptx(n), "bar2", 1, 64, b"", [])
    g, _ = _parity.assert_parity(w)
    release = max(16 + 4 * (n - 1) + 1, 16) + 20
    assert list(g.stats["cycles"]) == [release + 1] * 2


ZEROED_PTX = wl.HEADER + """.visible .entry z(.param .u64 out)
{
    .reg .b32 %r<6>;
    .reg .b64 %rd<4>;
    .shared .align 4 .b8 s[4096];
    ld.param.u64 %rd1, [out];
    mov.u32 %r1, %tid.x;
    mov.u32 %r2, %ctaid.x;
    shl.b32 %r3, %r1, 2;
    ld.shared.u32 %r4, [%r3];
    add.u32 %r5, %r4, %r2;
    st.shared.u32 [%r3], %r5;
    bar.sync 0;
    ld.shared.u32 %r4, [s+4];
    add.u32 %r5, %r5, %r4;
    mov.u32 %r3, %ntid.x;
    mad.lo.s32 %r3, %r2, %r3, %r1;
    cvt.u64.u32 %rd2, %r3;
    shl.b64 %rd2, %rd2, 2;
    add.s64 %rd3, %rd1, %rd2;
    st.global.u32 [%rd3], %r5;
    ret;
}
"""


def test_zeroed_shared_memory_and_partial_warps():
    ptx = ZEROED_PTX
    for grid, block in [(700, 48), (5, 256), (1, 1)]:
        out = np.zeros(grid * block, dtype=np.uint32)
        bufs = wl.place([("out", out, True)])
        w = wl.Workload("z", ptx, "z", grid, block, wl.pack_params([("u64", bufs[0].sim_base)]), bufs)
        g, _ = _parity.assert_parity(w)
        assert np.array_equal(g.buffers[0].view(np.uint32), np.repeat(2 * np.arange(grid, dtype=np.uint32), block))


def test_shared_statuses_match_the_oracle():
    for off, sym in [(4, "b"), (8, "b"), (2, "b"), (16, "a")]:
        ptx = wl.HEADER + f""".visible .entry lay()
{{
    .reg .b32 %r<4>;
    .shared .align 4 .b8 a[6];
    .shared .align 8 .b8 b[8];
    mov.u32 %r1, {sym};
    ld.shared.u32 %r2, [%r1+{off}];
    ret;
}}
"""
        _parity.assert_parity(wl.Workload("lay", ptx, "lay", 2, 64, b"", []))


def test_step_limit_inside_a_barrier_program():
    w = wl.smem_reduce(n=256 * 8, block=256)
    for limit in (5, 17, 40):
        _parity.assert_parity(w, cfg=ks.Config(max_ts=w.max_ts, step_limit=limit))


def test_barrier_release_far_ahead_of_a_warps_clock():
    # warp 0 runs a chain of dependent global loads of latency 2^24 (about
    # 2^30 cycles in all) before the barrier; warp 1 arrives at once, so its
    # release lies far beyond its own clock
    loads = "\n".join("    ld.global.u64 %rd2, [%rd2];" for _ in range(70))
    ptx = wl.HEADER + f""".visible .entry far(.param .u64 buf)
{{
    .reg .pred %p<2>;
    .reg .b32 %r<3>;
    .reg .b64 %rd<4>;
    ld.param.u64 %rd2, [buf];
    mov.u32 %r1, %tid.x;
    setp.lt.u32 %p1, %r1, 32;
    @!%p1 bra SKIP;
{loads}
SKIP:
    bar.sync 0;
    add.u32 %r2, %r1, 1;
    ret;
}}
"""
    buf = np.zeros(2, dtype=np.uint64)
    bufs = wl.place([("buf", buf, False)])
    buf[0] = bufs[0].sim_base  # every load reads the buffer's own address
    w = wl.Workload("far", ptx, "far", 3, 64, wl.pack_params([("u64", bufs[0].sim_base)]), bufs)
    lat = list(ks.DEFAULT_LAT)
    lat[2] = 1 << 24
    g, _ = _parity.assert_parity(w, cfg=ks.Config(lat=tuple(lat)))
    assert int(g.stats["cycles"][1]) > 1 << 30


def test_blocks_above_256_threads():
    """CTA mode for 9..32 warps per CTA (the 1024-thread configuration)."""
    from tests.test_gpu_parity import jit_memory
    for block in (512, 1024):
        w = wl.smem_reduce(n=block * 8, block=block)
        _parity.assert_parity(w)
        assert np.array_equal(_parity.gpu_run(w).buffers[1], jit_memory(w)[1])


@pytest.mark.parametrize("block", [640, 1000, 1024])
def test_lean_kernel_at_large_blocks(block):
    ptx = ZEROED_PTX
    grid = 5
    out = np.zeros(grid * block, dtype=np.uint32)
    bufs = wl.place([("out", out, True)])
    w = wl.Workload("z", ptx, "z", grid, block, wl.pack_params([("u64", bufs[0].sim_base)]), bufs)
    g, _ = _parity.assert_parity(w)
    assert np.array_equal(g.buffers[0].view(np.uint32), np.repeat(2 * np.arange(grid, dtype=np.uint32), block))


def cta_state_exceeds_smem(w: wl.Workload) -> bool:
    """The PAIR warp state of one CTA alone exceeds the SM's shared memory."""
    region = ks.Module(w.ptx).layout(w.kernel)[1]
    return region * ((w.block + 31) // 32) > torch.cuda.get_device_properties(0).shared_memory_per_block_optin


@pytest.mark.parametrize("i", [0, 1, 2, 7])
def test_cta_warp_state_in_global_memory(i):
    """Random shared programs at block 1024: 32 warps of about 11 KB of
    interpreter state each exceed an SM's shared memory, so the warps' state
    moves to global memory (the simulated shared arrays stay on chip); every
    warp's record, trace slot and byte of memory equals the oracle's."""
    w = wl.fuzz_shared(i, grid=4, block=1024)
    assert cta_state_exceeds_smem(w)
    _parity.assert_parity(w)


def test_cta_warp_state_in_global_memory_far_release():
    """As test_barrier_release_far_ahead_of_a_warps_clock, at block 1024 with
    40 more registers per thread: the barrier release moves the epochs of the
    waiting warps' clocks in global memory."""
    loads = "\n".join("    ld.global.u64 %rd2, [%rd2];" for _ in range(70))
    pads = "\n".join(f"    add.u32 %x{i}, %r1, {i};" for i in range(40))
    sums = "\n".join(f"    add.u32 %r2, %r2, %x{i};" for i in range(40))
    ptx = wl.HEADER + f""".visible .entry farbig(.param .u64 buf, .param .u64 out)
{{
    .reg .pred %p<2>;
    .reg .b32 %r<3>;
    .reg .b32 %x<40>;
    .reg .b64 %rd<6>;
    ld.param.u64 %rd2, [buf];
    mov.u32 %r1, %tid.x;
{pads}
    setp.lt.u32 %p1, %r1, 32;
    @!%p1 bra SKIP;
{loads}
SKIP:
    bar.sync 0;
    mov.u32 %r2, 0;
{sums}
    ld.param.u64 %rd3, [out];
    mov.u32 %r0, %ctaid.x;
    mad.lo.s32 %r0, %r0, 1024, %r1;
    cvt.u64.u32 %rd4, %r0;
    shl.b64 %rd4, %rd4, 2;
    add.s64 %rd5, %rd3, %rd4;
    st.global.u32 [%rd5], %r2;
    ret;
}}
"""
    buf = np.zeros(2, dtype=np.uint64)
    out = np.zeros(2 * 1024, dtype=np.uint32)
    bufs = wl.place([("buf", buf, False), ("out", out, True)])
    buf[0] = bufs[0].sim_base  # every load reads the buffer's own address
    w = wl.Workload("farbig", ptx, "farbig", 2, 1024,
                    wl.pack_params([("u64", bufs[0].sim_base), ("u64", bufs[1].sim_base)]), bufs)
    assert cta_state_exceeds_smem(w)
    lat = list(ks.DEFAULT_LAT)
    lat[2] = 1 << 24
    g, _ = _parity.assert_parity(w, cfg=ks.Config(lat=tuple(lat)))
    assert int(g.stats["cycles"][1]) > 1 << 30
    tid = np.arange(1024, dtype=np.uint64)
    want = (40 * tid + sum(range(40))) & 0xFFFFFFFF
    assert np.array_equal(g.buffers[1].view(np.uint32), np.tile(want.astype(np.uint32), 2))


def test_static_entry_refuses_global_warp_state():
    """The allocation-free entry point cannot take the global scratch such a
    launch needs: KS_ERR_LIMIT before any GPU work."""
    w = wl.fuzz_shared(0, grid=2, block=1024)
    m = ks.Module(w.ptx)
    dev = [(b.sim_base, torch.zeros(b.data.nbytes, dtype=torch.uint8).cuda()) for b in w.buffers]
    stats = torch.zeros(ks.stats_bytes(w.grid, w.block), dtype=torch.uint8, device="cuda")
    with pytest.raises(ks.KsError) as e:
        ks.simulate_static(m, w.kernel, w.grid, w.block, w.params, dev, stats)
    assert e.value.code == -6


# -------------------------------------------- the driver JIT as a third party ----

@pytest.mark.parametrize("block", [32, 64, 256])
def test_jit_crosscheck_smem_reduce(block):
    """The same PTX run natively through the driver JIT gives the same memory."""
    from tests.test_gpu_parity import jit_memory
    w = wl.smem_reduce(n=block * 64, block=block)
    sim = _parity.gpu_run(w).buffers
    nat = jit_memory(w)
    for b, x, y in zip(w.buffers, sim, nat):
        assert np.array_equal(x, y), b.name


@pytest.mark.parametrize("size", [4, 8])
@pytest.mark.parametrize("guard", ["all", "odd"])
@pytest.mark.parametrize("pattern", ["seq", "stride2", "stride32", "stride33", "reverse"])
def test_jit_crosscheck_shared_patterns(pattern, guard, size):
    # patterns whose stores never share an address (PTX leaves the winner of
    # same-address stores unspecified)
    from tests.test_gpu_parity import jit_memory
    w = shared_access_workload(pattern, guard, size)
    sim = _parity.gpu_run(w).buffers
    nat = jit_memory(w)
    assert np.array_equal(sim[0], nat[0])


@pytest.mark.parametrize("block", [32, 128, 256])
@pytest.mark.parametrize("i", range(24))
def test_random_shared_programs_match_the_oracle(i, block):
    _parity.assert_parity(wl.fuzz_shared(i, grid=16, block=block))


@pytest.mark.parametrize("i", range(0, 24, 3))
def test_jit_crosscheck_random_shared_programs(i):
    from tests.test_gpu_parity import jit_memory
    w = wl.fuzz_shared(i, grid=16, block=128)
    sim = _parity.gpu_run(w).buffers
    nat = jit_memory(w)
    assert np.array_equal(sim[1], nat[1])

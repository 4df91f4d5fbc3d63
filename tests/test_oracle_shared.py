"""Oracle pins for shared memory and barriers: the bank-conflict examples the
pages print, the pages' thread-count rule on a mixed bank, a barrier timing
closed form derived by hand, a shared-memory tree reduction against numpy,
warp mode against per-thread mode, the race checker, statuses, layout and the
forms the subset rejects. CPU only."""
import os
import struct

import numpy as np
import pytest

import oracle
from simt_ptx_interpretation_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
LAT = dict(zip(["alu", "fma", "ldg", "stg", "bra", "sfu", "ret", "lds", "sts", "bar"], oracle.DEFAULT_LAT))


def bank_probe_ptx(size: int = 4) -> str:
    """One warp: lane i reads its shared address from addr[i] and executes
    ld.shared of `size` bytes there when act[i] != 0."""
    ld = "ld.shared.u32 %r4, [%r3];" if size == 4 else "ld.shared.u64 %rd4, [%r3];"
    return wl.HEADER + f""".visible .entry probe(.param .u64 p_addr, .param .u64 p_act)
{{
    .reg .pred %p<2>;
    .reg .b32 %r<6>;
    .reg .b64 %rd<6>;
    .shared .align 8 .b8 smem[8192];
    ld.param.u64 %rd1, [p_addr];
    ld.param.u64 %rd2, [p_act];
    mov.u32 %r1, %tid.x;
    cvt.u64.u32 %rd3, %r1;
    shl.b64 %rd3, %rd3, 2;
    add.s64 %rd1, %rd1, %rd3;
    add.s64 %rd2, %rd2, %rd3;
    ld.global.u32 %r3, [%rd1];
    ld.global.u32 %r2, [%rd2];
    setp.ne.u32 %p1, %r2, 0;
    @%p1 {ld}
    ret;
}}
"""


def bank_degree(addresses, size=4):
    """Runs the probe with lanes 0..len-1 executing at `addresses`; returns
    (sh_req, sh_wavefronts) of the warp."""
    addr = np.zeros(32, dtype=np.uint32)
    act = np.zeros(32, dtype=np.uint32)
    addr[:len(addresses)] = addresses
    act[:len(addresses)] = 1
    bufs = wl.place([("addr", addr, False), ("act", act, False)])
    params = wl.pack_params([("u64", bufs[0].sim_base), ("u64", bufs[1].sim_base)])
    r = oracle.run(bank_probe_ptx(size), "probe", 1, 32, params, [(b.sim_base, b.data) for b in bufs])
    assert r.status == 0
    return int(r.stats[0]["sh_req"]), int(r.stats[0]["sh_wavefronts"])


def golden_rows():
    rows = []
    for line in open(os.path.join(GOLDEN, "kernelscope_shared_banks.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        name, addrs, degree = line.split()
        if addrs.startswith("i*"):
            k, _, off = addrs[2:].partition("+")
            addresses = [i * int(k) + int(off or 0) for i in range(32)]
        else:
            addresses = [int(a) for a in addrs.split(",")]
        rows.append((name, addresses, int(degree)))
    return rows


@pytest.mark.parametrize("name,addresses,degree", golden_rows(), ids=[r[0] for r in golden_rows()])
def test_bank_conflict_examples_from_the_pages(name, addresses, degree):
    assert bank_degree(addresses) == (1, degree)


def test_mixed_bank_counts_lanes_not_addresses():
    # The page's rule: a bank that is not a pure broadcast counts its lanes.
    # 16 lanes on address 0 and 16 on address 128 share bank 0 with two
    # addresses: degree 32 (a distinct-address count would give 2).
    assert bank_degree([0] * 16 + [128] * 16) == (1, 32)
    # three lanes in bank 5, two of them on one address: degree 3
    assert bank_degree([20, 20, 148, 4]) == (1, 3)


def test_bank_degree_brute_force_over_random_patterns():
    rng = np.random.default_rng(11)
    for _ in range(40):
        n = int(rng.integers(1, 33))
        # few distinct words so that broadcasts and mixed banks both occur
        addresses = [int(x) * 4 for x in rng.integers(0, 96, size=n)]
        banks = {}
        for a in addresses:
            banks.setdefault((a // 4) % 32, []).append(a)
        want = max([1] + [len(v) for v in banks.values() if len(set(v)) > 1])
        assert bank_degree(addresses) == (1, want)


def test_eight_byte_accesses_use_each_lanes_address():
    # lane i at 8i: lanes i and i+16 share bank (2i mod 32) on two addresses
    assert bank_degree([8 * i for i in range(32)], size=8) == (1, 2)
    assert bank_degree([8 * i for i in range(16)], size=8) == (1, 1)


def test_no_request_without_executing_lanes():
    assert bank_degree([]) == (0, 0)


# --------------------------------------------------------------- barriers ----

def barrier_ptx(n_fma: int) -> str:
    """Warp 0 runs a dependent chain of n_fma fma before bar.sync; warp 1 goes
    straight to it; both then ret."""
    body = "\n".join("    fma.rn.f32 %f1, %f1, %f1, %f1;" for _ in range(n_fma))
    return wl.HEADER + f""".visible .entry bar2()
{{
    .reg .pred %p<2>;
    .reg .b32 %r<3>;
    .reg .f32 %f<2>;
    mov.u32 %r1, %tid.x;
    setp.lt.u32 %p1, %r1, 32;
    @!%p1 bra SKIP;
{body}
SKIP:
    bar.sync 0;
    ret;
}}
"""


@pytest.mark.parametrize("n", [1, 3, 10])
def test_barrier_release_closed_form(n):
    # mov t=0 (ready 4); setp t=4 (ready 8); bra t=8, next issue 16.
    # warp 0: fma at 16, 20, ..., 16+4(n-1); bar.sync issues at 16+4(n-1)+1.
    # warp 1: taken branch, bar.sync at 16. Release R = max(both) + bar latency;
    # ret issues at R in both warps: cycles = R + 1.
    r = oracle.run(barrier_ptx(n), "bar2", 1, 64, b"", [])
    assert r.status == 0
    arrive0 = 16 + 4 * (n - 1) + 1
    release = max(arrive0, 16) + LAT["bar"]
    assert list(r.stats["cycles"]) == [release + 1, release + 1]
    assert list(r.stats["warp_insts"]) == [n + 5, 5]


def test_barrier_latency_is_a_parameter():
    lat = list(oracle.DEFAULT_LAT)
    lat[9] = 100
    r = oracle.run(barrier_ptx(2), "bar2", 1, 64, b"", [], lat=lat)
    assert list(r.stats["cycles"]) == [16 + 4 + 1 + 100 + 1] * 2


def test_finished_warps_do_not_hold_a_barrier():
    # warp 1 returns early; warp 0's barrier releases at its own arrival + latency
    ptx = wl.HEADER + """.visible .entry early()
{
    .reg .pred %p<2>;
    .reg .b32 %r<3>;
    mov.u32 %r1, %tid.x;
    setp.ge.u32 %p1, %r1, 32;
    @%p1 bra OUT;
    bar.sync 0;
OUT:
    ret;
}
"""
    r = oracle.run(ptx, "early", 1, 64, b"", [])
    # warp 0: mov 0, setp 4, bra 8 (not taken, next 16), bar at 16, release 36, ret 36
    assert r.stats["cycles"][0] == 16 + LAT["bar"] + 1
    # warp 1: bra taken at 8, ret at 16
    assert r.stats["cycles"][1] == 17


def test_ld_shared_latency_in_the_scoreboard():
    ptx = wl.HEADER + """.visible .entry lds()
{
    .reg .b32 %r<4>;
    .shared .align 4 .b8 s[128];
    mov.u32 %r1, s;
    ld.shared.u32 %r2, [%r1];
    add.u32 %r3, %r2, 1;
    st.shared.u32 [%r1+4], %r3;
    ret;
}
"""
    r = oracle.run(ptx, "lds", 1, 32, b"", [])
    # mov 0 (ready 4); ld.shared at 4 (ready 27); add at 27 (ready 31);
    # st.shared at 31, completes 31 + 23; ret at 32
    assert r.stats["cycles"][0] == 31 + LAT["sts"]


# --------------------------------------------------------- shared data flow ----

def reduction_sums(w) -> np.ndarray:
    x = w.buffers[0].data.astype(np.uint64).reshape(w.grid, w.block)
    return (x.sum(axis=1) & 0xFFFFFFFF).astype(np.uint32)


def test_tree_reduction_matches_numpy_and_per_thread_mode():
    w = wl.smem_reduce(n=1 << 12, block=256)
    want = reduction_sums(w)
    for mode in (oracle.MODE_WARP, oracle.MODE_PER_THREAD):
        bufs = w.fresh_buffers()
        r = oracle.run(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in bufs],
                       mode=mode)
        assert r.status == 0
        assert np.array_equal(bufs[1].data, want)


def test_tree_reduction_is_race_free_and_a_missing_barrier_is_a_race():
    w = wl.smem_reduce(n=1 << 10, block=128)
    bufs = w.fresh_buffers()
    r = oracle.run(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in bufs],
                   race_check=True)
    assert r.race_flags == 0
    broken = w.ptx.replace("    bar.sync 0;\n", "", 1)
    bufs = w.fresh_buffers()
    r = oracle.run(broken, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in bufs],
                   race_check=True)
    assert r.race_flags == oracle.RACE_CROSS_THREAD


def test_shared_memory_starts_zeroed_in_every_cta():
    ptx = wl.HEADER + """.visible .entry z(.param .u64 out)
{
    .reg .b32 %r<6>;
    .reg .b64 %rd<4>;
    .shared .align 4 .b8 s[1024];
    ld.param.u64 %rd1, [out];
    mov.u32 %r1, %tid.x;
    mov.u32 %r2, %ctaid.x;
    shl.b32 %r3, %r1, 2;
    ld.shared.u32 %r4, [%r3];
    add.u32 %r5, %r4, %r2;
    st.shared.u32 [%r3], %r5;
    mov.u32 %r3, %ntid.x;
    mad.lo.s32 %r3, %r2, %r3, %r1;
    cvt.u64.u32 %rd2, %r3;
    shl.b64 %rd2, %rd2, 2;
    add.s64 %rd3, %rd1, %rd2;
    st.global.u32 [%rd3], %r5;
    ret;
}
"""
    out = np.zeros(4 * 256, dtype=np.uint32)
    bufs = wl.place([("out", out, True)])
    oracle.run(ptx, "z", 4, 256, wl.pack_params([("u64", bufs[0].sim_base)]), [(b.sim_base, b.data) for b in bufs])
    assert np.array_equal(bufs[0].data, np.repeat(np.arange(4, dtype=np.uint32), 256))


def test_shared_layout_alignment_and_bounds():
    def kernel(off: int, sym: str = "b") -> str:
        return wl.HEADER + f""".visible .entry lay()
{{
    .reg .b32 %r<4>;
    .shared .align 4 .b8 a[6];
    .shared .align 8 .b8 b[8];
    mov.u32 %r1, {sym};
    ld.shared.u32 %r2, [%r1+{off}];
    ret;
}}
"""
    # a at 0..5, b aligned to 8: 8..15; 16 bytes in all
    assert oracle.run(kernel(4), "lay", 1, 32, b"", []).status == 0      # 12..15
    assert oracle.run(kernel(8), "lay", 1, 32, b"", []).status == 1      # 16: out of range
    assert oracle.run(kernel(2), "lay", 1, 32, b"", []).status == 2      # 10: misaligned
    assert oracle.run(kernel(12, "a"), "lay", 1, 32, b"", []).status == 0
    assert oracle.run(kernel(16, "a"), "lay", 1, 32, b"", []).status == 1


SHARED_BAD = [
    (".shared .align 4 .b8 s[49156];\n    ret;", -2),                                  # over 48 KiB
    ("bar.sync 1;\n    ret;", -2),                                                     # barrier 1
    ("bar.sync 0, 64;\n    ret;", -1),                                                 # thread count
    ("@%p1 bar.sync 0;\n    ret;", -2),                                                # guarded
    ("ld.shared.u32 %r1, [nowhere];\n    ret;", -1),                                   # unknown array
    (".shared .align 4 .b8 s[64];\n    mov.f32 %f1, s;\n    ret;", -1),                # float symbol
    (".shared .align 4 .b8 s[64];\n    ld.shared.u32 %r1, [%p1];\n    ret;", -1),      # predicate address
]


def bad_shared_kernel(body: str) -> str:
    return wl.HEADER + f""".visible .entry bad()
{{
    .reg .pred %p<2>;
    .reg .b32 %r<3>;
    .reg .f32 %f<2>;
    {body}
}}
"""


@pytest.mark.parametrize("body,code", SHARED_BAD)
def test_rejected_forms(body, code):
    assert oracle.parse_check(bad_shared_kernel(body), "bad")[0] == code


@pytest.mark.parametrize("i", range(0, 12, 3))
@pytest.mark.parametrize("block", [32, 256])
def test_random_shared_programs_are_race_free_and_mode_independent(i, block):
    """The shared-memory program generator's contract, checked on the oracle:
    no two threads of a CTA touch one word in one barrier interval with a
    write among them, and warp mode and per-thread mode store the same."""
    w = wl.fuzz_shared(i, grid=4, block=block)
    b1, b2 = w.fresh_buffers(), w.fresh_buffers()
    r1 = oracle.run(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in b1], race_check=True)
    r2 = oracle.run(w.ptx, w.kernel, w.grid, w.block, w.params, [(b.sim_base, b.data) for b in b2],
                    mode=oracle.MODE_PER_THREAD)
    assert r1.status == r2.status == 0 and r1.race_flags == 0
    assert np.array_equal(b1[1].data, b2[1].data)
    assert r1.stats["sh_wavefronts"].sum() >= r1.stats["sh_req"].sum() > 0

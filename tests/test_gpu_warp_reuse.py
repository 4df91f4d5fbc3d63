"""A real warp runs many simulated warps in one register region, one after
another. In the PAIR layout only the slots that some path may read before
writing them are cleared between them, and each later warp's clock starts
above every ready time the region still holds. These cases run grids far
larger than the GPU's resident warps (so every region is reused many times)
and must equal the oracle, which starts every warp from zeroed registers at
clock 0, byte for byte over the whole grid: registers written by some lanes
only, registers never written, loop-carried registers set inside a branch,
results still in flight when a warp ends, and random programs forced into
PAIR."""
import numpy as np
import pytest
import torch

import simt_ptx_interpretation_gb300 as ks
from simt_ptx_interpretation_gb300 import workloads as wl
from tests import _parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for -m gpu tests")
    from simt_ptx_interpretation_gb300 import _build
    _build.build_native()


def _kernel(name: str, body: list[str]) -> str:
    """out[gtid] (u32) from `body`, which starts with gtid in %r1, the
    output address in %rd3 and the input address in %rd4 (in[gtid], u32)."""
    lines = [f".visible .entry {name}(.param .u64 wr_out, .param .u64 wr_in)", "{",
             "    .reg .pred %p<4>;", "    .reg .b32 %r<16>;", "    .reg .f32 %f<4>;", "    .reg .b64 %rd<8>;",
             "    ld.param.u64 %rd1, [wr_out];", "    ld.param.u64 %rd2, [wr_in];",
             "    mov.u32 %r2, %ctaid.x;", "    mov.u32 %r3, %ntid.x;", "    mov.u32 %r4, %tid.x;",
             "    mad.lo.s32 %r1, %r2, %r3, %r4;", "    cvt.u64.u32 %rd5, %r1;", "    shl.b64 %rd5, %rd5, 2;",
             "    add.s64 %rd3, %rd1, %rd5;", "    add.s64 %rd4, %rd2, %rd5;"]
    lines += ["    " + x for x in body] + ["    ret;", "}", ""]
    return wl.HEADER + "\n".join(lines)


def _workload(name: str, body: list[str], grid: int = 1024, block: int = 256, seed: int = 11) -> wl.Workload:
    n = grid * block
    rng = np.random.default_rng(seed)
    inp = rng.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32)
    bufs = wl.place([("out", np.zeros(n, dtype=np.uint32), True), ("in", inp, False)])
    params = wl.pack_params([("u64", bufs[0].sim_base), ("u64", bufs[1].sim_base)])
    return wl.Workload(name, _kernel(name, body), name, grid, block, params, bufs)


CASES = {
    # %r5 written only by the odd lanes, read by all
    "some_lanes_write": [
        "and.b32 %r6, %r4, 1;", "setp.eq.u32 %p1, %r6, 0;", "@%p1 bra WR_JOIN;",
        "ld.global.u32 %r5, [%rd4];",
        "WR_JOIN:", "add.u32 %r7, %r5, %r1;", "st.global.u32 [%rd3], %r7;"],
    # %r9 and %f2 never written
    "never_written": [
        "cvt.rzi.u32.f32 %r8, %f2;", "add.u32 %r7, %r9, %r8;", "xor.b32 %r7, %r7, %r1;",
        "st.global.u32 [%rd3], %r7;"],
    # a guarded write does not make %r10 written
    "guarded_write": [
        "ld.global.u32 %r6, [%rd4];", "setp.lt.u32 %p2, %r6, 0x80000000;",
        "@%p2 mul.lo.u32 %r10, %r6, 3;", "add.u32 %r7, %r10, 1;", "st.global.u32 [%rd3], %r7;"],
    # loop-carried %r11 set inside a branch of the loop body
    "loop_carried": [
        "ld.global.u32 %r6, [%rd4];", "and.b32 %r6, %r6, 7;", "mov.u32 %r12, 0;",
        "WR_LOOP:", "setp.ge.u32 %p1, %r12, %r6;", "@%p1 bra WR_END;",
        "and.b32 %r13, %r12, 1;", "setp.eq.u32 %p2, %r13, 1;", "@%p2 bra WR_SKIP;",
        "add.u32 %r11, %r11, %r12;",
        "WR_SKIP:", "add.u32 %r12, %r12, 1;", "bra.uni WR_LOOP;",
        "WR_END:", "st.global.u32 [%rd3], %r11;"],
    # a load's result still in flight at the warp's end, and a store draining
    "in_flight_at_end": [
        "ld.global.u32 %r6, [%rd4];", "st.global.u32 [%rd3], %r1;", "ld.global.u32 %r14, [%rd4];"],
}


@pytest.mark.parametrize("layout", ["pair", "split"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_reused_regions_match_oracle(name, layout):
    w = _workload("wr_" + name, CASES[name])
    assert w.warps >= 8192  # far more than the resident warps
    _parity.assert_parity(w, cfg=ks.Config(max_ts=0, layout=layout))


@pytest.mark.parametrize("i", [0, 5, 9])
def test_random_programs_in_pair_over_many_waves(i):
    """Random programs forced into PAIR (regions of about 19 KB, some 1,700
    resident warps) on a grid of 4,096 warps."""
    w = wl.fuzz(i, grid=512, block=256)
    _parity.assert_parity(w, cfg=ks.Config(max_ts=w.max_ts, layout="pair"))

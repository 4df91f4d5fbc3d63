"""The occupancy post-pass (ks_occupancy) against the page's worked example,
hand-derived cases for each limiter, and the oracle's restatement over random
inputs on every architecture. CPU only: host code."""
import os
import random

import pytest

from oracle import occupancy as orc
from simt_ptx_interpretation_gb300 import api as ks

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kernelscope_occupancy.txt")


def golden():
    rows = {}
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            k, v = line.split(None, 1)
            rows[k] = v
    return rows


def lib_occ(arch, threads, regs, smem=0):
    return ks.occupancy(ks.gpu_limits(arch), threads, regs, smem)


def test_the_pages_worked_example():
    g = golden()
    r = lib_occ(g["arch"], int(g["threads_per_block"]), int(g["registers_per_thread"]))
    assert r["warps_by_registers"] == int(g["warps_by_registers"])
    assert r["warps_by_block_size"] == int(g["warps_by_block_size"])
    assert r["active_warps_per_sm"] == int(g["active_warps_per_sm"])
    assert r["occupancy_percent"] == float(g["occupancy_percent"])
    assert 32 * int(g["registers_per_thread"]) == int(g["regs_per_warp"])


def test_each_limiter_by_hand():
    # sm_80, 256 threads, 64 registers: 2048 per warp, 65536 / 2048 = 32 warps
    r = lib_occ("sm_80", 256, 64)
    assert (r["active_warps_per_sm"], r["limiter"], r["occupancy_percent"]) == (32, "registers", 50.0)
    # 33 registers: 1056 per warp rounds up to 1280; 65536 / 1280 = 51 warps
    assert lib_occ("sm_80", 256, 33)["warps_by_registers"] == 51
    # sm_80, 256 threads, 16 regs, 48 KB shared per block: 167936 / 49152 = 3
    # blocks = 24 warps, 37.5 %
    r = lib_occ("sm_80", 256, 16, 48 * 1024)
    assert (r["active_warps_per_sm"], r["limiter"], r["occupancy_percent"]) == (24, "shared_memory", 37.5)
    # 100 bytes of shared memory count as one 256-byte chunk
    assert lib_occ("sm_80", 256, 16, 100)["warps_by_shared_memory"] == (167936 // 256) * 8
    # sm_75, 96 threads, 16 registers: min(1024 // 96, 16) = 10 blocks x 3 warps = 30
    r = lib_occ("sm_75", 96, 16)
    assert (r["active_warps_per_sm"], r["limiter"]) == (30, "block_size")
    # sm_86, 32 threads: the 16-block limit binds at 16 warps of 48
    r = lib_occ("sm_86", 32, 0)
    assert (r["active_warps_per_sm"], r["limiter"]) == (16, "block_size")


def test_the_pages_tie_break():
    # no register or shared-memory demand: both limits equal the SM's warps, and
    # the page reports "registers" for the first limit that equals the result
    r = lib_occ("sm_80", 1024, 0, 0)
    assert (r["active_warps_per_sm"], r["limiter"]) == (64, "registers")
    r = lib_occ("sm_80", 1024, 64, 0)  # 32 warps by registers, 64 otherwise
    assert r["limiter"] == "registers"


def test_library_matches_the_oracle_on_random_inputs():
    rng = random.Random(21)
    for _ in range(2000):
        arch = rng.choice(sorted(orc.SPECS))
        max_threads = orc.SPECS[arch][0]
        threads = rng.randint(1, max_threads)
        regs = rng.choice([0, rng.randint(1, 255)])
        smem = rng.choice([0, rng.randint(1, orc.SPECS[arch][4])])
        want = orc.occupancy(arch, threads, regs, smem)
        got = lib_occ(arch, threads, regs, smem)
        for k, v in want.items():
            assert got[k] == v, (arch, threads, regs, smem, k)


def test_bad_arguments():
    with pytest.raises(ks.KsError):
        ks.gpu_limits("sm_12")
    with pytest.raises(ks.KsError):
        lib_occ("sm_75", 2048, 32)
    with pytest.raises(ks.KsError):
        lib_occ("sm_80", 0, 32)

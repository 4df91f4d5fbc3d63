"""GPU parity for the per-instruction profile behind the hints: the sm_103a
interpreter's counters (global coalescing efficiency, shared bank-conflict
degrees, divergent branches) against the same counters built from the
oracle's event list, byte for byte, through ks_simulate, ks_simulate_static
and ks_simulate_cached; and the hints that follow."""
import numpy as np
import pytest
import torch

import oracle
from oracle import hints as oh
import simt_ptx_interpretation_gb300 as ks
from simt_ptx_interpretation_gb300 import api
from simt_ptx_interpretation_gb300 import workloads as wl
from tests import test_hints as th

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def gpu():
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for -m gpu tests")
    from simt_ptx_interpretation_gb300 import _build
    _build.build_native()


WORKLOADS = {
    "vector_add": lambda: wl.vector_add(),
    "gather_s8": lambda: wl.gather(8, n_out=1 << 12),
    "divergent_k2": lambda: wl.divergent(2, n=1 << 11),
    "divergent_k32": lambda: wl.divergent(32, n=1 << 11),
    "fuzz3": lambda: wl.fuzz(3, grid=4, block=64),
    "fuzz7": lambda: wl.fuzz(7, grid=4, block=64),
    "smem_reduce": lambda: wl.smem_reduce(n=256 * 4, block=256),
    "fuzz_shared1": lambda: wl.fuzz_shared(1, grid=4, block=128),
    "fuzz_shared4": lambda: wl.fuzz_shared(4, grid=4, block=64),
}


def gpu_profile(w, how="plain"):
    mod = ks.Module(w.ptx)
    prof = torch.zeros(mod.profile_bytes(w.kernel), dtype=torch.uint8, device="cuda")
    dev = [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()]
    cfg = ks.Config(max_ts=w.max_ts, profile=prof)
    if how == "cached":
        r = ks.run(mod, w.kernel, w.grid, w.block, w.params, dev, config=cfg,
                   cache=ks.CacheConfig(max_accesses_per_warp=4096))
        status = r.totals.status
    else:
        st = torch.empty(ks.stats_bytes(w.grid, w.block), dtype=torch.uint8, device="cuda")
        f = ks.simulate_static if how == "static" else ks.simulate
        f(mod, w.kernel, w.grid, w.block, w.params, dev, st, None, cfg)
        status = ks.read_stats(st, w.warps).status
    torch.cuda.synchronize()
    assert status == 0
    return api.profile_array(prof)


def oracle_profile(w):
    r, e = oracle.run_events(w.ptx, w.kernel, w.grid, w.block, w.params,
                             [(b.sim_base, b.data) for b in w.fresh_buffers()])
    assert r.status == 0
    return oh.profile(e, len(oracle.ipdom(w.ptx, w.kernel))), e


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_profile_parity(name):
    w = WORKLOADS[name]()
    g = gpu_profile(w)
    o, e = oracle_profile(w)
    bad = np.nonzero(g.view(np.uint8).reshape(-1, 72) != o.view(np.uint8).reshape(-1, 72))[0]
    assert len(bad) == 0, f"profile differs at entries {np.unique(bad)[:5]}: gpu {g[bad[0]]} oracle {o[bad[0]]}"
    assert api.hints(g) == th.as_lib(oh.aggregate(e))


@pytest.mark.parametrize("how", ["static", "cached"])
@pytest.mark.parametrize("name", ["divergent_k2", "fuzz3", "smem_reduce"])
def test_profile_other_entry_points(name, how):
    w = WORKLOADS[name]()
    o, _ = oracle_profile(w)
    assert np.array_equal(gpu_profile(w, how).view(np.uint8), o.view(np.uint8))


@pytest.mark.parametrize("stride, message", [(4, None), (128, "32-way bank conflict"), (8, "2-way bank conflict")])
def test_page_bank_examples_on_gpu(stride, message):
    mod = ks.Module(th.BANKS)
    prof = torch.zeros(mod.profile_bytes("bk"), dtype=torch.uint8, device="cuda")
    r = ks.run(mod, "bk", 1, 32, wl.pack_params([("u32", stride)]), [], config=ks.Config(profile=prof))
    torch.cuda.synchronize()
    assert r.totals.status == 0
    got = [h["message"] for h in api.hints(prof)]
    assert got == ([message] if message else [])


def test_profile_too_small_is_refused():
    w = WORKLOADS["vector_add"]()
    mod = ks.Module(w.ptx)
    prof = torch.zeros(mod.profile_bytes(w.kernel) - 8, dtype=torch.uint8, device="cuda")
    dev = [(b.sim_base, torch.from_numpy(b.data.view(np.uint8)).cuda()) for b in w.fresh_buffers()]
    with pytest.raises(ks.KsError):
        ks.run(mod, w.kernel, w.grid, w.block, w.params, dev, config=ks.Config(profile=prof))


@pytest.mark.parametrize("block", [512, 1024])
def test_profile_large_blocks(block):
    w = wl.smem_reduce(n=block * 3, block=block)
    o, _ = oracle_profile(w)
    assert np.array_equal(gpu_profile(w).view(np.uint8), o.view(np.uint8))

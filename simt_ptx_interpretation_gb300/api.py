"""Python face of libks: argument marshalling around the C ABI only.

Device memory and streams come from PyTorch; every step of the simulation
runs in the library's sm_103a kernels.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass, field

import numpy as np
import torch

from . import _native

STATS_DTYPE = np.dtype(
    [("cycles", "<u8"), ("warp_insts", "<u8"), ("thread_insts", "<u8"), ("ld_req", "<u8"),
     ("ld_sectors", "<u8"), ("st_req", "<u8"), ("st_sectors", "<u8"), ("ld_lines", "<u8"),
     ("st_lines", "<u8"), ("status", "<i4"), ("max_stack_depth", "<u4"), ("sh_req", "<u8"),
     ("sh_wavefronts", "<u8")])
# ALU, FMA, ld.global, st.global, bra, div/sqrt, ret, ld.shared, st.shared,
# bar.sync, two reserved classes
DEFAULT_LAT = (4, 4, 400, 20, 8, 36, 1, 23, 23, 20, 0, 0)

ST_OOB, ST_MISALIGNED, ST_STEP_LIMIT, ST_SIMT_STACK, ST_TIMEOUT, ST_INJECTED = 1, 2, 3, 4, 5, 6
ST_CACHE_LOG, ST_CACHE_STREAM, ST_SCHED_LIMIT = 7, 8, 9

# SM issue model records (include/ks.h)
SCHED_WARP_DTYPE = np.dtype([("start", "<u8"), ("end", "<u8"), ("issued", "<u8"), ("not_selected", "<u8"),
                             ("stall_exec", "<u8"), ("stall_mem", "<u8"), ("stall_math", "<u8"),
                             ("stall_barrier", "<u8"), ("throttled", "<u8"), ("diverged", "<u8")])
SCHED_SM_DTYPE = np.dtype([("cycles", "<u8"), ("issued", "<u8"), ("ctas", "<u8"), ("status", "<i4"),
                           ("reserved", "<u4")])

# L1/L2 hit model: per-warp counts and logged accesses (include/ks.h)
CACHE_L1_HIT, CACHE_L2_HIT, CACHE_DRAM = 0, 1, 2
CACHE_WARP_DTYPE = np.dtype([("n_access", "<u4"), ("l1_hits", "<u4"), ("l2_hits", "<u4"), ("dram", "<u4")])
CACHE_ACCESS_DTYPE = np.dtype([("line", "<u8"), ("step", "<u4"), ("level", "<u4")])


class KsError(RuntimeError):
    def __init__(self, code: int, msg: str = ""):
        text = _native.lib().ks_status_string(code).decode()
        super().__init__(f"libks error {code} ({text}){': ' + msg if msg else ''}")
        self.code = code


def _check(rc: int, msg: str = ""):
    if rc != 0:
        raise KsError(rc, msg)


# ks_config.flags values of Config.layout (include/ks.h KS_FLAG_LAYOUT_*)
LAYOUT_FLAGS = {"auto": 0, "pair": 1, "split": 2}


@dataclass
class Config:
    lat: tuple = DEFAULT_LAT
    max_ts: int = 0
    stack_depth: int = 32
    step_limit: int = 1 << 26
    inject_warp: int = -1
    inject_step: int = 0
    profile: torch.Tensor | None = None  # uint8 cuda tensor of Module.profile_bytes(kernel), or None
    # register-file layout of the interpreter: "auto" (the library picks),
    # "pair" or "split" (KS_FLAG_LAYOUT_*); results are identical, speed differs
    layout: str = "auto"

    def to_c(self) -> _native.KsConfig:
        c = _native.KsConfig()
        _native.lib().ks_config_default(ctypes.byref(c))
        for i in range(12):
            c.lat[i] = self.lat[i] if i < len(self.lat) else 0
        c.max_ts_per_warp = self.max_ts
        c.simt_stack_depth = self.stack_depth
        c.step_limit = self.step_limit
        c.inject_warp = self.inject_warp
        c.inject_step = self.inject_step
        c.flags = LAYOUT_FLAGS[self.layout]
        if self.profile is not None:
            c.profile_buf = self.profile.data_ptr()
            c.profile_bytes = self.profile.numel() * self.profile.element_size()
        return c


@dataclass
class Totals:
    cycles_max: int
    cycles_sum: int
    warp_insts: int
    thread_insts: int
    ld_req: int
    ld_sectors: int
    st_req: int
    st_sectors: int
    ld_lines: int
    st_lines: int
    n_warps: int
    n_failed: int
    first_failed_warp: int
    status: int
    max_stack_depth: int
    sh_req: int = 0
    sh_wavefronts: int = 0


class Module:
    """A decoded PTX module (ks_load_module)."""

    def __init__(self, ptx: str):
        L = _native.lib()
        self._h = ctypes.c_void_p()
        err = ctypes.create_string_buffer(1024)
        data = ptx.encode()
        rc = L.ks_load_module(data, len(data), ctypes.byref(self._h), err, len(err))
        _check(rc, err.value.decode(errors="replace"))

    def close(self):
        if self._h:
            _native.lib().ks_free_module(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def handle(self):
        return self._h

    def info(self, kernel: str) -> dict:
        v = [ctypes.c_uint32() for _ in range(5)]
        _check(_native.lib().ks_kernel_info(self._h, kernel.encode(), *[ctypes.byref(x) for x in v]))
        return dict(zip(("n_params", "param_bytes", "n_events", "n_insns", "n_reg_slots"), (x.value for x in v)))

    def params(self, kernel: str) -> list[tuple[str, int, int]]:
        out = []
        for i in range(self.info(kernel)["n_params"]):
            off, size, name = ctypes.c_uint32(), ctypes.c_uint32(), ctypes.c_char_p()
            _check(_native.lib().ks_kernel_param(self._h, kernel.encode(), i, ctypes.byref(off), ctypes.byref(size),
                                                 ctypes.byref(name)))
            out.append((name.value.decode(), off.value, size.value))
        return out

    def record_bytes(self, kernel: str) -> int:
        """Trace record size of the kernel's slots: 4, 8 or 16 bytes."""
        b = ctypes.c_uint32()
        _check(_native.lib().ks_kernel_record_bytes(self._h, kernel.encode(), ctypes.byref(b)))
        return b.value

    def profile_bytes(self, kernel: str) -> int:
        """Bytes of the kernel's per-instruction profile (ks_profile_bytes)."""
        n = ctypes.c_size_t()
        _check(_native.lib().ks_profile_bytes(self._h, kernel.encode(), ctypes.byref(n)))
        return n.value

    def event_payload(self, kernel: str, event_id: int) -> int:
        """Payload bytes of an event: 0, 4 or 8."""
        b = ctypes.c_uint32()
        _check(_native.lib().ks_kernel_event_payload(self._h, kernel.encode(), event_id, ctypes.byref(b)))
        return b.value

    def events(self, kernel: str) -> list[tuple[int, str]]:
        out = []
        for i in range(self.info(kernel)["n_events"]):
            kind, name = ctypes.c_uint32(), ctypes.c_char_p()
            _check(_native.lib().ks_kernel_event(self._h, kernel.encode(), i, ctypes.byref(kind), ctypes.byref(name)))
            out.append((kind.value, name.value.decode()))
        return out

    def ipdom(self, kernel: str) -> list[int]:
        n = self.info(kernel)["n_insns"]
        arr = (ctypes.c_int32 * max(1, n))()
        cnt = ctypes.c_uint32()
        _check(_native.lib().ks_kernel_ipdom(self._h, kernel.encode(), arr, n, ctypes.byref(cnt)))
        return [arr[i] for i in range(cnt.value)]

    def fast_runs(self, kernel: str) -> list[tuple[int, bool, int]]:
        """Per program entry: (ops from it to the end of its fast-loop run,
        0 outside one; whether every one of them writes a row it reads; how
        many of them keep reading its b and c rows), PAIR layout."""
        n = self.info(kernel)["n_insns"]
        arr = (ctypes.c_uint32 * max(1, 3 * n))()
        cnt = ctypes.c_uint32()
        _check(_native.lib().ks_kernel_fast_runs(self._h, kernel.encode(), arr, n, ctypes.byref(cnt)))
        return [(arr[3 * i], bool(arr[3 * i + 1]), arr[3 * i + 2]) for i in range(cnt.value)]

    def layout(self, kernel: str, layout: str = "auto") -> tuple[str, int]:
        """The register-file layout a launch with Config(layout=layout) runs
        in ("pair" or "split") and the shared memory per simulated warp."""
        split, region = ctypes.c_uint32(), ctypes.c_uint32()
        _check(_native.lib().ks_kernel_layout(self._h, kernel.encode(), LAYOUT_FLAGS[layout], ctypes.byref(split),
                                              ctypes.byref(region)))
        return ("split" if split.value else "pair"), int(region.value)


def stats_bytes(grid: int, block: int) -> int:
    return int(_native.lib().ks_stats_bytes(grid, block))


def trace_to_json(module: "Module", kernel: str, grid: int, block: int, max_ts: int, trace, cycles_per_us: float) -> str:
    """Chrome trace-event JSON (Perfetto) of a launch's trace slots
    (ks_trace_to_json); `trace` is a host numpy uint8 array or a tensor."""
    data = trace.cpu().numpy() if isinstance(trace, torch.Tensor) else np.ascontiguousarray(trace)
    need = ctypes.c_size_t(0)
    L = _native.lib()
    rc = L.ks_trace_to_json(module._h, kernel.encode(), grid, block, max_ts, data.ctypes.data, data.nbytes,
                            cycles_per_us, None, 0, ctypes.byref(need))
    if rc not in (0, -3) or need.value == 0:
        _check(rc)
    buf = ctypes.create_string_buffer(need.value + 1)
    _check(L.ks_trace_to_json(module._h, kernel.encode(), grid, block, max_ts, data.ctypes.data, data.nbytes,
                              cycles_per_us, buf, len(buf), ctypes.byref(need)))
    return buf.value.decode()


LIMITERS = ("registers", "shared_memory", "block_size")

# per-instruction profile record (ks_pc_profile)
PROFILE_DTYPE = np.dtype([
    ("requests", "<u8"), ("poor", "<u8"), ("uncoalesced", "<u8"), ("conflicted", "<u8"), ("severe", "<u8"),
    ("divergent", "<u8"), ("high_divergence", "<u8"), ("degrees", "<u4"), ("poor_pcts", "<u4"),
    ("high_div_pcts", "<u8")])
HINT_SEVERITIES = ("info", "warning", "critical")
HINT_CATEGORIES = ("memory", "divergence", "occupancy", "registers")


def profile_array(profile) -> np.ndarray:
    """A profile buffer (tensor or uint8 array) as PROFILE_DTYPE records."""
    data = profile.cpu().numpy() if isinstance(profile, torch.Tensor) else np.ascontiguousarray(profile)
    return data.view(np.uint8).view(PROFILE_DTYPE)


def hints(profile, occupancy_result: dict | None = None) -> list[dict]:
    """The page's performance hints from a launch's per-instruction profile
    (ks_hints); occupancy_result as returned by occupancy()."""
    prof = np.ascontiguousarray(profile_array(profile))
    occ = None
    if occupancy_result is not None:
        occ = _native.KsOccupancy()
        for f, _ in _native.KsOccupancy._fields_:
            v = occupancy_result[f] if f != "limiter" else LIMITERS.index(occupancy_result["limiter"])
            setattr(occ, f, v)
    L = _native.lib()
    n = ctypes.c_uint32(0)
    rc = L.ks_hints(prof.ctypes.data if len(prof) else None, len(prof), ctypes.byref(occ) if occ else None, None, 0,
                    ctypes.byref(n))
    if rc not in (0, -3):
        _check(rc)
    out = (_native.KsHint * max(1, n.value))()
    _check(L.ks_hints(prof.ctypes.data if len(prof) else None, len(prof), ctypes.byref(occ) if occ else None, out,
                      n.value, ctypes.byref(n)))
    return [dict(category=HINT_CATEGORIES[h.category], severity=HINT_SEVERITIES[h.severity], pc=h.pc,
                 count=h.count, message=h.message.decode(), detail=h.detail.decode()) for h in out[:n.value]]


def gpu_limits(arch: str) -> dict:
    """Per-SM limits of an architecture (ks_gpu_limits_of)."""
    g = _native.KsGpuLimits()
    _check(_native.lib().ks_gpu_limits_of(arch.encode(), ctypes.byref(g)))
    return {f: getattr(g, f) for f, _ in _native.KsGpuLimits._fields_}


def occupancy(limits: dict, threads_per_block: int, registers_per_thread: int, shared_memory_per_block: int = 0) -> dict:
    """Resident warps per SM and the limiting resource (ks_occupancy)."""
    g = _native.KsGpuLimits(**limits)
    r = _native.KsOccupancy()
    _check(_native.lib().ks_occupancy(ctypes.byref(g), threads_per_block, registers_per_thread,
                                      shared_memory_per_block, ctypes.byref(r)))
    out = {f: getattr(r, f) for f, _ in _native.KsOccupancy._fields_}
    out["limiter"] = LIMITERS[out["limiter"]]
    return out


def trace_bytes(grid: int, block: int, max_ts: int, record_bytes: int = 4) -> int:
    if record_bytes == 4:
        return int(_native.lib().ks_trace_bytes(grid, block, max_ts))
    return int(_native.lib().ks_trace_bytes_records(grid, block, max_ts, record_bytes))


def _stream_handle(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def simulate(module: Module, kernel: str, grid: int, block: int, params: bytes, buffers, stats: torch.Tensor,
             trace: torch.Tensor | None = None, config: Config | None = None, stream=None) -> None:
    """Enqueues one simulation (ks_simulate). buffers: [(sim_base, cuda tensor)];
    stats / trace: uint8 cuda tensors of stats_bytes / trace_bytes."""
    bufs = (_native.KsBuffer * max(1, len(buffers)))()
    for i, (base, t) in enumerate(buffers):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("buffers must be contiguous CUDA tensors")
        bufs[i].sim_base = base
        bufs[i].dev_ptr = t.data_ptr()
        bufs[i].bytes = t.numel() * t.element_size()
    cfg = (config or Config()).to_c()
    pbuf = ctypes.create_string_buffer(bytes(params), max(1, len(params)))
    rc = _native.lib().ks_simulate(
        module.handle, kernel.encode(), grid, block, ctypes.cast(pbuf, ctypes.c_void_p), len(params), bufs,
        len(buffers), trace.data_ptr() if trace is not None else None,
        trace.numel() if trace is not None else 0, stats.data_ptr(), stats.numel(), ctypes.byref(cfg),
        _stream_handle(stream))
    _check(rc)


@dataclass
class BatchItem:
    """One launch of simulate_batch: simulate()'s arguments."""
    module: Module
    kernel: str
    grid: int
    block: int
    params: bytes
    buffers: list
    stats: torch.Tensor
    trace: torch.Tensor | None = None
    config: Config | None = None


def _fill_batch_item(a, it: BatchItem, keep: list) -> None:
    """Marshals one BatchItem into a ks_batch_item (the ctypes objects it
    points to go to `keep`)."""
    bufs = (_native.KsBuffer * max(1, len(it.buffers)))()
    for i, (base, t) in enumerate(it.buffers):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("buffers must be contiguous CUDA tensors")
        bufs[i].sim_base = base
        bufs[i].dev_ptr = t.data_ptr()
        bufs[i].bytes = t.numel() * t.element_size()
    cfg = (it.config or Config()).to_c()
    name = it.kernel.encode()
    pbuf = ctypes.create_string_buffer(bytes(it.params), max(1, len(it.params)))
    keep += [bufs, cfg, name, pbuf]
    a.mod = it.module.handle
    a.kernel = name
    a.grid, a.block = it.grid, it.block
    a.params = ctypes.cast(pbuf, ctypes.c_void_p)
    a.param_bytes = len(it.params)
    a.bufs = bufs
    a.n_bufs = len(it.buffers)
    a.trace_buf = it.trace.data_ptr() if it.trace is not None else None
    a.trace_bytes = it.trace.numel() if it.trace is not None else 0
    a.stats_buf = it.stats.data_ptr()
    a.stats_bytes = it.stats.numel()
    a.cfg = ctypes.pointer(cfg)


def simulate_batch(items, stream=None) -> int:
    """Enqueues several simulations as ks_simulate_batch (real grids of items
    of one kernel form); returns the number of real kernel launches. items:
    BatchItem list. On a refused item, KsError names it; nothing was
    launched."""
    items = list(items)
    arr = (_native.KsBatchItem * max(1, len(items)))()
    keep = []  # ctypes objects the C call reads
    for k, it in enumerate(items):
        _fill_batch_item(arr[k], it, keep)
    failed, launched = ctypes.c_uint32(0), ctypes.c_uint32(0)
    rc = _native.lib().ks_simulate_batch(arr, len(items), _stream_handle(stream), ctypes.byref(failed),
                                         ctypes.byref(launched))
    _check(rc, f"batch item {failed.value}" if failed.value < len(items) else "")
    return launched.value


def simulate_static(module: Module, kernel: str, grid: int, block: int, params: bytes, buffers, stats: torch.Tensor,
                    trace: torch.Tensor | None = None, config: Config | None = None, stream=None) -> None:
    """ks_simulate_static: like simulate(), but the library allocates no device
    memory (the program image goes to one fixed-size static device array shared
    by all calls; calls that overlap on the GPU race)."""
    bufs = (_native.KsBuffer * max(1, len(buffers)))()
    for i, (base, t) in enumerate(buffers):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("buffers must be contiguous CUDA tensors")
        bufs[i].sim_base = base
        bufs[i].dev_ptr = t.data_ptr()
        bufs[i].bytes = t.numel() * t.element_size()
    cfg = (config or Config()).to_c()
    pbuf = ctypes.create_string_buffer(bytes(params), max(1, len(params)))
    rc = _native.lib().ks_simulate_static(
        module.handle, kernel.encode(), grid, block, ctypes.cast(pbuf, ctypes.c_void_p), len(params), bufs,
        len(buffers), trace.data_ptr() if trace is not None else None,
        trace.numel() if trace is not None else 0, stats.data_ptr(), stats.numel(), ctypes.byref(cfg),
        _stream_handle(stream))
    _check(rc)


@dataclass
class CacheConfig:
    """The L1/L2 hit model's parameters (ks_cache_config)."""
    l1_lines: int = 1024
    l2_lines: int = 49152
    lat_l1: int = 28
    lat_l2: int = 150
    max_accesses_per_warp: int = 1024
    # 0: the second pass interprets again; > 0: a timing replay over a log of
    # this many issued runs per warp (kernels without shared memory / bar.sync)
    max_runs_per_warp: int = 0

    def to_c(self) -> _native.KsCacheConfig:
        c = _native.KsCacheConfig()
        _native.lib().ks_cache_config_default(ctypes.byref(c))
        c.l1_lines, c.l2_lines = self.l1_lines, self.l2_lines
        c.lat_l1, c.lat_l2 = self.lat_l1, self.lat_l2
        c.max_accesses_per_warp = self.max_accesses_per_warp
        c.max_runs_per_warp = self.max_runs_per_warp
        return c


@dataclass
class SchedConfig:
    """The SM issue model's parameters (ks_sched_config)."""
    n_sm: int = 152
    ctas_per_sm: int = 0
    schedulers_per_sm: int = 4
    max_runs_per_warp: int = 4096

    def to_c(self) -> _native.KsSchedConfig:
        c = _native.KsSchedConfig()
        _native.lib().ks_sched_config_default(ctypes.byref(c))
        c.n_sm, c.ctas_per_sm = self.n_sm, self.ctas_per_sm
        c.schedulers_per_sm, c.max_runs_per_warp = self.schedulers_per_sm, self.max_runs_per_warp
        return c


def sched_workspace_bytes(grid: int, block: int, sched: SchedConfig | None = None) -> int:
    sc = (sched or SchedConfig()).to_c()
    return int(_native.lib().ks_sched_workspace_bytes(grid, block, ctypes.byref(sc)))


def simulate_sched(module: Module, kernel: str, grid: int, block: int, params: bytes, buffers, stats: torch.Tensor,
                   sched_warps: torch.Tensor, sched_sms: torch.Tensor, workspace: torch.Tensor,
                   trace: torch.Tensor | None = None, config: Config | None = None,
                   sched: SchedConfig | None = None, stream=None) -> None:
    """ks_simulate_sched: simulate() plus the SM issue model; sched_warps /
    sched_sms / workspace are uint8 cuda tensors (80 B per warp, 32 B per SM,
    sched_workspace_bytes)."""
    bufs = (_native.KsBuffer * max(1, len(buffers)))()
    for i, (base, t) in enumerate(buffers):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("buffers must be contiguous CUDA tensors")
        bufs[i].sim_base = base
        bufs[i].dev_ptr = t.data_ptr()
        bufs[i].bytes = t.numel() * t.element_size()
    cfg = (config or Config()).to_c()
    sc = (sched or SchedConfig()).to_c()
    pbuf = ctypes.create_string_buffer(bytes(params), max(1, len(params)))
    rc = _native.lib().ks_simulate_sched(
        module.handle, kernel.encode(), grid, block, ctypes.cast(pbuf, ctypes.c_void_p), len(params), bufs,
        len(buffers), trace.data_ptr() if trace is not None else None,
        trace.numel() if trace is not None else 0, stats.data_ptr(), stats.numel(), ctypes.byref(cfg),
        ctypes.byref(sc), sched_warps.data_ptr(), sched_warps.numel(), sched_sms.data_ptr(), sched_sms.numel(),
        workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    _check(rc)


def cache_workspace_bytes(grid: int, block: int, cache: CacheConfig | None = None) -> int:
    """Device workspace of simulate_cached (0 when the configuration is invalid)."""
    cc = (cache or CacheConfig()).to_c()
    return int(_native.lib().ks_cache_workspace_bytes(grid, block, ctypes.byref(cc)))


def simulate_cached(module: Module, kernel: str, grid: int, block: int, params: bytes, buffers, stats: torch.Tensor,
                    workspace: torch.Tensor, trace: torch.Tensor | None = None, config: Config | None = None,
                    cache: CacheConfig | None = None, stream=None) -> None:
    """ks_simulate_cached: simulate() with the L1/L2 hit model; `workspace` is
    a uint8 cuda tensor of cache_workspace_bytes(grid, block, cache)."""
    bufs = (_native.KsBuffer * max(1, len(buffers)))()
    for i, (base, t) in enumerate(buffers):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("buffers must be contiguous CUDA tensors")
        bufs[i].sim_base = base
        bufs[i].dev_ptr = t.data_ptr()
        bufs[i].bytes = t.numel() * t.element_size()
    cfg = (config or Config()).to_c()
    cc = (cache or CacheConfig()).to_c()
    pbuf = ctypes.create_string_buffer(bytes(params), max(1, len(params)))
    rc = _native.lib().ks_simulate_cached(
        module.handle, kernel.encode(), grid, block, ctypes.cast(pbuf, ctypes.c_void_p), len(params), bufs,
        len(buffers), trace.data_ptr() if trace is not None else None,
        trace.numel() if trace is not None else 0, stats.data_ptr(), stats.numel(), ctypes.byref(cfg),
        ctypes.byref(cc), workspace.data_ptr(), workspace.numel(), _stream_handle(stream))
    _check(rc)



@dataclass
class CachedBatchItem:
    """One launch of simulate_cached_batch: a BatchItem, its hit model (None:
    the defaults) and its workspace (uint8 cuda tensor of
    cache_workspace_bytes)."""
    item: BatchItem
    cache: "CacheConfig | None"
    workspace: torch.Tensor


def simulate_cached_batch(items, stream=None) -> int:
    """ks_simulate_cached_batch: several cached simulations, their passes
    batched; returns the launches of the library's own kernels. items:
    CachedBatchItem list. On a refused item, KsError names it; nothing was
    launched."""
    items = list(items)
    arr = (_native.KsCachedItem * max(1, len(items)))()
    keep = []
    for k, it in enumerate(items):
        _fill_batch_item(arr[k].sim, it.item, keep)
        cc = (it.cache or CacheConfig()).to_c()
        keep.append(cc)
        arr[k].cache = ctypes.pointer(cc)
        arr[k].workspace = it.workspace.data_ptr()
        arr[k].workspace_bytes = it.workspace.numel()
    failed, launched = ctypes.c_uint32(0), ctypes.c_uint32(0)
    rc = _native.lib().ks_simulate_cached_batch(arr, len(items), _stream_handle(stream), ctypes.byref(failed),
                                                ctypes.byref(launched))
    _check(rc, f"batch item {failed.value}" if failed.value < len(items) else "")
    return launched.value

def cache_results(workspace: torch.Tensor, n_warps: int, cache: CacheConfig | None = None):
    """(per-warp counts, access log of shape (W, max_accesses_per_warp)) as numpy
    arrays, copied from a simulate_cached workspace."""
    cache = cache or CacheConfig()
    cap = cache.max_accesses_per_warp
    log_off = (n_warps * 16 + 255) // 256 * 256
    warps = workspace[:n_warps * 16].cpu().numpy().view(CACHE_WARP_DTYPE)
    log = workspace[log_off:log_off + n_warps * cap * 16].cpu().numpy().view(CACHE_ACCESS_DTYPE)
    return warps, log.reshape(n_warps, cap)


def read_stats(stats: torch.Tensor, n_warps: int, stream=None) -> Totals:
    """Launch totals (ks_read_stats); waits for the stream."""
    t = _native.KsTotals()
    _check(_native.lib().ks_read_stats(stats.data_ptr(), n_warps, _stream_handle(stream), ctypes.byref(t)))
    return Totals(**{f: getattr(t, f) for f, _ in _native.KsTotals._fields_})


def stats_array(stats: torch.Tensor) -> np.ndarray:
    """Per-warp records as a numpy structured array (copies to the host)."""
    return stats.cpu().numpy().view(STATS_DTYPE)


@dataclass
class Run:
    stats: torch.Tensor
    trace: torch.Tensor | None
    totals: Totals
    buffers: list = field(default_factory=list)
    cache_warps: np.ndarray | None = None  # CACHE_WARP_DTYPE per warp (cache model only)
    cache_log: np.ndarray | None = None    # CACHE_ACCESS_DTYPE, (W, max_accesses_per_warp)
    sched_warps: np.ndarray | None = None  # SCHED_WARP_DTYPE per warp (SM issue model only)
    sched_sms: np.ndarray | None = None    # SCHED_SM_DTYPE per SM


def run(module: Module, kernel: str, grid: int, block: int, params: bytes, buffers, config: Config | None = None,
        trace: bool = False, stream=None, cache: CacheConfig | None = None, sched: SchedConfig | None = None) -> Run:
    """Allocates the outputs, simulates (with the L1/L2 hit model when `cache`
    is given, with the SM issue model when `sched` is), and reduces the totals."""
    config = config or Config()
    dev = buffers[0][1].device if buffers else torch.device("cuda")
    st = torch.empty(stats_bytes(grid, block), dtype=torch.uint8, device=dev)
    tr = (torch.empty(trace_bytes(grid, block, config.max_ts, module.record_bytes(kernel)), dtype=torch.uint8, device=dev)
          if trace else None)
    n = grid * ((block + 31) // 32)
    if cache is not None and sched is not None:
        raise ValueError("the cache model and the SM issue model run separately")
    if sched is not None:
        sw = torch.empty(n * SCHED_WARP_DTYPE.itemsize, dtype=torch.uint8, device=dev)
        ss = torch.empty(sched.n_sm * 32, dtype=torch.uint8, device=dev)
        ws = torch.empty(max(1, sched_workspace_bytes(grid, block, sched)), dtype=torch.uint8, device=dev)
        simulate_sched(module, kernel, grid, block, params, buffers, st, sw, ss, ws, tr, config, sched, stream)
        totals = read_stats(st, n, stream)
        return Run(st, tr, totals, list(buffers), sched_warps=sw.cpu().numpy().view(SCHED_WARP_DTYPE),
                   sched_sms=ss.cpu().numpy().view(SCHED_SM_DTYPE))
    if cache is None:
        simulate(module, kernel, grid, block, params, buffers, st, tr, config, stream)
        return Run(st, tr, read_stats(st, n, stream), list(buffers))
    nbytes = cache_workspace_bytes(grid, block, cache)
    if nbytes == 0:
        raise KsError(-3, "invalid cache configuration")
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    simulate_cached(module, kernel, grid, block, params, buffers, st, ws, tr, config, cache, stream)
    totals = read_stats(st, n, stream)
    warps, log = cache_results(ws, n, cache)
    return Run(st, tr, totals, list(buffers), warps, log)

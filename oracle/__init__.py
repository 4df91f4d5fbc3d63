"""CPU oracle for the warp-level SIMT PTX interpreter — TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline /
``--impl reference`` legs may import this package. The product path never
does: it shares no code with the GPU interpreter (own parser, own
post-dominator sets, own per-lane semantics in ``ks_oracle.cpp``).

Parity status per function (pins live in ``tests/test_oracle_*.py``):
  * f32 add/sub/mul/fma/div/sqrt, int<->float cvt, integer ops, setp/selp —
    pinned against exact rational / big-integer arithmetic written in the
    tests, and against the hardware through the driver-JIT cross-check.
  * SIMT masking and reconvergence — pinned by per-thread mode (memory image),
    by the divergent workload's closed-form instruction counts and by
    hand-drawn CFGs whose post-dominators are brute-forced in the tests.
  * in-order scoreboard — pinned by closed forms (dependent chain 4N,
    k independent accumulators N+3, loop periods 141/48/16) and hand-derived
    cycle counts of vector_add.
  * sectors / lines — pinned by the coalescing examples of the KernelScope
    page and the strided closed form min(32, 4s).
  * trace slots — pinned by hand-derived vector_add records and the IKET slot
    size formula.
  * L1/L2 hit model (run_cached) — pinned by hand-derived hit sequences and
    cycle counts (reuse, L1-only and L1+L2 set conflicts, step order between
    warps, the lowest executing lane, stores installing lines, barrier
    release steps) and by a per-access replay of the pages' direct-mapped
    cache over the access stream in (step, warp) order.
  * cycles, sectors and traces of random (fuzz) programs beyond these rules:
    parity unpinned (oracle-vs-GPU agreement only).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ks_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

MODE_WARP = 0
MODE_PER_THREAD = 1
RACE_CROSS_THREAD = 1  # two threads touch one word, at least one writing
# ALU, FMA, ld.global, st.global, bra, div/sqrt, ret, ld.shared, st.shared,
# bar.sync, two reserved classes
DEFAULT_LAT = (4, 4, 400, 20, 8, 36, 1, 23, 23, 20, 0, 0)

STATS_DTYPE = np.dtype(
    [
        ("cycles", "<u8"),
        ("warp_insts", "<u8"),
        ("thread_insts", "<u8"),
        ("ld_req", "<u8"),
        ("ld_sectors", "<u8"),
        ("st_req", "<u8"),
        ("st_sectors", "<u8"),
        ("ld_lines", "<u8"),
        ("st_lines", "<u8"),
        ("status", "<i4"),
        ("max_stack_depth", "<u4"),
        ("sh_req", "<u8"),
        ("sh_wavefronts", "<u8"),
    ]
)
assert STATS_DTYPE.itemsize == 96


class _Buffer(ctypes.Structure):
    _fields_ = [("sim_base", ctypes.c_uint64), ("host", ctypes.c_void_p), ("bytes", ctypes.c_uint64)]


class _Config(ctypes.Structure):
    _fields_ = [
        ("lat", ctypes.c_uint32 * 12),
        ("max_ts_per_warp", ctypes.c_uint32),
        ("stack_depth", ctypes.c_uint32),
        ("step_limit", ctypes.c_uint64),
        ("inject_warp", ctypes.c_int64),
        ("inject_step", ctypes.c_uint64),
        ("mode", ctypes.c_uint32),
        ("threads", ctypes.c_uint32),
        ("race_check", ctypes.c_uint32),
        ("n_warp_list", ctypes.c_uint32),
        ("warp_list", ctypes.POINTER(ctypes.c_uint32)),
    ]


class _Cache(ctypes.Structure):
    _fields_ = [
        ("l1_lines", ctypes.c_uint32),
        ("l2_lines", ctypes.c_uint32),
        ("lat_l1", ctypes.c_uint32),
        ("lat_l2", ctypes.c_uint32),
        ("log_cap", ctypes.c_uint32),
        ("warps", ctypes.c_void_p),
        ("log", ctypes.c_void_p),
    ]


# L1/L2 hit model outputs: per-warp counts and the access log (line, step, level)
CACHE_L1_HIT, CACHE_L2_HIT, CACHE_DRAM = 0, 1, 2
CACHE_WARP_DTYPE = np.dtype([("n_access", "<u4"), ("l1_hits", "<u4"), ("l2_hits", "<u4"), ("dram", "<u4")])
CACHE_ACCESS_DTYPE = np.dtype([("line", "<u8"), ("step", "<u4"), ("level", "<u4")])


class OracleError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"oracle error {code}: {msg}")
        self.code = code


def build(force: bool = False) -> str:
    """Compiles the oracle with g++ (-ffp-contract=off, no fast-math)."""
    with _lock:
        if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
            return _LIB
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
               "-pthread", "-o", tmp, _SRC]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
        return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.orc_run.restype = ctypes.c_int
        lib.orc_run.argtypes = [
            ctypes.c_char_p, ctypes.c_char_p, ctypes.c_uint32, ctypes.c_uint32,
            ctypes.c_void_p, ctypes.c_uint64, ctypes.POINTER(_Buffer), ctypes.c_uint32,
            ctypes.POINTER(_Config), ctypes.c_void_p, ctypes.c_void_p,
            ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_uint32),
            ctypes.c_char_p, ctypes.c_uint64,
        ]
        lib.orc_run_cached.restype = ctypes.c_int
        lib.orc_run_cached.argtypes = [
            ctypes.c_char_p, ctypes.c_char_p, ctypes.c_uint32, ctypes.c_uint32,
            ctypes.c_void_p, ctypes.c_uint64, ctypes.POINTER(_Buffer), ctypes.c_uint32,
            ctypes.POINTER(_Config), ctypes.POINTER(_Cache), ctypes.c_void_p, ctypes.c_void_p,
            ctypes.POINTER(ctypes.c_int32), ctypes.c_char_p, ctypes.c_uint64,
        ]
        lib.orc_run_events.restype = ctypes.c_int
        lib.orc_run_events.argtypes = [
            ctypes.c_char_p, ctypes.c_char_p, ctypes.c_uint32, ctypes.c_uint32,
            ctypes.c_void_p, ctypes.c_uint64, ctypes.POINTER(_Buffer), ctypes.c_uint32,
            ctypes.POINTER(_Config), ctypes.c_void_p, ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32),
            ctypes.c_void_p, ctypes.c_uint64, ctypes.POINTER(ctypes.c_uint64), ctypes.c_char_p, ctypes.c_uint64,
        ]
        lib.orc_run_sched.restype = ctypes.c_int
        lib.orc_run_sched.argtypes = [
            ctypes.c_char_p, ctypes.c_char_p, ctypes.c_uint32, ctypes.c_uint32,
            ctypes.c_void_p, ctypes.c_uint64, ctypes.POINTER(_Buffer), ctypes.c_uint32,
            ctypes.POINTER(_Config), ctypes.POINTER(ctypes.c_uint32 * 3), ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_char_p, ctypes.c_uint64,
        ]
        lib.orc_ipdom.restype = ctypes.c_int
        lib.orc_ipdom.argtypes = [ctypes.c_char_p, ctypes.c_char_p, ctypes.POINTER(ctypes.c_int32),
                                  ctypes.c_uint32, ctypes.POINTER(ctypes.c_uint32), ctypes.c_char_p,
                                  ctypes.c_uint64]
        lib.orc_params.restype = ctypes.c_int
        lib.orc_params.argtypes = [ctypes.c_char_p, ctypes.c_char_p, ctypes.POINTER(ctypes.c_uint32),
                                   ctypes.POINTER(ctypes.c_uint32), ctypes.c_uint32,
                                   ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint32),
                                   ctypes.c_char_p, ctypes.c_uint64]
        lib.orc_event_info.restype = ctypes.c_int
        lib.orc_event_info.argtypes = [ctypes.c_char_p, ctypes.c_char_p, ctypes.c_uint32,
                                       ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint32),
                                       ctypes.c_char_p, ctypes.c_uint64, ctypes.c_char_p, ctypes.c_uint64]
        lib.orc_record_bytes.restype = ctypes.c_int
        lib.orc_record_bytes.argtypes = [ctypes.c_char_p, ctypes.c_char_p, ctypes.POINTER(ctypes.c_uint32),
                                         ctypes.c_char_p, ctypes.c_uint64]
        lib.orc_events.restype = ctypes.c_int
        lib.orc_events.argtypes = [ctypes.c_char_p, ctypes.c_char_p, ctypes.POINTER(ctypes.c_uint32),
                                   ctypes.c_uint32, ctypes.POINTER(ctypes.c_uint32), ctypes.c_char_p,
                                   ctypes.c_uint64]
        _lib = lib
    return _lib


def slot_bytes(max_ts: int, record_bytes: int = 4) -> int:
    return (16 + record_bytes * max_ts + 7) // 8 * 8


@dataclass
class Result:
    stats: np.ndarray      # STATS_DTYPE, one record per warp of the grid
    trace: np.ndarray | None  # uint8, W * slot_bytes(max_ts, record_bytes)
    status: int
    race_flags: int


def run(ptx: str, kernel: str, grid: int, block: int, params: bytes, buffers, *,
        lat=DEFAULT_LAT, max_ts: int = 0, trace: bool = False, stack_depth: int = 32,
        step_limit: int = 1 << 26, inject_warp: int = -1, inject_step: int = 0,
        mode: int = MODE_WARP, threads: int = 0, race_check: bool = False, warps=None) -> Result:
    """Interprets `kernel` on the CPU.

    buffers: sequence of (sim_base, numpy array); arrays must be C-contiguous
    and are updated in place with the simulated stores.
    warps: optional list of global warp ids to run (the others are skipped).
    """
    lib = _load()
    wpc = (block + 31) // 32
    W = grid * wpc
    bufs = (_Buffer * max(1, len(buffers)))()
    keep = []
    for i, (base, arr) in enumerate(buffers):
        if not arr.flags["C_CONTIGUOUS"]:
            raise ValueError("buffer arrays must be C-contiguous")
        keep.append(arr)
        bufs[i].sim_base = base
        bufs[i].host = arr.ctypes.data
        bufs[i].bytes = arr.nbytes
    cfg = _Config()
    for i in range(12):
        cfg.lat[i] = lat[i] if i < len(lat) else 0
    cfg.max_ts_per_warp = max_ts
    cfg.stack_depth = stack_depth
    cfg.step_limit = step_limit
    cfg.inject_warp = inject_warp
    cfg.inject_step = inject_step
    cfg.mode = mode
    cfg.threads = threads
    cfg.race_check = 1 if race_check else 0
    wl = None
    if warps is not None:
        wl = np.ascontiguousarray(np.asarray(warps, dtype=np.uint32))
        cfg.n_warp_list = len(wl)
        cfg.warp_list = wl.ctypes.data_as(ctypes.POINTER(ctypes.c_uint32))
    stats = np.zeros(W, dtype=STATS_DTYPE)
    tr = np.zeros(W * slot_bytes(max_ts, record_bytes(ptx, kernel)), dtype=np.uint8) if trace else None
    pbuf = ctypes.create_string_buffer(bytes(params), max(1, len(params)))
    status = ctypes.c_int32(0)
    race = ctypes.c_uint32(0)
    err = ctypes.create_string_buffer(512)
    rc = lib.orc_run(ptx.encode(), kernel.encode(), grid, block, ctypes.cast(pbuf, ctypes.c_void_p),
                     len(params), bufs, len(buffers), ctypes.byref(cfg), stats.ctypes.data,
                     tr.ctypes.data if tr is not None else None, ctypes.byref(status),
                     ctypes.byref(race), err, len(err))
    if rc != 0:
        raise OracleError(rc, err.value.decode(errors="replace"))
    return Result(stats=stats, trace=tr, status=status.value, race_flags=race.value)


# events the page's hints analyzer reads (orc_run_events)
EV_GLOBAL, EV_SHARED, EV_DIVERGE = 0, 1, 2
HINT_EVENT_DTYPE = np.dtype([("pc", "<u4"), ("kind", "<u4"), ("a", "<u4"), ("b", "<u4"), ("c", "<u4"),
                             ("pad", "<u4")])


def run_events(ptx: str, kernel: str, grid: int, block: int, params: bytes, buffers, *, lat=DEFAULT_LAT,
               step_limit: int = 1 << 26):
    """orc_run on one host thread that also returns the hint events in run
    order (HINT_EVENT_DTYPE): global requests (a lanes, b lines, c bytes),
    shared requests (a degree), divergent branches (a taken, b fall-through)."""
    lib = _load()
    W = grid * ((block + 31) // 32)
    bufs = (_Buffer * max(1, len(buffers)))()
    keep = []
    for i, (base, arr) in enumerate(buffers):
        keep.append(arr)
        bufs[i].sim_base = base
        bufs[i].host = arr.ctypes.data
        bufs[i].bytes = arr.nbytes
    cfg = _Config()
    for i in range(12):
        cfg.lat[i] = lat[i] if i < len(lat) else 0
    cfg.stack_depth = 32
    cfg.step_limit = step_limit
    cfg.inject_warp = -1
    cfg.mode = MODE_WARP
    stats = np.zeros(W, dtype=STATS_DTYPE)
    pbuf = ctypes.create_string_buffer(bytes(params), max(1, len(params)))
    status = ctypes.c_int32(0)
    n = ctypes.c_uint64(0)
    err = ctypes.create_string_buffer(512)
    args = (ptx.encode(), kernel.encode(), grid, block, ctypes.cast(pbuf, ctypes.c_void_p), len(params), bufs,
            len(buffers), ctypes.byref(cfg), stats.ctypes.data, None, ctypes.byref(status))
    fresh = [(base, arr.copy()) for base, arr in buffers]
    rc = lib.orc_run_events(*args, None, 0, ctypes.byref(n), err, len(err))
    if rc != 0:
        raise OracleError(rc, err.value.decode(errors="replace"))
    # run again into a buffer of the right size, from the original memory
    for (_, arr), (_, orig) in zip(buffers, fresh):
        arr[...] = orig
    ev = np.zeros(n.value, dtype=HINT_EVENT_DTYPE)
    rc = lib.orc_run_events(*args, ev.ctypes.data if n.value else None, n.value, ctypes.byref(n), err, len(err))
    if rc != 0:
        raise OracleError(rc, err.value.decode(errors="replace"))
    return Result(stats=stats, trace=None, status=status.value, race_flags=0), ev


# SM issue model outputs (orc_run_sched)
SCHED_WARP_DTYPE = np.dtype([("start", "<u8"), ("end", "<u8"), ("issued", "<u8"), ("not_selected", "<u8"),
                             ("stall_exec", "<u8"), ("stall_mem", "<u8"), ("stall_math", "<u8"),
                             ("stall_barrier", "<u8"), ("throttled", "<u8"), ("diverged", "<u8")])
SCHED_SM_DTYPE = np.dtype([("cycles", "<u8"), ("issued", "<u8"), ("ctas", "<u8"), ("status", "<i4"),
                           ("reserved", "<u4")])


def run_sched(ptx: str, kernel: str, grid: int, block: int, params: bytes, buffers, *, lat=DEFAULT_LAT,
              n_sm: int = 152, ctas_per_sm: int = 0, schedulers: int = 4, step_limit: int = 1 << 26,
              stats: np.ndarray | None = None):
    """The SM issue model, cycle by cycle on one host thread: (per-warp
    SCHED_WARP_DTYPE records, per-SM SCHED_SM_DTYPE records). Buffers are
    updated in place; `stats` (STATS_DTYPE, one per warp) gets the per-warp
    statistics, with this model's absolute ends as cycles."""
    lib = _load()
    W = grid * ((block + 31) // 32)
    bufs = (_Buffer * max(1, len(buffers)))()
    keep = []
    for i, (base, arr) in enumerate(buffers):
        keep.append(arr)
        bufs[i].sim_base = base
        bufs[i].host = arr.ctypes.data
        bufs[i].bytes = arr.nbytes
    cfg = _Config()
    for i in range(12):
        cfg.lat[i] = lat[i] if i < len(lat) else 0
    cfg.stack_depth = 32
    cfg.step_limit = step_limit
    cfg.inject_warp = -1
    cfg.mode = MODE_WARP
    sc = (ctypes.c_uint32 * 3)(n_sm, ctas_per_sm, schedulers)
    warps = np.zeros(W, dtype=SCHED_WARP_DTYPE)
    sms = np.zeros(n_sm, dtype=SCHED_SM_DTYPE)
    pbuf = ctypes.create_string_buffer(bytes(params), max(1, len(params)))
    err = ctypes.create_string_buffer(512)
    rc = lib.orc_run_sched(ptx.encode(), kernel.encode(), grid, block, ctypes.cast(pbuf, ctypes.c_void_p),
                           len(params), bufs, len(buffers), ctypes.byref(cfg), ctypes.byref(sc), warps.ctypes.data,
                           sms.ctypes.data, stats.ctypes.data if stats is not None else None, err, len(err))
    if rc != 0:
        raise OracleError(rc, err.value.decode(errors="replace"))
    return warps, sms


@dataclass
class CachedResult:
    stats: np.ndarray
    trace: np.ndarray | None
    status: int
    warps: np.ndarray  # CACHE_WARP_DTYPE, one record per warp
    log: np.ndarray    # CACHE_ACCESS_DTYPE, shape (W, log_cap)


def run_cached(ptx: str, kernel: str, grid: int, block: int, params: bytes, buffers, *,
               lat=DEFAULT_LAT, max_ts: int = 0, trace: bool = False, stack_depth: int = 32,
               step_limit: int = 1 << 26, l1_lines: int = 1024, l2_lines: int = 49152, lat_l1: int = 28,
               lat_l2: int = 150, log_cap: int = 256) -> CachedResult:
    """Interprets `kernel` with the L1/L2 hit model: the whole grid, stepped
    one instruction per warp per step on one host thread."""
    lib = _load()
    W = grid * ((block + 31) // 32)
    bufs = (_Buffer * max(1, len(buffers)))()
    keep = []
    for i, (base, arr) in enumerate(buffers):
        if not arr.flags["C_CONTIGUOUS"]:
            raise ValueError("buffer arrays must be C-contiguous")
        keep.append(arr)
        bufs[i].sim_base = base
        bufs[i].host = arr.ctypes.data
        bufs[i].bytes = arr.nbytes
    cfg = _Config()
    for i in range(12):
        cfg.lat[i] = lat[i] if i < len(lat) else 0
    cfg.max_ts_per_warp = max_ts
    cfg.stack_depth = stack_depth
    cfg.step_limit = step_limit
    cfg.inject_warp = -1
    cfg.mode = MODE_WARP
    warps = np.zeros(W, dtype=CACHE_WARP_DTYPE)
    log = np.zeros((W, log_cap), dtype=CACHE_ACCESS_DTYPE)
    cc = _Cache(l1_lines, l2_lines, lat_l1, lat_l2, log_cap, warps.ctypes.data, log.ctypes.data)
    stats = np.zeros(W, dtype=STATS_DTYPE)
    tr = np.zeros(W * slot_bytes(max_ts, record_bytes(ptx, kernel)), dtype=np.uint8) if trace else None
    pbuf = ctypes.create_string_buffer(bytes(params), max(1, len(params)))
    status = ctypes.c_int32(0)
    err = ctypes.create_string_buffer(512)
    rc = lib.orc_run_cached(ptx.encode(), kernel.encode(), grid, block, ctypes.cast(pbuf, ctypes.c_void_p),
                            len(params), bufs, len(buffers), ctypes.byref(cfg), ctypes.byref(cc),
                            stats.ctypes.data, tr.ctypes.data if tr is not None else None, ctypes.byref(status),
                            err, len(err))
    if rc != 0:
        raise OracleError(rc, err.value.decode(errors="replace"))
    return CachedResult(stats=stats, trace=tr, status=status.value, warps=warps, log=log)


def ipdom(ptx: str, kernel: str) -> list[int]:
    lib = _load()
    out = (ctypes.c_int32 * 65536)()
    n = ctypes.c_uint32(0)
    err = ctypes.create_string_buffer(512)
    rc = lib.orc_ipdom(ptx.encode(), kernel.encode(), out, 65536, ctypes.byref(n), err, len(err))
    if rc != 0:
        raise OracleError(rc, err.value.decode(errors="replace"))
    return [out[i] for i in range(n.value)]


def params_layout(ptx: str, kernel: str):
    lib = _load()
    offs = (ctypes.c_uint32 * 256)()
    sizes = (ctypes.c_uint32 * 256)()
    n = ctypes.c_uint32(0)
    total = ctypes.c_uint32(0)
    err = ctypes.create_string_buffer(512)
    rc = lib.orc_params(ptx.encode(), kernel.encode(), offs, sizes, 256, ctypes.byref(n),
                        ctypes.byref(total), err, len(err))
    if rc != 0:
        raise OracleError(rc, err.value.decode(errors="replace"))
    return [(offs[i], sizes[i]) for i in range(n.value)], total.value


def event_info(ptx: str, kernel: str) -> list[tuple[int, int, str]]:
    """(kind, payload bytes, name) of every event in id order."""
    lib = _load()
    out = []
    for i in range(len(events(ptx, kernel))):
        kind, pb = ctypes.c_uint32(0), ctypes.c_uint32(0)
        name = ctypes.create_string_buffer(256)
        err = ctypes.create_string_buffer(512)
        rc = lib.orc_event_info(ptx.encode(), kernel.encode(), i, ctypes.byref(kind), ctypes.byref(pb), name,
                                len(name), err, len(err))
        if rc != 0:
            raise OracleError(rc, err.value.decode(errors="replace"))
        out.append((kind.value, pb.value, name.value.decode()))
    return out


def record_bytes(ptx: str, kernel: str) -> int:
    """Bytes per trace record of the kernel's slots: 4, 8 or 16."""
    lib = _load()
    b = ctypes.c_uint32(0)
    err = ctypes.create_string_buffer(512)
    rc = lib.orc_record_bytes(ptx.encode(), kernel.encode(), ctypes.byref(b), err, len(err))
    if rc != 0:
        raise OracleError(rc, err.value.decode(errors="replace"))
    return b.value


def events(ptx: str, kernel: str) -> list[int]:
    lib = _load()
    kinds = (ctypes.c_uint32 * 256)()
    n = ctypes.c_uint32(0)
    err = ctypes.create_string_buffer(512)
    rc = lib.orc_events(ptx.encode(), kernel.encode(), kinds, 256, ctypes.byref(n), err, len(err))
    if rc != 0:
        raise OracleError(rc, err.value.decode(errors="replace"))
    return [kinds[i] for i in range(n.value)]


def parse_check(ptx: str, kernel: str) -> tuple[int, str]:
    """Returns (0, '') when the oracle accepts the program, else (code, message)."""
    try:
        params_layout(ptx, kernel)
        return 0, ""
    except OracleError as e:
        return e.code, str(e)

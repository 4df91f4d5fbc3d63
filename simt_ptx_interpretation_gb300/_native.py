"""ctypes declarations of libks (include/ks.h). Loading fails loudly: there is
no fallback path."""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libks.so")


class KsBuffer(ctypes.Structure):
    _fields_ = [("sim_base", ctypes.c_uint64), ("dev_ptr", ctypes.c_void_p), ("bytes", ctypes.c_uint64)]


class KsConfig(ctypes.Structure):
    _fields_ = [
        ("lat", ctypes.c_uint32 * 12),
        ("max_ts_per_warp", ctypes.c_uint32),
        ("simt_stack_depth", ctypes.c_uint32),
        ("step_limit", ctypes.c_uint64),
        ("inject_warp", ctypes.c_int64),
        ("inject_step", ctypes.c_uint64),
        ("flags", ctypes.c_uint32),
        ("reserved", ctypes.c_uint32),
        ("profile_buf", ctypes.c_void_p),
        ("profile_bytes", ctypes.c_uint64),
    ]


class KsTotals(ctypes.Structure):
    _fields_ = [(n, ctypes.c_uint64) for n in (
        "cycles_max", "cycles_sum", "warp_insts", "thread_insts", "ld_req", "ld_sectors", "st_req",
        "st_sectors", "ld_lines", "st_lines", "n_warps", "n_failed")] + [
        ("first_failed_warp", ctypes.c_int64), ("status", ctypes.c_int32), ("max_stack_depth", ctypes.c_uint32),
        ("sh_req", ctypes.c_uint64), ("sh_wavefronts", ctypes.c_uint64)]


class KsGpuLimits(ctypes.Structure):
    _fields_ = [("max_threads_per_sm", ctypes.c_uint32), ("max_warps_per_sm", ctypes.c_uint32),
                ("max_blocks_per_sm", ctypes.c_uint32), ("registers_per_sm", ctypes.c_uint32),
                ("shared_memory_per_sm", ctypes.c_uint32)]


class KsOccupancy(ctypes.Structure):
    _fields_ = [("active_warps_per_sm", ctypes.c_uint32), ("max_warps_per_sm", ctypes.c_uint32),
                ("warps_by_registers", ctypes.c_uint32), ("warps_by_shared_memory", ctypes.c_uint32),
                ("warps_by_block_size", ctypes.c_uint32), ("limiter", ctypes.c_int32),
                ("occupancy_percent", ctypes.c_double)]


class KsCacheConfig(ctypes.Structure):
    _fields_ = [("l1_lines", ctypes.c_uint32), ("l2_lines", ctypes.c_uint32), ("lat_l1", ctypes.c_uint32),
                ("lat_l2", ctypes.c_uint32), ("max_accesses_per_warp", ctypes.c_uint32),
                ("max_runs_per_warp", ctypes.c_uint32), ("reserved", ctypes.c_uint32 * 2)]


class KsSchedConfig(ctypes.Structure):
    _fields_ = [("n_sm", ctypes.c_uint32), ("ctas_per_sm", ctypes.c_uint32), ("schedulers_per_sm", ctypes.c_uint32),
                ("max_runs_per_warp", ctypes.c_uint32), ("reserved", ctypes.c_uint32 * 4)]


class KsHint(ctypes.Structure):
    _fields_ = [("category", ctypes.c_int32), ("severity", ctypes.c_int32), ("pc", ctypes.c_int32),
                ("reserved", ctypes.c_uint32), ("count", ctypes.c_uint64), ("message", ctypes.c_char * 64),
                ("detail", ctypes.c_char * 96)]


class KsBatchItem(ctypes.Structure):
    _fields_ = [("mod", ctypes.c_void_p), ("kernel", ctypes.c_char_p), ("grid", ctypes.c_uint32),
                ("block", ctypes.c_uint32), ("params", ctypes.c_void_p), ("param_bytes", ctypes.c_size_t),
                ("bufs", ctypes.POINTER(KsBuffer)), ("n_bufs", ctypes.c_uint32), ("reserved", ctypes.c_uint32),
                ("trace_buf", ctypes.c_void_p), ("trace_bytes", ctypes.c_size_t), ("stats_buf", ctypes.c_void_p),
                ("stats_bytes", ctypes.c_size_t), ("cfg", ctypes.POINTER(KsConfig))]


class KsCachedItem(ctypes.Structure):
    _fields_ = [("sim", KsBatchItem), ("cache", ctypes.POINTER(KsCacheConfig)), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t)]


EXPORTS = {
    "ks_config_default": (None, [ctypes.POINTER(KsConfig)]),
    "ks_load_module": (ctypes.c_int, [ctypes.c_char_p, ctypes.c_size_t, ctypes.POINTER(ctypes.c_void_p),
                                      ctypes.c_char_p, ctypes.c_size_t]),
    "ks_free_module": (None, [ctypes.c_void_p]),
    "ks_kernel_info": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_char_p] + [ctypes.POINTER(ctypes.c_uint32)] * 5),
    "ks_kernel_param": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_char_p, ctypes.c_uint32,
                                       ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint32),
                                       ctypes.POINTER(ctypes.c_char_p)]),
    "ks_kernel_event": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_char_p, ctypes.c_uint32,
                                       ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_char_p)]),
    "ks_kernel_ipdom": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_char_p, ctypes.POINTER(ctypes.c_int32),
                                       ctypes.c_uint32, ctypes.POINTER(ctypes.c_uint32)]),
    "ks_kernel_fast_runs": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_char_p, ctypes.POINTER(ctypes.c_uint32),
                                           ctypes.c_uint32, ctypes.POINTER(ctypes.c_uint32)]),
    "ks_kernel_layout": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_char_p, ctypes.c_uint32,
                                        ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint32)]),
    "ks_trace_bytes": (ctypes.c_size_t, [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]),
    "ks_stats_bytes": (ctypes.c_size_t, [ctypes.c_uint32, ctypes.c_uint32]),
    "ks_trace_to_json": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_char_p, ctypes.c_uint32, ctypes.c_uint32,
                                        ctypes.c_uint32, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_double,
                                        ctypes.c_char_p, ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t)]),
    "ks_gpu_limits_of": (ctypes.c_int, [ctypes.c_char_p, ctypes.POINTER(KsGpuLimits)]),
    "ks_occupancy": (ctypes.c_int, [ctypes.POINTER(KsGpuLimits), ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32,
                                    ctypes.POINTER(KsOccupancy)]),
    "ks_trace_bytes_records": (ctypes.c_size_t, [ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_uint32]),
    "ks_kernel_record_bytes": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_char_p, ctypes.POINTER(ctypes.c_uint32)]),
    "ks_kernel_event_payload": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_char_p, ctypes.c_uint32,
                                               ctypes.POINTER(ctypes.c_uint32)]),
    "ks_simulate": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_char_p, ctypes.c_uint32, ctypes.c_uint32,
                                   ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(KsBuffer), ctypes.c_uint32,
                                   ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_size_t,
                                   ctypes.POINTER(KsConfig), ctypes.c_void_p]),
    "ks_simulate_static": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_char_p, ctypes.c_uint32, ctypes.c_uint32,
                                          ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(KsBuffer),
                                          ctypes.c_uint32, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                          ctypes.c_size_t, ctypes.POINTER(KsConfig), ctypes.c_void_p]),
    "ks_simulate_batch": (ctypes.c_int, [ctypes.POINTER(KsBatchItem), ctypes.c_uint32, ctypes.c_void_p,
                                         ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint32)]),
    "ks_simulate_cached_batch": (ctypes.c_int, [ctypes.POINTER(KsCachedItem), ctypes.c_uint32, ctypes.c_void_p,
                                                ctypes.POINTER(ctypes.c_uint32), ctypes.POINTER(ctypes.c_uint32)]),
    "ks_cache_config_default": (None, [ctypes.POINTER(KsCacheConfig)]),
    "ks_cache_workspace_bytes": (ctypes.c_size_t, [ctypes.c_uint32, ctypes.c_uint32, ctypes.POINTER(KsCacheConfig)]),
    "ks_simulate_cached": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_char_p, ctypes.c_uint32, ctypes.c_uint32,
                                          ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(KsBuffer),
                                          ctypes.c_uint32, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                          ctypes.c_size_t, ctypes.POINTER(KsConfig), ctypes.POINTER(KsCacheConfig),
                                          ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "ks_profile_bytes": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_char_p, ctypes.POINTER(ctypes.c_size_t)]),
    "ks_hints": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint32, ctypes.POINTER(KsOccupancy), ctypes.POINTER(KsHint),
                                ctypes.c_uint32, ctypes.POINTER(ctypes.c_uint32)]),
    "ks_sched_config_default": (None, [ctypes.POINTER(KsSchedConfig)]),
    "ks_sched_workspace_bytes": (ctypes.c_size_t, [ctypes.c_uint32, ctypes.c_uint32, ctypes.POINTER(KsSchedConfig)]),
    "ks_simulate_sched": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_char_p, ctypes.c_uint32, ctypes.c_uint32,
                                         ctypes.c_void_p, ctypes.c_size_t, ctypes.POINTER(KsBuffer), ctypes.c_uint32,
                                         ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_size_t,
                                         ctypes.POINTER(KsConfig), ctypes.POINTER(KsSchedConfig), ctypes.c_void_p,
                                         ctypes.c_size_t, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p,
                                         ctypes.c_size_t, ctypes.c_void_p]),
    "ks_read_stats": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_uint64, ctypes.c_void_p, ctypes.POINTER(KsTotals)]),
    "ks_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}

_lib = None


def lib():
    """The loaded libks; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in EXPORTS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib

"""GB300-native warp-level SIMT PTX interpreter.

A host C++ decoder lowers a PTX subset into a packed instruction array; a
hand-written sm_103a kernel steps every simulated warp in lockstep and
produces the simulated memory, per-warp cycles from an in-order scoreboard,
32-byte sector counts per ld/st, shared-memory bank-conflict degrees,
IKET-style per-warp trace slots and, optionally, an L1/L2 hit model on load
latency; host post-passes compute occupancy and export traces. The C ABI
is include/ks.h (libks.so); this package marshals arguments to it.
"""
from .api import (CACHE_ACCESS_DTYPE, CACHE_WARP_DTYPE, DEFAULT_LAT, PROFILE_DTYPE, SCHED_SM_DTYPE, SCHED_WARP_DTYPE,
                  STATS_DTYPE, BatchItem, CacheConfig, CachedBatchItem, Config, KsError, Module, Run, SchedConfig, Totals, cache_results,
                  cache_workspace_bytes, gpu_limits, hints, occupancy, profile_array, read_stats, run,
                  sched_workspace_bytes, simulate, simulate_batch, simulate_cached, simulate_cached_batch, simulate_sched, simulate_static, stats_array,
                  stats_bytes, trace_bytes, trace_to_json)

__all__ = ["CACHE_ACCESS_DTYPE", "CACHE_WARP_DTYPE", "DEFAULT_LAT", "PROFILE_DTYPE", "SCHED_SM_DTYPE",
           "SCHED_WARP_DTYPE", "STATS_DTYPE", "BatchItem", "CacheConfig", "CachedBatchItem", "Config", "KsError", "Module", "Run", "SchedConfig",
           "Totals", "cache_results", "cache_workspace_bytes", "gpu_limits", "hints", "occupancy", "profile_array",
           "sched_workspace_bytes", "simulate_sched",
           "read_stats", "run", "simulate", "simulate_batch", "simulate_cached", "simulate_cached_batch", "simulate_static", "stats_array", "stats_bytes",
           "trace_bytes", "trace_to_json"]

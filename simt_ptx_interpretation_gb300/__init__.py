"""GB300-native warp-level SIMT PTX interpreter.

A host C++ decoder lowers a PTX subset into a packed instruction array; a
hand-written sm_103a kernel steps every simulated warp in lockstep and
produces the simulated memory, per-warp cycles from an in-order scoreboard,
32-byte sector counts per ld/st, shared-memory bank-conflict degrees and
IKET-style per-warp trace slots; host post-passes compute occupancy and
export traces. The C ABI
is include/ks.h (libks.so); this package marshals arguments to it.
"""
from .api import (DEFAULT_LAT, STATS_DTYPE, Config, KsError, Module, Run, Totals, gpu_limits, occupancy, read_stats,
                  run, simulate, simulate_static, stats_array, stats_bytes, trace_bytes, trace_to_json)

__all__ = ["DEFAULT_LAT", "STATS_DTYPE", "Config", "KsError", "Module", "Run", "Totals", "gpu_limits", "occupancy",
           "read_stats", "run", "simulate", "simulate_static", "stats_array", "stats_bytes", "trace_bytes",
           "trace_to_json"]

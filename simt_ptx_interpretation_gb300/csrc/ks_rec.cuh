// ks_rec.cuh — what the replays (the SM issue model's, ks_sched.cu, and the
// L1/L2 hit model's timing pass, ks_cache_replay.cu) need of a decoded
// program entry: its scoreboard terms and latencies, independent of the
// register layout its image was decoded for.
#pragma once

#include "ks_internal.h"

namespace ks {

// The predicate operands of a DevInsn: the guard, the predicate sources and
// the predicate destination (31 = none / the always-true predicate, whose
// ready entry never changes).
struct PredTerms {
  uint32_t guard, pa, pb, pc, pd;
};

__host__ __device__ inline PredTerms pred_terms(const DevInsn& d, uint32_t split, uint32_t pred_off) {
  auto pred = [&](uint32_t off) { return (off - pred_off) / 4u; };
  PredTerms t;
  if (split) {  // hazard halfwords 4..7: guard, sources; 3: the destination's term
    t.guard = pred(d.x[2] & 0xFFFFu);
    t.pa = pred(d.x[2] >> 16);
    t.pb = pred(d.x[3] & 0xFFFFu);
    t.pc = pred(d.x[3] >> 16);
    t.pd = (d.inc & INC_PDEST) ? pred(d.x[1] >> 16) : 31u;
  } else {  // guard, gneg, ha, hb, hc, hd
    t.guard = d.x[0];
    t.pa = pred(d.x[2]);
    t.pb = pred(d.x[3]);
    t.pc = pred(d.x[4]);
    t.pd = pred(d.x[5]);
  }
  return t;
}

// Latencies of an entry under a launch's table: its destination's (0 without
// one), a store's completion (0 if not a store), and the issue clock's advance
// (the latency for bra/ret, 1 otherwise, 0 for a pseudo-op) -- as the
// interpreter patches its staged copy.
struct EntryLat {
  uint32_t dest, store, next;
};

__host__ __device__ inline EntryLat entry_lat(const DevInsn& d, const uint32_t* lat) {
  const uint32_t f = d.wlat, l = lat[f & 0xFFu];
  EntryLat e;
  e.dest = (f & DEV_HAS_DEST) ? l : 0u;
  e.store = (f & DEV_IS_STORE) ? l : 0u;
  e.next = d.inc ? ((f & DEV_IS_CTRL) ? l : 1u) : 0u;
  return e;
}

}  // namespace ks

// ks_sched.cu — the SM-level issue model (KernelScope backend doc,
// simulator/engine.py and simulator/models.py — WarpStallReason,
// _determine_stall_reason, WarpScheduleInfo: warps that are ready but not
// picked, waiting on a load, on a result, on the math pipe, at a barrier).
//
// The interpreter's instrumented pass logs, per warp, the runs of program
// entries it consumed; values and control flow do not depend on timing, so
// the schedule can be replayed from those runs and the decoded program alone.
// One real warp replays one simulated SM: lane l holds the warp in resident
// slot l (CTA slot l / warps-per-CTA), its scoreboard (a ready time and the
// producer's kind per register row and predicate) in shared memory, and its
// position in its runs. Every step the lanes offer their next issue time
// max(own scoreboard time, their scheduler's free cycle); the earliest, and
// among equal times the lowest global warp id (the page's step() order),
// issues. Barriers release as in the interpreter (latest arrival + bar
// latency, finished warps do not hold them); a CTA whose warps are all done
// frees its slot, and the SM's next CTA (s, s + n_sm, s + 2 n_sm, ...) starts
// there at that cycle.
#include <cuda_runtime.h>

#include "ks_internal.h"
#include "ks_rec.cuh"

namespace ks {
namespace {

constexpr unsigned FULL = 0xFFFFFFFFu;
constexpr uint32_t NEVER = 0xFFFFFFFFu;
constexpr uint32_t CLOCK_LIMIT = 1u << 31;
enum : uint32_t { ST_EMPTY = 0, ST_RUNNING = 1, ST_WAITING = 2, ST_DONE = 3 };
enum : uint32_t { K_EXEC = 0, K_MATH = 1, K_MEM = 2 };  // what a stall waits on (priority order)

struct SchedLaunch {
  const uint8_t* image;  // DevInsn program (unpatched latencies)
  uint32_t n_insn;       // entries, the exit sentinel not included
  uint32_t n_rows;       // register, constant and zero rows of a warp region
  uint32_t pred_off;     // region offset of the predicate ready table
  uint32_t row_bytes;    // row size of the image's layout
  uint32_t split;        // the image's layout: 0 PAIR, 1 SPLIT (DevInsn::x differs)
  uint32_t cta_mode;     // the kernel has shared memory or bar.sync
  uint32_t lat[KS_NUM_LAT_CLASSES];
  uint32_t grid, wpc, n_sm, ctas_per_sm, schedulers;
  const uint32_t* log;
  const uint32_t* runs;
  uint32_t cap;
  ks_sched_warp* warps_out;
  ks_sched_sm* sms_out;
};

__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) { return __reduce_max_sync(FULL, v); }

// What the replay needs of a program entry, 32 bytes:
//   x: row a | row b << 16        y: row c | row d << 16
//   z: guard | pred a << 8 | pred b << 16 | pred c << 24
//   w: pred d | flags << 8 | kind of its result << 16
//   then dest latency, store latency, issue-clock advance
struct alignas(16) Rec {
  uint4 q;
  uint4 lat;
};
constexpr uint32_t F_ISSUE = 1, F_RDEST = 2, F_PDEST = 4, F_PHAZ = 8, F_BAR = 16, F_MCLASS = 32, F_MEMOP = 64;

struct Lane {
  uint32_t state, gw, cta_slot;
  uint32_t rank;                     // order of gw among the occupied lanes of my scheduler
  uint32_t pc, run_left, k, n_runs;  // next entry to issue; entries left in its run; next run index
  uint32_t t_next, t_last, max_ready, drain, base, start, e, bind, arrival, end;
  Rec r;                             // the record of the next entry
  uint32_t div;                      // the run of the next entry issues diverged (RUN_DIVERGED)
  uint32_t issued, not_selected, st_exec, st_mem, st_math, stall_bar;  // each below the 2^31 clock limit
  uint32_t throttled, diverged;      // the two labels (instructions)
  // the latest global / shared access (issue cycle, completion) and the one
  // before it: at cycle T the pending one is the latest issued before T
  uint32_t mem_at, mem_done, prev_done;
  bool has_mem, has_prev;
  __device__ __forceinline__ bool mem_pending(uint32_t T) const {
    return has_mem && (mem_at < T ? mem_done > T : (has_prev && prev_done > T));
  }
};

// ready table entry: ready time | kind of the producer << 32; the kind of a
// term counts when its time is the latest
__device__ __forceinline__ uint32_t kind_at(uint64_t v, uint32_t e) {
  return (uint32_t)v == e ? (uint32_t)(v >> 32) : K_EXEC;
}

// RUN_AHEAD: the form for kernels without barriers whose CTAs all reach
// their SMs at the start (every CTA slot filled at once, none left), where a
// warp alone on its scheduler runs ahead (below); the other form keeps the
// step loop alone (its code shape costs the other workloads 13 %).
template <bool RUN_AHEAD>
__global__ void __launch_bounds__(32) ks_sched_kernel(const __grid_constant__ SchedLaunch S) {
  extern __shared__ __align__(16) uint8_t sm[];
  const uint32_t lane = threadIdx.x;
  const uint32_t s_id = blockIdx.x;
  Rec* prog = reinterpret_cast<Rec*>(sm);
  const uint32_t NR = S.n_rows + 32u;  // rows, then the 32 predicates
  uint64_t* ready = reinterpret_cast<uint64_t*>(sm + (size_t)(S.n_insn + 1) * sizeof(Rec)) + (size_t)lane * NR;

  // the program's records with this launch's latencies (patched as the
  // interpreter patches its copy)
  for (uint32_t i = lane; i <= S.n_insn; i += 32) {
    const DevInsn d = reinterpret_cast<const DevInsn*>(S.image)[i];
    const uint32_t f = d.wlat, cls = f & 0xFFu;
    const EntryLat el = entry_lat(d, S.lat);
    const uint32_t kind = (cls == KS_LAT_LDG || cls == KS_LAT_LDS) ? K_MEM : cls == KS_LAT_SFU ? K_MATH : K_EXEC;
    uint32_t flags = 0;
    if (d.inc & INC_ISSUE) flags |= F_ISSUE;
    if (d.inc & INC_RDEST) flags |= F_RDEST;
    if (d.inc & INC_PDEST) flags |= F_PDEST;
    if (d.inc & INC_PHAZ) flags |= F_PHAZ;
    if (d.op == OP_BAR) flags |= F_BAR;
    if (d.inc & INC_MCLASS) flags |= F_MCLASS;
    if (d.inc & INC_MEMOP) flags |= F_MEMOP;
    // the guard, the predicate sources and the predicate destination (31:
    // none), from either layout's record
    const PredTerms pt = pred_terms(d, S.split, S.pred_off);
    const uint32_t guard = pt.guard, pa = pt.pa, pb = pt.pb, pc = pt.pc, pd = pt.pd;
    const uint32_t RB = S.row_bytes;
    Rec r;
    r.q.x = (d.a / RB) | ((d.b / RB) << 16);
    r.q.y = (d.c / RB) | ((d.d / RB) << 16);
    r.q.z = guard | (pa << 8) | (pb << 16) | (pc << 24);
    r.q.w = pd | (flags << 8) | (kind << 16);
    r.lat.x = el.dest;
    r.lat.y = el.store;
    r.lat.z = el.next;
    r.lat.w = 0u;
    prog[i] = r;
  }
  __syncwarp();

  const uint32_t slots = S.ctas_per_sm * S.wpc;  // resident warp slots (<= 32)
  const uint32_t my_sched = lane & (S.schedulers - 1u);  // schedulers: 1, 2 or 4
  // the lanes of my scheduler
  const uint32_t sched_lanes = (S.schedulers == 1u ? 0xFFFFFFFFu : S.schedulers == 2u ? 0x55555555u : 0x11111111u)
                               << my_sched;
  Lane L;
  L.state = ST_EMPTY;
  L.cta_slot = lane / S.wpc;
  L.has_mem = L.has_prev = false;
  L.mem_at = L.mem_done = L.prev_done = 0;
  uint32_t port = 0;  // next free cycle of my scheduler
  uint32_t next_cta_k = 0;
  uint32_t status = 0;
  uint64_t sm_issued = 0;
  uint32_t sm_end = 0, ctas = 0;
  bool ranks_dirty = true;  // a CTA was loaded since the ranks were taken

  // position at the next issued entry of the runs (its record in L.r);
  // false when none is left
  auto advance = [&](bool consume) -> bool {
    if (consume) {
      L.pc++;
      L.run_left--;
    }
    for (;;) {
      while (L.run_left == 0) {
        if (L.k >= L.n_runs) return false;
        const uint32_t r = S.log[(uint64_t)L.gw * S.cap + L.k++];
        L.pc = r >> 16;
        L.run_left = (r & (RUN_DIVERGED - 1u)) + 1u;
        L.div = r & RUN_DIVERGED;
      }
      L.r = prog[L.pc];
      if ((L.r.q.w >> 8) & F_ISSUE) return true;
      L.pc++;
      L.run_left--;
    }
  };
  // scoreboard time of the next entry and what binds it
  auto compute_e = [&]() {
    const uint4 q = L.r.q;
    const uint32_t P = S.n_rows;
    const uint64_t va = ready[q.x & 0xFFFFu], vb = ready[q.x >> 16], vc = ready[q.y & 0xFFFFu],
                   vd = ready[q.y >> 16], vg = ready[P + (q.z & 0xFFu)];
    uint32_t e = max(max(L.t_next, max((uint32_t)va, (uint32_t)vb)),
                     max(max((uint32_t)vc, (uint32_t)vd), (uint32_t)vg));
    uint64_t p0 = 0, p1 = 0, p2 = 0, p3 = 0;
    if ((q.w >> 8) & F_PHAZ) {
      p0 = ready[P + ((q.z >> 8) & 0xFFu)];
      p1 = ready[P + ((q.z >> 16) & 0xFFu)];
      p2 = ready[P + (q.z >> 24)];
      p3 = ready[P + (q.w & 0xFFu)];
      e = max(e, max(max((uint32_t)p0, (uint32_t)p1), max((uint32_t)p2, (uint32_t)p3)));
    }
    // the t_next term (a branch's latency) is an execution wait: kind 0
    const uint32_t kind = max(max(max(kind_at(va, e), kind_at(vb, e)), max(kind_at(vc, e), kind_at(vd, e))),
                              max(max(kind_at(vg, e), kind_at(p0, e)),
                                  max(max(kind_at(p1, e), kind_at(p2, e)), kind_at(p3, e))));
    L.e = e;
    L.bind = kind;
  };
  auto finish = [&]() {
    L.state = ST_DONE;
    L.end = L.issued ? max(max(L.t_last + 1u, L.max_ready), L.drain) : L.start;
    ks_sched_warp r;
    r.start = L.start;
    r.end = L.end;
    r.issued = L.issued;
    r.not_selected = L.not_selected;
    r.stall_exec = L.st_exec;
    r.stall_mem = L.st_mem;
    r.stall_math = L.st_math;
    r.stall_barrier = L.stall_bar;
    r.throttled = L.throttled;
    r.diverged = L.diverged;
    S.warps_out[L.gw] = r;
    sm_end = max(sm_end, L.end);
    sm_issued += L.issued;
  };
  // lanes of slot c (mine) load their warps of the SM's next CTA at cycle t0
  auto load_cta = [&](bool mine, uint32_t t0) {
    ranks_dirty = true;
    const uint32_t k = next_cta_k++;
    const uint64_t cta = (uint64_t)s_id + (uint64_t)k * S.n_sm;
    if (!mine) return;
    if (cta >= S.grid) {
      L.state = ST_EMPTY;
      return;
    }
    L.gw = (uint32_t)cta * S.wpc + (lane - L.cta_slot * S.wpc);
    for (uint32_t i = 0; i < NR; i++) ready[i] = 0ull;
    L.state = ST_RUNNING;
    L.k = 0;
    L.run_left = 0;
    L.n_runs = S.runs[L.gw];
    L.t_next = L.base = L.start = t0;
    L.t_last = t0;
    L.max_ready = L.drain = 0u;
    L.issued = L.not_selected = L.stall_bar = 0;
    L.st_exec = L.st_mem = L.st_math = 0;
    L.throttled = L.diverged = 0;
    L.has_mem = L.has_prev = false;
    L.mem_at = L.mem_done = L.prev_done = 0;
    L.div = 0;
    if (L.n_runs > S.cap) {
      status = KS_ST_SCHED_LIMIT;
      L.n_runs = 0;
    }
    if (advance(false)) compute_e();
    else finish();
  };
  // Settles CTA slot c after one of its warps arrived or finished: releases
  // its barrier when no warp runs, and when every warp is done starts the
  // SM's next CTA there (at once again if that CTA has nothing to issue).
  auto settle = [&](uint32_t c) {
    for (;;) {
      const bool mine = lane < slots && L.cta_slot == c;
      if (__any_sync(FULL, mine && L.state == ST_RUNNING)) return;
      const uint32_t waiting = __ballot_sync(FULL, mine && L.state == ST_WAITING);
      if (waiting) {
        const uint32_t latest = warp_max_u32(mine && L.state == ST_WAITING ? L.arrival : 0u);
        if (mine && L.state == ST_WAITING) {
          const uint32_t rel = latest + S.lat[KS_LAT_BAR];
          L.stall_bar += rel - (L.arrival + 1u);
          L.t_next = L.base = rel;
          L.state = ST_RUNNING;
          if (L.run_left != 0 || L.k < L.n_runs) compute_e();
          else finish();
        }
        continue;
      }
      if (!__any_sync(FULL, mine && L.state == ST_DONE)) return;  // an empty slot
      const uint32_t fin = warp_max_u32(mine ? L.end : 0u);
      ctas++;
      load_cta(mine, fin);
      if (!__any_sync(FULL, mine && L.state != ST_EMPTY)) return;
    }
  };

  // This lane's warp issues its next entry at cycle T: the waits it stood
  // (not selected, or stalled on what bound its scoreboard time), its
  // destination's ready entry, its clocks and counts. Returns the entry's
  // flags; the memory-class label and memory bookkeeping are the caller's.
  auto issue = [&](uint32_t T) -> uint32_t {
    L.not_selected += T - L.e;
    if (L.e > L.base) {
      const uint32_t d = L.e - L.base;
      if (L.bind == K_MEM) L.st_mem += d;
      else if (L.bind == K_MATH) L.st_math += d;
      else L.st_exec += d;
    }
    const uint4 q = L.r.q, lt = L.r.lat;
    const uint32_t flags = (q.w >> 8) & 0xFFu;
    const uint64_t wr = T + lt.x;
    const uint64_t entry = wr | ((uint64_t)(q.w >> 16) << 32);
    if (flags & F_RDEST) ready[q.y >> 16] = entry;
    if (flags & F_PDEST) ready[S.n_rows + (q.w & 0xFFu)] = entry;
    L.max_ready = max(L.max_ready, (uint32_t)wr);
    L.drain = max(L.drain, T + lt.y);
    L.t_last = T;
    L.t_next = T + lt.z;
    L.base = T + 1u;
    L.issued++;
    if (L.div) L.diverged++;
    return flags;
  };

  for (uint32_t c = 0; c < S.ctas_per_sm; c++) {
    const bool mine = lane < slots && L.cta_slot == c;
    load_cta(mine, 0u);
    if (__any_sync(FULL, mine && L.state != ST_EMPTY)) settle(c);
  }

  // Every step the earliest offer of all is found, and for each scheduler the
  // lowest global warp id offering it; those schedulers issue at once.
  // That is the order of one issue at a time: what an issue changes for other
  // warps (a barrier release, a new CTA) takes effect a cycle later at the
  // soonest, so issues of the same cycle on different schedulers do not see
  // each other. With a zero barrier latency a release takes effect in the
  // same cycle, and the schedulers take turns one issue at a time.
  const bool one_at_a_time = S.lat[KS_LAT_BAR] == 0u;
  const uint32_t per = 32u / S.schedulers;  // lanes of one scheduler
  const bool run_ahead = RUN_AHEAD && !one_at_a_time && S.cta_mode == 0u;
  for (;;) {
    // the earliest offer, then per scheduler the lowest warp id offering it
    const uint32_t cand = L.state == ST_RUNNING ? max(L.e, port) : NEVER;
    const uint32_t T = __reduce_min_sync(FULL, cand);
    if (T == NEVER) break;
    if (T >= CLOCK_LIMIT) {
      status = KS_ST_SCHED_LIMIT;
      break;
    }
    const bool at_T = cand == T;
    bool win;
    bool sched_won = false;  // (not one at a time) my scheduler issues at T
    if (one_at_a_time) {
      win = at_T && L.gw == __reduce_min_sync(FULL, at_T ? L.gw : NEVER);
    } else {
      // every scheduler's lowest warp id at T in one reduction: lane l sets
      // bit (scheduler * per + rank) where per = 32 / schedulers lanes share
      // a scheduler and rank orders their warp ids
      if (ranks_dirty) {
        const uint32_t key = L.state != ST_EMPTY ? L.gw : NEVER;
        uint32_t r = 0;
        for (uint32_t j = 0; j < per; j++) r += __shfl_sync(FULL, key, my_sched + j * S.schedulers) < key ? 1u : 0u;
        L.rank = r;
        ranks_dirty = false;
      }
      const uint32_t all = __reduce_or_sync(FULL, at_T ? 1u << (my_sched * per + L.rank) : 0u);
      const uint32_t mine_bits = per == 32u ? all : (all >> (my_sched * per)) & ((1u << per) - 1u);
      win = at_T && (uint32_t)(__ffs(mine_bits) - 1) == L.rank;
      sched_won = mine_bits != 0u;
    }
    // warps of this SM with a memory operation pending at T (issued earlier,
    // not yet complete), for the memory-throttle label
    const uint32_t pending = __ballot_sync(FULL, lane < slots && L.state != ST_EMPTY && L.mem_pending(T));
    uint32_t ev = 0;  // arrived at a barrier or finished
    if (win) {
      const uint32_t flags = issue(T);
      const uint4 lt = L.r.lat;
      if ((flags & F_MCLASS) && __popc(pending & ~(1u << lane)) >= 4) L.throttled++;
      if (flags & F_MEMOP) {
        L.has_prev = L.has_mem;
        L.prev_done = L.mem_done;
        L.has_mem = true;
        L.mem_at = T;
        L.mem_done = T + max(lt.x, lt.y);  // a load's result, a store's drain
      }
      const bool more = advance(true);
      if (flags & F_BAR) {
        L.state = ST_WAITING;
        L.arrival = T;
        ev = 1;
      } else if (more) {
        compute_e();
      } else {
        finish();
        ev = 1;
      }
    }
    // the winning schedulers' ports move on
    if (one_at_a_time ? (__ballot_sync(FULL, win) & sched_lanes) != 0u : sched_won) port = T + 1u;
    // settle every CTA slot in which a warp arrived or finished
    for (uint32_t m = __ballot_sync(FULL, ev != 0u); m;) {
      const uint32_t c = (uint32_t)(__ffs(m) - 1) / S.wpc;
      settle(c);
      const uint32_t lo = c * S.wpc;
      const uint32_t slot_mask = (S.wpc >= 32u ? FULL : ((1u << S.wpc) - 1u)) << lo;
      m &= ~slot_mask;
    }
    // Run-ahead. In a kernel without barriers, once no CTA is left to reach
    // this SM, a warp that is the only running one on its scheduler can be
    // contested by nothing: no warp can join its scheduler and no release
    // or dispatch depends on it. It issues on its own, at max(its scoreboard
    // time, its scheduler's port), exactly the cycles the steps would give
    // it, up to its next memory-class entry (whose throttle label counts the
    // other warps' memory operations pending at its cycle, known only in
    // step order) or its end.
    if (RUN_AHEAD && run_ahead && (uint64_t)s_id + (uint64_t)next_cta_k * S.n_sm >= S.grid) {
      const uint32_t busy = __ballot_sync(FULL, L.state == ST_RUNNING || L.state == ST_WAITING);
      uint32_t fin = 0;
      if (L.state == ST_RUNNING && __popc(busy & sched_lanes) == 1) {
        for (;;) {
          if (((L.r.q.w >> 8) & 0xFFu) & (F_MCLASS | F_BAR)) break;
          const uint32_t T1 = max(L.e, port);
          if (T1 >= CLOCK_LIMIT) break;  // the steps report it
          issue(T1);
          port = T1 + 1u;
          if (!advance(true)) {
            finish();
            fin = 1;
            break;
          }
          compute_e();
        }
      }
      for (uint32_t m = __ballot_sync(FULL, fin != 0u); m;) {
        const uint32_t c = (uint32_t)(__ffs(m) - 1) / S.wpc;
        settle(c);
        const uint32_t lo = c * S.wpc;
        const uint32_t slot_mask = (S.wpc >= 32u ? FULL : ((1u << S.wpc) - 1u)) << lo;
        m &= ~slot_mask;
      }
    }
  }

  // SM totals (each lane added its own warps)
  for (int o = 16; o > 0; o >>= 1) sm_issued += __shfl_xor_sync(FULL, sm_issued, o);
  sm_end = warp_max_u32(sm_end);
  status = warp_max_u32(status);
  if (lane == 0) {
    ks_sched_sm r;
    r.cycles = sm_end;
    r.issued = sm_issued;
    r.ctas = ctas;
    r.status = (int32_t)status;
    r.reserved = 0;
    S.sms_out[s_id] = r;
  }
}

}  // namespace

size_t sched_smem_bytes(uint32_t n_insn, uint32_t n_rows) {
  return (size_t)(n_insn + 1) * 32u + 32u * (size_t)(n_rows + 32u) * 8u;
}

int launch_sched(const KsLaunch& L, uint32_t n_rows, uint32_t n_sm, uint32_t ctas_per_sm, uint32_t schedulers,
                 ks_sched_warp* warps_out, ks_sched_sm* sms_out, void* stream) {
  SchedLaunch S;
  S.image = L.image;
  S.n_insn = L.n_insn;
  S.n_rows = n_rows;
  S.pred_off = L.layout.pred_off;
  S.row_bytes = L.layout.row_bytes;
  S.split = L.layout.split;
  S.cta_mode = L.cta_mode;
  for (int i = 0; i < KS_NUM_LAT_CLASSES; i++) S.lat[i] = L.lat[i];
  S.grid = L.grid;
  S.wpc = L.wpc;
  S.n_sm = n_sm;
  S.ctas_per_sm = ctas_per_sm;
  S.schedulers = schedulers;
  S.log = L.sched_log;
  S.runs = L.sched_runs;
  S.cap = L.sched_cap;
  S.warps_out = warps_out;
  S.sms_out = sms_out;
  const size_t smem = sched_smem_bytes(L.n_insn, n_rows);
  // every CTA on an SM at the start: grid <= simulated SMs x CTA slots
  const bool run_ahead = !L.cta_mode && L.lat[KS_LAT_BAR] != 0u && (uint64_t)L.grid <= (uint64_t)n_sm * ctas_per_sm;
  const void* fn = run_ahead ? (const void*)ks_sched_kernel<true> : (const void*)ks_sched_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  void* args[] = {&S};
  return (int)cudaLaunchKernel(fn, dim3(n_sm), dim3(32), args, smem, (cudaStream_t)stream);
}

}  // namespace ks

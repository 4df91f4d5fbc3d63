// ks_cache_replay.cu — the timing pass of the L1/L2 hit model's replay form
// (ks_simulate_cached with max_runs_per_warp > 0, kernels without shared
// memory or bar.sync).
//
// Timing never changes what a warp executes (which entries issue, with which
// lanes, at which addresses), only when. The one interpretation (cache_pass
// 3) is therefore the real run -- stores land, every output but the timing is
// final -- and it logs each warp's issued runs of program entries and its
// accesses (line, step); the level kernels give every access its level. Here
// one thread per simulated warp walks the warp's runs again with no values:
// the in-order scoreboard of the interpreter (each issued entry at the
// latest of the next issue cycle and its terms' ready times; a global load
// whose access hit L1 or L2 takes that level's latency), and rewrites what
// timing decides -- the cycles of the warp's stats record and trace header,
// the timestamps of its trace records, its hit counts. An access is matched
// to the entry that made it by its step, the number of entries the warp had
// issued before it (a guarded load with no executing lane made none).
#include <cuda_runtime.h>

#include <algorithm>

#include "ks_internal.h"
#include "ks_rec.cuh"

namespace ks {
namespace {

constexpr uint32_t RF_ISSUE = 1, RF_RDEST = 2, RF_PDEST = 4, RF_PHAZ = 8, RF_LDG = 16, RF_EVENT = 32;

// A program entry as the replay reads it (32 bytes): ready-table indices of
// rows a, b (x), c, d (y) -- register slots, every other row on the one
// entry that stays 0 -- the predicates' (z: guard, sources; w: destination
// | flags << 8), then the destination, store and issue-clock latencies.
struct alignas(16) RRec {
  uint4 q;
  uint4 lat;
};

struct ReplayLaunch {
  const uint8_t* image;  // DevInsn program (unpatched latencies)
  uint32_t n_insn;       // program entries, the exit sentinel not included
  uint32_t n_slots;      // register slots (ready entries 0..n_slots-1; n_slots: the zero entry)
  uint32_t pred_off, row_bytes, split;
  uint32_t lat[KS_NUM_LAT_CLASSES];
  uint32_t lat_l1, lat_l2;
  uint32_t n_warps;
  const uint32_t* runs;    // runs logged per warp
  const uint32_t* runlog;  // [n_warps * run_cap]
  uint32_t run_cap;
  const ks_cache_access* acc;  // [n_warps * acc_cap], levels set
  uint32_t acc_cap;
  ks_cache_warp* cw;
  uint8_t* stats;  // ks_warp_stats per warp
  uint8_t* trace;  // may be null
  uint64_t slot_bytes;
  uint32_t rec_bytes, max_ts;
};

__device__ __forceinline__ uint32_t ready_index(uint32_t row, uint32_t n_slots) { return row < n_slots ? row : n_slots; }

__global__ void __launch_bounds__(256) cache_replay_kernel(const __grid_constant__ ReplayLaunch R) {
  extern __shared__ __align__(16) uint8_t sm[];
  RRec* prog = reinterpret_cast<RRec*>(sm);
  const uint32_t NE = R.n_slots + 1u + 32u;  // register slots, the zero entry, the predicates
  const uint32_t P = R.n_slots + 1u;         // first predicate entry
  // ready times, [warp of the block][entry][lane]: lanes reading one entry
  // hit 32 banks
  uint64_t* ready = reinterpret_cast<uint64_t*>(sm + (size_t)(R.n_insn + 1u) * sizeof(RRec));

  for (uint32_t i = threadIdx.x; i <= R.n_insn; i += blockDim.x) {
    const DevInsn d = reinterpret_cast<const DevInsn*>(R.image)[i];
    const PredTerms pt = pred_terms(d, R.split, R.pred_off);
    const EntryLat el = entry_lat(d, R.lat);
    uint32_t flags = 0;
    if (d.inc & INC_ISSUE) flags |= RF_ISSUE;
    if (d.inc & INC_RDEST) flags |= RF_RDEST;
    if (d.inc & INC_PDEST) flags |= RF_PDEST;
    if (d.inc & INC_PHAZ) flags |= RF_PHAZ;
    if (d.op == OP_LDG32 || d.op == OP_LDG64) flags |= RF_LDG;
    if (d.op == OP_EVENT) flags |= RF_EVENT;
    const uint32_t RB = R.row_bytes;
    RRec r;
    r.q.x = ready_index(d.a / RB, R.n_slots) | (ready_index(d.b / RB, R.n_slots) << 16);
    r.q.y = ready_index(d.c / RB, R.n_slots) | (ready_index(d.d / RB, R.n_slots) << 16);
    r.q.z = pt.guard | (pt.pa << 8) | (pt.pb << 16) | (pt.pc << 24);
    r.q.w = pt.pd | (flags << 8);
    r.lat = make_uint4(el.dest, el.store, el.next, 0u);
    prog[i] = r;
  }
  __syncthreads();

  const uint32_t lane = threadIdx.x & 31u;
  uint64_t* rt = ready + (size_t)(threadIdx.x >> 5) * NE * 32u + lane;  // entry e at rt[32 e]
  for (uint64_t gw = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; gw < R.n_warps;
       gw += (uint64_t)gridDim.x * blockDim.x) {
    ks_warp_stats* st = reinterpret_cast<ks_warp_stats*>(R.stats + gw * sizeof(ks_warp_stats));
    const uint32_t n_runs = R.runs[gw];
    // a log too small: the interpretation reported it, its cycles stand
    if (st->status == KS_ST_CACHE_LOG || n_runs > R.run_cap) continue;
    const uint32_t n_acc = R.cw[gw].n_access;
    if (n_acc > R.acc_cap) continue;
    for (uint32_t e = 0; e < NE; e++) rt[32u * e] = 0ull;
    uint64_t t_next = 0, t_last = 0, max_ready = 0, drain = 0, issued = 0;
    uint32_t k = 0, l1 = 0, l2 = 0, n_rec = 0;
    const ks_cache_access* A = R.acc + gw * R.acc_cap;
    uint64_t next_step = n_acc ? A[0].step : ~0ull;
    uint8_t* slot = R.trace ? R.trace + gw * R.slot_bytes : nullptr;
    const uint32_t* log = R.runlog + gw * R.run_cap;
    for (uint32_t r = 0; r < n_runs; r++) {
      const uint32_t run = log[r];
      uint32_t pc = run >> 16;
      const uint32_t len = (run & (RUN_DIVERGED - 1u)) + 1u;
      if (pc + len > R.n_insn) break;  // not a run the interpretation could log
      for (uint32_t j = 0; j < len; j++, pc++) {
        const RRec x = prog[pc];
        const uint32_t flags = (x.q.w >> 8) & 0xFFu;
        if (!(flags & RF_ISSUE)) {  // a trace pseudo-op: its record's timestamp
          if (flags & RF_EVENT) {
            if (slot && n_rec < R.max_ts) {
              uint32_t* w = reinterpret_cast<uint32_t*>(slot + 16u + R.rec_bytes * n_rec);
              *w = (*w & 0xFF000000u) | ((uint32_t)t_next & 0xFFFFFFu);
            }
            n_rec++;
          }
          continue;
        }
        uint64_t t = max(max(t_next, max(rt[32u * (x.q.x & 0xFFFFu)], rt[32u * (x.q.x >> 16)])),
                         max(max(rt[32u * (x.q.y & 0xFFFFu)], rt[32u * (x.q.y >> 16)]),
                             rt[32u * (P + (x.q.z & 0xFFu))]));
        if (flags & RF_PHAZ)
          t = max(t, max(max(rt[32u * (P + ((x.q.z >> 8) & 0xFFu))], rt[32u * (P + ((x.q.z >> 16) & 0xFFu))]),
                         max(rt[32u * (P + (x.q.z >> 24))], rt[32u * (P + (x.q.w & 0xFFu))])));
        uint32_t lat = x.lat.x;
        if (issued == next_step) {  // this entry made the warp's next access
          const uint32_t level = A[k].level;
          l1 += level == KS_CACHE_L1_HIT;
          l2 += level == KS_CACHE_L2_HIT;
          if (flags & RF_LDG) lat = level == KS_CACHE_L1_HIT ? R.lat_l1 : level == KS_CACHE_L2_HIT ? R.lat_l2 : lat;
          k++;
          next_step = k < n_acc ? A[k].step : ~0ull;
        }
        const uint64_t wr = t + lat;
        if (flags & RF_RDEST) rt[32u * (x.q.y >> 16)] = wr;
        if (flags & RF_PDEST) rt[32u * (P + (x.q.w & 0xFFu))] = wr;
        max_ready = max(max_ready, wr);
        drain = max(drain, t + x.lat.y);
        t_last = t;
        t_next = t + x.lat.z;
        issued++;
      }
    }
    const uint64_t cycles = issued ? max(max(t_last + 1u, max_ready), drain) : 0ull;
    st->cycles = cycles;
    if (slot) *reinterpret_cast<uint64_t*>(slot + 8) = cycles;
    ks_cache_warp c = R.cw[gw];
    c.l1_hits = l1;
    c.l2_hits = l2;
    c.dram = n_acc - l1 - l2;
    R.cw[gw] = c;
  }
}

}  // namespace

int launch_cache_replay(const KsLaunch& L, int sms, int max_smem, void* stream) {
  ReplayLaunch R;
  R.image = L.image;
  R.n_insn = L.n_insn;
  R.n_slots = L.n_slots;
  R.pred_off = L.layout.pred_off;
  R.row_bytes = L.layout.row_bytes;
  R.split = L.layout.split;
  for (int i = 0; i < KS_NUM_LAT_CLASSES; i++) R.lat[i] = L.lat[i];
  R.lat_l1 = L.lat_l1;
  R.lat_l2 = L.lat_l2;
  R.n_warps = L.n_warps;
  R.runs = L.sched_runs;
  R.runlog = L.sched_log;
  R.run_cap = L.sched_cap;
  R.acc = L.cache_log;
  R.acc_cap = L.cache_cap;
  R.cw = L.cache_warps;
  R.stats = L.stats;
  R.trace = L.trace;
  R.slot_bytes = L.slot_bytes;
  R.rec_bytes = L.rec_bytes;
  R.max_ts = L.max_ts;
  // Warps of threads per block: as many as shared memory allows (records,
  // then each thread's ready table), at most 8, and no more than it takes to
  // spread the simulated warps over every SM (each thread walks one warp's
  // whole issue log, so a small grid wants its threads on many SMs)
  const size_t prog = (size_t)(L.n_insn + 1u) * sizeof(RRec);
  const size_t per_warp = (size_t)(L.n_slots + 33u) * 32u * 8u;
  if (prog + per_warp > (size_t)max_smem) return (int)cudaErrorInvalidValue;
  const uint64_t per_sm = (L.n_warps + (uint64_t)std::max(sms, 1) - 1u) / (uint64_t)std::max(sms, 1);
  const uint32_t spread = (uint32_t)std::max<uint64_t>(1, std::min<uint64_t>(8, (per_sm + 31u) / 32u));
  const uint32_t warps = (uint32_t)std::min<size_t>(spread, ((size_t)max_smem - prog) / per_warp);
  const size_t smem = prog + per_warp * warps;
  cudaError_t e = cudaFuncSetAttribute(cache_replay_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return (int)e;
  const uint32_t threads = warps * 32u;
  const uint64_t want = (L.n_warps + threads - 1u) / threads;
  const uint32_t blocks = (uint32_t)std::max<uint64_t>(1, std::min<uint64_t>(want, (uint64_t)std::max(sms, 1) * 4u));
  void* args[] = {&R};
  return (int)cudaLaunchKernel((const void*)cache_replay_kernel, dim3(blocks), dim3(threads), args, smem,
                               (cudaStream_t)stream);
}

}  // namespace ks

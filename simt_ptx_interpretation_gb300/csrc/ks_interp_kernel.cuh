// ks_interp_kernel.cuh — the sm_103a warp-level SIMT interpreter kernel.
//
// One real warp interprets one simulated warp at a time, one real lane per
// simulated lane (KernelScope backend doc, simulator/models.py: a warp is 32
// threads executing in lockstep under an active mask). Real warps are
// persistent: warp j of the launch takes simulated warps j, j + R, j + 2R...
// (R real warps in the grid), so the real launch shape is chosen for the GPU
// while the simulated grid and block only change what %tid/%ctaid read.
//
// Per real CTA, shared memory holds
//   [program: 64-byte DevInsn records | constant row values]
//   [parameter block | mbarrier | barrier-round control block]
//   [one region per warp: register rows | constant rows | zero row |
//    predicate ready table | reconvergence stack]   (layout in ks_internal.h)
//   [simulated shared memory of the CTA]             (CTA mode only)
// The program image is staged once per CTA with one cp.async.bulk
// global->shared copy completing on an mbarrier; the wait is bounded and
// reports KS_ST_TIMEOUT instead of hanging. The launch's latency table is then
// patched into the staged instructions.
//
// Every operand field of an instruction is the offset of a row of the warp's
// region, so registers, constants (replicated across the row) and "no
// operand" (the zero row) look the same. Two layouts (ks_internal.h; the
// SPLIT template parameter):
//  - PAIR: a 256-byte row holds one (value, ready) pair per lane, so lane l
//    reads an operand and its scoreboard entry with one 8-byte shared load at
//    (region + offset + 8l). A destination's ready time alone (the
//    write-after-write wait) is read from lane 0's pair by every lane: one
//    broadcast word instead of a strided load of two wavefronts.
//  - SPLIT: a 128-byte row holds the values (one 4-byte load per lane at
//    region + offset + 4l), and the warp-uniform ready times live apart, one
//    word per row and per predicate; an instruction's terms (its rows,
//    destination, guard and predicate sources) are gathered one per lane --
//    lane l loads the ready word named by halfword l mod 4 (fast and mid
//    loops) or l mod 8 (general path) of the record -- and one redux.sync max
//    gives the latest. Half the shared memory per warp, for kernels whose
//    regions would bound the resident warps; a few more instructions per
//    simulated instruction.
//
// Kernels with shared memory or bar.sync run in CTA mode (the CTA template
// instantiation): one real CTA per simulated CTA, one real warp per simulated
// warp, and barrier rounds between them (KernelScope backend doc,
// simulator/models.py Block and Warp.at_barrier).
//
// Warp-uniform state (pc, active mask, scoreboard clock, counters) lives in
// registers, identical in every lane; values every lane must agree on (ready
// times, stack entries) are written by all lanes with the same value, and the
// warp's shared-memory accesses complete in program order, so a lane may read
// any lane's copy (the predicate ready table and a destination's ready time
// are read as one broadcast word). Predicates are per-warp ballot
// masks, predicate p held by lane p (lane 31 holds the always-true predicate)
// and read with a shuffle. The scoreboard clock is 32-bit relative to a 64-bit
// epoch that moves forward before any clock reaches 2^31.
#pragma once

#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <type_traits>

#include "ks_internal.h"

namespace ks {

namespace {

constexpr uint32_t FULL = 0xFFFFFFFFu;
constexpr uint32_t WAIT_SPINS = 1u << 22;

__device__ __forceinline__ uint32_t cvta_shared(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(cvta_shared(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(cvta_shared(bar)), "r"(bytes)
               : "memory");
}

// Bulk (non-tensor) TMA copy global -> shared, completion counted on `bar`.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          cvta_shared(dst)),
      "l"(src), "r"(bytes), "r"(cvta_shared(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(cvta_shared(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait on phase 0 of the staging barrier.
__device__ __forceinline__ bool wait_staged(uint64_t* bar) {
  for (uint32_t i = 0; i < WAIT_SPINS; i++)
    if (mbar_try_wait(bar, 0)) return true;
  return false;
}

__device__ __forceinline__ uint32_t fbits(float f) {
  return (f != f) ? 0x7FFFFFFFu : __float_as_uint(f);  // canonical NaN
}

// The bits of an f32 result of one hardware FFMA / FADD / FMUL: every NaN
// such an instruction writes on this GPU is already the canonical 0x7FFFFFFF,
// whatever NaNs its operands hold (payloads, either sign, quiet or
// signalling), so the canonical-NaN rule costs no compare and select on the
// datapaths' chains (held by parity tests with NaN-payload operands in the
// fast, mid and general paths). Division and square root keep fbits.
__device__ __forceinline__ uint32_t fbits_hw(float f) { return __float_as_uint(f); }

__device__ __forceinline__ uint64_t f2i(float f, uint32_t flags) {
  if (f != f) return 0;
  const uint32_t rnd = flags >> 4, kind = flags & 15;
  float x = rnd == RND_RNI ? rintf(f) : rnd == RND_RZI ? truncf(f) : rnd == RND_RMI ? floorf(f) : ceilf(f);
  switch (kind) {
    case CVT_S32:
      if (x >= 2147483648.0f) return 0x7FFFFFFFull;
      if (x < -2147483648.0f) return 0x80000000ull;
      return (uint64_t)(uint32_t)(int32_t)x;
    case CVT_U32:
      if (x >= 4294967296.0f) return 0xFFFFFFFFull;
      if (x < 0.0f) return 0;
      return (uint64_t)(uint32_t)x;
    case CVT_S64:
      if (x >= 9223372036854775808.0f) return 0x7FFFFFFFFFFFFFFFull;
      if (x < -9223372036854775808.0f) return 0x8000000000000000ull;
      return (uint64_t)(int64_t)x;
    default:
      if (x >= 18446744073709551616.0f) return 0xFFFFFFFFFFFFFFFFull;
      if (x < 0.0f) return 0;
      return (uint64_t)x;
  }
}

// Comparison results from the three relations. Bit c of each mask is the
// result of comparison code c (eq, ne, lt, le, gt, ge) when that relation holds;
// an unordered f32 pair holds none of them, so every code is false (ordered
// comparisons).
constexpr uint32_t REL_LT = 0x0Eu;  // ne lt le
constexpr uint32_t REL_EQ = 0x29u;  // eq le ge
constexpr uint32_t REL_GT = 0x32u;  // ne gt ge
__device__ __forceinline__ bool rel_result(bool lt, bool eq, bool gt, uint32_t c) {
  return (((lt ? REL_LT : 0u) | (eq ? REL_EQ : 0u) | (gt ? REL_GT : 0u)) >> c) & 1u;
}

// Translates a simulated address for a `size`-byte access; 0 or a status.
__device__ __forceinline__ int translate(const KsLaunch& L, uint64_t va, uint32_t size, uint8_t** ptr) {
  if (va & (uint64_t)(size - 1)) return KS_ST_MISALIGNED;
#pragma unroll
  for (uint32_t b = 0; b < KS_MAX_BUFFERS; b++) {
    if (b < L.n_bufs) {
      const uint64_t base = L.bufs[b].sim_base, bytes = L.bufs[b].bytes;
      if (va >= base && bytes >= size && va - base <= bytes - size) {
        *ptr = L.bufs[b].ptr + (va - base);
        return 0;
      }
    }
  }
  return KS_ST_OOB;
}

// Predicated 32-bit shared store (no branch around the per-lane condition).
__device__ __forceinline__ void st_shared_if(bool p, uint32_t addr, uint32_t v) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %0, 0;\n\t@q st.shared.u32 [%1], %2;\n\t}" ::"r"((uint32_t)p),
      "r"(addr), "r"(v)
      : "memory");
}

// PAIR layout: stores (value, ready) for a lane that executes and only
// `ready` for one that does not (the scoreboard entry is written in every lane).
__device__ __forceinline__ void st_pair(bool on, uint32_t addr, uint32_t v, uint32_t ready) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %0, 0;\n\t"
      "@q st.shared.v2.u32 [%1], {%2, %3};\n\t"
      "@!q st.shared.u32 [%1+4], %3;\n\t}" ::"r"((uint32_t)on),
      "r"(addr), "r"(v), "r"(ready)
      : "memory");
}

#define SM32(off) (*reinterpret_cast<uint32_t*>(smem + (off)))
#define SM2(off) (*reinterpret_cast<const uint2*>(smem + (off)))
#define SM64(off) (*reinterpret_cast<uint64_t*>(smem + (off)))
// warp-region accesses (shared memory, or global memory under GREG)
#define RG32(off) (*reinterpret_cast<uint32_t*>(rg + (off)))
#define RG2(off) (*reinterpret_cast<const uint2*>(rg + (off)))
#define RG64(off) (*reinterpret_cast<uint64_t*>(rg + (off)))
// predicated region stores at lv + x / wb + x, and a (value, ready) pair at lv + x
#define ST_LANE_IF(p, x, v)                                    \
  do {                                                         \
    if constexpr (GREG) { if (p) RG32(lv + (x)) = (v); }       \
    else st_shared_if((p), s_lane + (x), (v));                 \
  } while (0)
#define ST_WB_IF(p, x, v)                                      \
  do {                                                         \
    if constexpr (GREG) { if (p) RG32(wb + (x)) = (v); }       \
    else st_shared_if((p), s_wb + (x), (v));                   \
  } while (0)
#define ST_LANE_PAIR(p, x, v, r)                               \
  do {                                                         \
    if constexpr (GREG) {                                      \
      if (p) RG32(lv + (x)) = (v);                             \
      RG32(lv + (x) + 4u) = (r);                               \
    } else {                                                   \
      st_pair((p), s_lane + (x), (v), (r));                    \
    }                                                          \
  } while (0)
// this lane's scoreboard-term offset in the record at `rec` (a const uint4*):
// halfword `hsel` (bytes) of its hazard words
#define HZ_AT(rec, hsel) \
  ((uint32_t)*reinterpret_cast<const uint16_t*>(reinterpret_cast<const uint8_t*>(rec) + (hsel)))

constexpr uint32_t REBASE_AT = 1u << 30;
constexpr uint64_t BUDGET_CHUNK = 1ull << 30;

// Barrier rounds of a CTA-mode launch: the latest bar.sync issue cycle of the
// round (absolute, two rounds in flight), the count of finished warps, and
// (cache model) 1 + the last step issued in the round by a warp that arrived
// or finished.
struct CtaCtl {
  unsigned long long latest[2];
  unsigned int done;
  unsigned int pad;
  unsigned long long step_end[2];
};
constexpr uint32_t CTL_BYTES = 48;

__host__ __device__ __forceinline__ uint32_t region0(uint32_t image_bytes) {
  return (image_bytes + KS_MAX_PARAM_BYTES + 16u + CTL_BYTES + 127u) / 128u * 128u;
}

__device__ __forceinline__ uint64_t pack_entry(uint32_t pc, uint32_t rpc, uint32_t mask) {
  return (uint64_t)(pc & 0xFFFFu) | ((uint64_t)(rpc & 0xFFFFu) << 16) | ((uint64_t)mask << 32);
}

}  // namespace

// CTA: the launch runs kernels with shared memory or bar.sync (one real CTA
// per simulated CTA, barrier rounds, shared-memory handlers); compiled apart
// so that the other kernels keep the register budget of the plain loop. BIG:
// CTA mode for blocks of 9..32 warps (a 1024-thread real CTA, at most 64
// registers a thread, so it spills: slower, used only for such blocks). The
// plain forms take CTAs of up to 12 warps.
// NB: launches per real grid (1, or KS_BATCH_ITEMS for ks_simulate_batch);
// each real CTA runs the item whose CTA range holds it, as if that item's
// CTAs were a grid of their own.
// CAP: compiled for more CTAs per SM where registers, not shared memory,
// bound the resident warps: plain, two CTAs of up to 10 warps (96
// registers, no spills, 21 warps an SM); CTA mode, three CTAs of up to 8
// warps (80 registers, a few spills, 24 warps an SM).
// SPLIT: the SPLIT register-file layout (plain mode only).
// GREG: CTA mode whose warps' state does not fit the SM's shared memory: the
// warp regions live in global memory (L.greg, one slice per real CTA, cached
// in L1/L2), the program, parameters, barrier control and simulated shared
// memory stay in shared memory (1024-thread form, single launches, PAIR).
template <bool CTA, bool BIG, bool INSTR, bool RUNLOG, uint32_t NB, bool CAP = false, bool SPLIT = false,
          bool GREG = false>
__global__ void __launch_bounds__(CAP ? (CTA ? 256 : 320) : (BIG ? 1024 : (CTA ? 256 : 384)), CAP ? (CTA ? 3 : 2) : 1)
    ks_interp_kernel(const __grid_constant__ KsGrid<NB> G) {
  static_assert(!(SPLIT && CTA), "CTA mode runs in the PAIR layout");
  static_assert(!GREG || (CTA && BIG && !SPLIT && NB == 1 && !CAP), "global warp state: single CTA-mode launches");
  uint32_t item = 0;
  if constexpr (NB > 1) {
    while (item + 1u < G.n && blockIdx.x >= G.cta_begin[item + 1u]) item++;  // uniform in the CTA
  }
  const KsLaunch& L = G.item[item];
  const uint32_t cta_x = NB > 1 ? blockIdx.x - G.cta_begin[item] : blockIdx.x;
  const uint32_t n_ctas = NB > 1 ? G.cta_begin[item + 1u] - G.cta_begin[item] : gridDim.x;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t wid = threadIdx.x >> 5;
  const uint32_t nwarps = blockDim.x >> 5;
  const DevLayout& Y = L.layout;

  uint8_t* s_params = smem + L.image_bytes;
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(smem + L.image_bytes + KS_MAX_PARAM_BYTES);
  CtaCtl* ctl = reinterpret_cast<CtaCtl*>(smem + L.image_bytes + KS_MAX_PARAM_BYTES + 16u);
  constexpr bool cta_mode = CTA;
  // simulated shared memory, after the warp regions (GREG: no regions here)
  const uint32_t sh_base = region0(L.image_bytes) + (GREG ? 0u : nwarps * Y.region_bytes);
  // the warp regions: shared memory from region0, or (GREG) this CTA's slice
  // of L.greg from 0; region accesses go through rg
  uint8_t* const rg = GREG ? L.greg + (uint64_t)cta_x * nwarps * Y.region_bytes : smem;
  const uint32_t wb = (GREG ? 0u : region0(L.image_bytes)) + wid * Y.region_bytes;  // this warp's region
  constexpr uint32_t RB = SPLIT ? ROW_SPLIT : ROW_PAIR;               // row bytes
  const uint32_t lv = wb + lane * (SPLIT ? 4u : 8u);                   // this lane's value in row 0
  [[maybe_unused]] const uint32_t s_lane = cvta_shared(smem) + lv;     // shared-window address of lv
  [[maybe_unused]] const uint32_t s_wb = cvta_shared(smem) + wb;       // ... of the region
  // where a lane reads a destination's ready time: lane 0's pair (one
  // broadcast word), or under GREG its own pair (global memory gives no
  // order between one lane's store and another lane's load)
  [[maybe_unused]] const uint32_t rdb = GREG ? lv : wb;
  [[maybe_unused]] const uint32_t pg = wb + Y.pred_off;                // predicate ready table
  // SPLIT: the scoreboard-term halfword this lane gathers: of four (fast and
  // mid loops: rows a, b, c, destination) or of eight (general path: then the
  // guard and the predicate sources); the lanes that hold the destination's
  // term write its ready time
  [[maybe_unused]] const uint32_t hs4 = DEV_HZ_OFF + 2u * (lane & 3u), hs8 = DEV_HZ_OFF + 2u * (lane & 7u);
  [[maybe_unused]] const bool is_d4 = (lane & 3u) == 3u, is_d8 = (lane & 7u) == 3u;

  // ---- stage the program once per CTA (a1) ----
  if (threadIdx.x == 0) {
    mbar_init(s_bar, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(s_bar, L.image_bytes);
    bulk_copy_g2s(smem, L.image, L.image_bytes, s_bar);
  }
  for (uint32_t i = threadIdx.x; i < KS_MAX_PARAM_BYTES / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(s_params)[i] = reinterpret_cast<const uint32_t*>(L.params)[i];
  const bool staged = __all_sync(FULL, wait_staged(s_bar));
  __syncthreads();
  // patch this launch's latencies into the program
  if (staged) {
    for (uint32_t i = threadIdx.x; i <= L.n_insn; i += blockDim.x) {
      DevInsn* p = reinterpret_cast<DevInsn*>(smem) + i;
      const uint32_t f = p->wlat, lat = L.lat[f & 0xFFu];
      p->wlat = (f & DEV_HAS_DEST) ? lat : 0u;
      p->x[DX_DLAT] = (f & DEV_IS_STORE) ? lat : 0u;
      p->x[DX_NLAT] = p->inc ? ((f & DEV_IS_CTRL) ? lat : 1u) : 0u;
    }
  }
  // constant rows and the zero row of this warp's region (read-only afterwards)
  {
    const uint32_t* vals = reinterpret_cast<const uint32_t*>(smem + L.prog_bytes);
    if constexpr (SPLIT) {
      for (uint32_t r = 0; r < Y.n_crows; r++) RG32(lv + Y.const_off + r * RB) = vals[r];
      RG32(lv + Y.zero_off) = 0u;
    } else {  // (value, ready = 0) pairs
      for (uint32_t r = 0; r < Y.n_crows; r++) RG64(lv + Y.const_off + r * RB) = (uint64_t)vals[r];
      RG64(lv + Y.zero_off) = 0ull;
    }
  }
  __syncthreads();

  const uint32_t exit_pc = L.n_insn;

  // simulated (CTA, warp-in-CTA) of this real warp's first simulated warp, and
  // the real-warp stride split the same way (no division per simulated warp)
  const uint32_t gw_stride = n_ctas * nwarps;
  const uint32_t step_cta = gw_stride / L.wpc, step_wic = gw_stride - step_cta * L.wpc;
  uint32_t cta = (cta_x * nwarps + wid) / L.wpc;
  uint32_t wic = (cta_x * nwarps + wid) - cta * L.wpc;
  uint32_t hint = 0;  // buffer of the last simulated access (tried first)
  // Outside CTA mode a real warp runs its simulated warps one after another
  // in one region. In the PAIR layout the first starts from a zeroed region
  // at clock 0; each later one zeroes only the slots it may read before
  // writing (the decoder's live-in set) and starts its clock at t_floor, the
  // latest time the region holds (every ready time left behind is at most
  // that, so none delays it), with its epoch at -t_floor so that its cycles
  // and timestamps still count from its own start. (The SPLIT form zeroes
  // every warp's region: the floor's registers would cost it resident warps.)
  constexpr bool FLOOR = !CTA && !SPLIT;
  bool region_fresh = false;
  uint32_t t_floor = 0;

  for (uint32_t gw = cta_x * nwarps + wid; gw < L.n_warps;
       gw += gw_stride, cta += step_cta, wic += step_wic, cta += (wic >= L.wpc), wic -= (wic >= L.wpc) ? L.wpc : 0u) {
    const uint32_t tid_sim = wic * 32u + lane;
    if (cta_mode) {
      // A new simulated CTA on this real CTA (one real warp per simulated
      // warp, so every warp of the CTA is here): zeroed shared memory, fresh
      // barrier rounds. The previous CTA's warps have all left its last round.
      for (uint32_t i = threadIdx.x; i < (L.shared_bytes + 3u) / 4u; i += blockDim.x) SM32(sh_base + 4u * i) = 0u;
      if (threadIdx.x == 0) {
        ctl->latest[0] = 0ull;
        ctl->latest[1] = 0ull;
        ctl->done = 0u;
        ctl->step_end[0] = 0ull;
        ctl->step_end[1] = 0ull;
      }
      __syncthreads();
    }

    // ---- warp set-up (a1): registers zero, predicates false, clock 0 ----
    if (!FLOOR || !region_fresh) {
      if constexpr (SPLIT) {
        for (uint32_t s = 0; s < Y.n_slots; s++) RG32(lv + s * RB) = 0u;
        for (uint32_t i = lane; i < Y.n_ready; i += 32u) RG32(wb + Y.ready_off + 4u * i) = 0u;
      } else {
        for (uint32_t s = 0; s < Y.n_slots; s++) RG64(lv + s * RB) = 0ull;
        RG32(pg + lane * 4u) = 0u;
      }
      region_fresh = true;
      t_floor = 0;
    } else {
      for (uint32_t w = 0; w < 4u; w++)
        for (uint32_t m = L.live_in[w]; m; m &= m - 1u) RG32(lv + (32u * w + (uint32_t)(__ffs(m) - 1)) * RB) = 0u;
    }
    __syncwarp();
    uint32_t my_pred = (lane == 31u) ? 0xFFFFFFFFu : 0u;  // predicate 31 is always true
    uint32_t pc = 0, rpc = exit_pc;
    uint32_t mask = __ballot_sync(FULL, tid_sim < L.block);
    uint32_t depth = 1, max_depth = 1;
    uint64_t sh_req = 0, sh_wf = 0;  // shared requests, their bank-conflict degrees
    bool at_bar = false, finished = false;
    uint64_t cyc_floor = 0;           // cycles owed to before a barrier's epoch move
    uint64_t epoch = 0ull - (uint64_t)t_floor;
    uint32_t t_next = t_floor, t_last = t_floor, max_ready = t_floor, drain = t_floor;
    uint64_t thread_insts = 0;
    uint64_t ld_req = 0, ld_sec = 0, st_req = 0, st_sec = 0, ld_lin = 0, st_lin = 0;
    uint32_t n_events = 0, n_rec = 0, n_dropped = 0;
    int status = staged ? 0 : KS_ST_TIMEOUT;
    // cache model: accesses made (c_k), hits, the first pass's count (c_n),
    // and the steps spent waiting at barriers (an access's step is c_off +
    // the instructions its warp issued before it)
    uint32_t c_k = 0, c_l1 = 0, c_l2 = 0, c_n = 0;
    uint64_t c_off = 0;
    // SM issue model: the run of consecutive program entries being consumed
    // [run_start, run_next) and the runs logged so far; `live` = the lanes
    // that have not executed ret, and run_div whether the run issues while
    // some of them wait on the stack (mask != live, the divergence label)
    uint32_t run_start = 0, run_next = 0, n_runs = 0;
    [[maybe_unused]] uint32_t live = mask, run_div = 0;
    if constexpr (INSTR) {
      if (L.cache_pass == 2) {
        c_n = L.cache_warps[gw].n_access;
        if (c_n > L.cache_cap && status == 0) status = KS_ST_CACHE_LOG;
      }
    }
    uint8_t* slot = L.trace ? L.trace + (uint64_t)gw * L.slot_bytes : nullptr;
    const bool injected = L.inject_warp >= 0 && (uint64_t)L.inject_warp == gw;
    const uint64_t stop_at = (injected && L.inject_step < L.step_limit) ? L.inject_step : L.step_limit;
    // Issued-instruction accounting: `budget` counts down the instructions
    // that may issue before the next check point (chunks of at most 2^30),
    // `left` those after it; issued = stop_at - left - budget. thread_insts
    // is accumulated at every active-mask change from the instructions issued
    // since `mark` (a budget value) times the lanes of the mask they ran with.
    uint32_t budget = (uint32_t)(stop_at < BUDGET_CHUNK ? stop_at : BUDGET_CHUNK);
    uint64_t left = stop_at - budget;
    uint32_t mark = budget;
#define FLUSH_THREADS()                                                 \
  do {                                                                  \
    thread_insts += (uint64_t)(mark - budget) * (uint64_t)__popc(mask); \
    mark = budget;                                                      \
  } while (0)

    for (uint32_t round = 0;; round++) {  // barrier rounds (one pass outside CTA mode)
    if (status == 0 && !finished) for (;;) {
      // pop finished entries (a6); every control condition below is warp-uniform
      // in value
      if (pc == rpc || mask == 0) {
        FLUSH_THREADS();
        if (depth == 1) break;
        depth--;
        const uint64_t e = RG64(wb + Y.stack_off + (depth - 1) * 8u);
        pc = (uint32_t)(e & 0xFFFFu);
        rpc = (uint32_t)((e >> 16) & 0xFFFFu);
        mask = (uint32_t)(e >> 32);
        continue;
      }
      // fetch (a2): the first half of the record decides the path. The active
      // mask is not empty and pc is not the reconvergence pc here; `fuel_in` =
      // instructions that may run before the reconvergence pc or the end of the
      // step budget.
      if constexpr (RUNLOG) {
        const uint32_t div = mask != live ? RUN_DIVERGED : 0u;
        if (pc != run_next || div != run_div) {  // a new run: log the one that ended
          if (run_next != run_start) {
            if (lane == 0 && n_runs < L.sched_cap)
              L.sched_log[(uint64_t)gw * L.sched_cap + n_runs] =
                  (run_start << 16) | run_div | (run_next - run_start - 1u);
            n_runs++;
          }
          run_start = run_next = pc;
          run_div = div;
        }
      }
      const uint4* ip = reinterpret_cast<const uint4*>(smem + pc * (uint32_t)sizeof(DevInsn));
      const uint4 q0 = ip[0], q1 = ip[1], q3 = ip[3];
      // PAIR: guard, gneg, ha, hb (SPLIT: the hazard halfwords, gathered per lane)
      const uint4 q2 = SPLIT ? make_uint4(0u, 0u, 0u, 0u) : ip[2];
      const uint32_t fuel_in = min(budget, rpc > pc ? rpc - pc : 0xFFFFFFFFu);
      const bool runnable = fuel_in != 0u && t_next < REBASE_AT;

      // ---- a setp fused with the bra after it (32-bit or f32 compare): the
      // setp issues here as the general path issues it, and the bra with it
      // when every active lane goes the same way (else the bra takes the
      // general path next), without the general path's operand loads and
      // dispatch. The setp is unguarded, so every active lane executes it.
      if (runnable && (q1.w & INC_FUSE) && (q0.x == OP_SETP_U32 || q0.x == OP_SETP_S32 || q0.x == OP_SETP_F32)) {
        // operands (PAIR: with their ready times); SPLIT: this lane's term
        // offset and term
        const uint2 sa2 = SPLIT ? make_uint2(RG32(lv + q1.x), 0u) : RG2(lv + q1.x);
        const uint2 sb2 = SPLIT ? make_uint2(RG32(lv + q1.y), 0u) : RG2(lv + q1.y);
        const uint32_t sa = sa2.x, sb = sb2.x;
        const uint32_t hk = SPLIT ? HZ_AT(ip, hs4) : 0u;
        const uint32_t hr = SPLIT ? RG32(wb + hk) : 0u;
        const uint32_t sop = q0.x, saux = q0.z, cmp = saux & 0xFFu, pd = (saux >> 8) & 0xFFu;
        bool lt, eq, gt;
        if (sop == OP_SETP_F32) {
          const float x = __uint_as_float(sa), y = __uint_as_float(sb);
          lt = x < y; eq = x == y; gt = x > y;
        } else {
          const uint32_t flip = sop == OP_SETP_S32 ? 0x80000000u : 0u;  // signed order
          const uint32_t x = sa ^ flip, y = sb ^ flip;
          lt = x < y; eq = x == y; gt = x > y;
        }
        const uint32_t bal = __ballot_sync(FULL, rel_result(lt, eq, gt, cmp));
        // its scoreboard: the sources, and the predicate it writes (the
        // other terms of an unguarded setp are the always-true predicate and
        // the zero row, ready at 0)
        uint32_t t, wr;
        if constexpr (SPLIT) {
          t = max(t_next, __reduce_max_sync(FULL, hr));
          wr = t + q0.y;
          ST_WB_IF(is_d4, hk, wr);
        } else {  // PAIR: ready times in the rows' pairs, the predicate's in q3.y (hd)
          t = max(max(t_next, sa2.y), max(sb2.y, RG32(wb + q3.y)));
          wr = t + q0.y;
          RG32(wb + q3.y) = wr;
        }
        if (lane == pd) my_pred = (my_pred & ~mask) | (bal & mask);
        max_ready = max(max_ready, wr);
        drain = max(drain, t + q3.z);
        t_last = t;
        t_next = t + q3.w;
        budget--;
        const uint32_t pc_setp = pc;
        pc++;
        const uint32_t taken = mask & (bal ^ (((saux >> 16) & 1u) ? 0xFFFFFFFFu : 0u));
        if ((taken == mask || taken == 0u) && budget != 0u && pc != rpc && t_next < REBASE_AT) {
          const uint32_t t2 = max(t_next, wr);  // the bra waits for its guard
          max_ready = max(max_ready, t2);
          drain = max(drain, t2);
          t_last = t2;
          t_next = t2 + L.lat[KS_LAT_BRA];
          budget--;
          pc = taken ? (saux >> 17) : pc + 1u;
          if constexpr (RUNLOG) run_next = pc_setp + 2u;
        } else {
          if constexpr (RUNLOG) run_next = pc_setp + 1u;
        }
        continue;
      }

      // ---- fast path: runs of unguarded routed FPU / IMAD instructions.
      // pc, budget and t_last are rebuilt when the run ends. Software-pipelined
      // in three stages: while instruction k executes, the operand rows (and
      // SPLIT: scoreboard terms) of k+1 are loaded and the record of k+2
      // fetched; k+1's loads may predate k's stores, so k's result goes into
      // any operand of k+1 that is k's destination and k's ready time into
      // k+1's scoreboard (PAIR: by comparing row offsets; SPLIT: as the
      // decoder's INC_FWD_* flags say).
      // The run is counted up front: at most the consecutive fast ops from pc
      // (inc >> 16), the fuel, and as many steps as keep every clock below
      // REBASE_AT (each step moves the clock by at most the largest fast-op
      // latency, which 2^fast_shift bounds).
      const uint32_t run_cap = max(t_next, max_ready) < REBASE_AT
                                   ? (REBASE_AT - max(t_next, max_ready)) >> L.fast_shift : 0u;
      const uint32_t run_n = min(min(fuel_in, q1.w >> INC_RUN_SHIFT), run_cap);
      if (t_next < REBASE_AT && run_n != 0u && (q0.x | 1u) == DOP_IMAD) {
        if constexpr (SPLIT) {
          uint32_t n = run_n;
          const bool on_all = (mask >> lane) & 1u;
          // instruction k: {op, wlat, aux, d}, {a, b, c, inc}; its operand
          // values, this lane's term offset and the latest term
          uint4 ka = q0, kb = q1;
          uint32_t a = RG32(lv + kb.x), b = RG32(lv + kb.y), c = RG32(lv + kb.z);
          uint32_t hk = HZ_AT(ip, hs4);
          uint32_t hm = __reduce_max_sync(FULL, RG32(wb + hk));
          // instruction k+1's record and term offset (the last instruction is
          // never a fast op, so k+1 and k+2 stay within the program and its
          // exit sentinel)
          uint4 na = ip[4], nb = ip[5];
          uint32_t hk1 = HZ_AT(ip + 4, hs4);
          for (;;) {
            uint32_t a1 = RG32(lv + nb.x), b1 = RG32(lv + nb.y), c1 = RG32(lv + nb.z);
            const uint32_t r1 = RG32(wb + hk1);
            const uint4 ma = ip[8], mb = ip[9];
            const uint32_t hk2 = HZ_AT(ip + 8, hs4);
            const uint32_t t = max(t_next, hm);
            const uint32_t wr = t + ka.y;
            max_ready = max(max_ready, wr);
            t_next = t + 1u;
            const uint32_t cx = c ^ ka.z;
            const uint32_t rf = fbits_hw(__fmaf_rn(__uint_as_float(a), __uint_as_float(b), __uint_as_float(cx)));
            const uint32_t ri = a * b + cx;
            const uint32_t res = ka.x == DOP_FPU ? rf : ri;
            ST_LANE_IF(on_all, ka.w, res);
            ST_WB_IF(is_d4, hk, wr);  // the destination's ready word
            // forward k into k+1 (in every lane: a lane outside the mask
            // stores nothing during the run)
            const uint32_t f = nb.w;
            a1 = (f & INC_FWD_A) ? res : a1;
            b1 = (f & INC_FWD_B) ? res : b1;
            c1 = (f & INC_FWD_C) ? res : c1;
            const uint32_t hm1 = __reduce_max_sync(FULL, r1);
            hm = (f & INC_FWD_T) ? max(hm1, wr) : hm1;
            ka = na;
            kb = nb;
            na = ma;
            nb = mb;
            a = a1;
            b = b1;
            c = c1;
            hk = hk1;
            hk1 = hk2;
            ip += 4;
            if (--n == 0u) break;  // uniform in value
          }
          pc += run_n;
          budget -= run_n;
          t_last = t_next - 1u;
          if constexpr (RUNLOG) run_next = pc;
          continue;
        } else {
          // The loop in three forms: with the destination's ready word as a
          // scoreboard term; without it (runs whose every op writes a row it
          // reads, INC_OWN_D: that term is one of the rows'); and, in such
          // runs, for a prefix that keeps reading the same b and c rows,
          // without their loads either (below). The register-capped forms
          // keep the first only (their launches are bound by registers,
          // which the other copies would raise).
          const bool on_all = (mask >> lane) & 1u;
          // n ops from ip on, the first one's record halves k0, k1
          auto pair_run = [&](auto with_rd, uint32_t n, const uint4 k0, const uint4 k1) {
            constexpr bool RD = decltype(with_rd)::value;
            // instruction k: {op, wlat, aux, d}, {a, b, c, inc}; its rows
            uint4 ka = k0, kb = k1;
            uint2 a = RG2(lv + kb.x), b = RG2(lv + kb.y), c = RG2(lv + kb.z);
            uint32_t rd = RD ? RG32(rdb + ka.w + 4u) : 0u;
            // instruction k+1 (the last instruction is never a fast op, so k+1
            // and k+2 stay within the program and its exit sentinel)
            uint4 na = ip[4], nb = ip[5];
            for (;;) {
              uint2 a1 = RG2(lv + nb.x), b1 = RG2(lv + nb.y), c1 = RG2(lv + nb.z);
              uint32_t rd1 = RD ? RG32(rdb + na.w + 4u) : 0u;
              const uint4 ma = ip[8], mb = ip[9];
              const uint32_t t = max(max(t_next, a.y), max(max(b.y, c.y), rd));
              const uint32_t wr = t + ka.y;
              max_ready = max(max_ready, wr);
              t_next = t + 1u;
              const uint32_t cx = c.x ^ ka.z;
              const uint32_t rf = fbits_hw(__fmaf_rn(__uint_as_float(a.x), __uint_as_float(b.x), __uint_as_float(cx)));
              const uint32_t ri = a.x * b.x + cx;
              const uint32_t res = ka.x == DOP_FPU ? rf : ri;
              ST_LANE_PAIR(on_all, ka.w, res, wr);
              // forward k into k+1 (the decoder's INC_FWD_* flags of k+1): the
              // value into each operand that is k's destination -- in every
              // lane: a lane outside the mask stores nothing during the run,
              // so what it computes from a forwarded value is never seen --
              // and k's ready time into k+1's scoreboard, through the
              // destination term (every term of k+1 is maxed together, and a
              // stale entry of k's destination is never later than k's own
              // ready time)
              const uint32_t f = nb.w;
              a1.x = (f & INC_FWD_A) ? res : a1.x;
              b1.x = (f & INC_FWD_B) ? res : b1.x;
              c1.x = (f & INC_FWD_C) ? res : c1.x;
              if constexpr (RD) rd1 = (f & INC_FWD_T) ? max(rd1, wr) : rd1;
              else rd1 = (f & INC_FWD_T) ? wr : 0u;
              ka = na;
              kb = nb;
              na = ma;
              nb = mb;
              a = a1;
              b = b1;
              c = c1;
              rd = rd1;
              ip += 4;
              if (--n == 0u) break;  // uniform in value
            }
          };
          if (CAP || !(q1.w & INC_OWN_D)) {
            pair_run(std::true_type{}, run_n, q0, q1);
          } else {
            // A run prefix whose ops read the same b and c rows (q3.x: hc of
            // a fast op), which no op of it but the last writes: those rows
            // are loaded once, and only a, the record and the result move
            // per op (then the rest of the run, its rows loaded afresh).
            const uint32_t keep = min(run_n, q3.x & KEEP_COUNT);
            // FPU: every op of the prefix is an f32 op (no integer datapath)
            auto keep_run = [&](auto fpu_only) {
              constexpr bool FPU = decltype(fpu_only)::value;
              uint32_t n = keep;
              uint4 ka = q0, kb = q1;
              uint2 a = RG2(lv + kb.x);
              const uint2 b = RG2(lv + kb.y), c = RG2(lv + kb.z);
              uint32_t rd = 0;
              uint4 na = ip[4], nb = ip[5];
              for (;;) {
                uint2 a1 = RG2(lv + nb.x);
                const uint4 ma = ip[8], mb = ip[9];
                const uint32_t t = max(max(t_next, a.y), max(max(b.y, c.y), rd));
                const uint32_t wr = t + ka.y;
                max_ready = max(max_ready, wr);
                t_next = t + 1u;
                const uint32_t cx = c.x ^ ka.z;
                const uint32_t rf =
                    fbits_hw(__fmaf_rn(__uint_as_float(a.x), __uint_as_float(b.x), __uint_as_float(cx)));
                uint32_t res = rf;
                if constexpr (!FPU) res = ka.x == DOP_FPU ? rf : a.x * b.x + cx;
                ST_LANE_PAIR(on_all, ka.w, res, wr);
                // forward k into k+1 (its b and c are not k's destination)
                const uint32_t f = nb.w;
                a1.x = (f & INC_FWD_A) ? res : a1.x;
                rd = (f & INC_FWD_T) ? wr : 0u;
                ka = na;
                kb = nb;
                na = ma;
                nb = mb;
                a = a1;
                ip += 4;
                if (--n == 0u) break;  // uniform in value
              }
            };
            if (keep < 2u) {
              pair_run(std::false_type{}, run_n, q0, q1);
            } else {
              if (q3.x & KEEP_FPU) keep_run(std::true_type{});
              else keep_run(std::false_type{});
              if (run_n > keep) pair_run(std::false_type{}, run_n - keep, ip[0], ip[1]);
            }
          }
          pc += run_n;
          budget -= run_n;
          t_last = t_next - 1u;
          if constexpr (RUNLOG) run_next = pc;
          continue;
        }
      }
      // ---- mid path: runs of the other unguarded register-to-register ops
      // (64-bit arithmetic, logic, shifts, conversions, specials, ld.param,
      // div, sqrt), bounded by `fuel` like the fast path, dispatched with one
      // uniform jump per instruction.
      if (runnable && (q1.w & INC_MID) != 0u) {
        uint32_t fuel = fuel_in;
        const bool on = (mask >> lane) & 1u;
        const uint4* mp = ip;
        uint4 ka = q0, kb = q1;
        [[maybe_unused]] uint32_t hk = SPLIT ? HZ_AT(mp, hs4) : 0u;  // SPLIT: this lane's term offset
        for (;;) {
          const uint4 na = mp[4], nb = mp[5];  // the next record, fetched early
          [[maybe_unused]] uint32_t hk1 = 0;
          uint32_t a0, b0, c0, t;
          if constexpr (SPLIT) {
            hk1 = HZ_AT(mp + 4, hs4);
            a0 = RG32(lv + kb.x);
            b0 = RG32(lv + kb.y);
            c0 = RG32(lv + kb.z);
            t = max(t_next, __reduce_max_sync(FULL, RG32(wb + hk)));
          } else {  // operands with their ready times, the destination's from lane 0's pair
            const uint2 pa = RG2(lv + kb.x), pb = RG2(lv + kb.y), pcc = RG2(lv + kb.z);
            const uint32_t rd = RG32(rdb + ka.w + 4u);
            t = max(max(t_next, pa.y), max(max(pb.y, pcc.y), rd));
            a0 = pa.x;
            b0 = pb.x;
            c0 = pcc.x;
          }
          const uint32_t wr = t + ka.y;
          max_ready = max(max_ready, wr);
          t_next = t + 1u;
          const uint32_t D = ka.w, aux = ka.z;
          const uint32_t A = kb.x, B = kb.y;
          uint32_t lo = 0, hi = 0;
          bool wide = false;
#define MA64() ((uint64_t)a0 | ((uint64_t)RG32(lv + A + RB) << 32))
#define MB64() ((uint64_t)b0 | ((uint64_t)RG32(lv + B + RB) << 32))
#define R64(v) do { const uint64_t v_ = (v); lo = (uint32_t)v_; hi = (uint32_t)(v_ >> 32); wide = true; } while (0)
          switch (__shfl_sync(FULL, ka.x, 0)) {
            case DOP_FPU: lo = fbits_hw(__fmaf_rn(__uint_as_float(a0), __uint_as_float(b0), __uint_as_float(c0 ^ aux))); break;
            case DOP_IMAD: lo = a0 * b0 + (c0 ^ aux); break;
            case DOP_MADI: lo = a0 * aux + c0; break;
            case DOP_MADII: lo = a0 * aux + mp[3].x; break;
            case OP_LDP32: lo = *reinterpret_cast<const uint32_t*>(s_params + aux); break;
            case OP_LDP64: R64(*reinterpret_cast<const uint64_t*>(s_params + aux)); break;
            case OP_MOV64: R64(MA64()); break;
            case OP_MOVSP:
              lo = aux == SP_TID ? tid_sim : aux == SP_NTID ? L.block : aux == SP_CTAID ? cta
                 : aux == SP_NCTAID ? L.grid : aux == SP_LANEID ? lane : aux == SP_ONE ? 1u : 0u;
              break;
            case OP_ADD64: R64(MA64() + MB64()); break;
            case OP_SUB64: R64(MA64() - MB64()); break;
            case OP_MUL64: R64(MA64() * MB64()); break;
            case OP_MAD64: R64(MA64() * MB64() + ((uint64_t)c0 | ((uint64_t)RG32(lv + kb.z + RB) << 32))); break;
            case OP_AND32: lo = a0 & (b0 | aux); break;
            case OP_OR32: lo = a0 | (b0 | aux); break;
            case OP_XOR32: lo = a0 ^ (b0 | aux); break;
            case OP_AND64: R64(MA64() & MB64()); break;
            case OP_OR64: R64(MA64() | MB64()); break;
            case OP_XOR64: R64(MA64() ^ MB64()); break;
            case OP_SHL32: lo = (b0 | aux) >= 32u ? 0u : a0 << (b0 | aux); break;
            case OP_SHR32U: lo = (b0 | aux) >= 32u ? 0u : a0 >> (b0 | aux); break;
            case OP_SHR32S: lo = (uint32_t)((b0 | aux) >= 32u ? ((int32_t)a0 >> 31) : ((int32_t)a0 >> (b0 | aux))); break;
            case OP_SHL64: R64((b0 | aux) >= 64u ? 0ull : MA64() << (b0 | aux)); break;
            case OP_SHR64U: R64((b0 | aux) >= 64u ? 0ull : MA64() >> (b0 | aux)); break;
            case OP_SHR64S: {
              const int64_t x = (int64_t)MA64();
              R64((uint64_t)((b0 | aux) >= 64u ? (x >> 63) : (x >> (b0 | aux))));
              break;
            }
            case OP_FDIV: lo = fbits(__fdiv_rn(__uint_as_float(a0), __uint_as_float(b0))); break;
            case OP_FSQRT: lo = fbits(__fsqrt_rn(__uint_as_float(a0))); break;
            case OP_CVT_F32_U32: lo = __float_as_uint(__uint2float_rn(a0)); break;
            case OP_CVT_F32_S32: lo = __float_as_uint(__int2float_rn((int32_t)a0)); break;
            case OP_CVT_F32_U64: lo = __float_as_uint(__ull2float_rn(MA64())); break;
            case OP_CVT_F32_S64: lo = __float_as_uint(__ll2float_rn((long long)MA64())); break;
            case OP_CVT_F2I: {
              const uint64_t v = f2i(__uint_as_float(a0), aux);
              if ((aux & 15u) == CVT_S64 || (aux & 15u) == CVT_U64) R64(v); else lo = (uint32_t)v;
              break;
            }
            case OP_CVT_ZX: R64((uint64_t)a0); break;
            case OP_CVT_SX: R64((uint64_t)(int64_t)(int32_t)a0); break;
            default: break;
          }
#undef MA64
#undef MB64
#undef R64
          if constexpr (SPLIT) {
            ST_LANE_IF(on, D, lo);
            ST_WB_IF(is_d4, hk, wr);  // the destination's ready word
            hk = hk1;
          } else {
            ST_LANE_PAIR(on, D, lo, wr);
          }
          ST_LANE_IF(on && wide, D + RB, hi);
          fuel--;
          mp += 4;
          ka = na;
          kb = nb;
          if (!(fuel != 0u && (kb.w & INC_MID) != 0u && t_next < REBASE_AT)) break;
        }
        const uint32_t steps = fuel_in - fuel;  // at least 1
        pc += steps;
        budget -= steps;
        t_last = t_next - 1u;
        if constexpr (RUNLOG) run_next = pc;
        continue;
      }
      // ---- general path: one instruction; every operand / ready-time load at once
      const uint32_t op = __shfl_sync(FULL, q0.x, 0), inc = q1.w;
      const uint32_t guard = SPLIT ? q3.x : q2.x, gneg = SPLIT ? q3.y : q2.y;
      [[maybe_unused]] const uint32_t pc_here = pc;  // the instrumented handlers' program entry
      [[maybe_unused]] uint32_t consumed = 1;        // program entries this step issues (2: setp + bra)
      const uint32_t A = q1.x, B = q1.y, C = q1.z, D = q0.w;
      const uint32_t aux = q0.z;
      uint32_t a0, b0, c0;
      // the scoreboard: SPLIT, the latest of all eight terms (rows a, b, c,
      // the destination, the guard, the predicate sources) gathered one per
      // lane; PAIR, the rows' ready times from their pairs, the
      // destination's from lane 0's pair, the guard's and (predicate
      // operands) the predicates' from the predicate table
      [[maybe_unused]] uint32_t hk = 0;
      uint32_t hr;
      if constexpr (SPLIT) {
        hk = HZ_AT(ip, hs8);
        a0 = RG32(lv + A);
        b0 = RG32(lv + B);
        c0 = RG32(lv + C);
        hr = RG32(wb + hk);
      } else {
        const uint2 pa = RG2(lv + A), pb = RG2(lv + B), pcc = RG2(lv + C);
        a0 = pa.x;
        b0 = pb.x;
        c0 = pcc.x;
        const uint32_t rd = RG32(rdb + D + 4u);
        uint32_t hmax = 0;
        if (inc & INC_PHAZ)
          hmax = max(max(RG32(wb + q2.z), RG32(wb + q2.w)), max(RG32(wb + q3.x), RG32(wb + q3.y)));
        const uint32_t rgd = RG32(pg + guard * 4u);  // the guard's ready time
        hr = max(max(max(pa.y, pb.y), pcc.y), max(max(rd, rgd), hmax));
      }
      const uint32_t pm = __shfl_sync(FULL, my_pred, guard);

      if ((inc & INC_ISSUE) == 0u || budget == 0u || t_next >= REBASE_AT) {  // rare path
        if (op == OP_EVENT) {  // trace record (a7), zero cost
          if (n_events != 0xFFFFFFFFu) n_events++;
          if (n_rec < L.max_ts) {
            // record: [id << 24 | ts] (4 B), + u32 payload (8 B), or + 0 + u64
            // payload (16 B); the payload is the lowest active lane's register
            const uint32_t src = (uint32_t)__ffs(mask) - 1u;
            const uint32_t plo = __shfl_sync(FULL, a0, src);
            const uint32_t phi = __shfl_sync(FULL, ((aux >> 8) & 0xFFu) == 8u ? RG32(lv + A + RB) : 0u, src);
            if (slot && lane == 0) {
              uint8_t* r = slot + 16u + L.rec_bytes * n_rec;
              *reinterpret_cast<uint32_t*>(r) = ((aux & 0xFFu) << 24) | (((uint32_t)epoch + t_next) & 0xFFFFFFu);
              if (L.rec_bytes == 8u) {
                *reinterpret_cast<uint32_t*>(r + 4) = plo;
              } else if (L.rec_bytes == 16u) {
                *reinterpret_cast<uint32_t*>(r + 4) = 0u;
                *reinterpret_cast<uint64_t*>(r + 8) = (uint64_t)plo | ((uint64_t)phi << 32);
              }
            }
            n_rec++;
          } else if (n_dropped < 0xFFFFu) {
            n_dropped++;
          }
          pc++;
          if constexpr (RUNLOG) run_next = pc;
          continue;
        }
        if (op == OP_EXIT) {  // reached the virtual exit: the remaining lanes finish
          FLUSH_THREADS();
          mask = 0;
          continue;
        }
        if (t_next >= REBASE_AT) {  // keep every clock below 2^31: move the epoch to t_last
          const uint32_t delta = t_last;
          if constexpr (SPLIT) {
            for (uint32_t i = lane; i < Y.n_ready; i += 32u) {
              const uint32_t e = RG32(wb + Y.ready_off + 4u * i);
              RG32(wb + Y.ready_off + 4u * i) = e > delta ? e - delta : 0u;
            }
          } else {
            for (uint32_t r = 0; r < Y.n_slots; r++) {
              const uint32_t e = RG32(lv + r * RB + 4u);
              RG32(lv + r * RB + 4u) = e > delta ? e - delta : 0u;
            }
            const uint32_t e = RG32(pg + lane * 4u);
            RG32(pg + lane * 4u) = e > delta ? e - delta : 0u;
          }
          __syncwarp();
          epoch += delta;
          t_last = 0;
          t_next -= delta;
          max_ready = max_ready > delta ? max_ready - delta : 0u;
          drain = drain > delta ? drain - delta : 0u;
          continue;  // reload the ready times
        }
        // budget == 0: a stop, or the next chunk
        FLUSH_THREADS();
        if (left == 0) {
          status = (injected && stop_at - left - budget == L.inject_step) ? KS_ST_INJECTED : KS_ST_STEP_LIMIT;
          break;
        }
        budget = (uint32_t)(left < BUDGET_CHUNK ? left : BUDGET_CHUNK);
        left -= budget;
        mark = budget;
        continue;
      }

      // cache model: one access per ld/st.global that a lane executes, at the
      // lowest executing lane's line; a load's latency follows the level
      uint32_t wlat = q0.y;
      if constexpr (INSTR) {
        const uint32_t ex = mask & (pm ^ gneg);
        if (L.cache_pass != 0u && op >= OP_LDG32 && op <= OP_STG64 && ex != 0u) {
          const uint64_t va_c =
              ((uint64_t)a0 | ((uint64_t)RG32(lv + A + RB) << 32)) + (uint64_t)(int64_t)(int32_t)aux;
          const uint64_t line = __shfl_sync(FULL, va_c, __ffs(ex) - 1) >> 7;
          const uint64_t step = c_off + (stop_at - left - budget);
          ks_cache_access* rec = L.cache_log + (uint64_t)gw * L.cache_cap + c_k;
          int cst = 0;
          if (step >= 0xFFFFFFFFull) {
            cst = KS_ST_CACHE_LOG;
          } else if (L.cache_pass != 2u) {  // a logging pass (1, or 3: the timing replay's)
            if (c_k < L.cache_cap && lane == 0) {
              rec->line = line;
              rec->step = (uint32_t)step;
              rec->level = KS_CACHE_DRAM;
            }
            c_k++;
          } else if (c_k >= c_n) {
            cst = KS_ST_CACHE_STREAM;
          } else {
            const ulonglong2 r = *reinterpret_cast<const ulonglong2*>(rec);
            const uint32_t level = (uint32_t)(r.y >> 32);
            if (r.x != line || (uint32_t)r.y != (uint32_t)step) {
              cst = KS_ST_CACHE_STREAM;
            } else {
              c_l1 += level == KS_CACHE_L1_HIT;
              c_l2 += level == KS_CACHE_L2_HIT;
              if (op == OP_LDG32 || op == OP_LDG64)
                wlat = level == KS_CACHE_L1_HIT ? L.lat_l1 : level == KS_CACHE_L2_HIT ? L.lat_l2 : q0.y;
              c_k++;
            }
          }
          if (cst != 0) {  // stop before issuing
            status = cst;
            FLUSH_THREADS();
            break;
          }
        }
      }

      // issue: in-order scoreboard (a3), epoch-relative 32-bit clock
      const uint32_t t = max(t_next, SPLIT ? __reduce_max_sync(FULL, hr) : hr);
      const uint32_t wr = t + wlat;
      if constexpr (SPLIT) {
        // the destination's ready word (a register row's, or the predicate's)
        if (inc & (INC_RDEST | INC_PDEST)) ST_WB_IF(is_d8, hk, wr);
      } else {
        if (inc & INC_RDEST) RG32(lv + D + 4u) = wr;  // register destination (every lane's pair)
        if (inc & INC_PDEST) RG32(wb + q3.y) = wr;    // predicate destination
      }
      max_ready = max(max_ready, wr);
      drain = max(drain, t + q3.z);
      t_last = t;
      t_next = t + q3.w;
      budget--;

      // guard (a2)
      const uint32_t exec = mask & (pm ^ gneg);
      const bool on = (exec >> lane) & 1u;
      // high words of 64-bit operands, loaded by the handlers that need them
#define A64() ((uint64_t)a0 | ((uint64_t)RG32(lv + A + RB) << 32))
#define B64() ((uint64_t)b0 | ((uint64_t)RG32(lv + B + RB) << 32))
#define C64() ((uint64_t)c0 | ((uint64_t)RG32(lv + C + RB) << 32))
#define W32(v) ST_LANE_IF(on, D, (v))
#define W64(v)                                                  \
  do {                                                          \
    const uint64_t v_ = (v);                                    \
    ST_LANE_IF(on, D, (uint32_t)v_);                            \
    ST_LANE_IF(on, D + RB, (uint32_t)(v_ >> 32));            \
  } while (0)

      // The most frequent general-path ops take plain branches ahead of the
      // switch (its indirect jump costs a lone warp more than the case itself);
      // each body sits in do { } while (0) so that `break` ends the instruction.
      if (op == OP_BRA) do {  // ---- control (a6)
          const uint32_t target = aux & 0xFFFFu, R = aux >> 16;
          const uint32_t taken = exec, fall = mask & ~exec;
          if (fall == 0) {
            pc = target;
          } else if (taken == 0) {
            pc = pc + 1;
          } else {
            FLUSH_THREADS();
            if (INSTR && L.profile && lane == 0) {  // a divergent branch (hints: divergence ratio)
              ks_pc_profile* pp = L.profile + pc_here;
              const uint32_t small = min(__popc(taken), __popc(fall)), act = __popc(mask);
              atomicAdd(reinterpret_cast<unsigned long long*>(&pp->divergent), 1ull);
              if (5u * small > 2u * act) {
                atomicAdd(reinterpret_cast<unsigned long long*>(&pp->high_divergence), 1ull);
                atomicOr(reinterpret_cast<unsigned long long*>(&pp->high_div_pcts), 1ull << (100u * small / act));
              }
            }
            const uint32_t sbase = wb + Y.stack_off;
            uint32_t n = depth;  // entries held in shared memory once the top is resolved
            if (rpc == R) {
              n = depth - 1;  // the top already waits at R below: replace it
            } else {
              RG64(sbase + (depth - 1) * 8u) = pack_entry(R, rpc, mask);
            }
            if (target != R) {
              if (n >= L.stack_depth) { status = KS_ST_SIMT_STACK; break; }
              RG64(sbase + n * 8u) = pack_entry(target, R, taken);
              n++;
            }
            if (pc + 1 != R) {
              if (n >= L.stack_depth) { status = KS_ST_SIMT_STACK; break; }
              RG64(sbase + n * 8u) = pack_entry(pc + 1, R, fall);
              n++;
            }
            if (n == 0) { depth = 1; pc = rpc = exit_pc; mask = 0; break; }
            depth = n;
            max_depth = max(max_depth, depth);
            const uint64_t e = RG64(sbase + (depth - 1) * 8u);
            pc = (uint32_t)(e & 0xFFFFu);
            rpc = (uint32_t)((e >> 16) & 0xFFFFu);
            mask = (uint32_t)(e >> 32);
          }
          break;
        } while (0);
      else if (op >= OP_SETP_U32 && op <= OP_SETP_F32) do {  // ---- predicates
          const uint32_t cmp = aux & 0xFFu, pd = (aux >> 8) & 0xFFu;
          bool lt, eq, gt;
          if (op == OP_SETP_F32) {
            const float x = __uint_as_float(a0), y = __uint_as_float(b0);
            lt = x < y; eq = x == y; gt = x > y;
          } else {
            // signed order = unsigned order with the sign bits flipped
            const bool sgn = op == OP_SETP_S32 || op == OP_SETP_S64;
            uint64_t x, y;
            if (op == OP_SETP_U64 || op == OP_SETP_S64) { x = A64(); y = B64(); }
            else if (sgn) { x = (uint64_t)(int64_t)(int32_t)a0; y = (uint64_t)(int64_t)(int32_t)b0; }
            else { x = a0; y = b0; }
            const uint64_t flip = sgn ? (1ull << 63) : 0ull;
            x ^= flip; y ^= flip;
            lt = x < y; eq = x == y; gt = x > y;
          }
          const uint32_t bal = __ballot_sync(FULL, rel_result(lt, eq, gt, cmp));
          // lane pd holds predicate pd
          if (lane == pd) my_pred = (my_pred & ~exec) | (bal & exec);
          if ((inc & INC_FUSE) && exec == mask && budget != 0u && pc + 1u != rpc && t_next < REBASE_AT) {
            // the next entry is `@[!]p bra` on this predicate: when every active
            // lane goes the same way it issues here, exactly as the general
            // path would (no register operands; its guard ready at wr)
            const uint32_t taken = mask & (bal ^ (((aux >> 16) & 1u) ? 0xFFFFFFFFu : 0u));
            if (taken == mask || taken == 0u) {
              const uint32_t t2 = max(t_next, wr);
              max_ready = max(max_ready, t2);
              drain = max(drain, t2);
              t_last = t2;
              t_next = t2 + L.lat[KS_LAT_BRA];
              budget--;
              pc = taken ? (aux >> 17) : pc + 2u;
              consumed = 2;
              break;
            }
          }
          pc++;
          break;
        } while (0);
      else if (op >= OP_LDG32 && op <= OP_STG64) do {  // ---- global memory (a5)
          const bool wide = (op == OP_LDG64 || op == OP_STG64);
          const bool is_ld = (op == OP_LDG32 || op == OP_LDG64);
          const uint32_t size = wide ? 8u : 4u;
          const uint64_t va = A64() + (uint64_t)(int64_t)(int32_t)aux;
          uint8_t* ptr = nullptr;
          int err = 0;
          {  // the buffer of the last access first, every buffer if any lane misses it
            const uint64_t base = L.bufs[hint].sim_base, bytes = L.bufs[hint].bytes;
            const bool hit = (va & (uint64_t)(size - 1)) == 0 && va >= base && bytes >= size && va - base <= bytes - size;
            if (__all_sync(FULL, hit || !on)) {
              ptr = L.bufs[hint].ptr + (va - base);
            } else {
              if (on) err = translate(L, va, size, &ptr);
              const uint32_t emask = __ballot_sync(FULL, err != 0);
              if (emask) {
                status = __shfl_sync(FULL, err, __ffs(emask) - 1);
                break;
              }
              uint32_t bi = 0;
              if (on) {
                for (uint32_t k = 0; k < L.n_bufs; k++)
                  if (ptr >= L.bufs[k].ptr && ptr < L.bufs[k].ptr + L.bufs[k].bytes) bi = k;
              }
              hint = __shfl_sync(FULL, bi, __ffs(exec ? exec : 1u) - 1);
            }
          }
          // Distinct 32-byte sectors and 128-byte lines over the executing lanes.
          // With every lane executing and addresses non-decreasing in lane order
          // (the coalesced case), equal sectors are adjacent and each change from
          // the lane below starts a new one; otherwise lanes are grouped by value.
          const uint64_t va_up = __shfl_up_sync(FULL, va, 1);
          const bool sorted = exec == FULL && __all_sync(FULL, lane == 0 || va >= va_up);
          uint32_t lines = 0;
          if (sorted) {
            const uint32_t sectors = 1u + __popc(__ballot_sync(FULL, lane != 0 && (va >> 5) != (va_up >> 5)));
            lines = 1u + __popc(__ballot_sync(FULL, lane != 0 && (va >> 7) != (va_up >> 7)));
            if (is_ld) { ld_req++; ld_sec += sectors; ld_lin += lines; }
            else { st_req++; st_sec += sectors; st_lin += lines; }
          } else if (exec) {
            const uint32_t ms = __match_any_sync(FULL, on ? (va >> 5) : ~0ull);
            const uint32_t sectors = __popc(__ballot_sync(FULL, on && (uint32_t)(__ffs(ms) - 1) == lane));
            const uint32_t ml = __match_any_sync(FULL, on ? (va >> 7) : ~0ull);
            lines = __popc(__ballot_sync(FULL, on && (uint32_t)(__ffs(ml) - 1) == lane));
            if (is_ld) { ld_req++; ld_sec += sectors; ld_lin += lines; }
            else { st_req++; st_sec += sectors; st_lin += lines; }
          }
          if (INSTR && L.profile && exec && lane == 0) {  // hints: coalescing efficiency min(1, ideal / lines)
            ks_pc_profile* pp = L.profile + pc_here;
            const uint32_t ideal = (__popc(exec) * size + 127u) / 128u;
            atomicAdd(reinterpret_cast<unsigned long long*>(&pp->requests), 1ull);
            if (4u * ideal < lines) {
              atomicAdd(reinterpret_cast<unsigned long long*>(&pp->poor), 1ull);
              atomicOr(&pp->poor_pcts, 1u << (100u * ideal / lines));
            } else if (2u * ideal < lines) {
              atomicAdd(reinterpret_cast<unsigned long long*>(&pp->uncoalesced), 1ull);
            }
          }
          if (is_ld) {
            if (on) {
              if (wide) {
                const uint64_t v = *reinterpret_cast<const uint64_t*>(ptr);
                RG32(lv + D) = (uint32_t)v;
                RG32(lv + D + RB) = (uint32_t)(v >> 32);
              } else {
                RG32(lv + D) = *reinterpret_cast<const uint32_t*>(ptr);
              }
            }
          } else {
            // the highest lane writing an address wins: in the sorted case the
            // last lane of each run of equal addresses
            const uint64_t va_dn = __shfl_down_sync(FULL, va, 1);
            const bool wins = sorted ? (lane == 31 || va_dn != va)
                                     : (31u - __clz(__match_any_sync(FULL, on ? va : ~0ull))) == lane;
            if (on && wins && !(INSTR && L.cache_pass == 1)) {  // the cache model's first pass stores nothing
              if (wide) *reinterpret_cast<uint64_t*>(ptr) = B64();
              else *reinterpret_cast<uint32_t*>(ptr) = b0;
            }
          }
          pc++;
          break;
        } while (0);
      else switch (op) {
        // ---- the routed datapaths (guarded, or outside a fast run) ----
        case DOP_FPU: case DOP_FPU | DOP_GUARDED:
          W32(fbits_hw(__fmaf_rn(__uint_as_float(a0), __uint_as_float(b0), __uint_as_float(c0 ^ aux))));
          pc++;
          break;
        case DOP_IMAD: case DOP_IMAD | DOP_GUARDED:
          W32(a0 * b0 + (c0 ^ aux));
          pc++;
          break;
        case DOP_MADI: W32(a0 * aux + c0); pc++; break;
        case DOP_MADII: W32(a0 * aux + q3.x); pc++; break;
        // ---- control (a6) ----

        case OP_RET: {
          FLUSH_THREADS();
          for (uint32_t i = 0; i + 1 < depth; i++) {
            const uint32_t at = wb + Y.stack_off + i * 8u;
            RG64(at) = RG64(at) & ~((uint64_t)exec << 32);
          }
          mask &= ~exec;
          if constexpr (RUNLOG) live &= ~exec;
          pc++;
          break;
        }
        // ---- memory (a5) ----
        case OP_LDP32: W32(*reinterpret_cast<const uint32_t*>(s_params + aux)); pc++; break;
        case OP_LDP64: W64(*reinterpret_cast<const uint64_t*>(s_params + aux)); pc++; break;

        // ---- shared memory: bank rule of analyze_shared_memory_access ----
        case OP_LDS32: case OP_LDS64: case OP_STS32: case OP_STS64: if constexpr (CTA) {
          const bool wide = (op == OP_LDS64 || op == OP_STS64);
          const bool is_ld = (op == OP_LDS32 || op == OP_LDS64);
          const uint32_t size = wide ? 8u : 4u;
          const uint64_t va = ((inc & INC_ADDR64) ? A64() : (uint64_t)a0) + (uint64_t)(int64_t)(int32_t)aux;
          int err = 0;
          if (on)
            err = (va & (uint64_t)(size - 1)) ? KS_ST_MISALIGNED
                  : (L.shared_bytes < size || va > (uint64_t)(L.shared_bytes - size)) ? KS_ST_OOB : 0;
          const uint32_t emask = __ballot_sync(FULL, err != 0);
          if (emask) {
            status = __shfl_sync(FULL, err, __ffs(emask) - 1);
            break;
          }
          const uint32_t sva = (uint32_t)va;
          // lanes on my address (the non-executing lanes get keys of their own)
          const uint32_t same_addr = __match_any_sync(FULL, on ? sva : (0x80000000u | lane));
          if (exec) {
            // lanes in my bank: a bank that is all one address counts 1, any
            // other bank its lanes; the request's degree is the largest
            const uint32_t same_bank = __match_any_sync(FULL, on ? ((sva >> 2) & 31u) : (32u + lane));
            const uint32_t deg = (on && same_addr != same_bank) ? (uint32_t)__popc(same_bank) : 1u;
            const uint32_t degree = __reduce_max_sync(FULL, deg);
            sh_req++;
            sh_wf += degree;
            if (INSTR && L.profile && lane == 0) {  // hints: bank-conflict degree
              ks_pc_profile* pp = L.profile + pc_here;
              atomicAdd(reinterpret_cast<unsigned long long*>(&pp->requests), 1ull);
              if (degree > 1u) atomicAdd(reinterpret_cast<unsigned long long*>(&pp->conflicted), 1ull);
              if (degree >= 8u) atomicAdd(reinterpret_cast<unsigned long long*>(&pp->severe), 1ull);
              atomicOr(&pp->degrees, 1u << (degree - 1u));
            }
          }
          uint8_t* sp = smem + sh_base + sva;  // dereferenced by executing lanes only
          if (is_ld) {
            if (on) {
              if (wide) {
                const uint2 v = *reinterpret_cast<const uint2*>(sp);
                RG32(lv + D) = v.x;
                RG32(lv + D + RB) = v.y;
              } else {
                RG32(lv + D) = *reinterpret_cast<const uint32_t*>(sp);
              }
            }
          } else if (on && (31u - __clz(same_addr)) == lane) {  // the highest lane on an address wins
            if (wide) {
              const uint64_t v = B64();
              *reinterpret_cast<uint2*>(sp) = make_uint2((uint32_t)v, (uint32_t)(v >> 32));
            } else {
              *reinterpret_cast<uint32_t*>(sp) = b0;
            }
          }
          pc++;
          break;
        }
        case OP_BAR:  // stop until the CTA's barrier releases
          if constexpr (CTA) at_bar = true;
          pc++;
          break;
        // ---- moves and integer ALU (a4) ----
        case OP_MOV32: W32(a0); pc++; break;
        case OP_MOV64: W64(A64()); pc++; break;
        case OP_MOVSP: {
          uint32_t v;
          switch (aux) {
            case SP_TID: v = tid_sim; break;
            case SP_NTID: v = L.block; break;
            case SP_CTAID: v = cta; break;
            case SP_NCTAID: v = L.grid; break;
            case SP_LANEID: v = lane; break;
            case SP_ONE: v = 1; break;
            default: v = 0; break;
          }
          W32(v);
          pc++;
          break;
        }
        case OP_ADD32: W32(a0 + b0); pc++; break;
        case OP_SUB32: W32(a0 - b0); pc++; break;
        case OP_MUL32: W32(a0 * b0); pc++; break;
        case OP_MAD32: W32(a0 * b0 + c0); pc++; break;
        case OP_ADD64: W64(A64() + B64()); pc++; break;
        case OP_SUB64: W64(A64() - B64()); pc++; break;
        case OP_MUL64: W64(A64() * B64()); pc++; break;
        case OP_MAD64: W64(A64() * B64() + C64()); pc++; break;
        case OP_AND32: W32(a0 & (b0 | aux)); pc++; break;
        case OP_OR32: W32(a0 | (b0 | aux)); pc++; break;
        case OP_XOR32: W32(a0 ^ (b0 | aux)); pc++; break;
        case OP_AND64: W64(A64() & B64()); pc++; break;
        case OP_OR64: W64(A64() | B64()); pc++; break;
        case OP_XOR64: W64(A64() ^ B64()); pc++; break;
        case OP_SHL32: W32((b0 | aux) >= 32u ? 0u : a0 << (b0 | aux)); pc++; break;
        case OP_SHR32U: W32((b0 | aux) >= 32u ? 0u : a0 >> (b0 | aux)); pc++; break;
        case OP_SHR32S: W32((uint32_t)((b0 | aux) >= 32u ? ((int32_t)a0 >> 31) : ((int32_t)a0 >> (b0 | aux)))); pc++; break;
        case OP_SHL64: W64((b0 | aux) >= 64u ? 0ull : A64() << (b0 | aux)); pc++; break;
        case OP_SHR64U: W64((b0 | aux) >= 64u ? 0ull : A64() >> (b0 | aux)); pc++; break;
        case OP_SHR64S: {
          const int64_t x = (int64_t)A64();
          W64((uint64_t)((b0 | aux) >= 64u ? (x >> 63) : (x >> (b0 | aux))));
          pc++;
          break;
        }
        // ---- f32 (a4), IEEE round-to-nearest-even, canonical NaN ----
        case OP_FADD: W32(fbits_hw(__fadd_rn(__uint_as_float(a0), __uint_as_float(b0)))); pc++; break;
        case OP_FSUB: W32(fbits_hw(__fsub_rn(__uint_as_float(a0), __uint_as_float(b0)))); pc++; break;
        case OP_FMUL: W32(fbits_hw(__fmul_rn(__uint_as_float(a0), __uint_as_float(b0)))); pc++; break;
        case OP_FFMA:
          W32(fbits_hw(__fmaf_rn(__uint_as_float(a0), __uint_as_float(b0), __uint_as_float(c0))));
          pc++;
          break;
        case OP_FDIV: W32(fbits(__fdiv_rn(__uint_as_float(a0), __uint_as_float(b0)))); pc++; break;
        case OP_FSQRT: W32(fbits(__fsqrt_rn(__uint_as_float(a0)))); pc++; break;
        // ---- predicates ----

        case OP_ANDP: case OP_ORP: case OP_XORP: {
          const uint32_t pa = __shfl_sync(FULL, my_pred, aux & 0xFFu);
          const uint32_t pb = __shfl_sync(FULL, my_pred, (aux >> 8) & 0xFFu);
          const uint32_t pd = (aux >> 16) & 0xFFu;
          const uint32_t r = op == OP_ANDP ? (pa & pb) : op == OP_ORP ? (pa | pb) : (pa ^ pb);
          if (lane == pd) my_pred = (my_pred & ~exec) | (r & exec);
          pc++;
          break;
        }
        case OP_SELP32: {
          const uint32_t sel = __shfl_sync(FULL, my_pred, aux);
          W32(((sel >> lane) & 1u) ? a0 : b0);
          pc++;
          break;
        }
        case OP_SELP64: {
          const uint32_t sel = __shfl_sync(FULL, my_pred, aux);
          W64(((sel >> lane) & 1u) ? A64() : B64());
          pc++;
          break;
        }
        // ---- conversions ----
        case OP_CVT_F32_U32: W32(__float_as_uint(__uint2float_rn(a0))); pc++; break;
        case OP_CVT_F32_S32: W32(__float_as_uint(__int2float_rn((int32_t)a0))); pc++; break;
        case OP_CVT_F32_U64: W32(__float_as_uint(__ull2float_rn(A64()))); pc++; break;
        case OP_CVT_F32_S64: W32(__float_as_uint(__ll2float_rn((long long)A64()))); pc++; break;
        case OP_CVT_F2I: {
          const uint64_t v = f2i(__uint_as_float(a0), aux);
          const uint32_t kind = aux & 15u;
          if (kind == CVT_S64 || kind == CVT_U64) W64(v);
          else W32((uint32_t)v);
          pc++;
          break;
        }
        case OP_CVT_ZX: W64((uint64_t)a0); pc++; break;
        case OP_CVT_SX: W64((uint64_t)(int64_t)(int32_t)a0); pc++; break;
        default:
          pc++;
          break;
      }
#undef W32
#undef W64
#undef A64
#undef B64
#undef C64
      if constexpr (RUNLOG) run_next = pc_here + consumed;
      if (status != 0) {
        FLUSH_THREADS();
        break;
      }
      if (at_bar) break;
    }
    if constexpr (!cta_mode) break;
    // ---- barrier round (CTA mode): each warp has stopped at bar.sync or
    // finished; the stopped ones resume at the latest arrival + latency ----
    if constexpr (INSTR) {
      // the release comes at the end of the step in which the last warp
      // arrived or finished: 1 + the last step issued by those warps
      const uint64_t issued = stop_at - left - budget;
      if (L.cache_pass != 0u && (at_bar || !finished) && issued != 0 && lane == 0)
        atomicMax(&ctl->step_end[round & 1u], (unsigned long long)(c_off + issued));
    }
    if (!at_bar && !finished) {
      finished = true;
      if (lane == 0) atomicAdd(&ctl->done, 1u);
    }
    // the bar.sync is the last instruction issued: it arrived at epoch + t_last
    if (at_bar && lane == 0) atomicMax(&ctl->latest[round & 1u], (unsigned long long)(epoch + t_last));
    __syncthreads();
    const unsigned long long latest = ctl->latest[round & 1u];
    const unsigned long long step_end = INSTR ? ctl->step_end[round & 1u] : 0ull;
    const bool all_done = ctl->done == nwarps;
    if (threadIdx.x == 0) {  // last read two rounds ago
      ctl->latest[(round + 1u) & 1u] = 0ull;
      if (INSTR) ctl->step_end[(round + 1u) & 1u] = 0ull;
    }
    __syncthreads();
    if (all_done) break;
    if (at_bar) {
      at_bar = false;
      if constexpr (INSTR) c_off = step_end - (stop_at - left - budget);
      const uint64_t rel = (uint64_t)latest + L.lat[KS_LAT_BAR] - epoch;
      if (rel < REBASE_AT) {
        t_next = (uint32_t)rel;
      } else {
        // Far ahead of this warp's clock: move the epoch to just before the
        // release. What the warp owes so far goes to cyc_floor; ready times
        // before the release no longer matter (saturate to 0); t_last stays
        // "none" (t_last + 1 == 0) until the next issue.
        cyc_floor = max(cyc_floor, epoch + (uint64_t)max(max(t_last + 1u, max_ready), drain));
        const uint64_t delta = rel - 1u;
        if constexpr (SPLIT) {
          for (uint32_t i = lane; i < Y.n_ready; i += 32u) {
            const uint32_t e = RG32(wb + Y.ready_off + 4u * i);
            RG32(wb + Y.ready_off + 4u * i) = (uint64_t)e > delta ? (uint32_t)(e - delta) : 0u;
          }
        } else {
          for (uint32_t r = 0; r < Y.n_slots; r++) {
            const uint32_t e = RG32(lv + r * RB + 4u);
            RG32(lv + r * RB + 4u) = (uint64_t)e > delta ? (uint32_t)(e - delta) : 0u;
          }
          const uint32_t e = RG32(pg + lane * 4u);
          RG32(pg + lane * 4u) = (uint64_t)e > delta ? (uint32_t)(e - delta) : 0u;
        }
        __syncwarp();
        epoch += delta;
        t_last = 0xFFFFFFFFu;
        t_next = 1u;
        max_ready = (uint64_t)max_ready > delta ? (uint32_t)(max_ready - delta) : 0u;
        drain = (uint64_t)drain > delta ? (uint32_t)(drain - delta) : 0u;
      }
    }
    }  // barrier rounds
#undef FLUSH_THREADS
    const uint64_t warp_insts = stop_at - left - budget;
    if constexpr (INSTR) {
      if constexpr (RUNLOG) {  // the last run, and the count
        if (run_next != run_start) {
          if (lane == 0 && n_runs < L.sched_cap)
            L.sched_log[(uint64_t)gw * L.sched_cap + n_runs] =
                (run_start << 16) | run_div | (run_next - run_start - 1u);
          n_runs++;
        }
        if (lane == 0) L.sched_runs[gw] = n_runs;
        if (n_runs > L.sched_cap && status == 0) status = L.cache_pass == 3u ? KS_ST_CACHE_LOG : KS_ST_SCHED_LIMIT;
      }
      if (L.cache_pass == 2 && status == 0 && c_k != c_n) status = KS_ST_CACHE_STREAM;
      // the timing replay needs every access's level
      if (L.cache_pass == 3 && status == 0 && c_k > L.cache_cap) status = KS_ST_CACHE_LOG;
      if (L.cache_pass != 0u && lane == 0) {
        ks_cache_warp cw;
        cw.n_access = c_k;
        cw.l1_hits = c_l1;
        cw.l2_hits = c_l2;
        cw.dram = c_k - c_l1 - c_l2;
        L.cache_warps[gw] = cw;
      }
    }

    // ---- write-back (a9) ----
    const uint64_t cycles =
        warp_insts ? max(cyc_floor, epoch + (uint64_t)max(max(t_last + 1u, max_ready), drain)) : 0ull;
    if (lane == 0) {
      ulonglong2* r = reinterpret_cast<ulonglong2*>(L.stats + (uint64_t)gw * sizeof(ks_warp_stats));
      r[0] = make_ulonglong2(cycles, warp_insts);
      r[1] = make_ulonglong2(thread_insts, ld_req);
      r[2] = make_ulonglong2(ld_sec, st_req);
      r[3] = make_ulonglong2(st_sec, ld_lin);
      r[4] = make_ulonglong2(st_lin, (uint64_t)(uint32_t)status | ((uint64_t)max_depth << 32));
      r[5] = make_ulonglong2(sh_req, sh_wf);
    }
    if (slot) {
      uint32_t* sw = reinterpret_cast<uint32_t*>(slot);
      const uint32_t words = (uint32_t)(L.slot_bytes / 4);
      if (lane == 0) {
        sw[0] = n_events;
        sw[1] = 1u | (L.rec_bytes << 8) | (n_dropped << 16);
        sw[2] = (uint32_t)cycles;
        sw[3] = (uint32_t)(cycles >> 32);
      }
      for (uint32_t i = 4 + n_rec * (L.rec_bytes / 4u) + lane; i < words; i += 32) sw[i] = 0u;
    }
    if constexpr (FLOOR) t_floor = max(max(t_next, t_last + 1u), max(max_ready, drain));
    __syncwarp();
  }
  // Leave no copy in flight: if staging timed out, wait once more (bounded).
  if (!staged) (void)wait_staged(s_bar);
}

}  // namespace ks

/*
 * ks_oracle.h — C interface of the CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. The oracle is a plain, slow, per-lane CPU
 * interpreter of the PTX subset that the GPU interpreter executes. Only the
 * test suite, the package's smoke() check and bench.py's CPU-baseline /
 * reference legs may load it. It shares no code, header, table or helper
 * with the GPU path: its parser, its post-dominator computation and its
 * instruction semantics are written separately here.
 *
 * Shared memory and barriers (KernelScope backend doc, simulator/models.py
 * Block: a per-block shared array and a barrier; simulator/engine.py
 * analyze_shared_memory_access: 32 banks of 4 bytes, broadcast rule;
 * latency/model.py: ld.shared/st.shared 23, bar.sync 20): a kernel that
 * declares .shared arrays or uses bar.sync runs CTA by CTA. A warp that issues
 * bar.sync 0 stops; once every warp of its CTA has stopped there or finished,
 * the stopped warps resume at (latest issue cycle of the bar.sync) + the
 * barrier latency. Shared memory starts zeroed for every CTA.
 *
 * Output formats that must match the GPU path byte for byte (written
 * independently on each side):
 *   - per-warp statistics record, 96 bytes (orc_warp_stats below);
 *   - per-warp trace slot: 16-byte header {u32 n_events, u8 format=1,
 *     u8 bytes_per_event, u16 n_dropped, u64 warp_cycles} followed by max_ts
 *     records of bytes_per_event (4, 8 or 16: no payload, a 4-byte payload,
 *     an 8-byte payload), slot size rounded up to 8 bytes
 *     (CuTeDSL IKET 浅析, §2 "buffer 是怎么定形的": warp_slot =
 *     align8(16B header + maxTsCntPerWarp × bytes_per_event)).
 */
#ifndef KS_ORACLE_H
#define KS_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes (same numbering as the library's device statuses). */
#define ORC_OK 0
#define ORC_ERR_PARSE (-1)
#define ORC_ERR_UNSUPPORTED (-2)
#define ORC_ERR_ARG (-3)
#define ORC_ERR_NOT_FOUND (-5)
#define ORC_ST_OOB 1
#define ORC_ST_MISALIGNED 2
#define ORC_ST_STEP_LIMIT 3
#define ORC_ST_SIMT_STACK 4
#define ORC_ST_TIMEOUT 5
#define ORC_ST_INJECTED 6

/* Latency classes (index into orc_config.lat). */
#define ORC_LAT_ALU 0 /* int/f32 add, sub, mul, mad, logic, shifts, cvt, mov, setp, selp, ld.param */
#define ORC_LAT_FMA 1 /* fma.rn.f32 */
#define ORC_LAT_LDG 2 /* ld.global */
#define ORC_LAT_STG 3 /* st.global */
#define ORC_LAT_BRA 4 /* bra */
#define ORC_LAT_SFU 5 /* div.rn.f32, sqrt.rn.f32 */
#define ORC_LAT_RET 6 /* ret, exit */
#define ORC_LAT_LDS 7 /* ld.shared */
#define ORC_LAT_STS 8 /* st.shared */
#define ORC_LAT_BAR 9 /* bar.sync: from the last arrival to the release */
#define ORC_NUM_LAT 12 /* slots 10 and 11 are reserved */

/* Simulated global buffer: caller-chosen simulated base address (4 KiB
 * aligned, non-overlapping) backed by host memory. */
typedef struct {
  uint64_t sim_base;
  void* host;
  uint64_t bytes;
} orc_buffer;

/* Run modes. */
#define ORC_MODE_WARP 0       /* warp-level SIMT with the reconvergence stack (the method) */
#define ORC_MODE_PER_THREAD 1 /* every thread alone, scalar (memory and status only) */

typedef struct {
  uint32_t lat[ORC_NUM_LAT];
  uint32_t max_ts_per_warp;
  uint32_t stack_depth;     /* SIMT stack entries per warp, base entry included */
  uint64_t step_limit;      /* max issued instructions per warp (per thread in per-thread mode) */
  int64_t inject_warp;      /* global warp id that posts ORC_ST_INJECTED, -1 = off */
  uint64_t inject_step;     /* ...when its issued-instruction count reaches this value */
  uint32_t mode;            /* ORC_MODE_* */
  uint32_t threads;         /* host worker threads, 0 = all hardware threads */
  uint32_t race_check;      /* 1 = shadow-memory race checker (forces one thread) */
  uint32_t n_warp_list;     /* 0 = every warp of the grid */
  const uint32_t* warp_list;/* global warp ids to run when n_warp_list > 0 */
} orc_config;

/* Per-warp statistics record, 96 bytes. */
typedef struct {
  uint64_t cycles;
  uint64_t warp_insts;
  uint64_t thread_insts;
  uint64_t ld_req;
  uint64_t ld_sectors;
  uint64_t st_req;
  uint64_t st_sectors;
  uint64_t ld_lines;
  uint64_t st_lines;
  int32_t status;
  uint32_t max_stack_depth;
  uint64_t sh_req;        /* ld/st.shared requests with at least one executing lane */
  uint64_t sh_wavefronts; /* sum over those requests of the bank-conflict degree */
} orc_warp_stats;

/* Race checker result bits: two threads touch one 4-byte word, at least one
 * writing (global memory: anywhere in the launch; shared memory: within one
 * barrier interval of one CTA). */
#define ORC_RACE_CROSS_THREAD 1u

/* Fill cfg with the defaults: latency table {4,4,400,20,8,36,1,23,23,20,0,0},
 * max_ts 0, stack depth 32, step limit 2^26, no injection, warp mode. */
void orc_config_default(orc_config* cfg);

/* Interpret `kernel` of the PTX module text over grid x block threads.
 * stats: W records (W = grid * ceil(block/32)), indexed by global warp id;
 *        only the warps that run are written.
 * trace: NULL, or W slots of align8(16 + 4*max_ts) bytes.
 * *status: status of the first warp (in run order) that stopped on an error.
 * Returns ORC_OK or a negative code with a message in err. */
int orc_run(const char* ptx, const char* kernel, uint32_t grid, uint32_t block,
            const void* params, uint64_t param_bytes, const orc_buffer* bufs,
            uint32_t n_bufs, const orc_config* cfg, void* stats, void* trace,
            int32_t* status, uint32_t* race_flags, char* err, uint64_t errlen);

/* L1/L2 hit model (KernelScope backend doc, simulator/engine.py — "Cache
 * parameters", SimpleCache, _execute_instruction): one direct-mapped L1 and
 * one direct-mapped L2 of 128-byte lines for the whole grid (set = line %
 * lines; a miss installs the line). Every ld/st.global with an executing lane
 * accesses L1 at its lowest executing lane's address, then L2 on a miss; a
 * load's destination is ready after lat_l1, lat_l2 or lat[ORC_LAT_LDG]. The
 * grid runs as the page's step() does: each step, every warp that is not done
 * or waiting at a barrier executes one instruction, blocks then warps in
 * order; a barrier releases at the end of the step in which its CTA's last
 * warp arrived or finished. */
#define ORC_CACHE_L1_HIT 0
#define ORC_CACHE_L2_HIT 1
#define ORC_CACHE_DRAM 2

typedef struct {
  uint32_t l1_lines, l2_lines;
  uint32_t lat_l1, lat_l2;
  uint32_t log_cap;  /* records per warp kept in `log` */
  void* warps;       /* W x {u32 n_access, u32 l1_hits, u32 l2_hits, u32 dram}, or NULL */
  void* log;         /* W x log_cap x {u64 line, u32 step, u32 level}, or NULL */
} orc_cache;

/* orc_run (warp mode, whole grid, one host thread) with the hit model. */
int orc_run_cached(const char* ptx, const char* kernel, uint32_t grid, uint32_t block,
                   const void* params, uint64_t param_bytes, const orc_buffer* bufs,
                   uint32_t n_bufs, const orc_config* cfg, const orc_cache* cache, void* stats,
                   void* trace, int32_t* status, char* err, uint64_t errlen);

/* orc_run (warp mode, one host thread) that also lists, in run order, the
 * events the page's hints analyzer reads (KernelScope backend doc,
 * hints/analyzer.py): 24-byte records {u32 pc, u32 kind, u32 a, u32 b, u32 c,
 * u32 0} — kind 0 a global ld/st request (a executing lanes, b distinct
 * 128-byte lines, c access bytes), kind 1 a shared request (a its
 * bank-conflict degree), kind 2 a branch that splits the active lanes (a
 * taken lanes, b fall-through lanes). At most events_cap records are copied;
 * *n_events gets the total. */
int orc_run_events(const char* ptx, const char* kernel, uint32_t grid, uint32_t block,
                   const void* params, uint64_t param_bytes, const orc_buffer* bufs,
                   uint32_t n_bufs, const orc_config* cfg, void* stats, void* trace,
                   int32_t* status, void* events, uint64_t events_cap, uint64_t* n_events,
                   char* err, uint64_t errlen);

/* SM-level issue model (KernelScope backend doc, simulator/engine.py and
 * simulator/models.py — WarpStallReason, WarpScheduleInfo), simulated cycle
 * by cycle: CTA c on SM c % n_sm, ctas_per_sm resident CTAs per SM (0 = as
 * many as fit in 32 warps) with the next CTA starting in a slot when the
 * slot's CTA has finished; warp slot i on scheduler i % schedulers; each cycle
 * each scheduler issues for its ready warp with the lowest global warp id.
 * Writes one 64-byte record per warp {start, end, issued, not_selected,
 * stall_exec, stall_mem, stall_math, stall_barrier} (u64 each) and one 32-byte
 * record per SM {cycles, issued, ctas, 0}. Memory is updated; `stats` (NULL
 * or W records) gets the per-warp statistics, whose cycles are this model's
 * absolute ends; no trace is written. */
typedef struct {
  uint32_t n_sm, ctas_per_sm, schedulers;
} orc_sched;

int orc_run_sched(const char* ptx, const char* kernel, uint32_t grid, uint32_t block,
                  const void* params, uint64_t param_bytes, const orc_buffer* bufs,
                  uint32_t n_bufs, const orc_config* cfg, const orc_sched* sched, void* sched_warps,
                  void* sched_sms, void* stats, char* err, uint64_t errlen);

/* Immediate post-dominator of every program entry (instructions and trace
 * pseudo-ops, in program order); the virtual exit is n (= *n_out). */
int orc_ipdom(const char* ptx, const char* kernel, int32_t* out, uint32_t cap,
              uint32_t* n_out, char* err, uint64_t errlen);

/* Parameter layout: offsets/sizes in declaration order, total block size. */
int orc_params(const char* ptx, const char* kernel, uint32_t* offsets,
               uint32_t* sizes, uint32_t cap, uint32_t* n_params,
               uint32_t* param_bytes, char* err, uint64_t errlen);

/* IKET record size of the kernel's trace slots (CuTeDSL IKET 浅析 §2, NativeDump:
 * 4 bytes without payload, 4 + payload for payloads under 8 bytes, else 16):
 * the largest record among its events. Slots are align8(16 + max_ts * bytes). */
int orc_record_bytes(const char* ptx, const char* kernel, uint32_t* bytes, char* err, uint64_t errlen);

/* Event `id`: kind (0 mark, 1 range_start, 2 range_end), payload bytes (0, 4
 * or 8) and name (NUL-terminated, truncated to cap). */
int orc_event_info(const char* ptx, const char* kernel, uint32_t id, uint32_t* kind, uint32_t* payload_bytes,
                   char* name, uint64_t cap, char* err, uint64_t errlen);

/* Event table: kinds (0 mark, 1 range_start, 2 range_end) in id order. */
int orc_events(const char* ptx, const char* kernel, uint32_t* kinds,
               uint32_t cap, uint32_t* n_events, char* err, uint64_t errlen);

#ifdef __cplusplus
}
#endif
#endif

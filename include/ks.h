/*
 * ks.h — C ABI of libks, a GB300 (sm_103a) warp-level SIMT PTX interpreter.
 *
 * What the library computes (KernelScope backend doc, simulator/engine.py and
 * simulator/models.py — PtxSimulator, Thread, Warp, Block, TraceEvent): it
 * steps every simulated warp of a simulated grid in lockstep over a decoded
 * PTX program, one real GPU lane per simulated lane, and produces
 *   1. the simulated global memory (the caller's device buffers, updated in
 *      place by the simulated stores);
 *   2. per-warp cycle counts from a fixed per-class latency table and an
 *      in-order scoreboard (KernelScope backend doc, latency/model.py);
 *   3. per-warp counts of 32-byte sectors and 128-byte lines touched by each
 *      ld/st request (KernelScope backend doc, simulator/engine.py —
 *      analyze_global_memory_access);
 *   4. per-warp trace slots in the IKET layout (CuTeDSL IKET 浅析, §2:
 *      16-byte header u32+u8+u8+u16+u64 then maxTsCntPerWarp records of the
 *      NativeDump size — 4 bytes, 4 + 4 with a 4-byte payload, 16 with an
 *      8-byte payload — slot size rounded up to 8 bytes, one slot per warp,
 *      no atomics);
 *   5. per-warp shared-memory requests and their bank-conflict degrees
 *      (KernelScope backend doc, simulator/engine.py —
 *      analyze_shared_memory_access: 32 banks of 4 bytes, bank =
 *      (address / 4) % 32, a bank whose lanes all use one address is a
 *      broadcast, any other bank's degree is its number of lanes, the
 *      request's degree is the largest).
 *
 * Supported PTX subset: add/sub (.u32 .s32 .u64 .s64 .f32), mul.lo/mad.lo
 * (integers), mul.f32, fma.rn.f32, div.rn.f32, sqrt.rn.f32, and/or/xor
 * (.b32 .b64 .pred), shl (.b32 .b64), shr (.b32 .b64 .u32 .u64 .s32 .s64),
 * cvt (int<->int, .rn f32<-int, .rni/.rzi/.rmi/.rpi int<-f32), mov, setp
 * (eq ne lt le gt ge, lo ls hi hs), selp, bra, ld.param, ld.global,
 * st.global (4- and 8-byte), ld.shared and st.shared (4- and 8-byte; address
 * [reg(+off)] with a 32- or 64-bit register, or [array(+off)]), .shared
 * arrays in the kernel body (at most 48 KiB per CTA; `mov` of an array name
 * gives its shared address), bar.sync 0 / barrier.sync 0 (unguarded, no
 * thread count), ret/exit; registers .b32 .u32 .s32 .f32 .b64
 * .u64 .s64 .pred; special registers %tid %ntid %ctaid %nctaid (.x; .y/.z
 * read 0 or 1) and %laneid; trace pseudo-ops written as comments
 * `//@iket mark NAME`, `//@iket range_start NAME`, `//@iket range_end NAME`,
 * each optionally followed by a 32- or 64-bit payload register.
 *
 * Semantics fixed where the pages are silent:
 *   - %tid.x is the thread's index in its CTA; lanes whose %tid.x >= block
 *     are inactive from the start.
 *   - Divergence: immediate post-dominator reconvergence stack; the
 *     fall-through path runs first; `ret` removes its lanes from every entry.
 *   - Cycles: t = max(t_next, ready[sources], ready[guard], ready[dests]);
 *     dests ready at t + lat; bra/ret set t_next = t + lat, others t + 1;
 *     a store completes at t + lat; cycles = max(last issue + 1, max ready,
 *     last store completion). Trace pseudo-ops cost nothing and are not
 *     counted. Guarded-off instructions still issue.
 *   - thread_insts adds the number of active lanes of every issued
 *     instruction; sectors are distinct addr>>5, lines distinct addr>>7, over
 *     the lanes that execute the access; a request counts when at least one
 *     lane executes it.
 *   - f32: IEEE binary32 round-to-nearest-even with subnormals; every NaN
 *     produced by add/sub/mul/fma/div/sqrt is stored as 0x7FFFFFFF.
 *   - Two lanes of one st.global writing the same address: the highest lane's
 *     value lands. Stores from different warps to the same address, or a load
 *     of a word another warp stores, are undefined (warps run concurrently).
 *   - Registers start at zero, predicates false.
 *   - Trace records: u32 (event_id << 24 | issue clock & 0xFFFFFF); with
 *     payloads the kernel's records are 8 bytes (+ u32 payload) or 16 bytes
 *     (+ u32 0 + u64 payload) for every event of the kernel (events without a
 *     payload store 0); the payload is the register in the warp's lowest
 *     active lane. The header's bytes_per_event holds the record size.
 *   - Shared memory and barriers (KernelScope backend doc, simulator/models.py
 *     Block: a shared array and a barrier per block; Warp.at_barrier): a
 *     kernel that declares .shared arrays or uses bar.sync runs CTA by CTA
 *     with every warp of the CTA resident (blocks above 256 threads run a
 *     slower 1024-thread configuration). When the warps' interpreter state
 *     and the shared arrays exceed one SM's shared memory, the warps' state
 *     moves to global memory (cached in L1/L2; the simulated shared arrays
 *     stay on chip): slower again, and the call then takes a stream-ordered
 *     device allocation of (real CTAs) x (warps per CTA) x (state per warp)
 *     for the launch (cudaMallocAsync / cudaFreeAsync on its stream).
 *     KS_ERR_LIMIT only when the shared arrays alone do not fit.
 *     Shared memory starts
 *     zeroed in every CTA. A warp that issues bar.sync (any active mask)
 *     stops; when every warp of the CTA has stopped at a barrier or finished,
 *     the stopped warps resume with t_next = latest bar.sync issue cycle +
 *     lat[KS_LAT_BAR]; a finished warp never holds a barrier. Shared accesses
 *     are checked like global ones (misaligned first, then outside the
 *     declared arrays). Bank conflicts are counted, not timed. Between two
 *     barriers, a shared word written by one warp and touched by another is
 *     undefined, as for global memory.
 */
#ifndef KS_H
#define KS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- return codes (host errors are negative) ---------------------------- */
#define KS_OK 0
#define KS_ERR_PARSE (-1)       /* malformed PTX */
#define KS_ERR_UNSUPPORTED (-2) /* valid PTX outside the supported subset */
#define KS_ERR_ARG (-3)         /* bad argument (null pointer, size, shape) */
#define KS_ERR_CUDA (-4)        /* a CUDA runtime call failed */
#define KS_ERR_NOT_FOUND (-5)   /* no such kernel / index */
#define KS_ERR_LIMIT (-6)       /* program or register file too large */

/* ---- per-warp device statuses (positive, in ks_warp_stats.status) ------- */
#define KS_ST_OOB 1          /* an address outside every buffer */
#define KS_ST_MISALIGNED 2   /* address not a multiple of the access size */
#define KS_ST_STEP_LIMIT 3   /* the warp tried to issue more than step_limit */
#define KS_ST_SIMT_STACK 4   /* reconvergence stack deeper than allowed */
#define KS_ST_TIMEOUT 5      /* a bounded wait inside the interpreter ran out */
#define KS_ST_INJECTED 6     /* the debug injection point was reached */
#define KS_ST_CACHE_LOG 7    /* cache model: a warp made more global accesses than the
                                log holds, or an access step reached 2^32 - 1 */
#define KS_ST_CACHE_STREAM 8 /* cache model: the second pass's global accesses differ
                                from the first pass's (see ks_simulate_cached) */
#define KS_ST_SCHED_LIMIT 9  /* SM issue model: a warp's issue log is full, or an SM's
                                clock reached 2^31 (see ks_simulate_sched) */

/* ---- latency classes (index of ks_config.lat) --------------------------- */
#define KS_NUM_LAT_CLASSES 12
#define KS_LAT_ALU 0 /* int & f32 add/sub/mul/mad, logic, shifts, cvt, mov, setp, selp, ld.param */
#define KS_LAT_FMA 1 /* fma.rn.f32 */
#define KS_LAT_LDG 2 /* ld.global */
#define KS_LAT_STG 3 /* st.global */
#define KS_LAT_BRA 4 /* bra */
#define KS_LAT_SFU 5 /* div.rn.f32, sqrt.rn.f32 */
#define KS_LAT_RET 6 /* ret, exit */
#define KS_LAT_LDS 7 /* ld.shared */
#define KS_LAT_STS 8 /* st.shared */
#define KS_LAT_BAR 9 /* bar.sync: last arrival to release */
/* classes 10 and 11 are reserved */

#define KS_MAX_BUFFERS 8
#define KS_MAX_PARAM_BYTES 256
#define KS_MAX_STACK 32
#define KS_MAX_SHARED_BYTES 49152   /* simulated shared memory per CTA */
#define KS_MAX_CTA_MODE_BLOCK 1024  /* block limit of kernels with shared memory or bar.sync */

/* ks_config.flags: the layout of each simulated warp's state in the
 * interpreter's shared memory. With neither flag the library picks: PAIR,
 * where every register row holds (value, ready time) pairs and one 8-byte
 * load per lane reads an operand with its scoreboard entry (fewest
 * instructions per simulated instruction), unless the kernel runs outside
 * CTA mode and its PAIR warp state exceeds 12 KiB, where SPLIT (value rows
 * and a separate table of ready times, half the shared memory per warp, so
 * more simulated warps resident) is taken. Results are identical in both
 * layouts; only speed differs. Both flags, or SPLIT forced on a kernel with
 * shared memory or bar.sync (CTA mode runs in PAIR only): KS_ERR_ARG /
 * KS_ERR_UNSUPPORTED. */
#define KS_FLAG_LAYOUT_PAIR 1u
#define KS_FLAG_LAYOUT_SPLIT 2u

typedef struct ks_module ks_module; /* opaque; owned by the library */

/* A simulated global buffer: the caller picks sim_base (4 KiB aligned,
 * buffers non-overlapping); simulated pointers passed in the kernel
 * parameters are sim_base-relative virtual addresses. dev_ptr is caller-owned
 * device memory of `bytes` bytes that the simulated loads read and the
 * simulated stores write. */
typedef struct {
  uint64_t sim_base;
  void* dev_ptr;
  uint64_t bytes;
} ks_buffer;

typedef struct {
  uint32_t lat[KS_NUM_LAT_CLASSES]; /* cycles per latency class, each <= 2^24 */
  uint32_t max_ts_per_warp;         /* trace records per warp slot */
  uint32_t simt_stack_depth;        /* 1..32 entries, base entry included */
  uint64_t step_limit;              /* max issued instructions per warp */
  int64_t inject_warp;              /* debug: global warp id that posts KS_ST_INJECTED; -1 off */
  uint64_t inject_step;             /* ...when its issued-instruction count reaches this */
  uint32_t flags;                   /* 0, or one KS_FLAG_LAYOUT_* (below) */
  uint32_t reserved;
  /* Optional per-instruction profile (device, NULL = none): one
   * ks_pc_profile per program entry, profile_bytes >= ks_profile_bytes();
   * the call zeroes it first. */
  void* profile_buf;
  uint64_t profile_bytes;
} ks_config;

/* Per-instruction profile record (72 bytes), indexed by program entry (the
 * order of ks_kernel_ipdom). It keeps what the page's hints analyzer reads
 * from each trace event (KernelScope backend doc, hints/analyzer.py —
 * analyze_trace_hints), counted per static instruction:
 *   global ld/st: efficiency = min(1, ideal / lines), ideal = ceil(executing
 *     lanes * access size / 128), lines = distinct 128-byte lines (the page's
 *     analyze_global_memory_access); "poor" below 0.25, "uncoalesced" in
 *     [0.25, 0.5); percentages are floor(100 * ideal / lines), exactly;
 *   shared ld/st: the bank-conflict degree (1 = none);
 *   bra: "divergent" when the guard splits the active lanes; the divergence
 *     ratio is the smaller side's lanes / the active lanes, "high" above 0.4,
 *     its percentage floor(100 * smaller / active). */
typedef struct {
  uint64_t requests;        /* ld/st (global or shared) with an executing lane */
  uint64_t poor;            /* global requests with efficiency < 0.25 */
  uint64_t uncoalesced;     /* global requests with 0.25 <= efficiency < 0.5 */
  uint64_t conflicted;      /* shared requests of degree > 1 */
  uint64_t severe;          /* shared requests of degree >= 8 */
  uint64_t divergent;       /* bra executions that split the active lanes */
  uint64_t high_divergence; /* ... with a divergence ratio above 0.4 */
  uint32_t degrees;         /* bit d - 1: a shared request of degree d */
  uint32_t poor_pcts;       /* bit p: a poor global request of efficiency p % */
  uint64_t high_div_pcts;   /* bit p: a high-divergence branch of ratio p % */
} ks_pc_profile;

/* Per-warp statistics record (96 bytes), indexed by global warp id
 * (ctaid * ceil(block/32) + warp index in the CTA). */
typedef struct {
  uint64_t cycles;
  uint64_t warp_insts;   /* issued instructions */
  uint64_t thread_insts; /* sum over issued instructions of the active lanes */
  uint64_t ld_req;
  uint64_t ld_sectors;
  uint64_t st_req;
  uint64_t st_sectors;
  uint64_t ld_lines;
  uint64_t st_lines;
  int32_t status;           /* 0 or a KS_ST_* code */
  uint32_t max_stack_depth; /* deepest reconvergence stack reached */
  uint64_t sh_req;          /* ld/st.shared requests with at least one executing lane */
  uint64_t sh_wavefronts;   /* sum over those requests of the bank-conflict degree */
} ks_warp_stats;

/* Launch totals reduced over every warp record. */
typedef struct {
  uint64_t cycles_max;
  uint64_t cycles_sum;
  uint64_t warp_insts;
  uint64_t thread_insts;
  uint64_t ld_req;
  uint64_t ld_sectors;
  uint64_t st_req;
  uint64_t st_sectors;
  uint64_t ld_lines;
  uint64_t st_lines;
  uint64_t n_warps;
  uint64_t n_failed;          /* warps with a nonzero status */
  int64_t first_failed_warp;  /* lowest failing warp id, -1 if none */
  int32_t status;             /* status of first_failed_warp, 0 if none */
  uint32_t max_stack_depth;
  uint64_t sh_req;
  uint64_t sh_wavefronts;
} ks_totals;

/* Fills the defaults: lat = {4, 4, 400, 20, 8, 36, 1, 23, 23, 20, 0, 0}, max_ts 0,
 * stack depth 32, step limit 2^26, injection off. */
void ks_config_default(ks_config* cfg);

/* Parses and decodes a PTX module (host only; no GPU work): the C form of the
 * page's two loading steps (KernelScope backend doc, "PTX Parser" —
 * ptx/parser.py parse_ptx, which turns the module text into kernels,
 * parameters and instructions with their optional predicates; and
 * simulator/engine.py PtxSimulator.load_kernel, which keeps the executable
 * instructions and builds the pc lookup table). Here the kernels are decoded
 * once into packed instruction records with their reconvergence points, and
 * any kernel of the module can be simulated by name (the page's load_kernel
 * takes the first). `len` bytes of `ptx` (need not be NUL-terminated). On
 * success *out owns the module; free it with ks_free_module. On failure
 * returns KS_ERR_PARSE / KS_ERR_UNSUPPORTED / KS_ERR_LIMIT / KS_ERR_ARG with
 * a message in err (NUL-terminated, truncated to errlen). */
int ks_load_module(const char* ptx, size_t len, ks_module** out, char* err, size_t errlen);

/* Frees the module and the device copies of its programs (which are created
 * lazily, once per device, by the first ks_simulate on that device). */
void ks_free_module(ks_module* mod);

/* Kernel introspection. Any output pointer may be NULL. */
int ks_kernel_info(const ks_module* mod, const char* kernel, uint32_t* n_params,
                   uint32_t* param_bytes, uint32_t* n_events, uint32_t* n_insns,
                   uint32_t* n_reg_slots);
/* Parameter `index` in declaration order: byte offset in the parameter block
 * (natural alignment), size in bytes, name (owned by the module). */
int ks_kernel_param(const ks_module* mod, const char* kernel, uint32_t index,
                    uint32_t* offset, uint32_t* size, const char** name);
/* Event `id`: kind 0 mark, 1 range_start, 2 range_end; ids number the
 * distinct (kind, name) pairs in order of first appearance. */
int ks_kernel_event(const ks_module* mod, const char* kernel, uint32_t id, uint32_t* kind,
                    const char** name);
/* Reconvergence point (immediate post-dominator) of every program entry
 * (instructions and pseudo-ops in order); the virtual exit is *n_out. */
int ks_kernel_ipdom(const ks_module* mod, const char* kernel, int32_t* out, uint32_t cap,
                    uint32_t* n_out);
/* The interpreter's fast-path runs in the PAIR register layout, per program
 * entry (order of ks_kernel_ipdom), three words each (no counterpart on the
 * pages: it describes how this library runs the kernel, not what it
 * computes): out[3i] = the consecutive unguarded FMA / IMAD-type ops from
 * entry i to the end of its run in the fast loop (0: entry i is not in
 * one); out[3i+1] = 1 when every one of them writes a row it also reads
 * (the loop then skips the destination's ready-time load); out[3i+2] = how
 * many of them, from i on, read entry i's b and c rows while none of them
 * but the last writes those (loaded once for all of them). cap is in
 * entries; *n_out receives the number of entries. */
int ks_kernel_fast_runs(const ks_module* mod, const char* kernel, uint32_t* out, uint32_t cap,
                        uint32_t* n_out);
/* The register-file layout a launch of `kernel` with these ks_config.flags
 * runs in (*split: 0 PAIR, 1 SPLIT; see KS_FLAG_LAYOUT_*) and the shared
 * memory each simulated warp's state takes in it (*region_bytes). Errors are
 * those the launch would return for the flags: KS_ERR_ARG (both flags or
 * unknown bits), KS_ERR_UNSUPPORTED (SPLIT forced on a CTA-mode kernel). */
int ks_kernel_layout(const ks_module* mod, const char* kernel, uint32_t flags, uint32_t* split,
                     uint32_t* region_bytes);

/* Size of the caller-owned trace buffer (CuTeDSL IKET 浅析, §2 "buffer
 * 是怎么定形的" — compute_warp_buffer_size_bytes: one slot per warp of
 * align8(16-byte header + maxTsCntPerWarp x bytes_per_event), warps per CTA
 * = ceil(block / 32)): W * align8(16 + 4 * max_ts_per_warp), W = grid *
 * ceil(block / 32). The page multiplies its total by 1.15 for launches whose
 * grid is not known in advance; the grid is an argument here, so the size is
 * exact and ks_simulate rejects anything smaller. */
size_t ks_trace_bytes(uint32_t grid, uint32_t block, uint32_t max_ts_per_warp);
/* The same for records of `record_bytes` (ks_kernel_record_bytes):
 * W * align8(16 + record_bytes * max_ts_per_warp). ks_simulate requires
 * trace_bytes >= this for the kernel's record size. */
size_t ks_trace_bytes_records(uint32_t grid, uint32_t block, uint32_t max_ts_per_warp, uint32_t record_bytes);
/* Trace record size of a kernel's slots: 4 (no payload events), 8 or 16. */
int ks_kernel_record_bytes(const ks_module* mod, const char* kernel, uint32_t* bytes);
/* Payload size of event `id`: 0, 4 or 8 bytes. */
int ks_kernel_event_payload(const ks_module* mod, const char* kernel, uint32_t id, uint32_t* bytes);
/* Size of the caller-owned stats buffer: W * 96 bytes, one ks_warp_stats
 * record per simulated warp. The record holds, per warp, what the page's
 * trace carries per executed instruction and its analyses count
 * (KernelScope backend doc, simulator/models.py — TraceEvent.active_threads,
 * the popcount of the active mask, summed into thread_insts; and
 * simulator/engine.py — analyze_global_memory_access sectors and lines,
 * analyze_shared_memory_access degrees), plus the cycle count and status. */
size_t ks_stats_bytes(uint32_t grid, uint32_t block);
/* Bytes of a kernel's per-instruction profile: 72 per program entry. */
int ks_profile_bytes(const ks_module* mod, const char* kernel, size_t* bytes);

/* Enqueues the interpretation of `kernel` over grid x block simulated
 * threads on `stream` (a cudaStream_t; NULL = the legacy default stream) of
 * the current device, and returns without waiting. This is the page's
 * simulation call (KernelScope backend doc: api/routes.py calls
 * simulate_kernel(parsed, sim_config), sim_config holding {grid_dim,
 * block_dim}; the simulation is simulator/engine.py PtxSimulator.run(), whose
 * step() executes one instruction of every unfinished warp until all have
 * finished), run to
 * completion for every warp of the grid: the page's max_steps bound becomes
 * the per-warp cfg->step_limit, and its trace list becomes the per-warp
 * statistics records and IKET trace slots.
 *   params      host pointer to the kernel's parameter block (layout from
 *               ks_kernel_param), param_bytes >= the kernel's block size,
 *               at most KS_MAX_PARAM_BYTES; copied at launch.
 *   bufs        host array of n_bufs <= 8 buffer descriptors (device memory).
 *   trace_buf   device buffer of trace_bytes >= ks_trace_bytes(...), or NULL
 *               (then no trace is written). Every byte of every slot is
 *               written (unused records as zero).
 *   stats_buf   device buffer of stats_bytes >= ks_stats_bytes(...); every
 *               record is written.
 *   cfg         host pointer; NULL = defaults.
 * Simulated faults do not fail the call: they are reported per warp in the
 * stats records (read them with ks_read_stats). Host-side errors: KS_ERR_ARG
 * (shapes, sizes, buffer table, undersized outputs), KS_ERR_NOT_FOUND,
 * KS_ERR_LIMIT (the real launch's shared memory does not fit: the program
 * and parameters, and for a kernel with shared memory or bar.sync its shared
 * arrays), KS_ERR_CUDA. The first call on a device
 * uploads the module's program there (one allocation per module per device);
 * a kernel with shared memory or bar.sync whose CTA's warp state does not fit
 * on chip also takes a stream-ordered scratch allocation per call (above).
 * Simulations that share output or store-target buffers must not overlap in
 * time; others may be enqueued on different streams and run concurrently
 * (they share only the read-only program copy), which is how small grids
 * fill the GPU. */
int ks_simulate(const ks_module* mod, const char* kernel, uint32_t grid, uint32_t block,
                const void* params, size_t param_bytes, const ks_buffer* bufs, uint32_t n_bufs,
                void* trace_buf, size_t trace_bytes, void* stats_buf, size_t stats_bytes,
                const ks_config* cfg, void* stream);

/* Allocation-free variant of ks_simulate. The pages have no counterpart: it
 * exists for callers that cannot let a library call cudaMalloc. Some
 * processes hand all of the GPU's memory to their own pool when they start
 * (a serving process that reserves its HBM up front), so a library
 * allocation would fail or fragment it; some run under a fixed device-memory
 * budget that is checked once at start-up and may not grow afterwards (a
 * tenant under an MPS memory limit, an embedded or certified deployment); and
 * some cannot afford the implicit device-wide synchronisation that
 * cudaMalloc / cudaFree may cause while other streams are busy. Instead of the
 * per-module device copy that ks_simulate allocates, the kernel's program
 * image (its decoded instructions and constant rows: 64 bytes per program
 * entry plus 4 per constant row) is copied with cudaMemcpyAsync on `stream`
 * into one file-scope device array of KS_STATIC_IMAGE_BYTES bytes, which every
 * GPU that loads the library holds until the process exits. Arguments,
 * outputs and errors are those of ks_simulate, plus KS_ERR_LIMIT when the
 * image exceeds KS_STATIC_IMAGE_BYTES (checked before any GPU work) and for
 * a kernel with shared memory or bar.sync whose CTA's warp state would need
 * ks_simulate's global scratch. The first
 * call on a device looks up the array's device address (cudaGetSymbolAddress)
 * and the device limits; make that first call before any stream capture.
 * Nothing in the array has to start at zero: each call writes every byte the
 * kernel reads. All calls share the array and it keeps the last call's image,
 * so calls whose copies and kernels overlap on the GPU (for example on two
 * streams) race: order them on one stream or synchronise between them. */
#define KS_STATIC_IMAGE_BYTES (64u * 1024u)
int ks_simulate_static(const ks_module* mod, const char* kernel, uint32_t grid, uint32_t block,
                       const void* params, size_t param_bytes, const ks_buffer* bufs, uint32_t n_bufs,
                       void* trace_buf, size_t trace_bytes, void* stats_buf, size_t stats_bytes,
                       const ks_config* cfg, void* stream);

/* ---- Batches (no counterpart on the pages) ----------------------------------
 * Several simulated launches in one call, each with ks_simulate's arguments
 * and each giving exactly ks_simulate's outputs (memory, stats, trace slots,
 * profile), but with the items' warps spread over one real grid: a simulated
 * grid of a few hundred warps leaves most of the GPU idle on its own, and one
 * of many warps ends in a tail where its slowest warps run alone. */
typedef struct ks_batch_item {
  const ks_module* mod;
  const char* kernel;
  uint32_t grid, block;
  const void* params;
  size_t param_bytes;
  const ks_buffer* bufs;
  uint32_t n_bufs;
  uint32_t reserved;      /* 0 */
  void* trace_buf;        /* device, may be NULL */
  size_t trace_bytes;
  void* stats_buf;        /* device, W x 96 bytes */
  size_t stats_bytes;
  const ks_config* cfg;   /* NULL: ks_config_default */
} ks_batch_item;

/* Enqueues n_items simulations on `stream`. Every item is checked first as
 * ks_simulate checks it; if one fails, its error is returned, *failed_item
 * (if not NULL) is set to its index and nothing is launched (modules may
 * still have been uploaded). Otherwise *failed_item = n_items and the items
 * run in real grids of one kernel form each (the same mode, lean or
 * profiled, and in CTA mode the same block), in the order of each grid's
 * first item: at most 32 items and at most 16 simulated warps per SM of the
 * GPU in a grid, so that a grid runs as one wave (an item larger than that
 * fills the GPU alone and is launched as ks_simulate launches it). Within a
 * grid the real CTAs are shared out in proportion to the items' simulated
 * warps (CTAs in CTA mode); when every simulated warp fits on the GPU at
 * once, the grid is a multiple of the SM count with the same number of real
 * warps on every SM. When the items take more than one real grid, the grids
 * run side by side on up to four streams that the library creates once per
 * device and keeps (one grid's last warps then overlap the next grid's work):
 * they start after everything enqueued on `stream` before the call, and
 * everything enqueued on `stream` after the call waits for all of them, as
 * for a launch on `stream` itself. While `stream` is capturing a graph, every
 * grid is launched on `stream`. Items must not share
 * output, trace, stats, profile or store-target buffers (they run at the same
 * time). *n_launched (if not NULL) receives the number of real kernel
 * launches enqueued. KS_ERR_ARG for items == NULL or n_items == 0, else the
 * errors of ks_simulate (a launch error after earlier grids were enqueued
 * leaves those enqueued). */
int ks_simulate_batch(const ks_batch_item* items, uint32_t n_items, void* stream, uint32_t* failed_item,
                      uint32_t* n_launched);

/* Reduces n_warps stats records (device pointer) on `stream`, waits for the
 * stream, and writes the totals to *out (host): the launch-wide sums of the
 * per-warp records (KernelScope backend doc, simulator/models.py —
 * TraceEvent.active_threads summed over the trace, here thread_insts), the
 * largest cycle count, and the first failing warp with its status. Uses a
 * small device accumulator that the library allocates once per device; calls
 * are serialised inside the library.
 * Shape: the call takes the stats buffer and its warp count rather than only
 * (stream, host totals, device status), because the library keeps no state
 * per simulation: the records live in the caller's buffer, any earlier
 * simulation's records can be reduced again, and the device status of the
 * launch is the `status` / first_failed_warp fields of *out (the status of the
 * lowest-indexed failing warp), so no separate status word is needed. */
int ks_read_stats(const void* stats_buf, uint64_t n_warps, void* stream, ks_totals* out);

/* ---- L1/L2 hit model (KernelScope backend doc, simulator/engine.py —
 * "Cache parameters", SimpleCache, _execute_instruction) ----------------------
 * Two direct-mapped caches of 128-byte lines, one L1 of l1_lines lines and one
 * L2 of l2_lines lines, each a single instance shared by the whole simulated
 * grid (as the page's simulator holds one of each). A line of address a is
 * a / 128; its set is line % lines; an access hits when the set holds that
 * line, and a miss installs it. Every ld.global / st.global with at least one
 * executing lane makes one access with the address of its lowest executing
 * lane (the page's "representative" address): L1 first, L2 on an L1 miss. A
 * load's destination is then ready lat_l1 (L1 hit), lat_l2 (L2 hit) or
 * lat[KS_LAT_LDG] (both miss: the DRAM latency) cycles after issue instead of
 * lat[KS_LAT_LDG]; stores keep lat[KS_LAT_STG]. Nothing else changes.
 *
 * Access order (the page's step(): one instruction of every warp per step,
 * blocks then warps in order): accesses are ordered by (step, global warp id),
 * where an instruction's step is the number of instructions its warp issued
 * before it, plus, after each bar.sync, the steps the warp spent waiting: a
 * barrier releases at the end of the step in which the last warp of the CTA
 * arrived or finished, and its warps issue again at the next step. Trace
 * pseudo-ops take no step.
 *
 * How it runs (two forms on `stream`; both give the same results where
 * both apply):
 *  - Re-interpretation (max_runs_per_warp == 0, and every kernel with shared
 *    memory or bar.sync): the library interprets the launch twice. The first
 *    pass suppresses the simulated stores and logs every access (line, step)
 *    per warp; two stable radix sorts of the log — by (L1 set, step, warp),
 *    then the L1 misses by their L2 set — put each set's accesses in order,
 *    and an access hits when the one before it in its set had the same line.
 *    The second pass is the real run: stores land, loads take the logged
 *    level's latency, and every access is checked against the log. If the
 *    addresses or the control flow depend on a value that the launch itself
 *    stored, the first pass may log other accesses than the second makes;
 *    such warps end with KS_ST_CACHE_STREAM rather than a wrong result.
 *  - Timing replay (max_runs_per_warp > 0, kernels without shared memory
 *    or bar.sync): timing never changes what a warp executes, so the one
 *    interpretation is the real run (stores land, loads read them) and also
 *    logs each warp's issued runs of program entries (at most
 *    max_runs_per_warp); after the same sorts, a replay kernel — one thread
 *    per simulated warp, no values — recomputes every warp's scoreboard from
 *    its runs with each load's level latency and rewrites what timing
 *    decides: the cycles of the stats record and trace header, the trace
 *    records' timestamps, the hit counts. About one interpretation instead
 *    of two. A warp reading back its own stores gets the values it stored
 *    (no KS_ST_CACHE_STREAM). A warp whose accesses or runs overflow their
 *    logs ends with KS_ST_CACHE_LOG, its stores done, its cycles those of
 *    DRAM latencies.
 */
typedef struct {
  uint32_t l1_lines;              /* default 1024 (128 KB); 1..65536 */
  uint32_t l2_lines;              /* default 49152 (6 MB); a multiple of l1_lines, l2/l1 <= 65535 */
  uint32_t lat_l1;                /* default 28 cycles, <= 2^24 */
  uint32_t lat_l2;                /* default 150 cycles, <= 2^24 */
  uint32_t max_accesses_per_warp; /* log capacity per warp (default 1024) */
  uint32_t max_runs_per_warp;     /* 0 (default): re-interpretation; > 0: timing replay with a run
                                     log of this many runs per warp (see above) */
  uint32_t reserved[2];
} ks_cache_config;

#define KS_CACHE_LINE_BYTES 128
#define KS_CACHE_L1_HIT 0
#define KS_CACHE_L2_HIT 1
#define KS_CACHE_DRAM 2

/* Per-warp cache counts, the first W records of the workspace. */
typedef struct {
  uint32_t n_access; /* global accesses made */
  uint32_t l1_hits;
  uint32_t l2_hits;
  uint32_t dram;     /* missed both */
} ks_cache_warp;

/* One logged access; warp w's k-th access is record w * max_accesses_per_warp
 * + k of the log, which starts at byte ceil(16 W / 256) * 256 of the workspace
 * (after the W ks_cache_warp records). */
typedef struct {
  uint64_t line;  /* representative address / 128 */
  uint32_t step;  /* position in the access order (see above) */
  uint32_t level; /* KS_CACHE_L1_HIT, KS_CACHE_L2_HIT or KS_CACHE_DRAM */
} ks_cache_access;

/* Defaults: 1024 and 49152 lines, 28 and 150 cycles, 1024 accesses per warp. */
void ks_cache_config_default(ks_cache_config* cc);

/* Bytes of the caller-owned device workspace of ks_simulate_cached: W
 * ks_cache_warp records, W * max_accesses_per_warp ks_cache_access records,
 * then the sort's scratch (its size is asked of the current CUDA device),
 * then (max_runs_per_warp > 0) W run counts and W * max_runs_per_warp runs.
 * 0 when the configuration is invalid, when the log would hold 2^31 records
 * or more, or when no CUDA device can be queried. */
size_t ks_cache_workspace_bytes(uint32_t grid, uint32_t block, const ks_cache_config* cc);

/* ks_simulate with the L1/L2 hit model. Arguments and errors as ks_simulate,
 * plus cc (host; NULL = defaults) and `workspace`, device memory of at least
 * ks_cache_workspace_bytes(grid, block, cc) bytes (KS_ERR_ARG otherwise, and
 * for an invalid cc; KS_ERR_LIMIT when ceil(log2(l1_lines)) + 32 +
 * ceil(log2(W)) > 64, the sort key's width). Unlike ks_simulate, this call
 * does not only enqueue: it enqueues the first pass, then BLOCKS the calling
 * host thread until `stream` has finished everything enqueued on it so far
 * (one cudaStreamSynchronize, to read the number of logged accesses, which
 * sizes the sorts: they cost in proportion to the accesses made, not to the
 * log's capacity), then enqueues the sorts and the second pass and returns;
 * so the call cannot be captured into a CUDA graph. Afterwards the workspace holds the per-warp
 * counts and the access log with each access's level; per-warp statuses
 * KS_ST_CACHE_LOG and KS_ST_CACHE_STREAM report a log that was too small or
 * an access stream that the first pass could not predict. */
int ks_simulate_cached(const ks_module* mod, const char* kernel, uint32_t grid, uint32_t block,
                       const void* params, size_t param_bytes, const ks_buffer* bufs, uint32_t n_bufs,
                       void* trace_buf, size_t trace_bytes, void* stats_buf, size_t stats_bytes,
                       const ks_config* cfg, const ks_cache_config* cc, void* workspace,
                       size_t workspace_bytes, void* stream);

/* Several cached simulations in one call (no counterpart on the pages), each
 * giving exactly ks_simulate_cached's outputs: the items' first passes run
 * as ks_simulate_batch runs its items (shared real grids), then each item's
 * levels (one stream wait each), then the second passes, again batched (the
 * timing replays side by side on ks_simulate_batch's helper streams).
 * Each item has its own hit model: cache NULL means ks_cache_config_default,
 * and its workspace is sized by ks_cache_workspace_bytes. Checks, failed_item
 * and the no-launch guarantee are those of ks_simulate_batch, plus the
 * cache arguments' checks of ks_simulate_cached. *n_launched (if not NULL)
 * receives the kernel launches of this library's own kernels (interpreter
 * grids and the level kernels; the sorts and the scan are CUB's). Items must
 * not share buffers or workspaces. */
typedef struct ks_cached_item {
  ks_batch_item sim;
  const ks_cache_config* cache;
  void* workspace;
  size_t workspace_bytes;
} ks_cached_item;
int ks_simulate_cached_batch(const ks_cached_item* items, uint32_t n_items, void* stream, uint32_t* failed_item,
                             uint32_t* n_launched);

/* ---- SM-level issue model (KernelScope backend doc, simulator/engine.py and
 * simulator/models.py — WarpStallReason, _determine_stall_reason,
 * WarpScheduleInfo) ------------------------------------------------------------
 * The launch's warps share simulated SMs: CTA c runs on SM c % n_sm; an SM
 * holds ctas_per_sm CTAs at once (at most 32 warps) and starts its next CTA in
 * a slot when the slot's CTA has finished (the latest end of its warps). Warp
 * slot i of an SM issues on scheduler i % schedulers_per_sm; a scheduler issues
 * at most one instruction per cycle, to the ready warp with the lowest global
 * warp id (the order of the page's step()). A warp is ready when the in-order
 * scoreboard of the per-warp model lets it issue; the per-warp rules stay as
 * they are (latencies, barriers, the store drain), with absolute cycles from
 * the SM's cycle 0. Cycles a warp waits are counted by what it waits for: the
 * scheduler picked another ready warp ("not selected"); a result of a load
 * (ld.global / ld.shared: "memory dependency"), of div/sqrt ("math pipe"), of
 * anything else or a branch's latency ("execution dependency"; when results of
 * several kinds arrive in the same cycle the load counts first, then div/sqrt);
 * a barrier's release ("barrier"). Per warp: start + issued + the waits + the
 * drain after its last issue = end.
 * Two more of the page's reasons are labels on issued instructions, as the
 * page's own step() attaches them (it never holds a warp back for them), so
 * they are counts of instructions, not cycles, and change no timing:
 * "memory throttle" (the page: an instruction of its memory class — ld, st,
 * mov — issued while 4 or more memory operations are pending), read per SM:
 * an ld.*, st.* or mov issued at a cycle when at least 4 other warps of its
 * SM have their latest global or shared load or store issued at an earlier
 * cycle and not yet complete (the load's result not yet ready, the store not
 * yet drained); and "divergence" (declared by the page, returned nowhere),
 * read as: an instruction issued while some of the warp's live lanes (lanes
 * that have not executed ret) wait on the reconvergence stack. */
typedef struct {
  uint32_t n_sm;              /* simulated SMs (default 152) */
  uint32_t ctas_per_sm;       /* resident CTAs per SM, ctas_per_sm * ceil(block / 32) <= 32;
                                 0 = as many as fit in 32 warps (default 0) */
  uint32_t schedulers_per_sm; /* 1, 2 or 4 (default 4) */
  uint32_t max_runs_per_warp; /* issue-log capacity: runs of consecutive program entries
                                 a warp consumes between control transfers (default 4096) */
  uint32_t reserved[4];
} ks_sched_config;

/* Per-warp schedule record (80 bytes), indexed by global warp id. */
typedef struct {
  uint64_t start, end;     /* the SM cycles at which the warp's CTA started, and its last
                              result or store completed */
  uint64_t issued;         /* instructions issued (= ks_warp_stats.warp_insts) */
  uint64_t not_selected;   /* ready, another warp of the scheduler issued */
  uint64_t stall_exec;     /* waiting on an ALU / FMA result or a branch's latency */
  uint64_t stall_mem;      /* waiting on a load's result */
  uint64_t stall_math;     /* waiting on a div / sqrt result */
  uint64_t stall_barrier;  /* waiting at bar.sync for the release */
  uint64_t throttled;      /* label: ld / st / mov issued with >= 4 other warps' memory
                              operations pending on the SM (instructions, not cycles) */
  uint64_t diverged;       /* label: instructions issued while live lanes of the warp
                              waited on the reconvergence stack */
} ks_sched_warp;

/* Per-SM record (32 bytes). */
typedef struct {
  uint64_t cycles;  /* the SM's last warp end (0 without CTAs) */
  uint64_t issued;  /* instructions its warps issued: IPC = issued / cycles */
  uint64_t ctas;    /* CTAs it ran */
  int32_t status;   /* 0 or KS_ST_SCHED_LIMIT */
  uint32_t reserved;
} ks_sched_sm;

void ks_sched_config_default(ks_sched_config* sc);

/* Device workspace of ks_simulate_sched (the issue log): W * (4 *
 * max_runs_per_warp + 4) bytes rounded up; 0 for an invalid configuration. */
size_t ks_sched_workspace_bytes(uint32_t grid, uint32_t block, const ks_sched_config* sc);

/* ks_simulate plus the SM-level issue model. The interpreter runs once (its
 * outputs are those of ks_simulate) and logs each warp's issued program
 * entries; a replay kernel then schedules the SMs. sched_warps: device, W
 * ks_sched_warp records; sched_sms: device, n_sm ks_sched_sm records;
 * workspace: device, ks_sched_workspace_bytes. KS_ERR_ARG for an invalid sc
 * or undersized buffers, KS_ERR_LIMIT when a replay's shared memory (the
 * program plus a ready table per warp slot) does not fit. Enqueues on `stream`
 * and returns. A warp whose issue log overflows ends with KS_ST_SCHED_LIMIT in
 * its stats, and its SM's record carries the same status. */
int ks_simulate_sched(const ks_module* mod, const char* kernel, uint32_t grid, uint32_t block,
                      const void* params, size_t param_bytes, const ks_buffer* bufs, uint32_t n_bufs,
                      void* trace_buf, size_t trace_bytes, void* stats_buf, size_t stats_bytes,
                      const ks_config* cfg, const ks_sched_config* sc, void* sched_warps,
                      size_t sched_warps_bytes, void* sched_sms, size_t sched_sms_bytes, void* workspace,
                      size_t workspace_bytes, void* stream);

/* ---- host post-pass: occupancy (KernelScope backend doc,
 * occupancy/calculator.py — calculate_occupancy) ----------------------------
 * Resident warps per SM from three limits, as the page computes them:
 * registers (threads' registers per warp rounded up to 256, the SM's file
 * divided by that), shared memory (per-block bytes rounded up to 256, blocks
 * that fit times warps per block) and block size (min(max threads / block,
 * max blocks) times warps per block), capped at the SM's warp limit. A limit
 * whose input is 0 does not bind. The limiter is the first of registers,
 * shared memory, block size whose warps equal the result. */
typedef struct {
  uint32_t max_threads_per_sm;
  uint32_t max_warps_per_sm;
  uint32_t max_blocks_per_sm;
  uint32_t registers_per_sm;
  uint32_t shared_memory_per_sm;
} ks_gpu_limits;

#define KS_LIMITER_REGISTERS 0
#define KS_LIMITER_SHARED_MEMORY 1
#define KS_LIMITER_BLOCK_SIZE 2

typedef struct {
  uint32_t active_warps_per_sm;
  uint32_t max_warps_per_sm;
  uint32_t warps_by_registers;
  uint32_t warps_by_shared_memory;
  uint32_t warps_by_block_size;
  int32_t limiter;           /* KS_LIMITER_* */
  double occupancy_percent;  /* 100 * active / max warps */
} ks_occupancy_result;

/* Limits of an architecture by name: "sm_75", "sm_80", "sm_86", "sm_89",
 * "sm_90" (the page's table; fields the page elides take the public CUDA
 * values), "sm_100", "sm_103". KS_ERR_NOT_FOUND for other names. */
int ks_gpu_limits_of(const char* arch, ks_gpu_limits* out);
/* KS_ERR_ARG for a null pointer, threads_per_block of 0 or above the SM's
 * threads, or a limits record with zero warps. */
int ks_occupancy(const ks_gpu_limits* limits, uint32_t threads_per_block, uint32_t registers_per_thread,
                 uint32_t shared_memory_per_block, ks_occupancy_result* out);

/* ---- host post-pass: trace export (CuTeDSL IKET 浅析 §3, "postprocess →
 * Perfetto trace") --------------------------------------------------------
 * Converts a host copy of a launch's trace slots into Chrome trace-event JSON,
 * which Perfetto opens: one process per CTA ("CTA c"), one thread per warp
 * ("warp w", w counted in its CTA), a complete event "warp" from 0 to the
 * slot's cycle count, and per record a "B" (range_start), "E" (range_end) or
 * thread-scoped instant "i" (mark) named after the event, with args {"id"}
 * and, for payload events, {"payload": raw bits as an unsigned integer}.
 * Record stamps hold the low 24 bits of the cycle; they are unwrapped in
 * record order (a warp's stamps never decrease, and consecutive stamps are
 * taken to be less than 2^24 cycles apart). ts and dur are cycles /
 * cycles_per_us (microseconds). grid, block and max_ts are the launch's.
 * *needed gets the length without the NUL; KS_ERR_ARG when out is NULL or
 * cap < *needed + 1 (call again with a larger buffer), when trace_bytes is
 * smaller than the launch's slots, or when a record names an unknown event. */
int ks_trace_to_json(const ks_module* mod, const char* kernel, uint32_t grid, uint32_t block, uint32_t max_ts,
                     const void* trace_host, size_t trace_bytes, double cycles_per_us, char* out, size_t cap,
                     size_t* needed);

/* ---- host post-pass: hints (KernelScope backend doc, hints/analyzer.py —
 * analyze_trace_hints) ---------------------------------------------------------
 * The page's rules, read from a per-instruction profile (a host copy of
 * ks_config.profile_buf) instead of from every trace event: the page emits
 * one hint per event, here one hint per (instruction, rule) stands for all of
 * that instruction's events, with their number in `count` and the worst
 * event's value in the message. In order, per program entry:
 *   shared degree >= 8:  CRITICAL MEMORY "<d>-way bank conflict" (largest d),
 *                        "Severe bank conflict causing serialized access";
 *   shared degree 2..7:  WARNING MEMORY "<d>-way bank conflict" (largest d),
 *                        "Bank conflict reducing throughput";
 *   global efficiency < 0.25: CRITICAL MEMORY "Poor memory efficiency (<p>%)"
 *                        (lowest p), "Scattered access causing many transactions";
 *   divergence ratio > 0.4: WARNING DIVERGENCE "High divergence (<p>%)" (largest
 *                        p), "Significant warp divergence at this branch";
 * then, with pc = -1: more than 5 shared requests of degree > 1 in the launch:
 * WARNING MEMORY "Shared memory bank conflicts (<n> events)", "Consider padding
 * arrays or restructuring access patterns"; more than 3 divergent branch
 * executions: WARNING DIVERGENCE "Branch divergence detected (<n> events)",
 * "Consider restructuring conditionals or using predication"; and with an
 * occupancy result: below 25 %: CRITICAL OCCUPANCY "Very low occupancy (<x>%)",
 * "Limited by <limiter>. Consider reducing resource usage."; below 50 %:
 * WARNING OCCUPANCY "Low occupancy (<x>%)", "Limited by <limiter>." (x printed
 * as the shortest decimal that reads back as the same double, with ".0" when
 * it is whole; limiter "registers", "shared_memory" or "block_size"). The
 * page also counts uncoalesced requests and register pressure but bases no
 * hint on them. */
#define KS_HINT_INFO 0
#define KS_HINT_WARNING 1
#define KS_HINT_CRITICAL 2
#define KS_HINT_MEMORY 0
#define KS_HINT_DIVERGENCE 1
#define KS_HINT_OCCUPANCY 2
#define KS_HINT_REGISTERS 3

typedef struct {
  int32_t category; /* KS_HINT_MEMORY ... */
  int32_t severity; /* KS_HINT_INFO ... */
  int32_t pc;       /* program entry, -1 for launch-wide hints */
  uint32_t reserved;
  uint64_t count;   /* events the hint stands for (1 for occupancy) */
  char message[64];
  char detail[96];
} ks_hint;

/* Hints of one launch. profile: host array of n_entries records (may be NULL
 * with n_entries 0); occupancy: NULL or a ks_occupancy result. Writes at most
 * cap hints to out and their number to *n_hints; KS_ERR_ARG when out is too
 * small (call again with *n_hints) or an argument is null. */
int ks_hints(const ks_pc_profile* profile, uint32_t n_entries, const ks_occupancy_result* occupancy,
             ks_hint* out, uint32_t cap, uint32_t* n_hints);

/* Text for any KS_* return code or status. */
const char* ks_status_string(int code);

#ifdef __cplusplus
}
#endif
#endif /* KS_H */

// ks_internal.h — decoded program format and launch block shared by the host
// decoder (ks_decode.cpp), the C ABI (ks_capi.cpp) and the sm_103a
// interpreter (ks_interp.cu).
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "../../include/ks.h"

namespace ks {

// Handler opcodes of the decoded program. Type and operand width are folded
// into the opcode so the interpreter dispatches once per instruction.
enum Op : uint8_t {
  OP_EVENT = 0,  // trace pseudo-op, zero cost
  OP_RET,
  OP_BRA,
  OP_LDP32, OP_LDP64,  // ld.param
  OP_LDG32, OP_LDG64,  // ld.global
  OP_STG32, OP_STG64,  // st.global
  OP_MOV32, OP_MOV64, OP_MOVSP,
  OP_ADD32, OP_SUB32, OP_MUL32, OP_MAD32,
  OP_ADD64, OP_SUB64, OP_MUL64, OP_MAD64,
  OP_AND32, OP_OR32, OP_XOR32, OP_AND64, OP_OR64, OP_XOR64,
  OP_ANDP, OP_ORP, OP_XORP,
  OP_SHL32, OP_SHR32U, OP_SHR32S, OP_SHL64, OP_SHR64U, OP_SHR64S,
  OP_FADD, OP_FSUB, OP_FMUL, OP_FFMA, OP_FDIV, OP_FSQRT,
  OP_SETP_U32, OP_SETP_S32, OP_SETP_U64, OP_SETP_S64, OP_SETP_F32,
  OP_SELP32, OP_SELP64,
  OP_CVT_F32_U32, OP_CVT_F32_S32, OP_CVT_F32_U64, OP_CVT_F32_S64,
  OP_CVT_F2I,          // flags: KS_CVT_* destination | rounding << 4
  OP_CVT_ZX, OP_CVT_SX,  // 32 -> 64 zero / sign extension
  OP_LDS32, OP_LDS64,  // ld.shared (flags: KS_SHA_*)
  OP_STS32, OP_STS64,  // st.shared
  OP_BAR,              // bar.sync 0
  OP_COUNT
};

// the interpreter tests these opcode ranges with two compares
static_assert(OP_LDG64 == OP_LDG32 + 1 && OP_STG32 == OP_LDG32 + 2 && OP_STG64 == OP_LDG32 + 3,
              "ld/st.global opcodes must be consecutive");
static_assert(OP_SETP_S32 == OP_SETP_U32 + 1 && OP_SETP_U64 == OP_SETP_U32 + 2 && OP_SETP_S64 == OP_SETP_U32 + 3 &&
                  OP_SETP_F32 == OP_SETP_U32 + 4,
              "setp opcodes must be consecutive");

// shared address form in KsInsn::flags of OP_LDS* / OP_STS*: a register base
// (KS_SHA_REG, 64-bit with KS_SHA_WIDE) plus KsInsn::imm, or imm alone
constexpr uint8_t KS_SHA_REG = 1, KS_SHA_WIDE = 2;
// KsInsn::flags of OP_MOV32 / OP_MOV64 / OP_MOVSP: written with the `mov`
// opcode (an integer cvt of one width decodes to a move as well)
constexpr uint8_t KS_MOV_OPCODE = 0x80;
// setp comparison in KsInsn::flags
enum Cmp : uint8_t { CMP_EQ = 0, CMP_NE, CMP_LT, CMP_LE, CMP_GT, CMP_GE };
// cvt float->int destination (low nibble) and rounding (high nibble)
enum CvtDst : uint8_t { CVT_S32 = 0, CVT_U32, CVT_S64, CVT_U64 };
enum CvtRnd : uint8_t { RND_RNI = 0, RND_RZI, RND_RMI, RND_RPI };
// special registers (KsInsn::imm of OP_MOVSP)
enum Special : uint8_t { SP_TID = 0, SP_NTID, SP_CTAID, SP_NCTAID, SP_LANEID, SP_ZERO, SP_ONE };

// Operand encoding: 0..KS_MAX_SLOTS-1 register slot (32-bit; a 64-bit
// register uses slots s and s+1), KS_CONST_BIT|i constant-pool entry i.
// Predicate operands are predicate indices 0..KS_MAX_PREDS-1.
constexpr uint32_t KS_MAX_SLOTS = 96;
constexpr uint32_t KS_MAX_PREDS = 31;
constexpr uint32_t KS_MAX_CONSTS = 128;
constexpr uint8_t KS_CONST_BIT = 0x80;
// a routed operand position that reads the zero row (its value travels in aux)
constexpr uint8_t OPND_ZERO = 0x7F;
// Scoreboard (ready-time table) indices: slots 0..95, predicates 96..126,
// 127 never written (always ready).
constexpr uint32_t KS_HZ_PRED0 = 96;
constexpr uint8_t KS_HZ_NONE = 127;
constexpr uint32_t KS_HZ_ENTRIES = 128;
constexpr uint8_t KS_NO_GUARD = 0xFF;
constexpr uint32_t KS_MAX_INSNS = 2048;
// Largest latency a class may have (keeps the 32-bit epoch-relative clock exact).
constexpr uint32_t KS_MAX_LATENCY = 1u << 24;

// One decoded instruction, 32 bytes (two 16-byte shared-memory loads).
struct alignas(16) KsInsn {
  uint8_t op;
  uint8_t lat;     // latency class
  uint8_t guard;   // predicate index or KS_NO_GUARD
  uint8_t gneg;    // 1: guard negated
  uint8_t d, a, b, c;
  uint8_t hd, ha, hb, hc;  // scoreboard indices of dest and sources
  uint8_t hg;              // scoreboard index of the guard
  uint8_t flags;
  uint16_t event;          // trace event id
  uint64_t imm;            // address offset / param offset / special id
  uint32_t target;         // branch target
  uint32_t rpc;            // reconvergence pc of a branch
};
static_assert(sizeof(KsInsn) == 32, "KsInsn must be 32 bytes");

// ---- device program format ---------------------------------------------
// The host resolves every KsInsn into a 64-byte DevInsn whose operand fields
// are byte offsets of rows inside a warp's shared-memory region. A row holds
// one simulated register (or constant) across the 32 lanes. Two layouts of
// the region exist; the decoder writes one program image for each and the
// launch takes one of them (ks::pick_layout):
//
// PAIR layout (rows of 256 B): a row holds one 8-byte pair per lane,
// (value, ready), where `ready` is the simulated cycle at which the register
// becomes available (the same in every lane), so one 64-bit shared load
// returns both an operand and its scoreboard entry:
//
//   warp region: [register rows: n_slots x 256 B]   row s = slot s
//                [constant rows: n_crows x 256 B]   (constant, 0) in every lane
//                [zero row: 256 B]                  operand "none": (0, 0), never written
//                [predicate ready table: 32 u32, padded to 256 B]
//                    entry p: predicate p (p = 31 is the always-true predicate and stays 0)
//                [reconvergence stack: 32 x 8 B]
//
// SPLIT layout (rows of 128 B): a row holds the values only, and the ready
// times live in a table of one word per row -- half the shared memory per
// warp, for kernels whose warp regions would otherwise bound the resident
// warps:
//
//   warp region: [register rows: n_slots x 128 B]
//                [constant rows: n_crows x 128 B]
//                [zero row: 128 B]
//                [ready table: one u32 per row]     (constant rows and the zero row: 0)
//                [predicate ready table: 32 u32]
//                [reconvergence stack: 32 x 8 B]
//
//   An instruction's scoreboard terms are gathered one per lane: lane l
//   loads the ready word named by halfword l mod 4 (fast and mid loops: rows
//   a, b, c, destination) or l mod 8 (general path: then the guard and the
//   predicate sources) of the record's hazard words, and one warp max
//   reduction gives the latest term.
//
// In both layouts a 64-bit register or constant uses two consecutive rows
// (low word first), so its high word is at row offset + row_bytes, and its
// scoreboard entry is the low row's.
constexpr uint32_t ROW_PAIR = 256, ROW_SPLIT = 128;

struct alignas(16) DevInsn {
  // q0, q1: everything the fast and mid loops read (both layouts)
  uint32_t op;
  uint32_t wlat;   // in the image: latency class | flags (below); patched to dest latency
  uint32_t aux;    // offset / param offset / special / event / cvt / cmp|pred / target|rpc<<16 / pred idx
  uint32_t d;      // destination row offset (the zero row if absent)
  uint32_t a, b, c;  // source row offsets (region-relative; the zero row if absent)
  uint32_t inc;    // bit 0: issued (0 for a trace pseudo-op or the exit sentinel);
                   // bit 1: has a register destination; bit 2: has a predicate destination
  // q2, q3 by layout (x[6] = dlat and x[7] = nlat in both):
  //   PAIR:  guard, gneg, ha, hb, hc, hd, dlat, nlat
  //          ha/hb/hc/hd: predicate-table offsets of predicate sources /
  //          destination (entry 31 if absent); DOP_MADII: hc = its immediate;
  //          a fast op in a run: hc = the ops from it on (itself included)
  //          that read the same b and c rows as it, which none of them but
  //          the last writes (the fast loop then loads those rows once), in
  //          KEEP_COUNT, and KEEP_FPU when all of them are DOP_FPU
  //   SPLIT: hz[0..3], guard, gneg, dlat, nlat
  //          hz: ready-word offsets (16 bits each, region-relative) of the
  //          scoreboard terms: halfwords 0..3 = rows a, b, c and the
  //          destination (the register's row, or the predicate written by
  //          setp / predicate logic), 4 = the guard predicate, 5..7 =
  //          predicate sources; an absent term names a word that stays 0.
  //          DOP_MADII: guard = its immediate (the mid loop runs every
  //          DOP_MADII; its guard term is in hz)
  //   guard: predicate lane 0..30, or 31 (always true); gneg: 0 or 0xFFFFFFFF
  //   dlat (patched): store completion latency (0 if not a store)
  //   nlat (patched): issue-clock advance (latency for bra/ret, 1 otherwise, 0 if inc == 0)
  uint32_t x[8];
};
static_assert(sizeof(DevInsn) == 64, "DevInsn must be 64 bytes");
// byte offset of the SPLIT layout's hazard halfwords inside a DevInsn
constexpr uint32_t DEV_HZ_OFF = 32;
// positions in DevInsn::x
constexpr uint32_t DX_DLAT = 6, DX_NLAT = 7;

// flags in DevInsn::wlat of the uploaded image
constexpr uint32_t DEV_HAS_DEST = 1u << 8;
constexpr uint32_t DEV_IS_STORE = 1u << 9;
constexpr uint32_t DEV_IS_CTRL = 1u << 10;
// bits of DevInsn::inc
constexpr uint32_t INC_ISSUE = 1u, INC_RDEST = 2u, INC_PDEST = 4u;
// INC_ADDR64: the address operand `a` is a 64-bit register (shared accesses)
constexpr uint32_t INC_ADDR64 = 32u;
// INC_FUSE: an unguarded setp whose next entry is a bra guarded by the setp's
// predicate; aux bit 16 = that guard's negation, aux bits 17..31 = the bra's
// target, so a uniform outcome issues the bra in the same step
constexpr uint32_t INC_FUSE = 64u;
// SM issue model labels: INC_MCLASS, an instruction of the page's memory
// class (ld, st, mov); INC_MEMOP, a global or shared load or store (a memory
// operation that stays pending until it completes)
constexpr uint32_t INC_MCLASS = 128u, INC_MEMOP = 256u;
// bit 15 of an issue-run log record: the run issued while some live lanes
// waited on the reconvergence stack (the divergence label); bits 0..14 hold
// its length - 1, bits 16..31 its first program entry
constexpr uint32_t RUN_DIVERGED = 1u << 15;
// bits 16..31 of DevInsn::inc of a fast-path op: the number of consecutive
// fast-path ops starting at it (a run's length, at most KS_MAX_INSNS)
constexpr uint32_t INC_RUN_SHIFT = 16u;
// Fast runs of at most this many ops carry INC_MID and a run length of 0: the
// mid loop runs them (DOP_FPU / DOP_IMAD cases) with the ops around them.
constexpr uint32_t MID_FAST_RUN = 2u;
// INC_MID: unguarded register-to-register op with no predicate operand, no
//          memory access and no control transfer (runs in the mid loop)
// INC_PHAZ: has a predicate source or destination (its ready entries matter)
constexpr uint32_t INC_MID = 8u, INC_PHAZ = 16u;
// Forwarding flags of a fast-path op relative to the entry before it (used
// only inside a fast run, where that entry is the previous instruction):
// INC_FWD_A/B/C, operand a / b / c is the previous entry's destination;
// INC_FWD_T, one of its scoreboard terms is that destination's ready word.
constexpr uint32_t INC_FWD_A = 1u << 9, INC_FWD_B = 1u << 10, INC_FWD_C = 1u << 11, INC_FWD_T = 1u << 12;
// INC_OWN_D: this fast op and every op after it in its run write a row they
// also read (d is a, b or c), so the destination's ready time is already one
// of the op's scoreboard terms (the PAIR fast loop then skips its load)
constexpr uint32_t INC_OWN_D = 1u << 13;
// the fields of a PAIR fast op's hc word (DevInsn::x[4])
constexpr uint32_t KEEP_COUNT = 0xFFFFu, KEEP_FPU = 1u << 31;
constexpr uint32_t OP_EXIT = 0xFE;  // sentinel at index n_insn: the remaining lanes finish
// Unified datapaths selected at resolve time (DevInsn::op only):
//   DOP_FPU:  d = fma.rn(a, b, c ^ aux)      add: b = 1.0, c = y;  sub: b = 1.0, c = y, aux = sign bit;
//                                            mul: c = -0.0;        fma: as is
//   DOP_IMAD: d = a * b + ((c ^ aux) - aux)  add: b = 1, c = y;    sub: aux = ~0;  mul: c = 0;
//                                            mad: as is;           mov: b = 1, c = 0
// Unguarded forms run in the interpreter's fast path; guarded ones add DOP_GUARDED.
constexpr uint32_t DOP_FPU = 0x40;
constexpr uint32_t DOP_IMAD = 0x41;
constexpr uint32_t DOP_GUARDED = 0x02;
// Unguarded mul.lo / mad.lo of a register by an immediate, in kernels with
// many constants (the immediates stay out of the constant rows; mid loop):
//   DOP_MADI:  d = a * aux + c             DOP_MADII: d = a * aux + hc
constexpr uint32_t DOP_MADI = 0x44;
constexpr uint32_t DOP_MADII = 0x45;

struct DevLayout {
  uint32_t split;      // 0: PAIR layout, 1: SPLIT layout
  uint32_t row_bytes;  // ROW_PAIR or ROW_SPLIT
  uint32_t n_slots, n_crows;
  uint32_t const_off, zero_off, pred_off, stack_off, region_bytes;
  // SPLIT: the ready table (one word per row, then the 32 predicates, which
  // start at pred_off), zeroed per warp
  uint32_t ready_off, n_ready;
  uint32_t pred_entry(uint32_t p) const { return pred_off + p * 4u; }
  // SPLIT: the ready word of the row at region offset `row`
  uint32_t ready_of(uint32_t row) const { return ready_off + row / row_bytes * 4u; }
  // rows: register, constant and zero rows of a region
  uint32_t n_rows() const { return zero_off / row_bytes + 1u; }
};

struct KsParam {
  std::string name;
  uint32_t offset, size;
};

struct KsEvent {
  std::string name;
  uint32_t kind;           // 0 mark, 1 range_start, 2 range_end
  uint32_t payload_bytes;  // 0, 4 or 8
};

struct KsKernel {
  std::string name;
  std::vector<KsParam> params;
  uint32_t param_bytes = 0;
  std::vector<KsEvent> events;
  std::vector<KsInsn> code;
  std::vector<uint64_t> cpool;
  uint32_t n_slots = 0;
  uint32_t n_preds = 0;
  std::vector<int32_t> ipdom;
  uint32_t shared_bytes = 0;  // simulated shared memory per CTA (.shared arrays)
  uint32_t record_bytes = 4;  // trace record size: 4, 8 (4-byte payloads) or 16 (8-byte payloads)
  bool has_bar = false;       // uses bar.sync
  // a CTA's warps share state: they run together, one real CTA per simulated CTA
  bool cta_mode() const { return shared_bytes > 0 || has_bar; }
  // Program images, [0] PAIR layout, [1] SPLIT layout:
  // [DevInsn x (n_insn + 1) | constant row values (u32 each), padded to 16]
  std::vector<uint8_t> image[2];
  DevLayout layout[2]{};
  uint32_t prog_bytes = 0;  // DevInsn part of an image
  uint32_t live_in[4]{};    // bit s: slot s may be read before it is written (starts at 0)
};

// The layout a launch of `k` runs in: forced by KS_FLAG_LAYOUT_PAIR /
// KS_FLAG_LAYOUT_SPLIT in ks_config.flags, else SPLIT for a kernel outside
// CTA mode whose PAIR warp region exceeds SPLIT_REGION_MIN bytes (its regions
// would bound the resident warps below what the registers allow), else PAIR.
// Returns 0 / 1, or a negative KS_ERR_* (both flags; SPLIT forced on a CTA-mode
// kernel, which runs in the PAIR layout only).
constexpr uint32_t SPLIT_REGION_MIN = 12u * 1024u;
int pick_layout(const KsKernel& k, uint32_t flags);

// Bytes of one warp's trace slot: align8(16-byte header + records).
inline uint64_t trace_slot_bytes(const KsKernel& k, const ks_config& cfg) {
  return (16ull + (uint64_t)k.record_bytes * cfg.max_ts_per_warp + 7ull) / 8ull * 8ull;
}
// The argument checks every simulation call makes (ks_simulate and the
// static, cached and SM-model calls, ks_capi.cpp): KS_OK with the layout the
// launch runs in (*lay), or the KS_ERR_* code of the first failed check.
int check_call(const KsKernel& k, uint32_t grid, uint32_t block, const void* params, size_t param_bytes,
               const ks_buffer* bufs, uint32_t n_bufs, const void* trace_buf, size_t trace_bytes,
               const void* stats_buf, size_t stats_bytes, const ks_config& cfg, int* lay);
struct KsLaunch;
// The launch block of a checked call whose program image of layout `lay`
// is at `image` (device memory).
void fill_launch(const KsKernel& k, int lay, const void* image, uint32_t grid, uint32_t block, const void* params,
                 size_t param_bytes, const ks_buffer* bufs, uint32_t n_bufs, void* trace_buf, void* stats_buf,
                 const ks_config& cfg, KsLaunch* L);

// Decoder entry point (ks_decode.cpp). Returns KS_OK or a KS_ERR_* code and
// fills `err` with a message.
int decode_module(const char* text, size_t len, std::vector<KsKernel>* out, std::string* err);

struct KsBufDev {
  uint64_t sim_base;
  uint64_t bytes;
  uint8_t* ptr;
};

// Everything one interpreter launch needs (752 bytes), passed by value in the
// kernel argument (KsGrid).
struct KsLaunch {
  const uint8_t* image;  // device: DevInsn program then constant row values
  uint32_t image_bytes;  // multiple of 16
  uint32_t prog_bytes;   // DevInsn part
  uint32_t n_insn;
  uint32_t n_slots;
  uint32_t n_crows;
  DevLayout layout;
  uint32_t grid, block, wpc;  // simulated grid, block, warps per simulated CTA
  uint32_t shared_bytes;      // simulated shared memory per CTA
  uint32_t cta_mode;          // 1: one real CTA per simulated CTA, one real warp per simulated warp
  uint32_t fast_shift;        // 2^fast_shift > the largest fast-path (ALU, FMA) latency
  uint32_t n_warps;           // grid * wpc
  uint32_t live_in[4];        // KsKernel::live_in
  uint32_t lat[KS_NUM_LAT_CLASSES];
  uint32_t max_ts;
  uint32_t rec_bytes;  // trace record size (4, 8 or 16)
  uint32_t stack_depth;
  uint64_t step_limit;
  int64_t inject_warp;
  uint64_t inject_step;
  uint32_t n_bufs;
  uint32_t param_bytes;
  KsBufDev bufs[KS_MAX_BUFFERS];
  uint8_t* trace;  // may be null
  uint64_t slot_bytes;
  uint8_t* stats;
  // L1/L2 hit model (ks_simulate_cached): 0 off; 1 first pass (stores
  // suppressed, accesses logged); 2 second pass (levels from the log); 3 the
  // one interpretation of the timing-replay form (stores land, accesses and
  // issued runs logged; cache_replay_kernel then retimes every warp)
  uint32_t cache_pass;
  uint32_t cache_cap;             // log records per warp
  uint32_t lat_l1, lat_l2;        // load latency on an L1 / L2 hit
  ks_cache_warp* cache_warps;     // [n_warps]
  ks_cache_access* cache_log;     // [n_warps * cache_cap]
  ks_pc_profile* profile;         // per-instruction profile, or null
  // SM issue model: each warp's issued program-entry runs, u32 (first entry
  // << 16 | length - 1), sched_cap per warp; their number per warp
  uint32_t* sched_log;
  uint32_t* sched_runs;
  uint32_t sched_cap;
  // CTA mode with the warps' state in global memory (LaunchShape::greg): the
  // regions of real CTA c at greg + c * wpc * region_bytes (set by launch_interp)
  uint8_t* greg;
  alignas(16) uint8_t params[KS_MAX_PARAM_BYTES];
};

// The kernel argument: up to NB launches interpreted by one real grid, real
// CTAs [cta_begin[i], cta_begin[i + 1]) running item[i] (ks_simulate_batch).
// Single launches use NB = 1 (one item, every CTA), batches NB =
// KS_BATCH_ITEMS (about 23 KB, under the 32 KB kernel-argument limit).
constexpr uint32_t KS_BATCH_ITEMS = 32;
template <uint32_t NB>
struct KsGrid {
  uint32_t n;
  uint32_t cta_begin[NB + 1];
  KsLaunch item[NB];
};
static_assert(sizeof(KsGrid<KS_BATCH_ITEMS>) <= 32764, "kernel argument too large");

// Shared-memory footprint of one real CTA of `warps` warps (plus the
// simulated shared memory of a CTA-mode launch).
size_t interp_smem_bytes(uint32_t image_bytes, uint32_t region_bytes, uint32_t warps, uint32_t shared_bytes);
// Offset of the first warp region in shared memory.
uint32_t interp_region0(uint32_t image_bytes);

// Kernel lookup by name in a module (ks_capi.cpp); nullptr if absent.
const KsKernel* module_kernel(const ks_module* mod, const char* name);

// Launchers (ks_interp.cu). Return a cudaError_t value.
// Real launch shape: real warps per CTA and real CTAs (persistent). A
// CTA-mode launch (L.cta_mode) takes one real warp per simulated warp of a
// CTA; otherwise 1..12 real warps per CTA over all simulated warps. KS_OK,
// KS_ERR_LIMIT (no shape fits the shared memory) or KS_ERR_CUDA.
// The real launch of one simulation: CTAs of warps_per_cta real warps, and
// whether the register-capped form runs it.
struct LaunchShape {
  uint32_t warps_per_cta;
  uint32_t ctas;
  bool reg_capped;
  // CTA mode whose warp regions do not fit the SM's shared memory with the
  // simulated shared memory: the regions go to global memory, a scratch of
  // ctas * wpc * region_bytes that launch_interp takes from the stream-ordered
  // allocator for the launch
  bool greg;
};
int choose_launch(const KsLaunch& L, int sms, int max_smem, LaunchShape* shape);
int launch_interp(const KsLaunch& L, const LaunchShape& shape, void* stream);
int interp_occupancy(const KsLaunch& L, uint32_t real_warps_per_cta, size_t smem, int* ctas_per_sm,
                     bool reg_capped = false, bool greg = false);
// Shared memory of a CTA-mode launch with every warp region in it; above the
// device limit the launch runs with its regions in global memory.
size_t cta_mode_smem(const KsLaunch& L);
// SPLIT-layout instantiations (ks_interp_split.cu; plain mode only): the
// single-launch kernel of a form (0 lean, 1 instrumented, 2 issue-logging),
// register-capped or not, and the batch kernel of a form.
const void* interp_fn_split(int form, bool reg_capped);
const void* batch_fn_split(int form);
// CTA mode with the warps' state in global memory (ks_interp_greg.cu): the
// 1024-thread single-launch kernel of a form.
const void* interp_fn_greg(int form);
// Instantiation form of a launch: 0 lean, 1 instrumented (cache model or
// profile), 2 instrumented with the issue-run log (SM model).
int interp_form(const KsLaunch& L);
// One real grid over G->n launches of one instantiation (the same mode and
// form; in CTA mode the same simulated block): picks the shape, shares the
// real CTAs out (G->cta_begin) and launches (ks_batch.cu). KS_OK, KS_ERR_ARG
// (mixed items), KS_ERR_LIMIT (shared memory), KS_ERR_CUDA.
int launch_batch(KsGrid<KS_BATCH_ITEMS>* G, int sms, int max_smem, void* stream);

// Workspace of the L1/L2 hit model (ks_cache.cu): per-warp counts, the log,
// and the sort's buffers, each at a 256-byte boundary.
struct CacheLayout {
  uint64_t warps_off, log_off, logged_off, offsets_off, keys_a, keys_b, vals_a, vals_b, temp_off, temp_bytes;
  uint64_t runs_off, runlog_off;  // timing replay (max_runs > 0): run counts, runs
  uint64_t total;
};
// KS_OK, KS_ERR_ARG (a log of 2^31 records or more) or KS_ERR_CUDA (the
// sort's scratch size could not be queried: it needs a current CUDA device).
int cache_layout(uint64_t n_warps, uint32_t cap, uint32_t max_runs, CacheLayout* out);
// The timing replay of the hit model (ks_cache_replay.cu): after the
// logging interpretation (cache_pass 3) and the levels, every warp's timing
// again from its logged runs and its accesses' levels -- the cycles of its
// stats record and trace header, its trace timestamps and hit counts.
// Returns a cudaError_t value.
int launch_cache_replay(const KsLaunch& L, int sms, int max_smem, void* stream);
// The hit computation between the two passes: the logged records packed,
// sorted by (L1 set, step, warp), L1 hits, a stable sort of the misses by
// their L2 set, L2 hits. Waits for the stream once (the sorts' length is the
// number of logged records). Returns a cudaError_t value; adds the kernels of
// its own that it launched to *own_kernels (if not null).
int launch_cache_levels(const KsLaunch& L, uint8_t* workspace, const CacheLayout& C, uint32_t l1_lines,
                        uint32_t l2_lines, void* stream, uint32_t* own_kernels = nullptr);

// SM issue model replay (ks_sched.cu): shared memory of one simulated SM's
// replay, and the launch (one 32-thread block per simulated SM). Returns a
// cudaError_t value.
size_t sched_smem_bytes(uint32_t n_insn, uint32_t n_rows);
int launch_sched(const KsLaunch& L, uint32_t n_rows, uint32_t n_sm, uint32_t ctas_per_sm, uint32_t schedulers,
                 ks_sched_warp* warps_out, ks_sched_sm* sms_out, void* stream);
int launch_reduce_stats(const void* stats, uint64_t n_warps, void* acc_dev, void* stream);

}  // namespace ks

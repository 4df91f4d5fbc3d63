// ks_interp.cu — the sm_103a warp-level SIMT interpreter and its launchers.
//
// One real warp interprets one simulated warp at a time, one real lane per
// simulated lane (KernelScope backend doc, simulator/models.py: a warp is 32
// threads executing in lockstep under an active mask). Real warps are
// persistent: warp j of the launch takes simulated warps j, j + R, j + 2R...
// (R real warps in the grid), so the real launch shape is chosen for the GPU
// while the simulated grid and block only change what %tid/%ctaid read.
//
// Per real CTA, shared memory holds
//   [program image | mbarrier | parameter block | latency table]
//   [register file: slot-major, one 32-bit word per real thread per slot]
//   [per warp: 128-entry ready-time table | 32-entry reconvergence stack].
// The program image (decoded instructions + constant pool) is staged once per
// CTA with one cp.async.bulk global->shared copy completing on an mbarrier;
// the wait is bounded and reports KS_ST_TIMEOUT instead of hanging.
//
// Warp-uniform state (pc, active mask, scoreboard clock, counters) lives in
// registers, identical in every lane; values every lane must agree on (ready
// times, stack entries) are written by all lanes with the same value, so each
// lane only ever reads back its own store. Predicates are per-warp ballot
// masks, predicate p held by lane p and read with a shuffle.
#include <cuda_runtime.h>

#include <cstdint>

#include "ks_internal.h"

namespace ks {

namespace {

constexpr uint32_t FULL = 0xFFFFFFFFu;
constexpr uint32_t HDR_BYTES = 384;  // mbarrier 16 + params 256 + latency table 32, padded
constexpr uint32_t HDR_PARAMS = 16;
constexpr uint32_t HDR_LAT = 16 + KS_MAX_PARAM_BYTES;
constexpr uint32_t STACK_ENTRIES = KS_MAX_STACK;
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

__device__ __forceinline__ uint64_t umax64(uint64_t a, uint64_t b) { return a > b ? a : b; }

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

__device__ __forceinline__ bool cmp_u(uint64_t a, uint64_t b, uint32_t c) {
  switch (c) {
    case CMP_EQ: return a == b;
    case CMP_NE: return a != b;
    case CMP_LT: return a < b;
    case CMP_LE: return a <= b;
    case CMP_GT: return a > b;
    default: return a >= b;
  }
}

__device__ __forceinline__ bool cmp_s(int64_t a, int64_t b, uint32_t c) {
  switch (c) {
    case CMP_EQ: return a == b;
    case CMP_NE: return a != b;
    case CMP_LT: return a < b;
    case CMP_LE: return a <= b;
    case CMP_GT: return a > b;
    default: return a >= b;
  }
}

__device__ __forceinline__ bool cmp_f(float a, float b, uint32_t c) {
  if (a != a || b != b) return false;  // ordered comparisons
  switch (c) {
    case CMP_EQ: return a == b;
    case CMP_NE: return a != b;
    case CMP_LT: return a < b;
    case CMP_LE: return a <= b;
    case CMP_GT: return a > b;
    default: return a >= b;
  }
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

__device__ __forceinline__ uint64_t pack_entry(uint32_t pc, uint32_t rpc, uint32_t mask) {
  return (uint64_t)(pc & 0xFFFFu) | ((uint64_t)(rpc & 0xFFFFu) << 16) | ((uint64_t)mask << 32);
}

}  // namespace

__global__ void __launch_bounds__(256) ks_interp_kernel(const __grid_constant__ KsLaunch L) {
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t lane = threadIdx.x & 31u;
  const uint32_t wid = threadIdx.x >> 5;
  const uint32_t nwarps = blockDim.x >> 5;
  const uint32_t stride = blockDim.x;  // register-file slot stride (words)

  uint8_t* s_image = smem;
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(smem + L.image_bytes);
  uint8_t* s_params = smem + L.image_bytes + HDR_PARAMS;
  uint32_t* s_lat = reinterpret_cast<uint32_t*>(smem + L.image_bytes + HDR_LAT);
  uint32_t* s_rf = reinterpret_cast<uint32_t*>(smem + L.image_bytes + HDR_BYTES);
  uint64_t* s_ready = reinterpret_cast<uint64_t*>(s_rf + (size_t)L.n_slots * stride);
  uint64_t* s_stack = s_ready + (size_t)nwarps * KS_HZ_ENTRIES;

  // ---- stage the program once per CTA (a1) ----
  if (threadIdx.x == 0) {
    mbar_init(s_bar, 1);
    mbar_init_fence();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(s_bar, L.image_bytes);
    bulk_copy_g2s(s_image, L.image, L.image_bytes, s_bar);
  }
  for (uint32_t i = threadIdx.x; i < KS_MAX_PARAM_BYTES / 4; i += blockDim.x)
    reinterpret_cast<uint32_t*>(s_params)[i] = reinterpret_cast<const uint32_t*>(L.params)[i];
  if (threadIdx.x < KS_NUM_LAT_CLASSES) s_lat[threadIdx.x] = L.lat[threadIdx.x];
  const bool staged = __all_sync(FULL, wait_staged(s_bar));
  __syncthreads();

  const KsInsn* prog = reinterpret_cast<const KsInsn*>(s_image);
  const uint64_t* cpool = reinterpret_cast<const uint64_t*>(s_image + (size_t)L.n_insn * sizeof(KsInsn));
  uint32_t* rf = s_rf + threadIdx.x;
  uint64_t* ready = s_ready + (size_t)wid * KS_HZ_ENTRIES;
  uint64_t* stk = s_stack + (size_t)wid * STACK_ENTRIES;
  const uint32_t exit_pc = L.n_insn;

#define RD32(o) (((o) & KS_CONST_BIT) ? (uint32_t)cpool[(o) & 0x7Fu] : rf[(uint32_t)(o) * stride])
#define RD64(o)                                                   \
  (((o) & KS_CONST_BIT) ? cpool[(o) & 0x7Fu]                      \
                        : ((uint64_t)rf[(uint32_t)(o) * stride] | \
                           ((uint64_t)rf[((uint32_t)(o) + 1u) * stride] << 32)))
#define WR32(o, v) (rf[(uint32_t)(o) * stride] = (v))
#define WR64(o, v)                                         \
  do {                                                     \
    const uint64_t v_ = (v);                               \
    rf[(uint32_t)(o) * stride] = (uint32_t)v_;             \
    rf[((uint32_t)(o) + 1u) * stride] = (uint32_t)(v_ >> 32); \
  } while (0)

  for (uint32_t gw = blockIdx.x * nwarps + wid; gw < L.n_warps; gw += gridDim.x * nwarps) {
    const uint32_t cta = gw / L.wpc;
    const uint32_t wic = gw - cta * L.wpc;
    const uint32_t tid_sim = wic * 32u + lane;

    // ---- warp set-up (a1): registers zero, predicates false, clock 0 ----
    for (uint32_t s = 0; s < L.n_slots; s++) rf[s * stride] = 0u;
    for (uint32_t i = lane; i < KS_HZ_ENTRIES; i += 32) ready[i] = 0ull;
    uint32_t my_pred = 0;
    uint32_t pc = 0, rpc = exit_pc;
    uint32_t mask = __ballot_sync(FULL, tid_sim < L.block);
    uint32_t depth = 1, max_depth = 1;
    uint64_t t_next = 0, t_last = 0, max_ready = 0, drain = 0;
    uint64_t warp_insts = 0, thread_insts = 0;
    uint64_t ld_req = 0, ld_sec = 0, st_req = 0, st_sec = 0, ld_lin = 0, st_lin = 0;
    uint32_t n_events = 0, n_rec = 0, n_dropped = 0;
    int status = staged ? 0 : KS_ST_TIMEOUT;
    uint8_t* slot = L.trace ? L.trace + (uint64_t)gw * L.slot_bytes : nullptr;

    while (status == 0) {
      // pop finished entries (a6)
      if (pc == rpc || mask == 0) {
        if (depth == 1) break;
        depth--;
        const uint64_t e = stk[depth - 1];
        pc = (uint32_t)(e & 0xFFFFu);
        rpc = (uint32_t)((e >> 16) & 0xFFFFu);
        mask = (uint32_t)(e >> 32);
        continue;
      }
      if (pc >= exit_pc) {  // reached the virtual exit: the remaining lanes finish
        mask = 0;
        continue;
      }
      // fetch (a2)
      const uint4 w0 = reinterpret_cast<const uint4*>(prog + pc)[0];
      const uint4 w1 = reinterpret_cast<const uint4*>(prog + pc)[1];
      const uint32_t op = w0.x & 0xFFu;
      if (op == OP_EVENT) {  // trace record (a7), zero cost
        const uint32_t ev = w0.w >> 16;
        if (n_events != 0xFFFFFFFFu) n_events++;
        if (n_rec < L.max_ts) {
          if (slot && lane == 0)
            *reinterpret_cast<uint32_t*>(slot + 16 + 4 * n_rec) =
                ((ev & 0xFFu) << 24) | (uint32_t)(t_next & 0xFFFFFFull);
          n_rec++;
        } else if (n_dropped < 0xFFFFu) {
          n_dropped++;
        }
        pc++;
        continue;
      }
      if (L.inject_warp >= 0 && (uint64_t)L.inject_warp == gw && warp_insts == L.inject_step) {
        status = KS_ST_INJECTED;
        break;
      }
      if (warp_insts == L.step_limit) {
        status = KS_ST_STEP_LIMIT;
        break;
      }
      const uint32_t latc = (w0.x >> 8) & 0xFFu;
      const uint32_t guard = (w0.x >> 16) & 0xFFu;
      const uint32_t gneg = w0.x >> 24;
      const uint32_t d = w0.y & 0xFFu, a = (w0.y >> 8) & 0xFFu, b = (w0.y >> 16) & 0xFFu, c = w0.y >> 24;
      const uint32_t hd = w0.z & 0xFFu;
      const uint32_t flags = (w0.w >> 8) & 0xFFu;
      const uint64_t imm = (uint64_t)w1.x | ((uint64_t)w1.y << 32);

      // issue: in-order scoreboard (a3)
      uint64_t t = t_next;
      t = umax64(t, ready[(w0.z >> 8) & 0xFFu]);
      t = umax64(t, ready[(w0.z >> 16) & 0xFFu]);
      t = umax64(t, ready[w0.z >> 24]);
      t = umax64(t, ready[w0.w & 0xFFu]);
      t = umax64(t, ready[hd]);
      const uint64_t lat = s_lat[latc];
      if (hd != KS_HZ_NONE) {
        ready[hd] = t + lat;
        max_ready = umax64(max_ready, t + lat);
      }
      if (op == OP_STG32 || op == OP_STG64) drain = umax64(drain, t + lat);
      t_last = t;
      t_next = (op == OP_BRA || op == OP_RET) ? t + lat : t + 1;
      warp_insts++;
      thread_insts += (uint64_t)__popc(mask);

      // guard (a2)
      uint32_t exec = mask;
      if (guard != KS_NO_GUARD) {
        const uint32_t pm = __shfl_sync(FULL, my_pred, guard);
        exec &= gneg ? ~pm : pm;
      }
      const bool on = (exec >> lane) & 1u;

      switch (op) {
        // ---- control (a6) ----
        case OP_BRA: {
          const uint32_t target = w1.z, R = w1.w;
          const uint32_t taken = exec, fall = mask & ~exec;
          if (fall == 0) {
            pc = target;
          } else if (taken == 0) {
            pc = pc + 1;
          } else {
            uint32_t n = depth;  // entries after the top is resolved, all in shared memory
            if (rpc == R) {
              n = depth - 1;  // the top already waits at R below: replace it
            } else {
              stk[depth - 1] = pack_entry(R, rpc, mask);
            }
            if (target != R) {
              if (n >= L.stack_depth) { status = KS_ST_SIMT_STACK; break; }
              stk[n++] = pack_entry(target, R, taken);
            }
            if (pc + 1 != R) {
              if (n >= L.stack_depth) { status = KS_ST_SIMT_STACK; break; }
              stk[n++] = pack_entry(pc + 1, R, fall);
            }
            if (n == 0) { depth = 1; pc = rpc = exit_pc; mask = 0; break; }
            depth = n;
            max_depth = max(max_depth, depth);
            const uint64_t e = stk[depth - 1];
            pc = (uint32_t)(e & 0xFFFFu);
            rpc = (uint32_t)((e >> 16) & 0xFFFFu);
            mask = (uint32_t)(e >> 32);
          }
          break;
        }
        case OP_RET: {
          for (uint32_t i = 0; i + 1 < depth; i++) stk[i] &= ~((uint64_t)exec << 32);
          mask &= ~exec;
          pc++;
          break;
        }
        // ---- memory (a5) ----
        case OP_LDP32: {
          const uint32_t v = *reinterpret_cast<const uint32_t*>(s_params + imm);
          if (on) WR32(d, v);
          pc++;
          break;
        }
        case OP_LDP64: {
          const uint64_t v = *reinterpret_cast<const uint64_t*>(s_params + imm);
          if (on) WR64(d, v);
          pc++;
          break;
        }
        case OP_LDG32: case OP_LDG64: case OP_STG32: case OP_STG64: {
          const bool wide = (op == OP_LDG64 || op == OP_STG64);
          const bool is_ld = (op == OP_LDG32 || op == OP_LDG64);
          const uint32_t size = wide ? 8u : 4u;
          const uint64_t va = RD64(a) + imm;
          uint8_t* ptr = nullptr;
          int err = 0;
          if (on) err = translate(L, va, size, &ptr);
          const uint32_t emask = __ballot_sync(FULL, err != 0);
          if (emask) {
            status = __shfl_sync(FULL, err, __ffs(emask) - 1);
            break;
          }
          if (exec) {
            const uint32_t ms = __match_any_sync(FULL, on ? (va >> 5) : ~0ull);
            const uint32_t sectors = __popc(__ballot_sync(FULL, on && (uint32_t)(__ffs(ms) - 1) == lane));
            const uint32_t ml = __match_any_sync(FULL, on ? (va >> 7) : ~0ull);
            const uint32_t lines = __popc(__ballot_sync(FULL, on && (uint32_t)(__ffs(ml) - 1) == lane));
            if (is_ld) { ld_req++; ld_sec += sectors; ld_lin += lines; }
            else { st_req++; st_sec += sectors; st_lin += lines; }
          }
          if (is_ld) {
            if (on) {
              if (wide) WR64(d, *reinterpret_cast<const uint64_t*>(ptr));
              else WR32(d, *reinterpret_cast<const uint32_t*>(ptr));
            }
          } else {
            // the highest lane writing an address wins
            const uint32_t mv = __match_any_sync(FULL, on ? va : ~0ull);
            if (on && (31u - __clz(mv)) == lane) {
              if (wide) *reinterpret_cast<uint64_t*>(ptr) = RD64(b);
              else *reinterpret_cast<uint32_t*>(ptr) = RD32(b);
            }
          }
          pc++;
          break;
        }
        // ---- moves and integer ALU (a4) ----
        case OP_MOV32: { const uint32_t v = RD32(a); if (on) WR32(d, v); pc++; break; }
        case OP_MOV64: { const uint64_t v = RD64(a); if (on) WR64(d, v); pc++; break; }
        case OP_MOVSP: {
          uint32_t v;
          switch ((uint32_t)imm) {
            case SP_TID: v = tid_sim; break;
            case SP_NTID: v = L.block; break;
            case SP_CTAID: v = cta; break;
            case SP_NCTAID: v = L.grid; break;
            case SP_LANEID: v = lane; break;
            case SP_ONE: v = 1; break;
            default: v = 0; break;
          }
          if (on) WR32(d, v);
          pc++;
          break;
        }
        case OP_ADD32: { const uint32_t v = RD32(a) + RD32(b); if (on) WR32(d, v); pc++; break; }
        case OP_SUB32: { const uint32_t v = RD32(a) - RD32(b); if (on) WR32(d, v); pc++; break; }
        case OP_MUL32: { const uint32_t v = RD32(a) * RD32(b); if (on) WR32(d, v); pc++; break; }
        case OP_MAD32: { const uint32_t v = RD32(a) * RD32(b) + RD32(c); if (on) WR32(d, v); pc++; break; }
        case OP_ADD64: { const uint64_t v = RD64(a) + RD64(b); if (on) WR64(d, v); pc++; break; }
        case OP_SUB64: { const uint64_t v = RD64(a) - RD64(b); if (on) WR64(d, v); pc++; break; }
        case OP_MUL64: { const uint64_t v = RD64(a) * RD64(b); if (on) WR64(d, v); pc++; break; }
        case OP_MAD64: { const uint64_t v = RD64(a) * RD64(b) + RD64(c); if (on) WR64(d, v); pc++; break; }
        case OP_AND32: { const uint32_t v = RD32(a) & RD32(b); if (on) WR32(d, v); pc++; break; }
        case OP_OR32: { const uint32_t v = RD32(a) | RD32(b); if (on) WR32(d, v); pc++; break; }
        case OP_XOR32: { const uint32_t v = RD32(a) ^ RD32(b); if (on) WR32(d, v); pc++; break; }
        case OP_AND64: { const uint64_t v = RD64(a) & RD64(b); if (on) WR64(d, v); pc++; break; }
        case OP_OR64: { const uint64_t v = RD64(a) | RD64(b); if (on) WR64(d, v); pc++; break; }
        case OP_XOR64: { const uint64_t v = RD64(a) ^ RD64(b); if (on) WR64(d, v); pc++; break; }
        case OP_SHL32: { const uint32_t s = RD32(b); const uint32_t v = s >= 32u ? 0u : RD32(a) << s; if (on) WR32(d, v); pc++; break; }
        case OP_SHR32U: { const uint32_t s = RD32(b); const uint32_t v = s >= 32u ? 0u : RD32(a) >> s; if (on) WR32(d, v); pc++; break; }
        case OP_SHR32S: {
          const uint32_t s = RD32(b);
          const int32_t x = (int32_t)RD32(a);
          const uint32_t v = (uint32_t)(s >= 32u ? (x >> 31) : (x >> s));
          if (on) WR32(d, v);
          pc++;
          break;
        }
        case OP_SHL64: { const uint32_t s = RD32(b); const uint64_t v = s >= 64u ? 0ull : RD64(a) << s; if (on) WR64(d, v); pc++; break; }
        case OP_SHR64U: { const uint32_t s = RD32(b); const uint64_t v = s >= 64u ? 0ull : RD64(a) >> s; if (on) WR64(d, v); pc++; break; }
        case OP_SHR64S: {
          const uint32_t s = RD32(b);
          const int64_t x = (int64_t)RD64(a);
          const uint64_t v = (uint64_t)(s >= 64u ? (x >> 63) : (x >> s));
          if (on) WR64(d, v);
          pc++;
          break;
        }
        // ---- f32 (a4), IEEE round-to-nearest-even, canonical NaN ----
        case OP_FADD: { const uint32_t v = fbits(__fadd_rn(__uint_as_float(RD32(a)), __uint_as_float(RD32(b)))); if (on) WR32(d, v); pc++; break; }
        case OP_FSUB: { const uint32_t v = fbits(__fsub_rn(__uint_as_float(RD32(a)), __uint_as_float(RD32(b)))); if (on) WR32(d, v); pc++; break; }
        case OP_FMUL: { const uint32_t v = fbits(__fmul_rn(__uint_as_float(RD32(a)), __uint_as_float(RD32(b)))); if (on) WR32(d, v); pc++; break; }
        case OP_FFMA: {
          const uint32_t v = fbits(__fmaf_rn(__uint_as_float(RD32(a)), __uint_as_float(RD32(b)), __uint_as_float(RD32(c))));
          if (on) WR32(d, v);
          pc++;
          break;
        }
        case OP_FDIV: { const uint32_t v = fbits(__fdiv_rn(__uint_as_float(RD32(a)), __uint_as_float(RD32(b)))); if (on) WR32(d, v); pc++; break; }
        case OP_FSQRT: { const uint32_t v = fbits(__fsqrt_rn(__uint_as_float(RD32(a)))); if (on) WR32(d, v); pc++; break; }
        // ---- predicates ----
        case OP_SETP_U32: case OP_SETP_S32: case OP_SETP_U64: case OP_SETP_S64: case OP_SETP_F32: {
          bool r;
          if (op == OP_SETP_U32) r = cmp_u(RD32(a), RD32(b), flags);
          else if (op == OP_SETP_S32) r = cmp_s((int32_t)RD32(a), (int32_t)RD32(b), flags);
          else if (op == OP_SETP_U64) r = cmp_u(RD64(a), RD64(b), flags);
          else if (op == OP_SETP_S64) r = cmp_s((int64_t)RD64(a), (int64_t)RD64(b), flags);
          else r = cmp_f(__uint_as_float(RD32(a)), __uint_as_float(RD32(b)), flags);
          const uint32_t bal = __ballot_sync(FULL, r);
          const uint32_t old = __shfl_sync(FULL, my_pred, d);
          if (lane == d) my_pred = (old & ~exec) | (bal & exec);
          pc++;
          break;
        }
        case OP_ANDP: case OP_ORP: case OP_XORP: {
          const uint32_t pa = __shfl_sync(FULL, my_pred, a);
          const uint32_t pb = __shfl_sync(FULL, my_pred, b);
          const uint32_t old = __shfl_sync(FULL, my_pred, d);
          const uint32_t r = op == OP_ANDP ? (pa & pb) : op == OP_ORP ? (pa | pb) : (pa ^ pb);
          if (lane == d) my_pred = (old & ~exec) | (r & exec);
          pc++;
          break;
        }
        case OP_SELP32: {
          const uint32_t pm = __shfl_sync(FULL, my_pred, c);
          const uint32_t v = ((pm >> lane) & 1u) ? RD32(a) : RD32(b);
          if (on) WR32(d, v);
          pc++;
          break;
        }
        case OP_SELP64: {
          const uint32_t pm = __shfl_sync(FULL, my_pred, c);
          const uint64_t v = ((pm >> lane) & 1u) ? RD64(a) : RD64(b);
          if (on) WR64(d, v);
          pc++;
          break;
        }
        // ---- conversions ----
        case OP_CVT_F32_U32: { const uint32_t v = __float_as_uint(__uint2float_rn(RD32(a))); if (on) WR32(d, v); pc++; break; }
        case OP_CVT_F32_S32: { const uint32_t v = __float_as_uint(__int2float_rn((int32_t)RD32(a))); if (on) WR32(d, v); pc++; break; }
        case OP_CVT_F32_U64: { const uint32_t v = __float_as_uint(__ull2float_rn(RD64(a))); if (on) WR32(d, v); pc++; break; }
        case OP_CVT_F32_S64: { const uint32_t v = __float_as_uint(__ll2float_rn((long long)RD64(a))); if (on) WR32(d, v); pc++; break; }
        case OP_CVT_F2I: {
          const uint64_t v = f2i(__uint_as_float(RD32(a)), flags);
          const uint32_t kind = flags & 15u;
          if (on) {
            if (kind == CVT_S64 || kind == CVT_U64) WR64(d, v);
            else WR32(d, (uint32_t)v);
          }
          pc++;
          break;
        }
        case OP_CVT_ZX: { const uint64_t v = (uint64_t)RD32(a); if (on) WR64(d, v); pc++; break; }
        case OP_CVT_SX: { const uint64_t v = (uint64_t)(int64_t)(int32_t)RD32(a); if (on) WR64(d, v); pc++; break; }
        default:
          pc++;
          break;
      }
    }

    // ---- write-back (a9) ----
    const uint64_t cycles = warp_insts ? umax64(umax64(t_last + 1, max_ready), drain) : 0ull;
    {
      uint64_t v = 0;
      switch (lane) {
        case 0: v = cycles; break;
        case 1: v = warp_insts; break;
        case 2: v = thread_insts; break;
        case 3: v = ld_req; break;
        case 4: v = ld_sec; break;
        case 5: v = st_req; break;
        case 6: v = st_sec; break;
        case 7: v = ld_lin; break;
        case 8: v = st_lin; break;
        case 9: v = (uint64_t)(uint32_t)status | ((uint64_t)max_depth << 32); break;
        default: v = 0; break;
      }
      if (lane < 12) reinterpret_cast<uint64_t*>(L.stats + (uint64_t)gw * sizeof(ks_warp_stats))[lane] = v;
    }
    if (slot) {
      uint32_t* sw = reinterpret_cast<uint32_t*>(slot);
      const uint32_t words = (uint32_t)(L.slot_bytes / 4);
      if (lane == 0) {
        sw[0] = n_events;
        sw[1] = 1u | (4u << 8) | (n_dropped << 16);
        sw[2] = (uint32_t)cycles;
        sw[3] = (uint32_t)(cycles >> 32);
      }
      for (uint32_t i = 4 + n_rec + lane; i < words; i += 32) sw[i] = 0u;
    }
  }
#undef RD32
#undef RD64
#undef WR32
#undef WR64
  // Leave no copy in flight: if staging timed out, wait once more (bounded).
  if (!staged) (void)wait_staged(s_bar);
}

// ---- launch-totals reduction -------------------------------------------------
// acc: [0] cycles max, [1] cycles sum, [2..9] counter sums, [10] failed warps,
// [11] max over failing warps of (2^64-1 - warp id), [12] max stack depth.
__global__ void ks_reduce_kernel(const ks_warp_stats* __restrict__ s, uint64_t n,
                                 unsigned long long* __restrict__ acc) {
  unsigned long long v[13] = {0};
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
    const ks_warp_stats r = s[i];
    v[0] = v[0] > r.cycles ? v[0] : r.cycles;
    v[1] += r.cycles;
    v[2] += r.warp_insts;
    v[3] += r.thread_insts;
    v[4] += r.ld_req;
    v[5] += r.ld_sectors;
    v[6] += r.st_req;
    v[7] += r.st_sectors;
    v[8] += r.ld_lines;
    v[9] += r.st_lines;
    if (r.status) {
      v[10] += 1;
      const unsigned long long inv = ~0ull - i;
      v[11] = v[11] > inv ? v[11] : inv;
    }
    v[12] = v[12] > r.max_stack_depth ? v[12] : r.max_stack_depth;
  }
#pragma unroll
  for (int k = 0; k < 13; k++) {
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long u = __shfl_down_sync(FULL, v[k], o);
      if (k == 0 || k == 11 || k == 12) v[k] = v[k] > u ? v[k] : u;
      else v[k] += u;
    }
  }
  if ((threadIdx.x & 31) == 0) {
#pragma unroll
    for (int k = 0; k < 13; k++) {
      if (k == 0 || k == 11 || k == 12) atomicMax(&acc[k], v[k]);
      else if (v[k]) atomicAdd(&acc[k], v[k]);
    }
  }
}

size_t interp_smem_bytes(uint32_t image_bytes, uint32_t n_slots, uint32_t warps) {
  return (size_t)image_bytes + HDR_BYTES + (size_t)n_slots * warps * 32 * 4 +
         (size_t)warps * (KS_HZ_ENTRIES + STACK_ENTRIES) * 8;
}

static int g_attr_done[64];

static int ensure_attr() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev < 64 && g_attr_done[dev]) return 0;
  int mx = 0;
  e = cudaDeviceGetAttribute(&mx, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return (int)e;
  e = cudaFuncSetAttribute(ks_interp_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
  if (e != cudaSuccess) return (int)e;
  if (dev < 64) g_attr_done[dev] = 1;
  return 0;
}

int interp_occupancy(uint32_t real_warps_per_cta, size_t smem, int* ctas_per_sm) {
  int e = ensure_attr();
  if (e) return e;
  return (int)cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, ks_interp_kernel,
                                                            (int)(real_warps_per_cta * 32), smem);
}

int launch_interp(const KsLaunch& L, uint32_t real_warps_per_cta, uint32_t real_ctas, void* stream) {
  int e = ensure_attr();
  if (e) return e;
  const size_t smem = interp_smem_bytes(L.image_bytes, L.n_slots, real_warps_per_cta);
  ks_interp_kernel<<<real_ctas, real_warps_per_cta * 32, smem, (cudaStream_t)stream>>>(L);
  return (int)cudaGetLastError();
}

int launch_reduce_stats(const void* stats, uint64_t n_warps, void* acc_dev, void* stream) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  uint64_t blocks = (n_warps + 255) / 256;
  const uint64_t cap = (uint64_t)(sms > 0 ? sms : 1) * 4;
  if (blocks > cap) blocks = cap;
  if (blocks == 0) blocks = 1;
  ks_reduce_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(
      reinterpret_cast<const ks_warp_stats*>(stats), n_warps, reinterpret_cast<unsigned long long*>(acc_dev));
  return (int)cudaGetLastError();
}

}  // namespace ks

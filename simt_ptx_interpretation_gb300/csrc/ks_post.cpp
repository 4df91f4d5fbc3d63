// ks_post.cpp — host post-passes of the C ABI: the occupancy calculator
// (KernelScope backend doc, occupancy/calculator.py) and the trace export.
#include <algorithm>
#include <cstring>
#include <string>

#include "ks_internal.h"

namespace {

struct NamedLimits {
  const char* name;
  ks_gpu_limits g;
};

// The page's GPU_SPECS table (max threads, max warps, max blocks, registers,
// shared memory per SM). sm_86 / sm_89 registers and shared memory and the
// sm_90 registers are elided on the page ("..."): those take the public
// CUDA values; sm_100 and sm_103 are not on the page.
const NamedLimits kLimits[] = {
    {"sm_75", {1024, 32, 16, 65536, 65536}},
    {"sm_80", {2048, 64, 32, 65536, 167936}},
    {"sm_86", {1536, 48, 16, 65536, 102400}},
    {"sm_89", {1536, 48, 24, 65536, 102400}},
    {"sm_90", {2048, 64, 32, 65536, 232448}},
    {"sm_100", {2048, 64, 32, 65536, 233472}},
    {"sm_103", {2048, 64, 32, 65536, 233472}},
};

}  // namespace

extern "C" {

int ks_gpu_limits_of(const char* arch, ks_gpu_limits* out) {
  if (!arch || !out) return KS_ERR_ARG;
  for (const NamedLimits& n : kLimits)
    if (std::strcmp(n.name, arch) == 0) {
      *out = n.g;
      return KS_OK;
    }
  return KS_ERR_NOT_FOUND;
}

int ks_occupancy(const ks_gpu_limits* g, uint32_t threads_per_block, uint32_t registers_per_thread,
                 uint32_t shared_memory_per_block, ks_occupancy_result* out) {
  if (!g || !out || g->max_warps_per_sm == 0 || threads_per_block == 0 ||
      threads_per_block > g->max_threads_per_sm)
    return KS_ERR_ARG;
  const uint64_t warps_per_block = (threads_per_block + 31u) / 32u;
  uint64_t by_regs = g->max_warps_per_sm;
  if (registers_per_thread > 0) {
    const uint64_t per_warp = ((uint64_t)registers_per_thread * 32u + 255u) / 256u * 256u;  // groups of 256
    by_regs = g->registers_per_sm / per_warp;
  }
  uint64_t by_smem = g->max_warps_per_sm;
  if (shared_memory_per_block > 0) {
    const uint64_t per_block = ((uint64_t)shared_memory_per_block + 255u) / 256u * 256u;  // 256-byte chunks
    by_smem = (g->shared_memory_per_sm / per_block) * warps_per_block;
  }
  const uint64_t blocks = std::min<uint64_t>(g->max_threads_per_sm / threads_per_block, g->max_blocks_per_sm);
  const uint64_t by_block = blocks * warps_per_block;
  const uint64_t active = std::min<uint64_t>(std::min(std::min(by_regs, by_smem), by_block), g->max_warps_per_sm);
  out->active_warps_per_sm = (uint32_t)active;
  out->max_warps_per_sm = g->max_warps_per_sm;
  out->warps_by_registers = (uint32_t)std::min<uint64_t>(by_regs, 0xFFFFFFFFu);
  out->warps_by_shared_memory = (uint32_t)std::min<uint64_t>(by_smem, 0xFFFFFFFFu);
  out->warps_by_block_size = (uint32_t)by_block;
  out->limiter = active == by_regs ? KS_LIMITER_REGISTERS
                 : active == by_smem ? KS_LIMITER_SHARED_MEMORY
                                     : KS_LIMITER_BLOCK_SIZE;
  out->occupancy_percent = (double)active / (double)g->max_warps_per_sm * 100.0;  // the page's order
  return KS_OK;
}

}  // extern "C"

// ks_post.cpp — host post-passes of the C ABI: the occupancy calculator
// (KernelScope backend doc, occupancy/calculator.py), the trace export and the
// hints (hints/analyzer.py).
#include <algorithm>
#include <charconv>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

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

void put_text(char* dst, size_t cap, const std::string& text) {
  const size_t n = std::min(text.size(), cap - 1);
  std::memcpy(dst, text.data(), n);
  dst[n] = 0;
}

// A double as Python prints it here: the shortest decimal that reads back as
// the same value, with ".0" when that has no fraction part (values 0..100).
std::string shortest(double v) {
  char buf[64];
  const auto r = std::to_chars(buf, buf + sizeof buf, v);
  std::string t(buf, r.ptr);
  if (t.find_first_of(".e") == std::string::npos) t += ".0";
  return t;
}

uint32_t highest_bit(uint64_t m) { return 63u - (uint32_t)__builtin_clzll(m); }
uint32_t lowest_bit(uint64_t m) { return (uint32_t)__builtin_ctzll(m); }

}  // namespace

extern "C" {

int ks_hints(const ks_pc_profile* profile, uint32_t n_entries, const ks_occupancy_result* occupancy,
             ks_hint* out, uint32_t cap, uint32_t* n_hints) {
  if (!n_hints || (n_entries && !profile)) return KS_ERR_ARG;
  std::vector<ks_hint> h;
  auto add = [&](int cat, int sev, int pc, uint64_t count, const std::string& msg, const std::string& detail) {
    ks_hint x;
    std::memset(&x, 0, sizeof x);
    x.category = cat;
    x.severity = sev;
    x.pc = pc;
    x.count = count;
    put_text(x.message, sizeof x.message, msg);
    put_text(x.detail, sizeof x.detail, detail);
    h.push_back(x);
  };
  uint64_t bank_events = 0, divergent_events = 0;
  for (uint32_t pc = 0; pc < n_entries; pc++) {
    const ks_pc_profile& p = profile[pc];
    bank_events += p.conflicted;
    divergent_events += p.divergent;
    if (p.severe)
      add(KS_HINT_MEMORY, KS_HINT_CRITICAL, (int)pc, p.severe, std::to_string(highest_bit(p.degrees) + 1) +
          "-way bank conflict", "Severe bank conflict causing serialized access");
    const uint32_t mild = p.degrees & 0x7Eu;  // degrees 2..7
    if (p.conflicted > p.severe && mild)
      add(KS_HINT_MEMORY, KS_HINT_WARNING, (int)pc, p.conflicted - p.severe,
          std::to_string(highest_bit(mild) + 1) + "-way bank conflict", "Bank conflict reducing throughput");
    if (p.poor && p.poor_pcts)
      add(KS_HINT_MEMORY, KS_HINT_CRITICAL, (int)pc, p.poor,
          "Poor memory efficiency (" + std::to_string(lowest_bit(p.poor_pcts)) + "%)",
          "Scattered access causing many transactions");
    if (p.high_divergence && p.high_div_pcts)
      add(KS_HINT_DIVERGENCE, KS_HINT_WARNING, (int)pc, p.high_divergence,
          "High divergence (" + std::to_string(highest_bit(p.high_div_pcts)) + "%)",
          "Significant warp divergence at this branch");
  }
  if (bank_events > 5)
    add(KS_HINT_MEMORY, KS_HINT_WARNING, -1, bank_events,
        "Shared memory bank conflicts (" + std::to_string(bank_events) + " events)",
        "Consider padding arrays or restructuring access patterns");
  if (divergent_events > 3)
    add(KS_HINT_DIVERGENCE, KS_HINT_WARNING, -1, divergent_events,
        "Branch divergence detected (" + std::to_string(divergent_events) + " events)",
        "Consider restructuring conditionals or using predication");
  if (occupancy) {
    static const char* const kNames[] = {"registers", "shared_memory", "block_size"};
    const int li = occupancy->limiter;
    const std::string lim = (li >= 0 && li < 3) ? kNames[li] : "";
    const double pct = occupancy->occupancy_percent;
    if (pct < 25)
      add(KS_HINT_OCCUPANCY, KS_HINT_CRITICAL, -1, 1, "Very low occupancy (" + shortest(pct) + "%)",
          "Limited by " + lim + ". Consider reducing resource usage.");
    else if (pct < 50)
      add(KS_HINT_OCCUPANCY, KS_HINT_WARNING, -1, 1, "Low occupancy (" + shortest(pct) + "%)",
          "Limited by " + lim + ".");
  }
  *n_hints = (uint32_t)h.size();
  if (!out || cap < h.size()) return h.empty() ? KS_OK : KS_ERR_ARG;
  std::copy(h.begin(), h.end(), out);
  return KS_OK;
}

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

int ks_trace_to_json(const ks_module* mod, const char* kernel, uint32_t grid, uint32_t block, uint32_t max_ts,
                     const void* trace_host, size_t trace_bytes, double cycles_per_us, char* out, size_t cap,
                     size_t* needed) {
  if (!mod || !kernel) return KS_ERR_ARG;
  const ks::KsKernel* k = ks::module_kernel(mod, kernel);
  if (!k) return KS_ERR_NOT_FOUND;
  if (!trace_host || !needed || grid == 0 || block == 0 || !(cycles_per_us > 0.0)) return KS_ERR_ARG;
  const uint64_t rb = k->record_bytes;
  const uint64_t slot = (16ull + rb * max_ts + 7ull) / 8ull * 8ull;
  const uint64_t wpc = (block + 31u) / 32u;
  if ((uint64_t)trace_bytes < (uint64_t)grid * wpc * slot) return KS_ERR_ARG;
  const uint8_t* t = static_cast<const uint8_t*>(trace_host);
  auto u32 = [&](uint64_t off) { uint32_t v; std::memcpy(&v, t + off, 4); return v; };
  auto u64 = [&](uint64_t off) { uint64_t v; std::memcpy(&v, t + off, 8); return v; };
  std::string js;
  js.reserve(256 + (size_t)grid * wpc * (64 + 96 * std::min<uint64_t>(max_ts, 64)));
  char num[64];
  auto dbl = [&](double v) {
    std::snprintf(num, sizeof num, "%.17g", v);
    return std::string(num);
  };
  auto ids = [&](uint32_t cta, uint32_t w) {
    return "\"pid\":" + std::to_string(cta) + ",\"tid\":" + std::to_string(w);
  };
  bool first = true;
  auto emit = [&](const std::string& ev) {
    if (!first) js += ',';
    first = false;
    js += ev;
  };
  js += "{\"traceEvents\":[";
  for (uint32_t cta = 0; cta < grid; cta++) {
    emit("{\"name\":\"process_name\",\"ph\":\"M\"," + ids(cta, 0) + ",\"args\":{\"name\":\"CTA " +
         std::to_string(cta) + "\"}}");
    for (uint32_t w = 0; w < wpc; w++) {
      const uint64_t base = ((uint64_t)cta * wpc + w) * slot;
      const uint32_t n_events = u32(base);
      const uint64_t cycles = u64(base + 8);
      emit("{\"name\":\"thread_name\",\"ph\":\"M\"," + ids(cta, w) + ",\"args\":{\"name\":\"warp " +
           std::to_string(w) + "\"}}");
      emit("{\"name\":\"warp\",\"ph\":\"X\"," + ids(cta, w) + ",\"ts\":" + dbl(0.0 / cycles_per_us) +
           ",\"dur\":" + dbl((double)cycles / cycles_per_us) + "}");
      // record stamps hold the cycle's low 24 bits: unwrap in record order
      uint64_t full = 0;
      const uint32_t n = std::min<uint32_t>(n_events, max_ts);
      for (uint32_t i = 0; i < n; i++) {
        const uint64_t r = base + 16u + rb * i;
        const uint32_t word = u32(r), eid = word >> 24, ts24 = word & 0xFFFFFFu;
        full += (uint64_t)((ts24 - (uint32_t)(full & 0xFFFFFFu)) & 0xFFFFFFu);
        if (eid >= k->events.size()) return KS_ERR_ARG;
        const ks::KsEvent& e = k->events[eid];
        const char* ph = e.kind == 1 ? "B" : e.kind == 2 ? "E" : "i";
        std::string ev = "{\"name\":\"" + e.name + "\",\"ph\":\"" + ph + "\"," + ids(cta, w) +
                         ",\"ts\":" + dbl((double)full / cycles_per_us);
        if (e.kind == 0) ev += ",\"s\":\"t\"";
        ev += ",\"args\":{\"id\":" + std::to_string(eid);
        if (e.payload_bytes) ev += ",\"payload\":" + std::to_string(rb == 8 ? (uint64_t)u32(r + 4) : u64(r + 8));
        ev += "}}";
        emit(ev);
      }
    }
  }
  js += "],\"displayTimeUnit\":\"ns\"}";
  *needed = js.size();
  if (!out || cap < js.size() + 1) return KS_ERR_ARG;
  std::memcpy(out, js.data(), js.size());
  out[js.size()] = 0;
  return KS_OK;
}

}  // extern "C"

// ks_capi.cpp — the extern "C" boundary of libks (declared in include/ks.h).
//
// Host work only: argument checks, the module registry, one lazy upload of
// each kernel's program image per device, the real launch shape, and the
// stats-reduction call. Every step of the simulation itself runs in
// ks_interp.cu on the GPU.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "ks_internal.h"

struct ks_module {
  std::vector<ks::KsKernel> kernels;
  std::mutex mu;
  std::map<std::tuple<size_t, int, int>, void*> images;  // (kernel index, device, layout) -> device copy
};

namespace {

void put_err(const std::string& m, char* err, size_t errlen) {
  if (!err || errlen == 0) return;
  size_t n = std::min(m.size(), errlen - 1);
  std::memcpy(err, m.data(), n);
  err[n] = 0;
}

const ks::KsKernel* find_kernel(const ks_module* mod, const char* name, size_t* index) {
  if (!mod || !name) return nullptr;
  for (size_t i = 0; i < mod->kernels.size(); i++)
    if (mod->kernels[i].name == name) {
      if (index) *index = i;
      return &mod->kernels[i];
    }
  return nullptr;
}

struct DevInfo {
  int sms = 0;
  int max_smem = 0;
};

std::mutex g_dev_mu;
std::map<int, DevInfo> g_dev;

int device_info(DevInfo* out, int* dev_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KS_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  auto it = g_dev.find(dev);
  if (it == g_dev.end()) {
    DevInfo d;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KS_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return KS_ERR_CUDA;
    it = g_dev.emplace(dev, d).first;
  }
  *out = it->second;
  *dev_out = dev;
  return KS_OK;
}

// Device accumulator for ks_read_stats, one per device, allocated once.
std::mutex g_acc_mu;
std::map<int, void*> g_acc;
constexpr size_t ACC_WORDS = 15;

uint64_t warps_of(uint32_t grid, uint32_t block) { return (uint64_t)grid * ((block + 31u) / 32u); }

}  // namespace

namespace ks {
const KsKernel* module_kernel(const ks_module* mod, const char* name) { return find_kernel(mod, name, nullptr); }

int pick_layout(const KsKernel& k, uint32_t flags) {
  const bool pair = (flags & KS_FLAG_LAYOUT_PAIR) != 0, split = (flags & KS_FLAG_LAYOUT_SPLIT) != 0;
  if ((flags & ~(KS_FLAG_LAYOUT_PAIR | KS_FLAG_LAYOUT_SPLIT)) != 0 || (pair && split)) return KS_ERR_ARG;
  if (split) return k.cta_mode() ? KS_ERR_UNSUPPORTED : 1;
  if (pair) return 0;
  return (!k.cta_mode() && k.layout[0].region_bytes > SPLIT_REGION_MIN) ? 1 : 0;
}

int check_call(const KsKernel& k, uint32_t grid, uint32_t block, const void* params, size_t param_bytes,
               const ks_buffer* bufs, uint32_t n_bufs, const void* trace_buf, size_t trace_bytes,
               const void* stats_buf, size_t stats_bytes, const ks_config& cfg, int* lay) {
  if (grid == 0 || block == 0 || block > 1024) return KS_ERR_ARG;
  const uint64_t W = (uint64_t)grid * ((block + 31u) / 32u);
  if (W >= (1ull << 31)) return KS_ERR_ARG;
  if (param_bytes < k.param_bytes || param_bytes > KS_MAX_PARAM_BYTES) return KS_ERR_ARG;
  if (k.param_bytes && !params) return KS_ERR_ARG;
  if (n_bufs > KS_MAX_BUFFERS || (n_bufs && !bufs)) return KS_ERR_ARG;
  for (uint32_t i = 0; i < n_bufs; i++) {
    const ks_buffer& b = bufs[i];
    if (b.sim_base % 4096 != 0 || b.bytes == 0 || !b.dev_ptr) return KS_ERR_ARG;
    if (b.sim_base + b.bytes < b.sim_base) return KS_ERR_ARG;
    for (uint32_t j = 0; j < i; j++) {
      const ks_buffer& o = bufs[j];
      if (!(b.sim_base + b.bytes <= o.sim_base || o.sim_base + o.bytes <= b.sim_base)) return KS_ERR_ARG;
    }
  }
  if (!stats_buf || stats_bytes < W * sizeof(ks_warp_stats)) return KS_ERR_ARG;
  if (cfg.simt_stack_depth == 0 || cfg.simt_stack_depth > KS_MAX_STACK) return KS_ERR_ARG;
  if (cfg.max_ts_per_warp > (1u << 24)) return KS_ERR_ARG;
  for (uint32_t i = 0; i < KS_NUM_LAT_CLASSES; i++)
    if (cfg.lat[i] > KS_MAX_LATENCY) return KS_ERR_ARG;
  if (trace_buf && trace_bytes < W * trace_slot_bytes(k, cfg)) return KS_ERR_ARG;
  // shared memory / bar.sync: every warp of a CTA resident on one real CTA
  if (k.cta_mode() && block > KS_MAX_CTA_MODE_BLOCK) return KS_ERR_LIMIT;
  if (cfg.profile_buf && cfg.profile_bytes < k.code.size() * sizeof(ks_pc_profile)) return KS_ERR_ARG;
  const int l = pick_layout(k, cfg.flags);
  if (l < 0) return l;
  *lay = l;
  return KS_OK;
}

void fill_launch(const KsKernel& k, int lay, const void* image, uint32_t grid, uint32_t block, const void* params,
                 size_t param_bytes, const ks_buffer* bufs, uint32_t n_bufs, void* trace_buf, void* stats_buf,
                 const ks_config& cfg, KsLaunch* Lp) {
  KsLaunch& L = *Lp;
  std::memset(&L, 0, sizeof L);
  L.image = static_cast<const uint8_t*>(image);
  L.image_bytes = (uint32_t)k.image[lay].size();
  L.prog_bytes = k.prog_bytes;
  L.n_insn = (uint32_t)k.code.size();
  L.n_slots = k.n_slots;
  L.n_crows = k.layout[lay].n_crows;
  L.layout = k.layout[lay];
  L.grid = grid;
  L.block = block;
  L.wpc = (block + 31u) / 32u;
  L.n_warps = grid * L.wpc;
  std::memcpy(L.live_in, k.live_in, sizeof L.live_in);
  L.shared_bytes = k.shared_bytes;
  L.cta_mode = k.cta_mode() ? 1u : 0u;
  {
    const uint32_t lmax = std::max(std::max(cfg.lat[KS_LAT_ALU], cfg.lat[KS_LAT_FMA]), 1u);
    L.fast_shift = 32u - (uint32_t)__builtin_clz(lmax);  // 2^shift > lmax
  }
  std::memcpy(L.lat, cfg.lat, sizeof L.lat);
  L.max_ts = cfg.max_ts_per_warp;
  L.rec_bytes = k.record_bytes;
  L.stack_depth = cfg.simt_stack_depth;
  L.step_limit = cfg.step_limit;
  L.inject_warp = cfg.inject_warp;
  L.inject_step = cfg.inject_step;
  L.n_bufs = n_bufs;
  for (uint32_t i = 0; i < n_bufs; i++) {
    L.bufs[i].sim_base = bufs[i].sim_base;
    L.bufs[i].bytes = bufs[i].bytes;
    L.bufs[i].ptr = static_cast<uint8_t*>(bufs[i].dev_ptr);
  }
  L.trace = static_cast<uint8_t*>(trace_buf);
  L.slot_bytes = trace_slot_bytes(k, cfg);
  L.stats = static_cast<uint8_t*>(stats_buf);
  L.param_bytes = (uint32_t)param_bytes;
  if (param_bytes) std::memcpy(L.params, params, param_bytes);
  L.profile = static_cast<ks_pc_profile*>(cfg.profile_buf);
}
}  // namespace ks

extern "C" {

void ks_config_default(ks_config* cfg) {
  if (!cfg) return;
  std::memset(cfg, 0, sizeof *cfg);
  const uint32_t lat[KS_NUM_LAT_CLASSES] = {4, 4, 400, 20, 8, 36, 1, 23, 23, 20, 0, 0};
  std::memcpy(cfg->lat, lat, sizeof lat);
  cfg->max_ts_per_warp = 0;
  cfg->simt_stack_depth = 32;
  cfg->step_limit = 1ull << 26;
  cfg->inject_warp = -1;
  cfg->inject_step = 0;
}

int ks_load_module(const char* ptx, size_t len, ks_module** out, char* err, size_t errlen) {
  if (!ptx || !out) {
    put_err("null argument", err, errlen);
    return KS_ERR_ARG;
  }
  *out = nullptr;
  std::vector<ks::KsKernel> ks;
  std::string msg;
  int rc = ks::decode_module(ptx, len, &ks, &msg);
  if (rc != KS_OK) {
    put_err(msg, err, errlen);
    return rc;
  }
  ks_module* m = new ks_module;
  m->kernels = std::move(ks);
  *out = m;
  put_err("", err, errlen);
  return KS_OK;
}

void ks_free_module(ks_module* mod) {
  if (!mod) return;
  int cur = -1;
  cudaGetDevice(&cur);
  for (auto& kv : mod->images) {
    cudaSetDevice(std::get<1>(kv.first));
    cudaFree(kv.second);
  }
  if (cur >= 0 && !mod->images.empty()) cudaSetDevice(cur);
  delete mod;
}

int ks_kernel_info(const ks_module* mod, const char* kernel, uint32_t* n_params, uint32_t* param_bytes,
                   uint32_t* n_events, uint32_t* n_insns, uint32_t* n_reg_slots) {
  const ks::KsKernel* k = find_kernel(mod, kernel, nullptr);
  if (!k) return mod && kernel ? KS_ERR_NOT_FOUND : KS_ERR_ARG;
  if (n_params) *n_params = (uint32_t)k->params.size();
  if (param_bytes) *param_bytes = k->param_bytes;
  if (n_events) *n_events = (uint32_t)k->events.size();
  if (n_insns) *n_insns = (uint32_t)k->code.size();
  if (n_reg_slots) *n_reg_slots = k->n_slots;
  return KS_OK;
}

int ks_kernel_param(const ks_module* mod, const char* kernel, uint32_t index, uint32_t* offset, uint32_t* size,
                    const char** name) {
  const ks::KsKernel* k = find_kernel(mod, kernel, nullptr);
  if (!k) return mod && kernel ? KS_ERR_NOT_FOUND : KS_ERR_ARG;
  if (index >= k->params.size()) return KS_ERR_NOT_FOUND;
  if (offset) *offset = k->params[index].offset;
  if (size) *size = k->params[index].size;
  if (name) *name = k->params[index].name.c_str();
  return KS_OK;
}

int ks_kernel_event(const ks_module* mod, const char* kernel, uint32_t id, uint32_t* kind, const char** name) {
  const ks::KsKernel* k = find_kernel(mod, kernel, nullptr);
  if (!k) return mod && kernel ? KS_ERR_NOT_FOUND : KS_ERR_ARG;
  if (id >= k->events.size()) return KS_ERR_NOT_FOUND;
  if (kind) *kind = k->events[id].kind;
  if (name) *name = k->events[id].name.c_str();
  return KS_OK;
}

int ks_kernel_ipdom(const ks_module* mod, const char* kernel, int32_t* out, uint32_t cap, uint32_t* n_out) {
  const ks::KsKernel* k = find_kernel(mod, kernel, nullptr);
  if (!k) return mod && kernel ? KS_ERR_NOT_FOUND : KS_ERR_ARG;
  if (n_out) *n_out = (uint32_t)k->ipdom.size();
  if (out)
    for (size_t i = 0; i < k->ipdom.size() && i < cap; i++) out[i] = k->ipdom[i];
  return KS_OK;
}

int ks_kernel_fast_runs(const ks_module* mod, const char* kernel, uint32_t* out, uint32_t cap, uint32_t* n_out) {
  const ks::KsKernel* k = find_kernel(mod, kernel, nullptr);
  if (!k) return mod && kernel ? KS_ERR_NOT_FOUND : KS_ERR_ARG;
  const size_t n = k->code.size();
  if (n_out) *n_out = (uint32_t)n;
  if (out) {
    const ks::DevInsn* d = reinterpret_cast<const ks::DevInsn*>(k->image[0].data());
    for (size_t i = 0; i < n && i < cap; i++) {
      const uint32_t len = d[i].inc >> ks::INC_RUN_SHIFT;
      out[3 * i] = len;
      out[3 * i + 1] = (len && (d[i].inc & ks::INC_OWN_D)) ? 1u : 0u;
      out[3 * i + 2] = len ? (d[i].x[4] & ks::KEEP_COUNT) : 0u;
    }
  }
  return KS_OK;
}

int ks_kernel_layout(const ks_module* mod, const char* kernel, uint32_t flags, uint32_t* split,
                     uint32_t* region_bytes) {
  const ks::KsKernel* k = find_kernel(mod, kernel, nullptr);
  if (!k) return mod && kernel ? KS_ERR_NOT_FOUND : KS_ERR_ARG;
  const int lay = ks::pick_layout(*k, flags);
  if (lay < 0) return lay;
  if (split) *split = (uint32_t)lay;
  if (region_bytes) *region_bytes = k->layout[lay].region_bytes;
  return KS_OK;
}

size_t ks_trace_bytes(uint32_t grid, uint32_t block, uint32_t max_ts_per_warp) {
  const uint64_t slot = (16ull + 4ull * max_ts_per_warp + 7ull) / 8ull * 8ull;
  return (size_t)(warps_of(grid, block) * slot);
}

size_t ks_trace_bytes_records(uint32_t grid, uint32_t block, uint32_t max_ts_per_warp, uint32_t record_bytes) {
  const uint64_t slot = (16ull + (uint64_t)record_bytes * max_ts_per_warp + 7ull) / 8ull * 8ull;
  return (size_t)(warps_of(grid, block) * slot);
}

int ks_kernel_record_bytes(const ks_module* mod, const char* kernel, uint32_t* bytes) {
  const ks::KsKernel* k = find_kernel(mod, kernel, nullptr);
  if (!k) return mod && kernel ? KS_ERR_NOT_FOUND : KS_ERR_ARG;
  if (!bytes) return KS_ERR_ARG;
  *bytes = k->record_bytes;
  return KS_OK;
}

int ks_kernel_event_payload(const ks_module* mod, const char* kernel, uint32_t id, uint32_t* bytes) {
  const ks::KsKernel* k = find_kernel(mod, kernel, nullptr);
  if (!k) return mod && kernel ? KS_ERR_NOT_FOUND : KS_ERR_ARG;
  if (id >= k->events.size()) return KS_ERR_NOT_FOUND;
  if (!bytes) return KS_ERR_ARG;
  *bytes = k->events[id].payload_bytes;
  return KS_OK;
}

size_t ks_stats_bytes(uint32_t grid, uint32_t block) {
  return (size_t)(warps_of(grid, block) * sizeof(ks_warp_stats));
}

}  // extern "C"

namespace {

// Argument checks, the lazy program upload and the launch block shared by
// ks_simulate and ks_simulate_cached.
int prepare(const ks_module* mod_c, const char* kernel, uint32_t grid, uint32_t block, const void* params,
            size_t param_bytes, const ks_buffer* bufs, uint32_t n_bufs, void* trace_buf, size_t trace_bytes,
            void* stats_buf, size_t stats_bytes, const ks_config* cfg_in, ks::KsLaunch* Lp, DevInfo* dip,
            bool host_checks_only = false) {
  ks_module* mod = const_cast<ks_module*>(mod_c);
  size_t kidx = 0;
  const ks::KsKernel* k = find_kernel(mod, kernel, &kidx);
  if (!mod || !kernel) return KS_ERR_ARG;
  if (!k) return KS_ERR_NOT_FOUND;
  ks_config cfg;
  if (cfg_in) cfg = *cfg_in; else ks_config_default(&cfg);
  int lay = 0;
  const int rc = ks::check_call(*k, grid, block, params, param_bytes, bufs, n_bufs, trace_buf, trace_bytes, stats_buf,
                                stats_bytes, cfg, &lay);
  if (rc != KS_OK) return rc;

  if (host_checks_only) return KS_OK;
  DevInfo& di = *dip;
  int dev = 0;
  if (device_info(&di, &dev) != KS_OK) return KS_ERR_CUDA;

  // ---- program image of the chosen layout on this device (uploaded once) ----
  const std::vector<uint8_t>& img = k->image[lay];
  void* image = nullptr;
  {
    std::lock_guard<std::mutex> lk(mod->mu);
    auto key = std::make_tuple(kidx, dev, lay);
    auto it = mod->images.find(key);
    if (it == mod->images.end()) {
      if (cudaMalloc(&image, img.size()) != cudaSuccess) return KS_ERR_CUDA;
      if (cudaMemcpy(image, img.data(), img.size(), cudaMemcpyHostToDevice) != cudaSuccess) {
        cudaFree(image);
        return KS_ERR_CUDA;
      }
      mod->images[key] = image;
    } else {
      image = it->second;
    }
  }
  ks::fill_launch(*k, lay, image, grid, block, params, param_bytes, bufs, n_bufs, trace_buf, stats_buf, cfg, Lp);
  return KS_OK;
}

// Zeroes the profile (if any) on the stream before the launch that fills it.
int clear_profile(const ks::KsLaunch& L, void* stream) {
  if (!L.profile) return KS_OK;
  return cudaMemsetAsync(L.profile, 0, (size_t)L.n_insn * sizeof(ks_pc_profile), static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? KS_OK
             : KS_ERR_CUDA;
}

// Real launch shape (persistent real warps, see ks::choose_launch) and launch.
int shape_and_launch(const ks::KsLaunch& L, const DevInfo& di, void* stream) {
  ks::LaunchShape shape;
  const int rc = ks::choose_launch(L, di.sms, di.max_smem, &shape);
  if (rc != KS_OK) return rc;
  if (ks::launch_interp(L, shape, stream) != 0) return KS_ERR_CUDA;
  return KS_OK;
}

bool cache_config_ok(const ks_cache_config& c) {
  return c.l1_lines >= 1 && c.l1_lines <= 65536 && c.l2_lines >= c.l1_lines && c.l2_lines % c.l1_lines == 0 &&
         c.l2_lines / c.l1_lines <= 65535 && c.lat_l1 <= ks::KS_MAX_LATENCY && c.lat_l2 <= ks::KS_MAX_LATENCY &&
         c.max_accesses_per_warp >= 1;
}

uint32_t bits_for(uint64_t max_value) {
  uint32_t b = 0;
  while (b < 64 && (max_value >> b) != 0) b++;
  return b;
}

// The cache model's own argument checks (ks_simulate_cached): the
// configuration (defaults for NULL), the key width, then (not with
// host_checks_only: the sorts' scratch size asks the device) the workspace
// layout and size.
int cache_checks(const ks_cache_config* cc_in, const void* workspace, size_t workspace_bytes, uint32_t grid,
                 uint32_t block, ks_cache_config* cc, ks::CacheLayout* C, bool host_checks_only = false) {
  if (cc_in) *cc = *cc_in; else ks_cache_config_default(cc);
  if (!cache_config_ok(*cc) || !workspace) return KS_ERR_ARG;
  if (grid == 0 || block == 0 || block > 1024) return KS_ERR_ARG;
  const uint64_t W = warps_of(grid, block);
  if (bits_for(cc->l1_lines - 1u) + 32u + bits_for(W - 1u) > 64u) return KS_ERR_LIMIT;
  if (host_checks_only) return KS_OK;
  const int lc = ks::cache_layout(W, cc->max_accesses_per_warp, cc->max_runs_per_warp, C);
  if (lc != KS_OK) return lc;
  if (workspace_bytes < C->total) return KS_ERR_ARG;
  return KS_OK;
}

// Points a prepared launch at its cache-model workspace for its first pass
// and returns whether the launch takes the timing-replay form: then the pass
// is the real run (cache_pass 3: stores land, accesses and issued runs
// logged, the profile collected); else the accesses are logged with the
// stores suppressed and no profile (cache_pass 1), and a second
// interpretation follows.
bool cache_first_pass(ks::KsLaunch* L, const ks_cache_config& cc, uint8_t* ws, const ks::CacheLayout& C) {
  L->cache_cap = cc.max_accesses_per_warp;
  L->lat_l1 = cc.lat_l1;
  L->lat_l2 = cc.lat_l2;
  L->cache_warps = reinterpret_cast<ks_cache_warp*>(ws + C.warps_off);
  L->cache_log = reinterpret_cast<ks_cache_access*>(ws + C.log_off);
  if (cc.max_runs_per_warp > 0 && !L->cta_mode) {
    L->sched_runs = reinterpret_cast<uint32_t*>(ws + C.runs_off);
    L->sched_log = reinterpret_cast<uint32_t*>(ws + C.runlog_off);
    L->sched_cap = cc.max_runs_per_warp;
    L->cache_pass = 3;
    return true;
  }
  L->profile = nullptr;
  L->cache_pass = 1;
  return false;
}

// Helper streams of one device, created on first use and kept for the
// library's lifetime: the grids of one call that do not share a real grid run
// on them side by side, so that one grid's last warps overlap the next grid's
// work instead of leaving SMs idle (the 64 fuzz kernels: 182 -> 166 ms a step
// on four streams). They start when the caller's stream reaches the call and
// the caller's stream waits for all of them, so the call keeps the ordering
// of a single-stream launch.
constexpr int FORK_STREAMS = 4;
struct ForkPool {
  cudaStream_t s[FORK_STREAMS];
  cudaEvent_t fork, join[FORK_STREAMS];
};
std::mutex g_fork_mu;  // held while a call enqueues its fork and join
std::map<int, ForkPool> g_fork;

// The current device's pool, or null if it cannot be made (the call then
// launches everything on the caller's stream). Needs g_fork_mu.
ForkPool* fork_pool() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  auto it = g_fork.find(dev);
  if (it != g_fork.end()) return &it->second;
  ForkPool P;
  if (cudaEventCreateWithFlags(&P.fork, cudaEventDisableTiming) != cudaSuccess) return nullptr;
  for (int j = 0; j < FORK_STREAMS; j++) {
    if (cudaStreamCreateWithFlags(&P.s[j], cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&P.join[j], cudaEventDisableTiming) != cudaSuccess)
      return nullptr;  // (what was made stays unused)
  }
  return &g_fork.emplace(dev, P).first->second;
}

// Runs launch(k, stream) for k = 0 .. n-1: with n > 1 on the helper streams,
// forked from and joined back to `stream` (unless it is capturing a graph,
// or no pool can be made: then all on `stream`, in order). Returns the first
// launch's error; the join is enqueued whatever happened.
template <class F>
int fork_launches(size_t n, void* stream, F&& launch) {
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (n > 1 && cudaStreamIsCapturing(cs, &cap) != cudaSuccess) return KS_ERR_CUDA;
  std::unique_lock<std::mutex> lk(g_fork_mu, std::defer_lock);
  ForkPool* P = nullptr;
  if (n > 1 && cap == cudaStreamCaptureStatusNone) {
    lk.lock();
    P = fork_pool();
    if (!P) lk.unlock();
  }
  if (!P) {
    for (size_t k = 0; k < n; k++) {
      const int rc = launch(k, stream);
      if (rc != KS_OK) return rc;
    }
    return KS_OK;
  }
  const int used = (int)std::min<size_t>(n, FORK_STREAMS);
  if (cudaEventRecord(P->fork, cs) != cudaSuccess) return KS_ERR_CUDA;
  for (int j = 0; j < used; j++)
    if (cudaStreamWaitEvent(P->s[j], P->fork, 0) != cudaSuccess) return KS_ERR_CUDA;
  int rc = KS_OK;
  for (size_t k = 0; k < n && rc == KS_OK; k++) rc = launch(k, P->s[k % used]);
  for (int j = 0; j < used; j++) {
    if (cudaEventRecord(P->join[j], P->s[j]) != cudaSuccess || cudaStreamWaitEvent(cs, P->join[j], 0) != cudaSuccess)
      rc = rc == KS_OK ? KS_ERR_CUDA : rc;
  }
  return rc;
}

// Launches prepared simulations as real grids of one instantiation each (mode,
// form, layout, and in CTA mode the block), in the order of their first items, at
// most KS_BATCH_ITEMS and at most BATCH_WARPS_PER_SM simulated warps per SM
// of them, so that a grid runs as one wave and ends with its slowest warp
// (items are not weighted by their unknown cost per warp). An item larger
// than that fills the GPU alone and is launched as ks_simulate launches it.
// Several grids go to the helper streams (above) unless the caller's stream
// is capturing a graph. Adds the real launches to *n_launched (if not null).
int launch_items(const std::vector<ks::KsLaunch>& Ls, const DevInfo& di, void* stream, uint32_t* n_launched) {
  constexpr uint64_t BATCH_WARPS_PER_SM = 16;
  const uint64_t budget = BATCH_WARPS_PER_SM * (uint64_t)std::max(di.sms, 1);
  auto key = [](const ks::KsLaunch& L) {
    return ((uint64_t)L.cta_mode << 40) | ((uint64_t)L.layout.split << 36) | ((uint64_t)ks::interp_form(L) << 32) |
           (L.cta_mode ? L.wpc : 0u);
  };
  // a CTA-mode item whose warps' state does not fit shared memory runs alone
  // (its regions in global scratch, ks::LaunchShape::greg)
  auto alone = [&](const ks::KsLaunch& L) {
    return L.cta_mode && ks::cta_mode_smem(L) > (size_t)di.max_smem;
  };
  // the real grids: the items of each, in call order
  const size_t n_items = Ls.size();
  std::vector<char> done(n_items, 0);
  std::vector<std::vector<size_t>> grids;
  for (size_t i = 0; i < n_items; i++) {
    if (done[i]) continue;
    std::vector<size_t> g;
    uint64_t warps = 0;
    for (size_t j = i; j < n_items && g.size() < ks::KS_BATCH_ITEMS; j++) {
      if (done[j] || key(Ls[j]) != key(Ls[i]) || (!g.empty() && (alone(Ls[i]) || alone(Ls[j])))) continue;
      if (!g.empty() && (Ls[j].n_warps > budget || warps + Ls[j].n_warps > budget)) continue;
      g.push_back(j);
      warps += Ls[j].n_warps;
      done[j] = 1;
      if (warps > budget) break;  // a large first item goes alone
    }
    grids.push_back(std::move(g));
  }
  auto G = std::make_unique<ks::KsGrid<ks::KS_BATCH_ITEMS>>();
  auto launch = [&](const std::vector<size_t>& g, void* st) {
    if (g.size() == 1) return shape_and_launch(Ls[g[0]], di, st);
    G->n = 0;
    for (size_t j : g) G->item[G->n++] = Ls[j];
    return ks::launch_batch(G.get(), di.sms, di.max_smem, st);
  };
  return fork_launches(grids.size(), stream, [&](size_t g, void* st) {
    const int rc = launch(grids[g], st);
    if (rc == KS_OK && n_launched) ++*n_launched;
    return rc;
  });
}

}  // namespace

extern "C" {

int ks_simulate(const ks_module* mod, const char* kernel, uint32_t grid, uint32_t block, const void* params,
                size_t param_bytes, const ks_buffer* bufs, uint32_t n_bufs, void* trace_buf, size_t trace_bytes,
                void* stats_buf, size_t stats_bytes, const ks_config* cfg, void* stream) {
  ks::KsLaunch L;
  DevInfo di;
  const int rc = prepare(mod, kernel, grid, block, params, param_bytes, bufs, n_bufs, trace_buf, trace_bytes,
                         stats_buf, stats_bytes, cfg, &L, &di);
  if (rc != KS_OK) return rc;
  if (clear_profile(L, stream) != KS_OK) return KS_ERR_CUDA;
  return shape_and_launch(L, di, stream);
}

int ks_simulate_batch(const ks_batch_item* items, uint32_t n_items, void* stream, uint32_t* failed_item,
                      uint32_t* n_launched) {
  if (failed_item) *failed_item = n_items;
  if (n_launched) *n_launched = 0;
  if (!items || n_items == 0) return KS_ERR_ARG;
  std::vector<ks::KsLaunch> Ls(n_items);
  DevInfo di;
  // every item's host-side checks first, then the device work of each
  for (int pass = 0; pass < 2; pass++) {
    for (uint32_t i = 0; i < n_items; i++) {
      const ks_batch_item& it = items[i];
      const int rc = it.reserved ? KS_ERR_ARG
                                 : prepare(it.mod, it.kernel, it.grid, it.block, it.params, it.param_bytes, it.bufs,
                                           it.n_bufs, it.trace_buf, it.trace_bytes, it.stats_buf, it.stats_bytes,
                                           it.cfg, &Ls[i], &di, pass == 0);
      if (rc != KS_OK) {
        if (failed_item) *failed_item = i;
        return rc;
      }
    }
  }
  for (uint32_t i = 0; i < n_items; i++)
    if (clear_profile(Ls[i], stream) != KS_OK) return KS_ERR_CUDA;
  return launch_items(Ls, di, stream, n_launched);
}

int ks_profile_bytes(const ks_module* mod, const char* kernel, size_t* bytes) {
  const ks::KsKernel* k = find_kernel(mod, kernel, nullptr);
  if (!k) return mod && kernel ? KS_ERR_NOT_FOUND : KS_ERR_ARG;
  if (!bytes) return KS_ERR_ARG;
  *bytes = k->code.size() * sizeof(ks_pc_profile);
  return KS_OK;
}

void ks_sched_config_default(ks_sched_config* sc) {
  if (!sc) return;
  std::memset(sc, 0, sizeof *sc);
  sc->n_sm = 152;
  sc->ctas_per_sm = 0;
  sc->schedulers_per_sm = 4;
  sc->max_runs_per_warp = 4096;
}

size_t ks_sched_workspace_bytes(uint32_t grid, uint32_t block, const ks_sched_config* sc_in) {
  ks_sched_config sc;
  if (sc_in) sc = *sc_in; else ks_sched_config_default(&sc);
  if (grid == 0 || block == 0 || block > 1024 || sc.max_runs_per_warp == 0) return 0;
  const uint64_t W = warps_of(grid, block);
  return (size_t)((W * 4 + 255) / 256 * 256 + W * (uint64_t)sc.max_runs_per_warp * 4);
}

int ks_simulate_sched(const ks_module* mod, const char* kernel, uint32_t grid, uint32_t block, const void* params,
                      size_t param_bytes, const ks_buffer* bufs, uint32_t n_bufs, void* trace_buf,
                      size_t trace_bytes, void* stats_buf, size_t stats_bytes, const ks_config* cfg,
                      const ks_sched_config* sc_in, void* sched_warps, size_t sched_warps_bytes, void* sched_sms,
                      size_t sched_sms_bytes, void* workspace, size_t workspace_bytes, void* stream) {
  ks_sched_config sc;
  if (sc_in) sc = *sc_in; else ks_sched_config_default(&sc);
  if (grid == 0 || block == 0 || block > 1024) return KS_ERR_ARG;
  const uint32_t wpc = (block + 31u) / 32u;
  if (sc.n_sm == 0 || sc.max_runs_per_warp == 0 ||
      !(sc.schedulers_per_sm == 1 || sc.schedulers_per_sm == 2 || sc.schedulers_per_sm == 4))
    return KS_ERR_ARG;
  const uint32_t ctas = sc.ctas_per_sm ? sc.ctas_per_sm : 32u / wpc;
  if (ctas == 0 || ctas * wpc > 32u) return KS_ERR_ARG;
  const uint64_t W = warps_of(grid, block);
  if (!sched_warps || sched_warps_bytes < W * sizeof(ks_sched_warp)) return KS_ERR_ARG;
  if (!sched_sms || sched_sms_bytes < (uint64_t)sc.n_sm * sizeof(ks_sched_sm)) return KS_ERR_ARG;
  const size_t need = ks_sched_workspace_bytes(grid, block, &sc);
  if (!workspace || need == 0 || workspace_bytes < need) return KS_ERR_ARG;
  if (W * (uint64_t)sc.max_runs_per_warp >= (1ull << 40)) return KS_ERR_ARG;
  ks::KsLaunch L;
  DevInfo di;
  int rc = prepare(mod, kernel, grid, block, params, param_bytes, bufs, n_bufs, trace_buf, trace_bytes, stats_buf,
                   stats_bytes, cfg, &L, &di);
  if (rc != KS_OK) return rc;
  const uint32_t n_rows = L.layout.n_rows();
  if (ks::sched_smem_bytes(L.n_insn, n_rows) > (size_t)di.max_smem) return KS_ERR_LIMIT;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  L.sched_runs = reinterpret_cast<uint32_t*>(ws);
  L.sched_log = reinterpret_cast<uint32_t*>(ws + (W * 4 + 255) / 256 * 256);
  L.sched_cap = sc.max_runs_per_warp;
  if (clear_profile(L, stream) != KS_OK) return KS_ERR_CUDA;
  rc = shape_and_launch(L, di, stream);
  if (rc != KS_OK) return rc;
  if (ks::launch_sched(L, n_rows, sc.n_sm, ctas, sc.schedulers_per_sm, static_cast<ks_sched_warp*>(sched_warps),
                       static_cast<ks_sched_sm*>(sched_sms), stream) != 0)
    return KS_ERR_CUDA;
  return KS_OK;
}

void ks_cache_config_default(ks_cache_config* cc) {
  if (!cc) return;
  std::memset(cc, 0, sizeof *cc);
  cc->l1_lines = 1024;
  cc->l2_lines = 49152;
  cc->lat_l1 = 28;
  cc->lat_l2 = 150;
  cc->max_accesses_per_warp = 1024;
}

size_t ks_cache_workspace_bytes(uint32_t grid, uint32_t block, const ks_cache_config* cc_in) {
  ks_cache_config cc;
  if (cc_in) cc = *cc_in; else ks_cache_config_default(&cc);
  if (grid == 0 || block == 0 || block > 1024 || !cache_config_ok(cc)) return 0;
  ks::CacheLayout C;
  if (ks::cache_layout(warps_of(grid, block), cc.max_accesses_per_warp, cc.max_runs_per_warp, &C) != KS_OK) return 0;
  return (size_t)C.total;
}

int ks_simulate_cached(const ks_module* mod, const char* kernel, uint32_t grid, uint32_t block, const void* params,
                       size_t param_bytes, const ks_buffer* bufs, uint32_t n_bufs, void* trace_buf,
                       size_t trace_bytes, void* stats_buf, size_t stats_bytes, const ks_config* cfg,
                       const ks_cache_config* cc_in, void* workspace, size_t workspace_bytes, void* stream) {
  ks_cache_config cc;
  ks::CacheLayout C;
  const int lc = cache_checks(cc_in, workspace, workspace_bytes, grid, block, &cc, &C);
  if (lc != KS_OK) return lc;
  ks::KsLaunch L;
  DevInfo di;
  int rc = prepare(mod, kernel, grid, block, params, param_bytes, bufs, n_bufs, trace_buf, trace_bytes, stats_buf,
                   stats_bytes, cfg, &L, &di);
  if (rc != KS_OK) return rc;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  ks_pc_profile* profile = L.profile;
  const bool replay = cache_first_pass(&L, cc, ws, C);
  if (replay && clear_profile(L, stream) != KS_OK) return KS_ERR_CUDA;
  rc = shape_and_launch(L, di, stream);
  if (rc != KS_OK) return rc;
  if (ks::launch_cache_levels(L, ws, C, cc.l1_lines, cc.l2_lines, stream) != 0) return KS_ERR_CUDA;
  if (replay) return ks::launch_cache_replay(L, di.sms, di.max_smem, stream) != 0 ? KS_ERR_CUDA : KS_OK;
  L.cache_pass = 2;  // the real run, latencies from the levels
  L.profile = profile;
  if (clear_profile(L, stream) != KS_OK) return KS_ERR_CUDA;
  return shape_and_launch(L, di, stream);
}

int ks_simulate_cached_batch(const ks_cached_item* items, uint32_t n_items, void* stream, uint32_t* failed_item,
                             uint32_t* n_launched) {
  if (failed_item) *failed_item = n_items;
  if (n_launched) *n_launched = 0;
  if (!items || n_items == 0) return KS_ERR_ARG;
  std::vector<ks::KsLaunch> Ls(n_items);
  std::vector<ks_cache_config> ccs(n_items);
  std::vector<ks::CacheLayout> Cs(n_items);
  std::vector<ks_pc_profile*> profiles(n_items);
  DevInfo di;
  // every item's host-side checks first, then the device work of each
  for (int pass = 0; pass < 2; pass++) {
    for (uint32_t i = 0; i < n_items; i++) {
      const ks_batch_item& it = items[i].sim;
      int rc = it.reserved ? KS_ERR_ARG
                           : cache_checks(items[i].cache, items[i].workspace, items[i].workspace_bytes, it.grid,
                                          it.block, &ccs[i], &Cs[i], pass == 0);
      if (rc == KS_OK)
        rc = prepare(it.mod, it.kernel, it.grid, it.block, it.params, it.param_bytes, it.bufs, it.n_bufs,
                     it.trace_buf, it.trace_bytes, it.stats_buf, it.stats_bytes, it.cfg, &Ls[i], &di, pass == 0);
      if (rc != KS_OK) {
        if (failed_item) *failed_item = i;
        return rc;
      }
    }
  }
  // first pass of every item, then every item's levels, then the second
  // passes: timing replays, and the other items' interpretations batched
  std::vector<char> replay(n_items, 0);
  for (uint32_t i = 0; i < n_items; i++) {
    profiles[i] = Ls[i].profile;
    replay[i] = cache_first_pass(&Ls[i], ccs[i], static_cast<uint8_t*>(items[i].workspace), Cs[i]) ? 1 : 0;
    if (replay[i] && clear_profile(Ls[i], stream) != KS_OK) return KS_ERR_CUDA;
  }
  int rc = launch_items(Ls, di, stream, n_launched);
  if (rc != KS_OK) return rc;
  for (uint32_t i = 0; i < n_items; i++)
    if (ks::launch_cache_levels(Ls[i], static_cast<uint8_t*>(items[i].workspace), Cs[i], ccs[i].l1_lines,
                                ccs[i].l2_lines, stream, n_launched) != 0)
      return KS_ERR_CUDA;
  // the timing replays side by side (each fills few SMs)
  std::vector<uint32_t> rep;
  for (uint32_t i = 0; i < n_items; i++)
    if (replay[i]) rep.push_back(i);
  rc = fork_launches(rep.size(), stream, [&](size_t k, void* st) {
    if (ks::launch_cache_replay(Ls[rep[k]], di.sms, di.max_smem, st) != 0) return (int)KS_ERR_CUDA;
    if (n_launched) ++*n_launched;
    return (int)KS_OK;
  });
  if (rc != KS_OK) return rc;
  std::vector<ks::KsLaunch> second;
  for (uint32_t i = 0; i < n_items; i++) {
    if (replay[i]) continue;
    Ls[i].cache_pass = 2;
    Ls[i].profile = profiles[i];
    if (clear_profile(Ls[i], stream) != KS_OK) return KS_ERR_CUDA;
    second.push_back(Ls[i]);
  }
  return second.empty() ? KS_OK : launch_items(second, di, stream, n_launched);
}

int ks_read_stats(const void* stats_buf, uint64_t n_warps, void* stream, ks_totals* out) {
  if (!stats_buf || !out || n_warps == 0) return KS_ERR_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return KS_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_acc_mu);
  void*& acc = g_acc[dev];
  if (!acc && cudaMalloc(&acc, ACC_WORDS * sizeof(uint64_t)) != cudaSuccess) {
    acc = nullptr;
    return KS_ERR_CUDA;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(acc, 0, ACC_WORDS * sizeof(uint64_t), s) != cudaSuccess) return KS_ERR_CUDA;
  if (ks::launch_reduce_stats(stats_buf, n_warps, acc, stream) != 0) return KS_ERR_CUDA;
  uint64_t h[ACC_WORDS];
  if (cudaMemcpyAsync(h, acc, sizeof h, cudaMemcpyDeviceToHost, s) != cudaSuccess) return KS_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return KS_ERR_CUDA;
  std::memset(out, 0, sizeof *out);
  out->cycles_max = h[0];
  out->cycles_sum = h[1];
  out->warp_insts = h[2];
  out->thread_insts = h[3];
  out->ld_req = h[4];
  out->ld_sectors = h[5];
  out->st_req = h[6];
  out->st_sectors = h[7];
  out->ld_lines = h[8];
  out->st_lines = h[9];
  out->n_warps = n_warps;
  out->n_failed = h[10];
  out->max_stack_depth = (uint32_t)h[12];
  out->sh_req = h[13];
  out->sh_wavefronts = h[14];
  out->first_failed_warp = -1;
  out->status = 0;
  if (h[10]) {
    const uint64_t w = ~0ull - h[11];
    out->first_failed_warp = (int64_t)w;
    int32_t st = 0;
    const char* p = static_cast<const char*>(stats_buf) + w * sizeof(ks_warp_stats) + offsetof(ks_warp_stats, status);
    if (cudaMemcpyAsync(&st, p, sizeof st, cudaMemcpyDeviceToHost, s) != cudaSuccess) return KS_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return KS_ERR_CUDA;
    out->status = st;
  }
  return KS_OK;
}

const char* ks_status_string(int code) {
  switch (code) {
    case KS_OK: return "ok";
    case KS_ERR_PARSE: return "malformed PTX";
    case KS_ERR_UNSUPPORTED: return "PTX outside the supported subset";
    case KS_ERR_ARG: return "bad argument";
    case KS_ERR_CUDA: return "CUDA runtime error";
    case KS_ERR_NOT_FOUND: return "not found";
    case KS_ERR_LIMIT: return "program or register file too large";
    case KS_ST_OOB: return "simulated address outside every buffer";
    case KS_ST_MISALIGNED: return "simulated address not aligned to the access size";
    case KS_ST_STEP_LIMIT: return "warp exceeded the step limit";
    case KS_ST_SIMT_STACK: return "reconvergence stack overflow";
    case KS_ST_TIMEOUT: return "bounded wait ran out";
    case KS_ST_INJECTED: return "injected fault";
    case KS_ST_CACHE_LOG: return "cache model: access log full or access step too large";
    case KS_ST_CACHE_STREAM: return "cache model: accesses differ between the two passes";
    case KS_ST_SCHED_LIMIT: return "SM issue model: issue log full or SM clock too large";
    default: return "unknown status";
  }
}

}  // extern "C"

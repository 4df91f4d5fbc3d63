// ks_static.cu — ks_simulate_static: ks_simulate without any device
// allocation.
//
// ks_simulate keeps each kernel's program image (decoded instructions and
// constant rows) in device memory that the library allocates on first use
// per device. Some callers cannot let a library call cudaMalloc: processes
// that give all of the GPU's memory to their own pool at start-up (the
// library's allocation would fail or fragment it), deployments with a fixed
// device-memory budget that may not grow after start-up, and callers that
// cannot afford the implicit device-wide synchronisation cudaMalloc /
// cudaFree may cause. For them this entry point stages the image into the
// file-scope array below instead, which every GPU that loads the library
// holds until the process exits. It calls no allocating routine: the array's
// address comes from cudaGetSymbolAddress, the launch shape from device
// attributes and the occupancy calculator.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "ks_internal.h"

// One image of at most KS_STATIC_IMAGE_BYTES, shared by every call on a device.
static __device__ __align__(256) uint8_t ks_static_image[KS_STATIC_IMAGE_BYTES];

namespace {

constexpr int MAX_DEVICES = 64;
std::mutex g_static_mu;
void* g_static_addr[MAX_DEVICES];  // device address of ks_static_image, per device
int g_static_sms[MAX_DEVICES];
int g_static_smem[MAX_DEVICES];

// Set-up, once per device, with that device current: the device address of
// the array (host code only sees a host-side stand-in for its name) and the
// device limits used to shape the launch.
int static_setup(int dev) {
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (g_static_addr[dev]) return KS_OK;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, ks_static_image) != cudaSuccess || !p) return KS_ERR_CUDA;
  int sms = 0, smem = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return KS_ERR_CUDA;
  if (cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return KS_ERR_CUDA;
  g_static_sms[dev] = sms;
  g_static_smem[dev] = smem;
  g_static_addr[dev] = p;
  return KS_OK;
}

}  // namespace

extern "C" int ks_simulate_static(const ks_module* mod, const char* kernel, uint32_t grid, uint32_t block,
                                  const void* params, size_t param_bytes, const ks_buffer* bufs, uint32_t n_bufs,
                                  void* trace_buf, size_t trace_bytes, void* stats_buf, size_t stats_bytes,
                                  const ks_config* cfg_in, void* stream) {
  if (!mod || !kernel) return KS_ERR_ARG;
  const ks::KsKernel* k = ks::module_kernel(mod, kernel);
  if (!k) return KS_ERR_NOT_FOUND;
  ks_config cfg;
  if (cfg_in) cfg = *cfg_in; else ks_config_default(&cfg);

  // ---- the same argument checks as ks_simulate ----
  if (grid == 0 || block == 0 || block > 1024) return KS_ERR_ARG;
  const uint64_t W = (uint64_t)grid * ((block + 31u) / 32u);
  if (W >= (1ull << 31)) return KS_ERR_ARG;
  if (param_bytes < k->param_bytes || param_bytes > KS_MAX_PARAM_BYTES) return KS_ERR_ARG;
  if (k->param_bytes && !params) return KS_ERR_ARG;
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
    if (cfg.lat[i] > ks::KS_MAX_LATENCY) return KS_ERR_ARG;
  const uint64_t slot = (16ull + (uint64_t)k->record_bytes * cfg.max_ts_per_warp + 7ull) / 8ull * 8ull;
  if (trace_buf && trace_bytes < W * slot) return KS_ERR_ARG;
  // shared memory / bar.sync: every warp of a CTA resident on one real CTA
  if (k->cta_mode() && block > KS_MAX_CTA_MODE_BLOCK) return KS_ERR_LIMIT;
  if (cfg.profile_buf && cfg.profile_bytes < k->code.size() * sizeof(ks_pc_profile)) return KS_ERR_ARG;
  // ---- the program image of the layout ks_simulate would take must fit the static array ----
  const int lay = ks::pick_layout(*k, cfg.flags);
  if (lay < 0) return lay;
  const std::vector<uint8_t>& img = k->image[lay];
  if (img.size() > KS_STATIC_IMAGE_BYTES) return KS_ERR_LIMIT;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return KS_ERR_CUDA;
  if (static_setup(dev) != KS_OK) return KS_ERR_CUDA;
  // a kernel with shared memory or bar.sync whose CTA's warp state does not
  // fit on chip needs ks_simulate's global scratch: refused before any GPU work
  if (k->cta_mode() && ks::interp_smem_bytes((uint32_t)img.size(), k->layout[lay].region_bytes, (block + 31u) / 32u,
                                             k->shared_bytes) > (size_t)g_static_smem[dev])
    return KS_ERR_LIMIT;
  void* image = g_static_addr[dev];
  if (cudaMemcpyAsync(image, img.data(), img.size(), cudaMemcpyHostToDevice,
                      static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KS_ERR_CUDA;

  ks::KsLaunch L;
  std::memset(&L, 0, sizeof L);
  L.image = static_cast<const uint8_t*>(image);
  L.image_bytes = (uint32_t)img.size();
  L.prog_bytes = k->prog_bytes;
  L.n_insn = (uint32_t)k->code.size();
  L.n_slots = k->n_slots;
  L.n_crows = k->layout[lay].n_crows;
  L.layout = k->layout[lay];
  L.grid = grid;
  L.block = block;
  L.wpc = (block + 31u) / 32u;
  L.n_warps = (uint32_t)W;
  L.shared_bytes = k->shared_bytes;
  L.cta_mode = k->cta_mode() ? 1u : 0u;
  {
    const uint32_t lmax = std::max(std::max(cfg.lat[KS_LAT_ALU], cfg.lat[KS_LAT_FMA]), 1u);
    L.fast_shift = 32u - (uint32_t)__builtin_clz(lmax);  // 2^shift > lmax
  }
  std::memcpy(L.lat, cfg.lat, sizeof L.lat);
  L.max_ts = cfg.max_ts_per_warp;
  L.rec_bytes = k->record_bytes;
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
  L.slot_bytes = slot;
  L.stats = static_cast<uint8_t*>(stats_buf);
  L.param_bytes = (uint32_t)param_bytes;
  if (param_bytes) std::memcpy(L.params, params, param_bytes);
  L.profile = static_cast<ks_pc_profile*>(cfg.profile_buf);
  if (L.profile && cudaMemsetAsync(L.profile, 0, k->code.size() * sizeof(ks_pc_profile),
                                   static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return KS_ERR_CUDA;

  ks::LaunchShape shape;
  const int rc = ks::choose_launch(L, g_static_sms[dev], g_static_smem[dev], &shape);
  if (rc != KS_OK) return rc;
  // a CTA whose warps' state needs global scratch cannot run without an allocation
  if (shape.greg) return KS_ERR_LIMIT;
  if (ks::launch_interp(L, shape, stream) != 0) return KS_ERR_CUDA;
  return KS_OK;
}

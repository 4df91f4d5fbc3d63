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

  // ---- the checks every simulation call makes, and the layout ----
  int lay = 0;
  const int ck = ks::check_call(*k, grid, block, params, param_bytes, bufs, n_bufs, trace_buf, trace_bytes, stats_buf,
                                stats_bytes, cfg, &lay);
  if (ck != KS_OK) return ck;
  // ---- the program image of that layout must fit the static array ----
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
  if (cudaMemcpyAsync(image, img.data(), img.size(), cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return KS_ERR_CUDA;

  ks::KsLaunch L;
  ks::fill_launch(*k, lay, image, grid, block, params, param_bytes, bufs, n_bufs, trace_buf, stats_buf, cfg, &L);
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

// ks_interp.cu — launchers of the interpreter kernel (ks_interp_kernel.cuh)
// for single launches, and the launch-totals reduction.

#include <map>
#include <mutex>
#include <tuple>

#include "ks_interp_kernel.cuh"

namespace ks {

// ---- launch-totals reduction -------------------------------------------------
// acc: [0] cycles max, [1] cycles sum, [2..9] counter sums, [10] failed warps,
// [11] max over failing warps of (2^64-1 - warp id), [12] max stack depth,
// [13] shared requests, [14] shared wavefronts.
__global__ void ks_reduce_kernel(const ks_warp_stats* __restrict__ s, uint64_t n,
                                 unsigned long long* __restrict__ acc) {
  unsigned long long v[15] = {0};
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
    v[13] += r.sh_req;
    v[14] += r.sh_wavefronts;
  }
#pragma unroll
  for (int k = 0; k < 15; k++) {
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long u = __shfl_down_sync(FULL, v[k], o);
      if (k == 0 || k == 11 || k == 12) v[k] = v[k] > u ? v[k] : u;
      else v[k] += u;
    }
  }
  if ((threadIdx.x & 31) == 0) {
#pragma unroll
    for (int k = 0; k < 15; k++) {
      if (k == 0 || k == 11 || k == 12) atomicMax(&acc[k], v[k]);
      else if (v[k]) atomicAdd(&acc[k], v[k]);
    }
  }
}

uint32_t interp_region0(uint32_t image_bytes) { return region0(image_bytes); }

size_t interp_smem_bytes(uint32_t image_bytes, uint32_t region_bytes, uint32_t warps, uint32_t shared_bytes) {
  return (size_t)region0(image_bytes) + (size_t)region_bytes * warps + (size_t)(shared_bytes + 15u) / 16u * 16u;
}

static int g_attr_done[64];

// The instantiation that runs a launch: CTA mode (9..32 warps: the 1024-thread
// form); the instrumented form for the cache model's passes and the
// per-instruction profile, and that form with the issue-run log for the SM
// issue model (the lean forms carry none of it).
template <bool CTA, bool BIG, bool CAP>
static const void* interp_fn_of(int form) {
  return form == 0   ? (const void*)ks_interp_kernel<CTA, BIG, false, false, 1u, CAP>
         : form == 1 ? (const void*)ks_interp_kernel<CTA, BIG, true, false, 1u, CAP>
                     : (const void*)ks_interp_kernel<CTA, BIG, true, true, 1u, CAP>;
}

static const void* interp_fn(bool cta, uint32_t real_warps_per_cta, int form, bool reg_capped, bool split,
                             bool greg = false) {
  if (greg) return interp_fn_greg(form);                // CTA mode, warp regions in global memory
  if (split) return interp_fn_split(form, reg_capped);  // plain mode only
  if (!cta) return reg_capped ? interp_fn_of<false, false, true>(form) : interp_fn_of<false, false, false>(form);
  if (real_warps_per_cta > 8) return interp_fn_of<true, true, false>(form);
  return reg_capped ? interp_fn_of<true, false, true>(form) : interp_fn_of<true, false, false>(form);
}

int interp_form(const KsLaunch& L) {
  if (L.sched_log != nullptr) return 2;
  return (L.cache_pass != 0 || L.profile != nullptr) ? 1 : 0;
}

static int form_of(const KsLaunch& L) { return interp_form(L); }

static int ensure_attr() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev < 64 && g_attr_done[dev]) return 0;
  int mx = 0;
  e = cudaDeviceGetAttribute(&mx, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return (int)e;
  for (int split = 0; split < 2; split++)
    for (int cta = 0; cta < 2; cta++)
      for (int big = 0; big < 2; big++)
        for (int capped = 0; capped < 2; capped++)
          for (int form = 0; form < 3; form++) {
            if (!cta && big) continue;
            if (big && capped) continue;
            if (split && cta) continue;
            e = cudaFuncSetAttribute(interp_fn(cta, big ? 32u : 1u, form, capped, split),
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
            if (e != cudaSuccess) return (int)e;
          }
  for (int form = 0; form < 3; form++) {
    e = cudaFuncSetAttribute(interp_fn_greg(form), cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
    if (e != cudaSuccess) return (int)e;
  }
  if (dev < 64) g_attr_done[dev] = 1;
  return 0;
}

// Resident CTAs per SM of one instantiation at one CTA size and shared-memory
// size, asked of the runtime once per device and remembered (the shape
// choice asks for several candidates at every launch).
int interp_occupancy(const KsLaunch& L, uint32_t real_warps_per_cta, size_t smem, int* ctas_per_sm,
                     bool reg_capped, bool greg) {
  int e = ensure_attr();
  if (e) return e;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return (int)cudaErrorInvalidDevice;
  const void* fn = interp_fn(L.cta_mode != 0, real_warps_per_cta, form_of(L), reg_capped, L.layout.split != 0, greg);
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, uint32_t, size_t>, int> known;
  const auto key = std::make_tuple(dev, fn, real_warps_per_cta, smem);
  {
    std::lock_guard<std::mutex> lk(mu);
    const auto it = known.find(key);
    if (it != known.end()) {
      *ctas_per_sm = it->second;
      return 0;
    }
  }
  e = (int)cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, fn, (int)(real_warps_per_cta * 32), smem);
  if (e) return e;
  std::lock_guard<std::mutex> lk(mu);
  known[key] = *ctas_per_sm;
  return 0;
}

size_t cta_mode_smem(const KsLaunch& L) {
  return interp_smem_bytes(L.image_bytes, L.layout.region_bytes, L.wpc, L.shared_bytes);
}

int choose_launch(const KsLaunch& L, int sms, int max_smem, LaunchShape* shape) {
  const uint64_t n_warps = L.n_warps;
  shape->greg = false;
  if (L.cta_mode) {
    // one real CTA per simulated CTA at a time, one real warp per simulated warp
    const size_t smem = cta_mode_smem(L);
    if (smem > (size_t)max_smem) {
      // the warps' state does not fit next to the simulated shared memory:
      // regions in global memory, the rest in shared memory
      const size_t smem_g = interp_smem_bytes(L.image_bytes, 0u, L.wpc, L.shared_bytes);
      if (smem_g > (size_t)max_smem) return KS_ERR_LIMIT;
      int per_sm = 0;
      if (interp_occupancy(L, L.wpc, smem_g, &per_sm, false, true)) return KS_ERR_CUDA;
      if (per_sm < 1) return KS_ERR_LIMIT;
      shape->warps_per_cta = L.wpc;
      shape->ctas = (uint32_t)std::min<uint64_t>(L.grid, (uint64_t)sms * (uint64_t)per_sm);
      shape->reg_capped = false;
      shape->greg = true;
      return KS_OK;
    }
    int per_sm = 0, per_sm_capped = 0;
    if (interp_occupancy(L, L.wpc, smem, &per_sm)) return KS_ERR_CUDA;
    // the register-capped form (blocks of up to 8 warps) where it holds
    // more CTAs
    if (L.wpc <= 8 && interp_occupancy(L, L.wpc, smem, &per_sm_capped, true)) return KS_ERR_CUDA;
    const bool capped = per_sm_capped > per_sm;
    if (capped) per_sm = per_sm_capped;
    if (per_sm < 1) return KS_ERR_LIMIT;
    shape->warps_per_cta = L.wpc;
    shape->ctas = (uint32_t)std::min<uint64_t>(L.grid, (uint64_t)sms * (uint64_t)per_sm);
    shape->reg_capped = capped;
    return KS_OK;
  }
  // Candidates: 1..12 real warps per CTA (one CTA of many warps holds one
  // program copy where large warp regions leave room for few CTAs). While
  // the simulated grid is small, keep at least two CTAs per SM so that every
  // SM gets work; among the rest
  // take the shape with the most resident real warps (shared memory,
  // registers and the CTA limit all count), then the larger CTA (fewer
  // program copies). The register-capped form (CTAs of up to 10 warps) is
  // taken only where it holds strictly more warps.
  uint32_t best_w = 0, best_ctas = 0;
  bool best_capped = false;
  uint64_t best_res = 0;
  bool any_fit = false;
  for (int capped = 0; capped < 2; capped++) {
    for (uint32_t w = 1; w <= (capped ? 10u : 12u); w++) {
      const size_t smem = interp_smem_bytes(L.image_bytes, L.layout.region_bytes, w, 0);
      if (smem > (size_t)max_smem) break;
      any_fit = true;
      const uint64_t want = (n_warps + w - 1) / w;
      if (w > 1 && want < 2ull * (uint64_t)sms) break;
      int per_sm = 0;
      const int e = interp_occupancy(L, w, smem, &per_sm, capped != 0);
      if (e) return KS_ERR_CUDA;
      if (per_sm < 1) continue;
      const uint64_t cap = (uint64_t)sms * (uint64_t)per_sm;
      const uint64_t res = std::min<uint64_t>(n_warps, cap * w);
      if (capped ? res > best_res : res >= best_res) {
        best_res = res;
        best_w = w;
        best_ctas = (uint32_t)std::min<uint64_t>(want, cap);
        best_capped = capped != 0;
      }
    }
  }
  if (!any_fit || best_w == 0) return KS_ERR_LIMIT;
  shape->warps_per_cta = best_w;
  shape->ctas = best_ctas;
  shape->reg_capped = best_capped;
  return KS_OK;
}

int launch_interp(const KsLaunch& L, const LaunchShape& shape, void* stream) {
  int e = ensure_attr();
  if (e) return e;
  const size_t smem = interp_smem_bytes(L.image_bytes, shape.greg ? 0u : L.layout.region_bytes, shape.warps_per_cta,
                                       L.cta_mode ? L.shared_bytes : 0u);
  KsGrid<1> G;
  G.n = 1;
  G.cta_begin[0] = 0;
  G.cta_begin[1] = shape.ctas;
  G.item[0] = L;
  void* scratch = nullptr;
  if (shape.greg) {  // the warp regions of every real CTA, for this launch only
    const size_t bytes = (size_t)shape.ctas * shape.warps_per_cta * L.layout.region_bytes;
    e = (int)cudaMallocAsync(&scratch, bytes, (cudaStream_t)stream);
    if (e) return e;
    G.item[0].greg = static_cast<uint8_t*>(scratch);
  }
  void* args[] = {&G};
  e = (int)cudaLaunchKernel(interp_fn(L.cta_mode != 0, shape.warps_per_cta, form_of(L), shape.reg_capped,
                                      L.layout.split != 0, shape.greg),
                            dim3(shape.ctas), dim3(shape.warps_per_cta * 32), args, smem, (cudaStream_t)stream);
  if (scratch) {
    const int f = (int)cudaFreeAsync(scratch, (cudaStream_t)stream);
    if (!e) e = f;
  }
  return e;
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

// ks_cache.cu — levels of the L1/L2 hit model, between the interpreter's two
// passes (KernelScope backend doc, simulator/engine.py — "Cache parameters"
// and SimpleCache: direct-mapped caches of 128-byte lines, set = line % lines,
// an access hits when its set holds the line, a miss installs it).
//
// A direct-mapped set's content after any prefix of its accesses is the line
// of the last one, so an access hits exactly when the access before it in
// the same set (in the global order) had the same line. The first pass logged
// every access (line, step) per warp; here the log is ordered by (L1 set,
// step, warp) with one radix sort, each access compared with its predecessor,
// and the L1 misses reordered by a stable sort on their L2 set's high part
// (line / l1_lines) % (l2_lines / l1_lines): as l1_lines divides l2_lines, an
// L2 set lies inside one L1 set, so the misses of one L2 set come out
// contiguous and still in (step, warp) order, and the same neighbour test
// gives the L2 hits.
#include <cub/device/device_radix_sort.cuh>
#include <cub/device/device_scan.cuh>
#include <cuda_runtime.h>

#include <algorithm>

#include "ks_internal.h"

namespace ks {
namespace {

constexpr uint64_t NO_KEY = ~0ull;

__host__ __device__ inline uint32_t bits_for(uint64_t max_value) {  // bits to hold 0..max_value
  uint32_t b = 0;
  while (b < 64 && (max_value >> b) != 0) b++;
  return b;
}

inline uint64_t align256(uint64_t x) { return (x + 255u) / 256u * 256u; }

// Records each warp logged (its count, at most the log's capacity).
__global__ void cache_logged_kernel(const ks_cache_warp* __restrict__ warps, uint64_t n_warps, uint32_t cap,
                                    uint32_t* __restrict__ logged) {
  for (uint64_t w = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; w < n_warps;
       w += (uint64_t)gridDim.x * blockDim.x)
    logged[w] = min(warps[w].n_access, cap);
}

// The logged records packed densely (warp w's at offsets[w]): key (L1 set,
// step, warp) packed from the top, value the record's log index. One real
// warp per simulated warp's records.
__global__ void cache_keys_kernel(const uint32_t* __restrict__ logged, const uint32_t* __restrict__ offsets,
                                  const ks_cache_access* __restrict__ log, uint64_t n_warps, uint32_t cap,
                                  uint32_t l1_lines, uint32_t warp_bits, uint64_t* __restrict__ keys,
                                  uint32_t* __restrict__ vals) {
  const uint64_t lane = threadIdx.x & 31u;
  for (uint64_t w = ((uint64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; w < n_warps;
       w += ((uint64_t)gridDim.x * blockDim.x) >> 5) {
    const uint32_t n = logged[w], off = offsets[w];
    for (uint32_t k = (uint32_t)lane; k < n; k += 32) {
      const uint64_t i = w * cap + k;
      const ks_cache_access a = log[i];
      keys[off + k] = ((a.line % l1_lines) << (32 + warp_bits)) | ((uint64_t)a.step << warp_bits) | w;
      vals[off + k] = (uint32_t)i;
    }
  }
}

// L1: hit when the previous access of the set had the same line. Misses get
// the sort key of their L2 set's high part; hits go last.
__global__ void cache_l1_kernel(const uint64_t* __restrict__ keys, const uint32_t* __restrict__ vals, uint64_t n,
                                ks_cache_access* __restrict__ log, uint32_t l1_lines, uint32_t n_l2_parts,
                                uint32_t* __restrict__ keys2) {
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
    uint32_t k2 = n_l2_parts;  // after every real part
    if (keys[i] != NO_KEY) {
      const uint64_t line = log[vals[i]].line;
      const bool hit = i > 0 && keys[i - 1] != NO_KEY && log[vals[i - 1]].line == line;
      if (hit) {
        log[vals[i]].level = KS_CACHE_L1_HIT;
      } else {
        log[vals[i]].level = KS_CACHE_DRAM;
        k2 = (uint32_t)((line / l1_lines) % n_l2_parts);
      }
    }
    keys2[i] = k2;
  }
}

// L2 over the L1 misses, ordered by (L2 part, L1 set, step, warp).
__global__ void cache_l2_kernel(const uint32_t* __restrict__ keys2, const uint32_t* __restrict__ vals, uint64_t n,
                                ks_cache_access* __restrict__ log, uint32_t n_l2_parts) {
  for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (uint64_t)gridDim.x * blockDim.x) {
    const uint32_t k2 = keys2[i];
    if (k2 == n_l2_parts) continue;
    const uint64_t line = log[vals[i]].line;
    if (i > 0 && keys2[i - 1] == k2 && log[vals[i - 1]].line == line) log[vals[i]].level = KS_CACHE_L2_HIT;
  }
}

unsigned grid_for(uint64_t n) {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  uint64_t blocks = (n + 255) / 256;
  const uint64_t cap = (uint64_t)(sms > 0 ? sms : 1) * 8;
  if (blocks > cap) blocks = cap;
  return (unsigned)(blocks ? blocks : 1);
}

}  // namespace

int cache_layout(uint64_t n_warps, uint32_t cap, uint32_t max_runs, CacheLayout* out) {
  const uint64_t n = n_warps * (uint64_t)cap;
  if (n == 0 || n >= (1ull << 31)) return KS_ERR_ARG;
  size_t t1 = 0, t2 = 0, t3 = 0;
  if (cub::DeviceRadixSort::SortPairs(nullptr, t1, (const uint64_t*)nullptr, (uint64_t*)nullptr,
                                      (const uint32_t*)nullptr, (uint32_t*)nullptr, (int)n) != cudaSuccess)
    return KS_ERR_CUDA;
  if (cub::DeviceRadixSort::SortPairs(nullptr, t2, (const uint32_t*)nullptr, (uint32_t*)nullptr,
                                      (const uint32_t*)nullptr, (uint32_t*)nullptr, (int)n) != cudaSuccess)
    return KS_ERR_CUDA;
  if (cub::DeviceScan::ExclusiveSum(nullptr, t3, (const uint32_t*)nullptr, (uint32_t*)nullptr, (int)n_warps + 1) !=
      cudaSuccess)
    return KS_ERR_CUDA;
  CacheLayout C;
  C.warps_off = 0;
  C.log_off = align256(n_warps * sizeof(ks_cache_warp));
  C.logged_off = C.log_off + align256(n * sizeof(ks_cache_access));
  C.offsets_off = C.logged_off + align256((n_warps + 1) * 4);
  C.keys_a = C.offsets_off + align256((n_warps + 1) * 4);
  C.keys_b = C.keys_a + align256(n * 8);
  C.vals_a = C.keys_b + align256(n * 8);
  C.vals_b = C.vals_a + align256(n * 4);
  C.temp_off = C.vals_b + align256(n * 4);
  C.temp_bytes = align256(std::max(std::max(t1, t2), t3));
  C.runs_off = C.temp_off + C.temp_bytes;
  C.runlog_off = C.runs_off + (max_runs ? align256(n_warps * 4) : 0);
  const uint64_t nr = n_warps * (uint64_t)max_runs;
  if (nr >= (1ull << 34)) return KS_ERR_ARG;
  C.total = C.runlog_off + align256(nr * 4);
  *out = C;
  return KS_OK;
}

int launch_cache_levels(const KsLaunch& L, uint8_t* ws, const CacheLayout& C, uint32_t l1_lines, uint32_t l2_lines,
                        void* stream_v, uint32_t* own_kernels) {
  cudaStream_t stream = (cudaStream_t)stream_v;
  const uint64_t W = L.n_warps;
  const uint32_t warp_bits = bits_for(W - 1u);
  const uint32_t key_bits = bits_for(l1_lines - 1u) + 32u + warp_bits;
  const uint32_t n_parts = l2_lines / l1_lines;
  uint32_t* logged = reinterpret_cast<uint32_t*>(ws + C.logged_off);
  uint32_t* offsets = reinterpret_cast<uint32_t*>(ws + C.offsets_off);
  uint64_t* keys_a = reinterpret_cast<uint64_t*>(ws + C.keys_a);
  uint64_t* keys_b = reinterpret_cast<uint64_t*>(ws + C.keys_b);
  uint32_t* vals_a = reinterpret_cast<uint32_t*>(ws + C.vals_a);
  uint32_t* vals_b = reinterpret_cast<uint32_t*>(ws + C.vals_b);
  // the second sort's u32 keys reuse the first sort's key buffers
  uint32_t* keys2_a = reinterpret_cast<uint32_t*>(ws + C.keys_a);
  uint32_t* keys2_b = reinterpret_cast<uint32_t*>(ws + C.keys_b);
  void* temp = ws + C.temp_off;
  size_t temp_bytes = C.temp_bytes;

  // per-warp record counts, their exclusive prefix (offsets[W] = the total),
  // and the total on the host: the sorts run over the logged records only
  cache_logged_kernel<<<grid_for(W), 256, 0, stream>>>(L.cache_warps, W, L.cache_cap, logged);
  if (own_kernels) *own_kernels += 1;
  cudaError_t e = cudaMemsetAsync(logged + W, 0, 4, stream);
  if (e != cudaSuccess) return (int)e;
  e = cub::DeviceScan::ExclusiveSum(temp, temp_bytes, logged, offsets, (int)W + 1, stream);
  if (e != cudaSuccess) return (int)e;
  uint32_t total = 0;
  e = cudaMemcpyAsync(&total, offsets + W, 4, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return (int)e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return (int)e;
  if (total == 0) return 0;
  if (own_kernels) *own_kernels += 3;
  const uint64_t n = total;
  const unsigned g = grid_for(n);

  cache_keys_kernel<<<grid_for(W * 32), 256, 0, stream>>>(logged, offsets, L.cache_log, W, L.cache_cap, l1_lines,
                                                          warp_bits, keys_a, vals_a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return (int)e;
  e = cub::DeviceRadixSort::SortPairs(temp, temp_bytes, keys_a, keys_b, vals_a, vals_b, (int)n, 0, (int)key_bits,
                                      stream);
  if (e != cudaSuccess) return (int)e;
  cache_l1_kernel<<<g, 256, 0, stream>>>(keys_b, vals_b, n, L.cache_log, l1_lines, n_parts, keys2_a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return (int)e;
  e = cub::DeviceRadixSort::SortPairs(temp, temp_bytes, keys2_a, keys2_b, vals_b, vals_a, (int)n, 0,
                                      (int)bits_for(n_parts), stream);
  if (e != cudaSuccess) return (int)e;
  cache_l2_kernel<<<g, 256, 0, stream>>>(keys2_b, vals_a, n, L.cache_log, n_parts);
  return (int)cudaGetLastError();
}

}  // namespace ks

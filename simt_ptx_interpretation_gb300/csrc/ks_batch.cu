// ks_batch.cu — one real grid over several simulated launches
// (ks_simulate_batch).
//
// A simulated launch of a few hundred warps leaves most of the GPU idle (one
// simulated warp per real warp, a real warp per SM sub-partition or fewer),
// and a launch of many warps ends in a tail where its slowest warps run alone.
// A batch gives every item a range of the real grid's CTAs; each real CTA
// runs its item exactly as a single launch would run it on a grid of that
// range's size (ks_interp_kernel.cuh, NB = KS_BATCH_ITEMS), so results do
// not depend on the batching. The items of one real grid share the kernel
// instantiation: the same mode, form and layout, and in CTA mode the same
// block.

#include "ks_interp_kernel.cuh"

namespace ks {

namespace {

constexpr uint32_t NB = KS_BATCH_ITEMS;

template <bool CTA, bool BIG>
const void* batch_fn_of(int form) {
  return form == 0   ? (const void*)ks_interp_kernel<CTA, BIG, false, false, NB>
         : form == 1 ? (const void*)ks_interp_kernel<CTA, BIG, true, false, NB>
                     : (const void*)ks_interp_kernel<CTA, BIG, true, true, NB>;
}

const void* batch_fn(bool cta, uint32_t real_warps_per_cta, int form, bool split) {
  if (split) return batch_fn_split(form);  // plain mode only
  if (!cta) return batch_fn_of<false, false>(form);
  if (real_warps_per_cta > 8) return batch_fn_of<true, true>(form);
  return batch_fn_of<true, false>(form);
}

int g_batch_attr_done[64];

int ensure_batch_attr() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev < 64 && g_batch_attr_done[dev]) return 0;
  int mx = 0;
  e = cudaDeviceGetAttribute(&mx, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return (int)e;
  for (int split = 0; split < 2; split++)
    for (int cta = 0; cta < 2; cta++)
      for (int big = 0; big < 2; big++)
        for (int form = 0; form < 3; form++) {
          if (!cta && big) continue;
          if (split && cta) continue;
          e = cudaFuncSetAttribute(batch_fn(cta, big ? 32u : 1u, form, split),
                                   cudaFuncAttributeMaxDynamicSharedMemorySize, mx);
          if (e != cudaSuccess) return (int)e;
        }
  if (dev < 64) g_batch_attr_done[dev] = 1;
  return 0;
}

int occupancy(bool cta, uint32_t w, int form, bool split, size_t smem, int* per_sm) {
  *per_sm = 0;
  return (int)cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, batch_fn(cta, w, form, split), (int)(w * 32u),
                                                            smem);
}

// Shared memory of a real CTA of w warps that may run any item.
size_t batch_smem(const KsGrid<NB>& G, uint32_t w) {
  size_t m = 0;
  for (uint32_t i = 0; i < G.n; i++) {
    const KsLaunch& L = G.item[i];
    m = std::max(m, interp_smem_bytes(L.image_bytes, L.layout.region_bytes, w, L.cta_mode ? L.shared_bytes : 0u));
  }
  return m;
}

}  // namespace

int launch_batch(KsGrid<NB>* Gp, int sms, int max_smem, void* stream) {
  KsGrid<NB>& G = *Gp;
  if (G.n == 0 || G.n > NB || sms < 1) return KS_ERR_ARG;
  const KsLaunch& L0 = G.item[0];
  const bool cta = L0.cta_mode != 0;
  const int form = interp_form(L0);
  const bool split = L0.layout.split != 0;
  for (uint32_t i = 1; i < G.n; i++) {
    const KsLaunch& L = G.item[i];
    if ((L.cta_mode != 0) != cta || interp_form(L) != form || (L.layout.split != 0) != split ||
        (cta && L.wpc != L0.wpc))
      return KS_ERR_ARG;
  }
  int e = ensure_batch_attr();
  if (e) return KS_ERR_CUDA;

  // units an item's CTAs share out: simulated warps (plain mode) or
  // simulated CTAs (CTA mode); useful = the most real CTAs an item can use
  uint64_t units[NB], useful[NB], total = 0;
  uint32_t w = 0;
  uint64_t ctas = 0;
  size_t smem = 0;
  if (cta) {
    w = L0.wpc;
    smem = batch_smem(G, w);
    if (smem > (size_t)max_smem) return KS_ERR_LIMIT;
    int per_sm = 0;
    if (occupancy(true, w, form, split, smem, &per_sm)) return KS_ERR_CUDA;
    if (per_sm < 1) return KS_ERR_LIMIT;
    for (uint32_t i = 0; i < G.n; i++) total += units[i] = useful[i] = G.item[i].grid;
    ctas = std::min<uint64_t>(total, (uint64_t)sms * (uint64_t)per_sm);
  } else {
    for (uint32_t i = 0; i < G.n; i++) total += units[i] = G.item[i].n_warps;
    // Every simulated warp resident at once if it fits: k CTAs of w warps
    // on each SM, k * w >= the simulated warps per SM, the grid a multiple
    // of the SM count so that every SM gets the same share.
    const uint64_t m = (total + (uint64_t)sms - 1) / (uint64_t)sms;
    const uint64_t k = (m + 7) / 8;
    if (k <= 32) {
      const uint32_t wk = (uint32_t)((m + k - 1) / k);
      const size_t s = batch_smem(G, wk);
      int per_sm = 0;
      if (s <= (size_t)max_smem) {
        if (occupancy(false, wk, form, split, s, &per_sm)) return KS_ERR_CUDA;
        if ((uint64_t)per_sm >= k) {
          w = wk;
          smem = s;
          ctas = k * (uint64_t)sms;
        }
      }
    }
    if (w == 0) {
      // persistent: the shape with the most resident real warps (then the
      // larger CTA), every CTA of it resident
      uint64_t best_res = 0;
      for (uint32_t c = 1; c <= 8; c++) {
        const size_t s = batch_smem(G, c);
        if (s > (size_t)max_smem) break;
        int per_sm = 0;
        if (occupancy(false, c, form, split, s, &per_sm)) return KS_ERR_CUDA;
        if (per_sm < 1) continue;
        const uint64_t cap = (uint64_t)sms * (uint64_t)per_sm;
        const uint64_t res = std::min<uint64_t>(total, cap * c);
        if (res >= best_res) {
          best_res = res;
          w = c;
          smem = s;
          ctas = std::min<uint64_t>(cap, (total + c - 1) / c);
        }
      }
      if (w == 0) return KS_ERR_LIMIT;
    }
    for (uint32_t i = 0; i < G.n; i++) useful[i] = (units[i] + w - 1) / w;
  }

  // Share the CTAs out in proportion to the units (at least one each, at
  // most what an item can use), the remainder one by one to the item with
  // the most units per CTA.
  uint64_t alloc[NB], given = 0;
  for (uint32_t i = 0; i < G.n; i++) {
    alloc[i] = std::max<uint64_t>(1, std::min<uint64_t>(useful[i], ctas * units[i] / std::max<uint64_t>(total, 1)));
    given += alloc[i];
  }
  while (given < ctas) {
    int best = -1;
    for (uint32_t i = 0; i < G.n; i++) {
      if (alloc[i] >= useful[i]) continue;
      if (best < 0 || units[i] * alloc[best] > units[best] * alloc[i]) best = (int)i;
    }
    if (best < 0) break;
    alloc[best]++;
    given++;
  }
  if (given > 0xFFFFFFFFull) return KS_ERR_LIMIT;
  G.cta_begin[0] = 0;
  for (uint32_t i = 0; i < G.n; i++) G.cta_begin[i + 1] = G.cta_begin[i] + (uint32_t)alloc[i];
  void* args[] = {Gp};
  return cudaLaunchKernel(batch_fn(cta, w, form, split), dim3(G.cta_begin[G.n]), dim3(w * 32u), args, smem,
                          (cudaStream_t)stream) == cudaSuccess
             ? KS_OK
             : KS_ERR_CUDA;
}

}  // namespace ks

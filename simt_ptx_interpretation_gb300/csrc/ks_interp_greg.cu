// ks_interp_greg.cu — the CTA-mode instantiations of the interpreter kernel
// (ks_interp_kernel.cuh) whose warp regions live in global memory, for
// kernels with shared memory or bar.sync whose CTA's warp state does not fit
// an SM's shared memory next to its simulated shared memory (lean,
// instrumented and issue-logging forms; single launches). Compiled apart so
// that the build stays parallel.

#include "ks_interp_kernel.cuh"

namespace ks {

const void* interp_fn_greg(int form) {
  return form == 0   ? (const void*)ks_interp_kernel<true, true, false, false, 1u, false, false, true>
         : form == 1 ? (const void*)ks_interp_kernel<true, true, true, false, 1u, false, false, true>
                     : (const void*)ks_interp_kernel<true, true, true, true, 1u, false, false, true>;
}

}  // namespace ks

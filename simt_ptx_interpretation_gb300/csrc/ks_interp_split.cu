// ks_interp_split.cu — the SPLIT-layout instantiations of the interpreter
// kernel (ks_interp_kernel.cuh): plain mode, single launches (lean,
// instrumented and issue-logging forms, with and without the register cap)
// and batches. Compiled apart from ks_interp.cu and ks_batch.cu so that the
// build stays parallel.

#include "ks_interp_kernel.cuh"

namespace ks {

namespace {

template <uint32_t NB, bool CAP>
const void* split_fn_of(int form) {
  return form == 0   ? (const void*)ks_interp_kernel<false, false, false, false, NB, CAP, true>
         : form == 1 ? (const void*)ks_interp_kernel<false, false, true, false, NB, CAP, true>
                     : (const void*)ks_interp_kernel<false, false, true, true, NB, CAP, true>;
}

}  // namespace

const void* interp_fn_split(int form, bool reg_capped) {
  return reg_capped ? split_fn_of<1u, true>(form) : split_fn_of<1u, false>(form);
}

const void* batch_fn_split(int form) { return split_fn_of<KS_BATCH_ITEMS, false>(form); }

}  // namespace ks

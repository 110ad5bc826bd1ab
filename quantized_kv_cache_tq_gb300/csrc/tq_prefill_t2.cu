// turbo2 instantiation of the tcgen05 inline-dequant prefill kernel.
#include "tq_prefill.cuh"

namespace tq {
cudaError_t launch_prefill_t2(const PrefillArgs &a, cudaStream_t s) { return pf::launch_type<2>(a, s); }
}  // namespace tq

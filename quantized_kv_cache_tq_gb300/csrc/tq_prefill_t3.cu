// turbo3 instantiation of the tcgen05 inline-dequant prefill kernel.
#include "tq_prefill.cuh"

namespace tq {
cudaError_t launch_prefill_t3(const PrefillArgs &a, cudaStream_t s) { return pf::launch_type<3>(a, s); }
}  // namespace tq

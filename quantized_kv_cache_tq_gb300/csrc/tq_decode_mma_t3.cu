// turbo3 instantiation of the tensor-core decode kernel.
#include "tq_decode_mma.cuh"

namespace tq {
cudaError_t launch_decode_mma_t3(const DecodeArgs &a, cudaStream_t s) { return mmadec::launch_type<3>(a, s); }
}  // namespace tq

// turbo4 instantiation of the tensor-core decode kernel.
#include "tq_decode_mma.cuh"

namespace tq {
cudaError_t launch_decode_mma_t4(const DecodeArgs &a, cudaStream_t s) { return mmadec::launch_type<4>(a, s); }
}  // namespace tq

// Dispatch of the tensor-core decode (kernel in tq_decode_mma.cuh; one
// translation unit per code type so they compile in parallel).
#include "tq_internal.h"

namespace tq {

// group: query heads per KV head (any size; see mma_group)
bool decode_mma_supported(int ktype, int vtype, int group, int nbk, int nbv) {
  if (ktype != vtype || group < 1) return false;
  return (nbk == 1 && nbv == 1) || (nbk == 2 && (nbv == 1 || nbv == 2));
}

// a.group: query heads per launch head (1, 2 or 4)
cudaError_t launch_decode_mma(int ktype, int vtype, const DecodeArgs &a, cudaStream_t s) {
  if (mma_group(a.group) != a.group || !decode_mma_supported(ktype, vtype, a.group, a.nbk, a.nbv))
    return cudaErrorNotSupported;
  switch (ktype) {
    case TQ_TURBO2: return launch_decode_mma_t2(a, s);
    case TQ_TURBO3: return launch_decode_mma_t3(a, s);
    default: return launch_decode_mma_t4(a, s);
  }
}

}  // namespace tq

// Dispatch of the tcgen05 prefill kernel (tq_prefill.cuh; one translation unit
// per code type so they compile in parallel).
#include "tq_internal.h"

namespace tq {

cudaError_t launch_prefill_t2(const PrefillArgs &a, cudaStream_t s);
cudaError_t launch_prefill_t3(const PrefillArgs &a, cudaStream_t s);
cudaError_t launch_prefill_t4(const PrefillArgs &a, cudaStream_t s);

bool prefill_supported(int ktype, int vtype, int group, int nbk, int nbv) {
  if (ktype != vtype) return false;
  if (group <= 0 || group > 128 || (group & (group - 1)) != 0) return false;   // power of two
  return (nbk == 1 && nbv == 1) || (nbk == 2 && (nbv == 1 || nbv == 2));
}

cudaError_t launch_prefill(int ktype, const PrefillArgs &a, cudaStream_t s) {
  switch (ktype) {
    case TQ_TURBO2: return launch_prefill_t2(a, s);
    case TQ_TURBO3: return launch_prefill_t3(a, s);
    default: return launch_prefill_t4(a, s);
  }
}

}  // namespace tq

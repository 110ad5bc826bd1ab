// Decode entry point that allocates nothing and needs no caller workspace.
//
// Some callers cannot allocate device memory at the point where they call
// decode: code running inside a custom allocator or memory-pool callback, a
// runtime that forbids cudaMalloc once it has reserved all device memory, or a
// plugin host that only hands out input and output buffers.  For them the split
// partials, the split counters and the status word live in one fixed array in
// the library's own device memory.
//
// Properties callers must know:
//   - The array holds kNoAllocScratchBytes (4 MiB).  Every GPU that loads the
//     library keeps that much device memory reserved until the process exits.
//   - Shapes whose decode workspace would exceed it are rejected with
//     TQ_ERR_WORKSPACE before anything is launched.
//   - The first call on each device looks up the array's device address (with
//     that device current).  Make that first call before any stream capture.
//   - All calls share the array and it keeps the last call's contents.  Each call
//     clears the split counters itself (cudaMemsetAsync on the caller's stream,
//     after its argument checks).  The status word at the start of the array
//     collects the first device-side error (e.g. a bounded wait that timed out)
//     until tq_noalloc_status reads and clears it.  Calls that overlap on the
//     GPU, on different streams, race on the array and produce wrong results.
#include <atomic>

#include "tq_internal.h"

namespace tq {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;

// Host code must not use this symbol as a device address: it names a host-side
// stand-in.  The device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

static std::atomic<void *> g_scratch_ptr[64];

// Device address of the scratch array on the current device (looked up once per device).
static cudaError_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  void *p = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (!p) {
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev].store(p, std::memory_order_release);
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace tq

using namespace tq;

extern "C" tq_status tq_fattn_decode_noalloc(const tq_cache *k, const tq_cache *v, const tq_codebook *cbk,
                                              const tq_codebook *cbv, const float *q, int n_q_heads,
                                              int64_t kv_len, float scale, int algo, float *out,
                                              tq_stream stream) {
  const size_t need = tq_fattn_decode_workspace(k, v, n_q_heads, kv_len);
  if (need == 0) return TQ_ERR_INVALID_ARG;
  if (need > kNoAllocScratchBytes) return TQ_ERR_WORKSPACE;
  void *ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) {
    cudaGetLastError();
    return TQ_ERR_CUDA;
  }
  // the counters start at zero: they are cleared on the stream once every argument
  // has passed its check, just before the kernel; the epochs carry on from call to
  // call and the status word keeps the first device-side error until
  // tq_noalloc_status reads it
  return decode_counters_cleared(k, v, cbk, cbv, q, n_q_heads, kv_len, scale, algo, out, ws,
                                 kNoAllocScratchBytes, stream);
}

extern "C" tq_status tq_noalloc_status(int32_t *status_out, tq_stream stream) {
  if (!status_out) return TQ_ERR_INVALID_ARG;
  void *ws = nullptr;
  if (scratch_address(&ws) != cudaSuccess) {
    cudaGetLastError();
    return TQ_ERR_CUDA;
  }
  return tq_workspace_status(ws, kNoAllocScratchBytes, status_out, stream);
}

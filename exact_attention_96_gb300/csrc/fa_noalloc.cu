// fa_noalloc.cu -- fa_bwd_noalloc: the backward pass for callers that cannot allocate
// device memory.
//
// fa_bwd needs a caller-provided workspace (D, LSE*log2e and the fp32 dQ accumulator).
// Some callers cannot obtain one: embedders whose device memory is wholly owned by another
// allocator they cannot call from here, and code that must not trigger the implicit device
// synchronisation a cudaMalloc/cudaFree can cause.  For them this entry point uses a fixed
// scratch array that lives in the library's static device memory instead: it allocates
// nothing and frees nothing.
//
// The array is FA_NOALLOC_SCRATCH_BYTES (64 MiB) on every device that loads the library
// and stays allocated until the process exits.  Host code cannot use the array's name as a
// device address, so the first call on each device (with that device current) looks the
// address up with cudaGetSymbolAddress and caches it for later calls.  All calls share the
// one array: calls that overlap on the GPU (different streams, or several host threads
// without ordering) race on it and give undefined results.  The array keeps the previous call's contents; everything that must
// start at zero (the dQ accumulator) is cleared by the backward pass itself on every call.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include "fa_internal.h"

namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

}  // namespace

extern "C" fa_status fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o,
                                    const void* dout, const float* lse, void* dq, void* dk, void* dv,
                                    int B, int H, int N, int d, float scale, int causal,
                                    fa_stream_t stream) {
  const fa_status sizes = fa::check_problem_sizes(B, H, N, d);
  if (sizes != FA_OK) return sizes;
  if (fa_bwd_workspace_bytes(B, H, N, d) > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return FA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return FA_ERR_CUDA;
      g_scratch_ptr[dev] = p;
    }
    scratch = g_scratch_ptr[dev];
  }
  return fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, B, H, N, d, scale, causal, scratch,
                FA_NOALLOC_SCRATCH_BYTES, stream);
}

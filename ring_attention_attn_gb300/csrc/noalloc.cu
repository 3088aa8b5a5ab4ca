// factored_attn_static: factored video attention for callers that may not
// allocate device memory (their device memory belongs to a pool set up at
// start-up, or an allocation and its implicit synchronisation are not allowed
// where they call us).  The scratch factored_attn asks its caller for lives
// here instead, in a fixed array compiled into the library.
#include <stdint.h>

#include <mutex>

#include "ra_internal.h"
#include "ringattn.h"

namespace {

// The scratch: RA_STATIC_SCRATCH_BYTES on every device that loads the
// library, held until the process exits.  In host code this name is only a
// host-side stand-in for the symbol, never a device address: kernels get the
// address that cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_factored_scratch[RA_STATIC_SCRATCH_BYTES];

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.  nullptr on failure, with the
// CUDA error recorded.  The runtime loads the library's device code lazily,
// so this first lookup is also where the array is placed in device memory.
// The cache is never refreshed: after cudaDeviceReset (or the primary context
// being torn down) the cached address is stale, which the header states.
void *scratch_on_current_device() {
  static void *addr[64] = {};
  static std::mutex mu;
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    ra::record_cuda_error(e);
    return nullptr;
  }
  if (dev < 0 || dev >= 64) {
    ra::record_cuda_error(cudaErrorInvalidDevice);
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_factored_scratch);
    if (e != cudaSuccess || p == nullptr) {
      ra::record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" int factored_attn_static(const void *q, const void *k, const void *v, void *out_s,
                                    float *lse_s, void *out_t, float *lse_t, int B, int H, int T,
                                    int N, int d, int P, void *stream) {
  // Sizes beyond the fixed scratch are refused before anything runs.  The
  // count is the one this P needs: chunks of up to 128 frames use no scratch
  // whatever T is.  (Invalid sizes count 0 here; factored_attn then reports
  // the argument error itself.)
  const size_t need = ra::factored_scratch_bytes(B, H, T, N, d, P);
  if (need > RA_STATIC_SCRATCH_BYTES) return RA_ERR_WORKSPACE;
  // Sizes that need no scratch do not look the array up, so they never make
  // the runtime place it in device memory.
  void *ws = nullptr;
  if (need > 0) {
    ws = scratch_on_current_device();
    if (ws == nullptr) return RA_ERR_CUDA;
  }
  // Every scratch byte factored_attn reads it has first written in the same
  // call, so nothing is cleared here.
  return factored_attn(q, k, v, out_s, lse_s, out_t, lse_t, B, H, T, N, d, P, ws,
                       need > 0 ? RA_STATIC_SCRATCH_BYTES : 0, stream);
}

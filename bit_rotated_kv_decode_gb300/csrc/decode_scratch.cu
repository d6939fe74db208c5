// Fixed, statically allocated decode scratch for oscar_decode_attention_noalloc:
// q_rot and the partials of the decode kernels.
//
// Some callers cannot allocate device memory around a decode step: a serving
// engine that hands all free HBM to its KV pools at start-up and owns no
// allocator it may call per step, or a plain C host that has no allocator to
// pass at all.  For them q_rot and the partials of the decode kernels
// live in one file-scope device array, loaded with the module, instead of a
// caller-owned workspace.  Nothing here calls cudaMalloc, cudaFree or any
// library routine that allocates.
//
// The array is one per device.  Set-up, once per device with that device
// current, takes its address with cudaGetSymbolAddress and zeroes it on the
// caller's stream (the decode itself needs no initial contents).  Two calls
// that use the array at the same time on one device -- on different streams,
// or from different caches -- race.
#include <mutex>

#include "internal.h"

static __device__ __align__(256) unsigned char g_decode_scratch[oscar::DECODE_SCRATCH_BYTES];

namespace oscar {
namespace {

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
void* g_addr[MAX_DEVICES] = {};

}  // namespace

cudaError_t decode_scratch_address(void** ptr, cudaStream_t s) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(p, 0, DECODE_SCRATCH_BYTES, s);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *ptr = g_addr[dev];
  return cudaSuccess;
}

}  // namespace oscar

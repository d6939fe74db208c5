// Fixed, statically allocated decode scratch for oscar_decode_attention_noalloc:
// the partial records (o, m, l per query head) of the decode kernel.
//
// Some callers cannot allocate device memory around a decode step: a serving
// engine that hands all free HBM to its KV pools at start-up and owns no
// allocator it may call per step, or a plain C host that has no allocator to
// pass at all.  For them the partial records of the decode kernel live in one
// file-scope device array, loaded with the module, instead of a
// caller-owned workspace.  Nothing here calls cudaMalloc, cudaFree or any
// library routine that allocates.
//
// The array is one per device.  Every call takes its address afresh with
// cudaGetSymbolAddress (with the caller's device current), so a module that was
// reloaded -- after cudaDeviceReset, say -- is never reached through a stale
// pointer.  The first call on a device also zeroes the array on the caller's
// stream; the decode needs no initial contents, so a reload that leaves other
// contents does no harm.  Two calls that use the array at the same time on one
// device -- on different streams, or from different caches -- race.
#include <mutex>

#include "internal.h"

static __device__ __align__(256) unsigned char g_decode_scratch[oscar::DECODE_SCRATCH_BYTES];

namespace oscar {
namespace {

constexpr int MAX_DEVICES = 64;
std::mutex g_mu;
bool g_zeroed[MAX_DEVICES] = {};

}  // namespace

cudaError_t decode_scratch_address(void** ptr, cudaStream_t s) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_decode_scratch);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_zeroed[dev]) {
    e = cudaMemsetAsync(p, 0, DECODE_SCRATCH_BYTES, s);
    if (e != cudaSuccess) return e;
    g_zeroed[dev] = true;
  }
  *ptr = p;
  return cudaSuccess;
}

}  // namespace oscar

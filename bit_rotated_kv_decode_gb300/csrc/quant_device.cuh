// Device-side INT2 quantiser of one 128-channel token-head group.
//
// Write path of "Together AI Open-Sources OSCAR" (MarkTechPost), section "The
// Serving System: Mixed-Precision Cache Layout": rotate, clip to the stored
// threshold, per-token asymmetric INT2 with a scale and a zero point ("scale /
// zero point" in "TogetherAI开源OSCAR" (ModelScope), section "OSCAR的设计"),
// four codes per byte.  Every decision is taken in IEEE fp32 / fp16
// round-to-nearest-even arithmetic:
//   xc = clip(x, -tau, tau) + 0          (signed zero canonicalised to +0)
//   z  = fp16_rn(min xc)
//   s  = fp16_rn(fl32(fl32(max xc - min xc) / 3))
//   code = clamp(rint(fl32(fl32(xc - z) / s)), 0, 3), 0 when s == 0
#pragma once

#include <cuda_fp16.h>

#include "internal.h"

namespace oscar {

struct GroupCode {
  uint32_t byte;      // packed codes of this lane's 4 channels
  uint16_t s_bits;    // fp16 scale
  uint16_t z_bits;    // fp16 zero point
};

__device__ __forceinline__ float clip_canon(float x, float tau) {
  return __fadd_rn(fminf(fmaxf(x, -tau), tau), 0.0f);
}

__device__ __forceinline__ uint32_t code_of(float xc, float z, float s) {
  const float t = __fdiv_rn(__fsub_rn(xc, z), s);
  const float r = fminf(fmaxf(rintf(t), 0.0f), 3.0f);
  return static_cast<uint32_t>(r);
}

// A full warp holds the group: lane l owns channels 4l .. 4l+3 (already
// rotated, not yet clipped).  Every lane returns its packed byte and the
// group's (s, z).
__device__ __forceinline__ GroupCode quantize_group_warp(float4 x, float tau) {
  x.x = clip_canon(x.x, tau);
  x.y = clip_canon(x.y, tau);
  x.z = clip_canon(x.z, tau);
  x.w = clip_canon(x.w, tau);
  float mn = fminf(fminf(x.x, x.y), fminf(x.z, x.w));
  float mx = fmaxf(fmaxf(x.x, x.y), fmaxf(x.z, x.w));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  const __half zh = __float2half_rn(mn);
  const float z = __half2float(zh);
  const float r = __fdiv_rn(__fsub_rn(mx, mn), 3.0f);
  const __half sh = __float2half_rn(r);
  const float s = __half2float(sh);
  GroupCode g;
  g.byte = 0;
  if (s != 0.0f) {
    g.byte = code_of(x.x, z, s) | (code_of(x.y, z, s) << 2) | (code_of(x.z, z, s) << 4) |
             (code_of(x.w, z, s) << 6);
  }
  g.s_bits = __half_as_ushort(sh);
  g.z_bits = __half_as_ushort(zh);
  return g;
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

}  // namespace oscar

// Device-side INT2 quantiser of one 128-channel token-head group.
//
// Write path of "Together AI Open-Sources OSCAR" (MarkTechPost), section "The
// Serving System: Mixed-Precision Cache Layout": rotate, clip to the stored
// threshold, per-token asymmetric INT2 with a scale and a zero point ("scale /
// zero point" in "TogetherAI开源OSCAR" (ModelScope), section "OSCAR的设计"),
// four codes per byte.  The decisions are defined on x = fp32_rn(k . R), the
// exactly rounded rotated value, in IEEE fp32 / fp16 round-to-nearest-even:
//   xc = clip(x, -tau, tau) + 0          (signed zero canonicalised to +0)
//   z  = fp16_rn(min xc)
//   s  = fp16_rn(fl32(fl32(max xc - min xc) / 3))
//   code = clamp(rint(fl32(fl32(xc - z) / s)), 0, 3), 0 when s == 0
//
// The kernels compute x with an fp32 FMA chain of 128 steps, whose error is at
// most gamma_128 * sum_i |k_i R_ij| <= gamma_128 * |k|_2 * |R_:j|_2 (recursive
// summation bound, one rounding per step), plus half an ulp for the final
// rounding.  Every decision is taken on the interval [x - e, x + e]; the steps
// above are monotone in x, so equal decisions at both ends are the exact
// decision.  Where the ends differ (rare), the value is recomputed exactly: a
// compensated (TwoSum) double-precision dot product -- each bf16 x fp32 product
// is exact in double -- rounded once to fp32.  That result equals
// fp32_rn(k . R) unless the exact value lies within ~2^-90 sum|k_i R_ij| of an
// fp32 rounding midpoint.
#pragma once

#include <cuda_fp16.h>

#include "internal.h"

namespace oscar {

struct GroupCode {
  uint32_t byte;      // packed codes of this lane's 4 channels
  uint16_t s_bits;    // fp16 scale
  uint16_t z_bits;    // fp16 zero point
  int exact_calls;    // values recomputed exactly by this lane
};

// gamma_128 = 128 u / (1 - 128 u), u = 2^-24, rounded up with margin.
constexpr float GAMMA_128 = 7.6295e-6f;

__device__ __forceinline__ float clip_canon(float x, float tau) {
  return __fadd_rn(fminf(fmaxf(x, -tau), tau), 0.0f);
}

__device__ __forceinline__ uint32_t code_of(float xc, float z, float s) {
  if (s == 0.0f) return 0u;
  const float t = __fdiv_rn(__fsub_rn(xc, z), s);
  return static_cast<uint32_t>(fminf(fmaxf(rintf(t), 0.0f), 3.0f));
}

__device__ __forceinline__ float scale_of(float mx, float mn) {
  return __half2float(__float2half_rn(__fdiv_rn(__fsub_rn(mx, mn), 3.0f)));
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ void two_sum(double a, double b, double& s, double& e) {
  s = a + b;
  const double bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

// fp32_rn of sum_i k_i * r_i over 128 terms held by a whole warp, lane l holding
// terms 4l .. 4l+3 (k exactly bf16-valued, r fp32).  Every product is exact in
// double; the terms are added with TwoSum in a butterfly, so every lane ends
// with the same (s, c), s + c within ~2^-100 * sum |k_i r_i| of the exact sum.
__device__ __forceinline__ float warp_exact_dot(float4 k, float4 r) {
  double s = static_cast<double>(k.x) * static_cast<double>(r.x);
  double c = 0.0, e;
  two_sum(s, static_cast<double>(k.y) * static_cast<double>(r.y), s, e);
  c += e;
  two_sum(s, static_cast<double>(k.z) * static_cast<double>(r.z), s, e);
  c += e;
  two_sum(s, static_cast<double>(k.w) * static_cast<double>(r.w), s, e);
  c += e;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const double s2 = __shfl_xor_sync(0xffffffffu, s, off);
    const double c2 = __shfl_xor_sync(0xffffffffu, c, off);
    two_sum(s, s2, s, e);
    c = (c + c2) + e;
  }
  double hi, lo;
  two_sum(s, c, hi, lo);   // hi + lo == s + c exactly
  float f = __double2float_rn(hi);
  const double fd = static_cast<double>(f);
  if (hi != fd && lo != 0.0) {
    // hi may sit exactly on an fp32 rounding midpoint; then the remainder decides
    const float nb = nextafterf(f, hi > fd ? INFINITY : -INFINITY);
    const double mid = 0.5 * (fd + static_cast<double>(nb));
    if (hi == mid) f = (lo > 0.0) ? fmaxf(f, nb) : fminf(f, nb);
  }
  return f;
}

// A full warp holds the group: lane l owns channels 4l .. 4l+3 with rotated
// values x (fast path) and error bounds err; k holds the token's input
// channels 4l .. 4l+3 and rt points at R^T (row ch = column ch of R), so the
// exact value of channel ch is warp_exact_dot(k, rt[ch][4l .. 4l+3]).
__device__ __forceinline__ GroupCode quantize_group_warp(float4 xv, float4 ev, float tau, float4 k,
                                                         const float* __restrict__ rt) {
  const int lane = threadIdx.x & 31;
  const float x[4] = {xv.x, xv.y, xv.z, xv.w};
  const float er[4] = {ev.x, ev.y, ev.z, ev.w};
  float lo[4], hi[4];
  GroupCode g;
  g.exact_calls = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float e = __fmaf_ru(fabsf(x[i]), 0x1.0001p-24f, er[i]);
    lo[i] = clip_canon(__fsub_rd(x[i], e), tau);
    hi[i] = clip_canon(__fadd_ru(x[i], e), tau);
  }
  auto reduce_min = [](float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
  };
  auto reduce_max = [](float v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    return v;
  };
  auto exact = [&](int ch) {
    const float4 r = __ldg(reinterpret_cast<const float4*>(rt + (size_t)ch * D) + lane);
    return warp_exact_dot(k, r);
  };
  float mn_lo = reduce_min(fminf(fminf(lo[0], lo[1]), fminf(lo[2], lo[3])));
  float mn_hi = reduce_min(fminf(fminf(hi[0], hi[1]), fminf(hi[2], hi[3])));
  float mx_lo = reduce_max(fmaxf(fmaxf(lo[0], lo[1]), fmaxf(lo[2], lo[3])));
  float mx_hi = reduce_max(fmaxf(fmaxf(hi[0], hi[1]), fmaxf(hi[2], hi[3])));
  const bool meta_sure = __half_as_ushort(__float2half_rn(mn_lo)) == __half_as_ushort(__float2half_rn(mn_hi)) &&
                         scale_of(mx_lo, mn_hi) == scale_of(mx_hi, mn_lo);
  if (!meta_sure) {
    // (warp-uniform, rare) the group's min or max is too close to an fp16
    // rounding boundary: take exactly every value that could be the min (its
    // interval reaches below mn_hi) or the max (reaches above mx_lo).  The
    // others lie strictly inside, so the extremes become exact.
    uint32_t cand = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (lo[i] <= mn_hi || hi[i] >= mx_lo) cand |= 1u << i;
    uint32_t todo = __ballot_sync(0xffffffffu, cand != 0);
    while (todo) {
      const int src = __ffs(todo) - 1;
      const int i = __ffs(__shfl_sync(0xffffffffu, cand, src)) - 1;
      const float xe = clip_canon(exact(4 * src + i), tau);
      if (lane == src) {
        lo[i] = hi[i] = xe;
        cand &= ~(1u << i);
        g.exact_calls += 1;
      }
      todo = __ballot_sync(0xffffffffu, cand != 0);
    }
    mn_lo = reduce_min(fminf(fminf(lo[0], lo[1]), fminf(lo[2], lo[3])));
    mx_lo = reduce_max(fmaxf(fmaxf(lo[0], lo[1]), fmaxf(lo[2], lo[3])));
  }
  const __half zh = __float2half_rn(mn_lo);
  const float z = __half2float(zh);
  const __half sh = __float2half_rn(__fdiv_rn(__fsub_rn(mx_lo, mn_lo), 3.0f));
  const float s = __half2float(sh);
  uint32_t code[4];
  uint32_t unsure = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    code[i] = code_of(lo[i], z, s);
    if (code[i] != code_of(hi[i], z, s)) unsure |= 1u << i;
  }
  // resolve the undecided codes one at a time, the whole warp computing each
  uint32_t pending = __ballot_sync(0xffffffffu, unsure != 0);
  while (pending) {
    const int src = __ffs(pending) - 1;
    const uint32_t bits = __shfl_sync(0xffffffffu, unsure, src);
    const int i = __ffs(bits) - 1;
    const float xe = clip_canon(exact(4 * src + i), tau);
    if (lane == src) {
      code[i] = code_of(xe, z, s);
      unsure &= ~(1u << i);
      g.exact_calls += 1;
    }
    pending = __ballot_sync(0xffffffffu, unsure != 0);
  }
  g.byte = code[0] | (code[1] << 2) | (code[2] << 4) | (code[3] << 6);
  g.s_bits = __half_as_ushort(sh);
  g.z_bits = __half_as_ushort(zh);
  return g;
}

// gamma_n bound of an FMA chain / sum with n roundings, rounded up with margin.
__device__ __forceinline__ float gamma_n(int n) {
  const float u = 0x1p-24f;
  return __fdiv_ru(n * u, 1.0f - n * u) * 1.0001f;
}

// Cauchy-Schwarz form of the chain bound for a token with |k|_2^2 = knorm2
// and a matrix whose columns have norm at most colnorm.
__device__ __forceinline__ float chain_error_bound(float knorm2, float colnorm) {
  return GAMMA_128 * 1.0001f * sqrtf(knorm2 * 1.0001f) * colnorm;
}

}  // namespace oscar

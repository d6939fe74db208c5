// Device-side INT2 quantiser of the groups of one 128-channel token-head: one
// group of 128 channels, or two of 64 (G_K = 64: channels 0..63 and 64..127,
// each with its own scale and zero; "Together AI Open-Sources OSCAR"
// (MarkTechPost), section "What OSCAR Does Differently").
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
// fp32 rounding midpoint.  Before that, an undecided value is narrowed by a
// compensated fp32 dot product (Dot2) with a rigorous bound; the fp64 path runs
// only if the narrow interval still leaves the decision open.
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

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

__device__ __forceinline__ void two_sum_f(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Compensated fp32 dot product over the same 128 terms as warp_exact_dot
// (Ogita, Rump and Oishi's Dot2): each product is split exactly into
// p + q with an FMA, the p are added by error-free TwoSum steps (lane, then a
// butterfly across the warp) and every error term is accumulated in c.  s + c
// differs from the exact sum by at most gamma_16 * 9 u * S <= 144 u^2 S, with
// S >= sum_i |k_i r_i| (16 = deepest chain of additions into c, 9 u S = bound on
// the error terms' magnitudes).  Returns fp32 bounds lo <= exact <= hi, widened
// by 2^-36 S (a 28x margin) and rounded outwards; fp32_rn(exact) lies in
// [lo, hi] since rounding is monotone.
__device__ __forceinline__ void warp_dot2(float4 k, float4 r, float S, float& lo, float& hi) {
  const float kk[4] = {k.x, k.y, k.z, k.w}, rr[4] = {r.x, r.y, r.z, r.w};
  float s = __fmul_rn(kk[0], rr[0]);
  float c = __fmaf_rn(kk[0], rr[0], -s);
#pragma unroll
  for (int i = 1; i < 4; ++i) {
    const float p = __fmul_rn(kk[i], rr[i]);
    const float q = __fmaf_rn(kk[i], rr[i], -p);
    float t;
    two_sum_f(s, p, s, t);
    c = __fadd_rn(c, __fadd_rn(t, q));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
    const float c2 = __shfl_xor_sync(0xffffffffu, c, off);
    float t;
    two_sum_f(s, s2, s, t);
    c = __fadd_rn(c, __fadd_rn(c2, t));
  }
  const float E = __fmul_ru(S, 0x1p-36f);
  lo = __fsub_rd(__fadd_rd(s, c), E);
  hi = __fadd_ru(__fadd_ru(s, c), E);
}

// A full warp holds the token-head: lane l owns channels 4l .. 4l+3 with rotated
// values x (fast path), their error bounds ev and S >= sum_i |k_i R_i,ch| (sv);
// k holds the token's input channels 4l .. 4l+3 and rt points at R^T (row ch =
// column ch of R).  A value whose interval leaves a decision open is narrowed
// first by warp_dot2 (cheap, fp32) and only then, if still open, computed
// exactly by warp_exact_dot (fp64).  With GK = 64, lanes 0..15 hold group 0 and
// lanes 16..31 group 1: the min / max reductions stay within a half-warp, each
// lane's scale and zero are its group's, and the warp-wide narrowing loops run
// when either group needs them (only that group's values are candidates).
template <int GK = 128>
__device__ __forceinline__ GroupCode quantize_group_warp(float4 xv, float4 ev, float4 sv, float tau, float4 k,
                                                         const float* __restrict__ rt) {
  static_assert(GK == 128 || GK == 64, "group of 128 or 64 channels");
  constexpr int RED0 = GK / 8;   // first butterfly offset: lanes of one group
  const int lane = threadIdx.x & 31;
  const float x[4] = {xv.x, xv.y, xv.z, xv.w};
  const float er[4] = {ev.x, ev.y, ev.z, ev.w};
  const float sb[4] = {sv.x, sv.y, sv.z, sv.w};
  float lo[4], hi[4];
  GroupCode g;
  g.exact_calls = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float e = __fmaf_ru(fabsf(x[i]), 0x1.0001p-24f, er[i]);
    lo[i] = clip_canon(__fsub_rd(x[i], e), tau);
    hi[i] = clip_canon(__fadd_ru(x[i], e), tau);
  }
  // min / max over the group's lanes: one warp-wide redux.sync (f32, sm_100 family)
  // for a 128-channel group, a half-warp butterfly for 64 (no -0 or NaN reaches here:
  // the values are clipped and canonicalised)
  auto reduce_min = [](float v) {
    if constexpr (GK == 128) {
      float r;
      asm volatile("redux.sync.min.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
      return r;
    } else {
#pragma unroll
      for (int off = RED0; off > 0; off >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, off));
      return v;
    }
  };
  auto reduce_max = [](float v) {
    if constexpr (GK == 128) {
      float r;
      asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
      return r;
    } else {
#pragma unroll
      for (int off = RED0; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
      return v;
    }
  };
  auto exact = [&](int ch) {
    const float4 r = __ldg(reinterpret_cast<const float4*>(rt + (size_t)ch * D) + lane);
    return warp_exact_dot(k, r);
  };
  // value (src, i) narrowed by warp_dot2, clipped: every lane computes, lane src keeps
  auto narrow = [&](int src, int i, float& nlo, float& nhi) {
    const float4 r = __ldg(reinterpret_cast<const float4*>(rt + (size_t)(4 * src + i) * D) + lane);
    // select, not an indexed load (which would put sb in local memory)
    const float own = i == 0 ? sb[0] : i == 1 ? sb[1] : i == 2 ? sb[2] : sb[3];
    const float S = __shfl_sync(0xffffffffu, own, src);
    warp_dot2(k, r, S, nlo, nhi);
    nlo = clip_canon(nlo, tau);
    nhi = clip_canon(nhi, tau);
  };
  float mn_lo = reduce_min(fminf(fminf(lo[0], lo[1]), fminf(lo[2], lo[3])));
  float mn_hi = reduce_min(fminf(fminf(hi[0], hi[1]), fminf(hi[2], hi[3])));
  float mx_lo = reduce_max(fmaxf(fmaxf(lo[0], lo[1]), fmaxf(lo[2], lo[3])));
  float mx_hi = reduce_max(fmaxf(fmaxf(hi[0], hi[1]), fmaxf(hi[2], hi[3])));
  bool meta_sure = __half_as_ushort(__float2half_rn(mn_lo)) == __half_as_ushort(__float2half_rn(mn_hi)) &&
                   scale_of(mx_lo, mn_hi) == scale_of(mx_hi, mn_lo);
  if (__any_sync(0xffffffffu, !meta_sure)) {
    // a group's min or max is too close to an fp16 rounding boundary: narrow
    // every value of that group that could be the min (its interval reaches
    // below mn_hi) or the max (reaches above mx_lo) and is not already a single
    // point (a clipped value is); then decide again.
    uint32_t cand = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (!meta_sure && lo[i] != hi[i] && (lo[i] <= mn_hi || hi[i] >= mx_lo)) cand |= 1u << i;
    uint32_t todo = __ballot_sync(0xffffffffu, cand != 0);
    while (todo) {
      const int src = __ffs(todo) - 1;
      const int i = __ffs(__shfl_sync(0xffffffffu, cand, src)) - 1;
      float nlo, nhi;
      narrow(src, i, nlo, nhi);
      if (lane == src) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j == i) {
            lo[j] = nlo;
            hi[j] = nhi;
          }
        cand &= ~(1u << i);
      }
      todo = __ballot_sync(0xffffffffu, cand != 0);
    }
    mn_lo = reduce_min(fminf(fminf(lo[0], lo[1]), fminf(lo[2], lo[3])));
    mn_hi = reduce_min(fminf(fminf(hi[0], hi[1]), fminf(hi[2], hi[3])));
    mx_lo = reduce_max(fmaxf(fmaxf(lo[0], lo[1]), fmaxf(lo[2], lo[3])));
    mx_hi = reduce_max(fmaxf(fmaxf(hi[0], hi[1]), fmaxf(hi[2], hi[3])));
    meta_sure = __half_as_ushort(__float2half_rn(mn_lo)) == __half_as_ushort(__float2half_rn(mn_hi)) &&
                scale_of(mx_lo, mn_hi) == scale_of(mx_hi, mn_lo);
  }
  if (__any_sync(0xffffffffu, !meta_sure)) {
    // (rare) still open: take exactly every candidate of the min or the max.  The
    // others lie strictly inside, so the extremes become exact.
    uint32_t cand = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (!meta_sure && lo[i] != hi[i] && (lo[i] <= mn_hi || hi[i] >= mx_lo)) cand |= 1u << i;
    uint32_t todo = __ballot_sync(0xffffffffu, cand != 0);
    while (todo) {
      const int src = __ffs(todo) - 1;
      const int i = __ffs(__shfl_sync(0xffffffffu, cand, src)) - 1;
      const float xe = clip_canon(exact(4 * src + i), tau);
      if (lane == src) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (j == i) lo[j] = hi[j] = xe;
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
  // Fast decision of a whole interval [lo, hi] with the approximate reciprocal:
  // q' = fl(d rcp(s)) is within |d / s| 2^-21 of the IEEE quotient fl(d / s)
  // (rcp.approx: 1 ulp; two roundings of 2^-24), and M = (|q'| + 1) 2^-19 also
  // covers the roundings of q' -/+ M + 1/2.  If both ends land in one rounding
  // cell after the clamp, every value of the interval has that code; otherwise
  // the IEEE quotient decides, as before.
  const float rs = s == 0.0f ? 0.0f : rcp_approx(s);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float qa = __fmul_rn(__fsub_rn(lo[i], z), rs), qb = __fmul_rn(__fsub_rn(hi[i], z), rs);
    const float ma = __fmul_rn(fabsf(qa) + 1.0f, 0x1p-19f), mb = __fmul_rn(fabsf(qb) + 1.0f, 0x1p-19f);
    const float ca = fminf(fmaxf(floorf(qa - ma + 0.5f), 0.0f), 3.0f);
    const float cb = fminf(fmaxf(floorf(qb + mb + 0.5f), 0.0f), 3.0f);
    if (ca == cb) {
      code[i] = static_cast<uint32_t>(ca);
    } else {
      code[i] = code_of(lo[i], z, s);
      if (code[i] != code_of(hi[i], z, s)) unsure |= 1u << i;
    }
  }
  // resolve the undecided codes one at a time, the whole warp computing each:
  // narrowed first, exactly only if the narrow interval still straddles a boundary
  uint32_t pending = __ballot_sync(0xffffffffu, unsure != 0);
  while (pending) {
    const int src = __ffs(pending) - 1;
    const uint32_t bits = __shfl_sync(0xffffffffu, unsure, src);
    const int i = __ffs(bits) - 1;
    float nlo, nhi;
    narrow(src, i, nlo, nhi);
    const uint32_t clo = code_of(nlo, z, s), chi = code_of(nhi, z, s);
    const bool open = __shfl_sync(0xffffffffu, clo != chi ? 1 : 0, src) != 0;
    uint32_t ce = clo;
    if (open) {
      ce = code_of(clip_canon(exact(4 * src + i), tau), z, s);
      if (lane == src) g.exact_calls += 1;
    }
    if (lane == src) {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (j == i) code[j] = ce;
      unsure &= ~(1u << i);
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

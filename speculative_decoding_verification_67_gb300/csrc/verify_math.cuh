// Device arithmetic shared by the kernels that produce and consume softmax
// statistics: float-float (double-float) sums and the exponent map.
//
// exp(z/T) is evaluated as 2^(z*c) with c = log2(e)/T carried as a pair of
// floats, so z*c is exact to ~1e-14 and no rounded temperature or log2(e)
// scales every exponent the same way.  A partial sum is kept against an
// integer reference k (at or a few units above its largest exponent): bringing
// partials to a common reference is then an exact power of two.  Sums are
// compensated (TwoSum), so the normalisers carry no systematic error larger
// than ~1e-12; the only per-token error left is the f32 rounding of one
// exponent and one exp2f, which is random across tokens.
#pragma once

#include <cuda_runtime.h>

#include <cmath>

namespace sv {

struct ff {
  float hi, lo;
};

// a + b exactly as hi + lo (Knuth's TwoSum).
__device__ __forceinline__ ff two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  const float e = (a - (s - bb)) + (b - bb);
  return {s, e};
}

__device__ __forceinline__ ff ff_norm(float hi, float lo) {
  const float s = hi + lo;
  return {s, lo - (s - hi)};
}

__device__ __forceinline__ ff ff_add(ff a, ff b) {
  const ff s = two_sum(a.hi, b.hi);
  return ff_norm(s.hi, s.lo + a.lo + b.lo);
}

__device__ __forceinline__ ff ff_add_f(ff a, float b) {
  const ff s = two_sum(a.hi, b);
  return ff_norm(s.hi, s.lo + a.lo);
}

// Running compensated sum: add b to (hi, lo) without renormalising (the
// caller normalises once at the end with ff_norm).
__device__ __forceinline__ void ff_accumulate(float& hi, float& lo, float b) {
  const ff s = two_sum(hi, b);
  hi = s.hi;
  lo += s.lo;
}

// a > b for normalised pairs.
__device__ __forceinline__ bool ff_gt(ff a, ff b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }

// 2^e for an integer-valued float e <= 0 (exact; 0 below the normal range,
// and for e = -inf).
__device__ __forceinline__ float pow2_int(float e) {
  return e >= -126.f ? __int_as_float((static_cast<int>(e) + 127) << 23) : 0.f;
}

// The same for an integer-valued e <= 0 (0 at or below -127, also for -inf
// and NaN) without a float-to-int conversion, which issues ~12x slower than
// a float add on sm_103: adding 1.5 * 2^23 leaves the integer in the low
// mantissa bits, from which the exponent field is built.
__device__ __forceinline__ float pow2_nonpos(float e) {
  const float c = __fadd_rn(fmaxf(e, -127.f), 12582912.f);
  return __int_as_float((__float_as_int(c) - (0x4B400000 - 127)) << 23);
}

// An integer-valued reference k with h <= k <= h + 4 for any finite h, from
// float adds only (ceilf issues ~12x slower than an add on sm_103).  Adding
// and removing m = +-1.5 * 2^23 (the sign of h) rounds to an integer: the
// nearest one for |h| < 2^22, so k = rint(h) + 1 in [h + 1/2, h + 3/2]; one
// within 1 of h for 2^22 <= |h| < 2^23; beyond that h itself is an integer
// and the max and min keep k within [h, h + 4] (h + 2 may round up by 2).
// NaN and infinities pass through (as NaN or infinity).
__device__ __forceinline__ float ref_above(float h) {
  const float m = __int_as_float((__float_as_int(h) & 0x80000000) | 0x4B400000);  // copysign(1.5 * 2^23, h)
  const float r = __fadd_rn(__fadd_rn(h, m), -m);
  return fminf(fmaxf(__fadd_rn(r, 1.f), h), __fadd_rn(h, 2.f));
}

// a * 2^e, exact (barring underflow).
__device__ __forceinline__ ff ff_scale2(ff a, int e) { return {ldexpf(a.hi, e), ldexpf(a.lo, e)}; }

__device__ __forceinline__ ff ff_mul_f(ff a, float b) {
  const float p = a.hi * b;
  const float e = fmaf(a.hi, b, -p);
  return ff_norm(p, e + a.lo * b);
}

// a / b to ~1e-14 (one correction step of the f32 quotient).
__device__ __forceinline__ ff ff_div(ff a, ff b) {
  const float q1 = a.hi / b.hi;
  const ff qb = ff_mul_f(b, q1);
  const ff r = ff_add(a, {-qb.hi, -qb.lo});
  const float q2 = r.hi / b.hi;
  return ff_norm(q1, q2);
}

__device__ __forceinline__ ff shfl_xor_ff(ff v, int off) {
  return {__shfl_xor_sync(0xffffffffu, v.hi, off), __shfl_xor_sync(0xffffffffu, v.lo, off)};
}

__device__ __forceinline__ ff warp_sum_ff(ff v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = ff_add(v, shfl_xor_ff(v, off));
  return v;
}

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

// ------------------------------------------------------------ exponent map
// z * c as a float pair (unnormalised: hi = fl(z*ch), lo = the rest).
struct Expo {
  float ch, cl;
};

__device__ __forceinline__ float expo_hi(float z, Expo c) { return z * c.ch; }

__device__ __forceinline__ float expo_lo(float z, float hi, Expo c) { return fmaf(z, c.cl, fmaf(z, c.ch, -hi)); }

// 2^(z*c - k) for an integer-valued float k (<= 1 when k >= ceil(z*c)).
__device__ __forceinline__ float pow2_rel(float z, Expo c, float k) {
  const float h = expo_hi(z, c);
  return exp2f((h - k) + expo_lo(z, h, c));
}

// ------------------------------------------------------------ partials
// A softmax-normaliser partial: sum of 2^(z*c - k) over some tokens, as a
// float pair, against the integer reference k (-inf when empty).
struct Partial {
  float k;
  ff s;
  int bad;
};

__device__ __forceinline__ Partial partial_empty() { return {-INFINITY, {0.f, 0.f}, 0}; }

// Bring two partials to the larger reference and add (exact rescaling).
__device__ __forceinline__ Partial partial_merge(Partial a, Partial b) {
  Partial r;
  r.bad = a.bad | b.bad;
  if (b.k == -INFINITY || b.s.hi == 0.f) {
    r.k = a.k;
    r.s = a.s;
    return r;
  }
  if (a.k == -INFINITY || a.s.hi == 0.f) {
    r.k = b.k;
    r.s = b.s;
    return r;
  }
  r.k = fmaxf(a.k, b.k);
  // differences below -300 underflow to zero either way; the clamp keeps the
  // float-to-int conversion in range
  const int ea = static_cast<int>(fmaxf(a.k - r.k, -300.f));
  const int eb = static_cast<int>(fmaxf(b.k - r.k, -300.f));
  r.s = ff_add(ff_scale2(a.s, ea), ff_scale2(b.s, eb));
  return r;
}

__device__ __forceinline__ Partial warp_merge(Partial p) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    Partial o;
    o.k = __shfl_xor_sync(0xffffffffu, p.k, off);
    o.s = shfl_xor_ff(p.s, off);
    o.bad = __shfl_xor_sync(0xffffffffu, p.bad, off);
    p = partial_merge(p, o);
  }
  return p;
}

}  // namespace sv

// Double-float ("df64") arithmetic on the FP32 pipe.
//
// GB300 executes fp64 FMA at about 1/70 of its fp32 FMA rate, so fp64-accurate
// recurrences are carried here as unevaluated sums hi + lo of two floats, with
// error-free transformations (Knuth's TwoSum; the FMA form of Dekker's exact
// product).  A value (h, l) is kept unnormalised between steps: |l| is a few
// units in the last place of h at most, which is all the exact products need.
// Relative accuracy is about 2^-47 (h carries 24 bits, l another ~23).
//
// Every operation whose rounding matters is written with the _rn intrinsics so
// that the compiler cannot fuse or reorder it; fmaf is used only where a fused
// multiply-add is intended.
//
// Conversions between fp64 and df64 use integer bit manipulation instead of
// the fp64<->fp32 conversion instructions, which share the slow fp64 pipe.
// Dynamic range: values with 2^-100 < |v| < 2^127 convert with full accuracy;
// smaller magnitudes (including zero) become tiny values of magnitude below
// 2^-126; larger ones are out of range.  Solutions are therefore accurate
// relative to the largest entry of a system as long as that entry lies inside
// the range.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace pent {
namespace df {

struct D2 {
  float h, l;
};

// exact product a*b = p + e
__device__ __forceinline__ void two_prod(float a, float b, float& p, float& e) {
  p = __fmul_rn(a, b);
  e = __fmaf_rn(a, b, -p);
}

// exact sum a+b = s + e (no magnitude precondition)
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float ap = __fsub_rn(s, bb);
  e = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bb));
}

// s = f + c1*y1 + c2*y2 + c3*y3 with f, c_k, y_k double-floats; f may be scaled
// by a coefficient too (see axpy3).  Products use only the hi part of y in the
// exact step; the hi*lo and lo*hi cross terms are accumulated in the low word.
// The lo*lo terms (relative 2^-48) are dropped.
__device__ __forceinline__ D2 sum3(D2 f, D2 c1, D2 y1, D2 c2, D2 y2) {
  float p1, e1, p2, e2, s1, t1, s2, t2;
  two_prod(c1.h, y1.h, p1, e1);
  two_prod(c2.h, y2.h, p2, e2);
  two_sum(f.h, p1, s1, t1);
  two_sum(s1, p2, s2, t2);
  float lo = __fadd_rn(f.l, e1);
  lo = __fadd_rn(lo, e2);
  lo = __fadd_rn(lo, t1);
  lo = __fadd_rn(lo, t2);
  lo = __fmaf_rn(c1.h, y1.l, lo);
  lo = __fmaf_rn(c1.l, y1.h, lo);
  lo = __fmaf_rn(c2.h, y2.l, lo);
  lo = __fmaf_rn(c2.l, y2.h, lo);
  return D2{s2, lo};
}

// r*f + c1*y1 + c2*y2  (three products)
__device__ __forceinline__ D2 sum3p(D2 r, D2 f, D2 c1, D2 y1, D2 c2, D2 y2) {
  float p0, e0;
  two_prod(r.h, f.h, p0, e0);
  float lo0 = __fmaf_rn(r.h, f.l, e0);
  lo0 = __fmaf_rn(r.l, f.h, lo0);
  return sum3(D2{p0, lo0}, c1, y1, c2, y2);
}

// a + c*y (one product), used for low-rank corrections
__device__ __forceinline__ D2 axpy(D2 a, D2 c, D2 y) {
  float p, e, s, t;
  two_prod(c.h, y.h, p, e);
  two_sum(a.h, p, s, t);
  float lo = __fadd_rn(a.l, e);
  lo = __fadd_rn(lo, t);
  lo = __fmaf_rn(c.h, y.l, lo);
  lo = __fmaf_rn(c.l, y.h, lo);
  return D2{s, lo};
}

// a * b (exact product of the hi words, cross terms in the low word)
__device__ __forceinline__ D2 mul(D2 a, D2 b) {
  float p, e;
  two_prod(a.h, b.h, p, e);
  float lo = __fmaf_rn(a.h, b.l, e);
  lo = __fmaf_rn(a.l, b.h, lo);
  return D2{p, lo};
}

// a + b
__device__ __forceinline__ D2 add(D2 a, D2 b) {
  float s, t;
  two_sum(a.h, b.h, s, t);
  return D2{s, __fadd_rn(__fadd_rn(a.l, b.l), t)};
}

__device__ __forceinline__ D2 neg(D2 a) { return D2{-a.h, -a.l}; }

// ---------------------------------------------------------------------------
// fp64 <-> df64 by integer operations
// ---------------------------------------------------------------------------

// Split a double into hi (its leading 24 significant bits, truncated) and lo
// (the next 23 bits), both floats with the sign of v.
__device__ __forceinline__ D2 from_double(double v) {
  const uint32_t hi = (uint32_t)__double2hiint(v);
  const uint32_t lo = (uint32_t)__double2loint(v);
  const uint32_t sign = hi & 0x80000000u;
  // magnitude bits of the high word, exponent clamped to the float range
  uint32_t mag = hi & 0x7FFFFFFFu;
  mag = max(mag, 0x38000000u);          // |v| < 2^-127 -> exponent field 0 below
  mag = min(mag, 0x47EFFFFFu);          // |v| >= 2^128 -> largest finite float range
  const uint32_t t = mag - 0x38000000u;  // re-bias 1023 -> 127 (in place, 11-bit field)
  // float bits: 8-bit exponent and 23 mantissa bits = (t:lo) << 3, high word
  const uint32_t hbits = __funnelshift_l(lo, t, 3) | sign;
  // remaining 29 mantissa bits, top 23 of them, scaled by 2^(e-23): built as
  // (2^(e-23) * 1.m) - 2^(e-23), exact in fp32.
  uint32_t ebits = hbits & 0x7F800000u;
  ebits = max(ebits, 0x0C000000u);       // keep e-23 >= 1 (tiny values only)
  const uint32_t base = (ebits - 0x0B800000u) | sign;
  const uint32_t m = (lo >> 6) & 0x007FFFFFu;
  const float l = __fsub_rn(__uint_as_float(base | m), __uint_as_float(base));
  return D2{__uint_as_float(hbits), l};
}

// Bits of the double equal to the float x (x normal).  A zero or subnormal x
// maps to a double of magnitude 2^-127 or less, never to a large value.
__device__ __forceinline__ double float_bits_to_double(float x) {
  const uint32_t b = __float_as_uint(x);
  const uint32_t sh = (uint32_t)((int32_t)b >> 3);          // sign replicated into 31..28
  const uint32_t hi = sh + (0x38000000u ^ (sh & 0xF0000000u));
  return __hiloint2double((int)hi, (int)(b << 29));
}

// hi + lo as a correctly rounded double (one fp64 add).
__device__ __forceinline__ double to_double(D2 v) {
  return __dadd_rn(float_bits_to_double(v.h), float_bits_to_double(v.l));
}

__device__ __forceinline__ D2 ld_coef(const float2 c) { return D2{c.x, c.y}; }

}  // namespace df
}  // namespace pent

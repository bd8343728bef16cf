// Fixed-grid double-float arithmetic for the partitioned solves.
//
// A value v is held as a pair (a, l) of floats with v = (a - B) + l, where the
// bias B = 1.5 * 2^(k+23) puts every a in the binade [2^(k+23), 2^(k+24)), so
// a is v rounded to the grid of multiples of 2^k and l carries the rest.  As
// long as every partial sum stays below 2^(k+22) in magnitude (the plan derives
// k from bounds on the solve's intermediate values, for a right-hand side
// scaled so that max |f| lies in [1, 2)), rounding to the grid happens at one
// fixed exponent, so
//   t = fma(c, y, a)            is a + c y rounded to the grid,
//   a - t                       is exact (same binade), and
//   fma(c, y, a - t)            recovers the rounding error,
// and a multiply-add costs six FP32 instructions instead of the twelve of a
// TwoSum-based double-float one.  The error of each operation is about
// 2^(k-24): about 2^-46 of the largest intermediate value of the solve.
//
// Conversions between fp64 and the pair use integer operations (the fp64 <->
// fp32 conversion instructions share GB300's slow fp64 pipe), with a
// per-system power-of-two scale folded into the exponent arithmetic: a system
// is converted as f * 2^-s with s chosen so that its largest entry lies in
// [1, 2), and its solution converted back as x * 2^s, both exactly.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

namespace pent {
namespace fg {

// acc += c * y:  c = (ch, cl) a double-float coefficient, y = (yh, yl) with yh
// on the grid (unbiased), acc = (a, l) biased.  In a recurrence y is the
// previous row's result: its low word enters one FMA and one add before the
// new low word, so a row costs two dependent FP32 latencies on either word.
__device__ __forceinline__ void madd(float& a, float& l, float ch, float cl, float yh, float yl) {
  const float t = __fmaf_rn(ch, yh, a);
  const float e = __fmaf_rn(ch, yh, __fsub_rn(a, t));
  float m = __fmaf_rn(cl, yh, l);
  m = __fmaf_rn(ch, yl, m);
  l = __fadd_rn(m, e);
  a = t;
}

// acc += c * y for a response |c| < 2^-24: the product lands in the low word
// alone (its rounding there is below 2^-48 of |y|).
__device__ __forceinline__ void madd_low(float& l, float ch, float yh) { l = __fmaf_rn(ch, yh, l); }

// acc = B + r * f:  r = (rh, rl), f = (fh, fl) a split double
__device__ __forceinline__ void start(float& a, float& l, float B, float rh, float rl, float fh, float fl) {
  a = __fmaf_rn(rh, fh, B);
  const float e = __fmaf_rn(rh, fh, __fsub_rn(B, a));
  l = __fmaf_rn(rl, fh, __fmaf_rn(rh, fl, e));
}

// Exponent field of the largest |v| seen: the high word's magnitude bits.
__device__ __forceinline__ uint32_t mag_bits(double v) {
  return (uint32_t)__double2hiint(v) & 0x7FFFFFFFu;
}

// Rebias constant for a system whose largest entry has the (biased) fp64
// exponent field e: a value with exponent field ev converts to a float with
// exponent field ev - e + 127, i.e. f * 2^-(e - 1023).  Any 1 <= e <= 2046
// works: for e < 127 the unsigned difference wraps and the signed value of
// (magnitude - offset) in split() is still exact.
__device__ __forceinline__ uint32_t in_offset(uint32_t e) { return (e - 127u) << 20; }

// Split v * 2^-s into hi (its leading 24 significant bits, truncated) and lo
// (the next 23 bits) as floats; `off` = in_offset(e) of the system.  Values
// more than 2^126 below the system's largest entry become zero-like (|.| <
// 2^-126 after scaling), which is below any solution error.
__device__ __forceinline__ void split(double v, uint32_t off, float& h, float& lo) {
  const uint32_t hw = (uint32_t)__double2hiint(v);
  const uint32_t lw = (uint32_t)__double2loint(v);
  const uint32_t sign = hw & 0x80000000u;
  int32_t t = (int32_t)(hw - sign - off);   // magnitude word minus the rebias
  t = max(t, 0);
  const uint32_t hb = __funnelshift_l(lw, (uint32_t)t, 3) | sign;
  uint32_t eb = hb & 0x7F800000u;
  eb = max(eb, 0x0C000000u);            // e - 23 >= 1 for the low word's base
  const uint32_t base = (eb - 0x0B800000u) | sign;
  const uint32_t m = (lw >> 6) & 0x007FFFFFu;
  lo = __fsub_rn(__uint_as_float(base | m), __uint_as_float(base));
  h = __uint_as_float(hb);
}

// Output constant of a system with largest-entry exponent field e: a float
// with exponent field fe becomes the double with exponent field fe - 127 + e.
__device__ __forceinline__ uint32_t out_offset(uint32_t e) { return (e - 127u) << 20; }

// Bits of the double x * 2^s for the float x (x normal; zero and subnormal x
// map to doubles of magnitude 2^(s-126) or less, far below the solution).
__device__ __forceinline__ double scaled_double(float x, uint32_t off) {
  const uint32_t b = __float_as_uint(x);
  const uint32_t sh = (uint32_t)((int32_t)b >> 3);   // sign replicated into bits 31..28
  // positive: sh + off; negative: the sign bit back in place of the replicated ones
  const uint32_t hi = sh + off - (sh & 0x70000000u);
  return __hiloint2double((int)hi, (int)(b << 29));
}

// (h + l) * 2^s rounded to fp64 (one fp64 add).
__device__ __forceinline__ double join(float h, float l, uint32_t off) {
  return __dadd_rn(scaled_double(h, off), scaled_double(l, off));
}

// (h + l) * 2^s as a double without the fp64 pipe, for h and l as join()
// takes them.  s1 = h + l rounded toward zero, so that e1 = (h + l) - s1 has the
// sign of s1 and |e1| <= one float ulp of s1; the double of s1 comes from its
// bits as in scaled_double(); e1, rounded to a multiple of 2^8 double ulps of
// s1 (at most 2^21 of them, by the magic-number float add), is added to its
// magnitude bits (carrying into the exponent where the sum reaches the next
// binade).  Error: at most 2^-45 of |s1| beyond the rounding of e1's own two
// float adds (2^-24 of |e1|), against 2^-53 for join().  Eleven integer and
// five FP32 operations: a kernel that joins many outputs can split them
// between this and join() to balance the FP32/integer lanes against GB300's
// slow fp64 pipe.
__device__ __forceinline__ double join_int(float h, float l, uint32_t off) {
  const float s1 = __fadd_rz(h, l);
  const float e1 = __fadd_rn(__fsub_rn(h, s1), l);
  const uint32_t b = __float_as_uint(s1);
  const uint32_t sh = (uint32_t)((int32_t)b >> 3);
  const uint32_t hi = sh + off - (sh & 0x70000000u);
  // 2^(171 - E) for the float exponent field E of s1 (E >= 44: smaller s1 are
  // below 2^-83 of the system's largest value, where e1 cannot matter)
  const uint32_t es = max(b & 0x7F800000u, 44u << 23);
  const float fac = __uint_as_float((298u << 23) - es);
  const float t = __fadd_rn(__fmul_rn(e1, fac), 12582912.0f);      // + 1.5 * 2^23: round to an integer
  const unsigned long long n = (unsigned long long)abs((int)__float_as_uint(t) - 0x4B400000);
  const unsigned long long bits =
      (((unsigned long long)hi << 32) | (unsigned long long)(b << 29)) + (n << 8);
  return __longlong_as_double((long long)bits);
}

// Streaming store of v to *p where pred holds, as one predicated instruction:
// an unrolled output loop stays one basic block (a branch per row would cut
// it into blocks whose latency chains cannot overlap).
__device__ __forceinline__ void store_cs_if(double* p, double v, bool pred) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t@q st.global.cs.f64 [%0], %1;\n\t}" ::"l"(p), "d"(v),
      "r"((int)pred));
}

// Exponent window (fp64 biased exponent field of a system's largest entry) of
// the scaled double-float paths; Cahn–Hilliard also needs 2^(2s) (the factor of
// its cubic) in float range at the top.  Systems outside go to native fp64.
constexpr uint32_t kEMin = 1023 - 860, kEMax = 1023 + 1000, kEMaxCH = 1023 + 50;

// 2^d as a double, exact, for -1022 <= d <= 1023
__device__ __forceinline__ double pow2i(int d) { return __hiloint2double((1023 + d) << 20, 0); }

// What a linear solve does with one system, from the largest magnitude word of
// its entries (fp64 high word without sign, with bit 0 set if any low word is
// nonzero, so that only an all-zero system gives 0):
//   fast  largest exponent e in the window: converted in with 2^-s and out
//         with 2^s, s = e - 1023;
//   zero  every entry +-0: the solution is zero (an in-place solve has
//         nothing to store);
//   resc  a finite largest entry above the window: converted in the same way
//         (the integer split is exact for normal entries, and subnormal ones
//         are then far below the largest and flushed), but converted out with
//         the window's top eo (the join needs its outputs' exponents in range)
//         and then multiplied by 2^(e - eo) in fp64;
//   otherwise (largest entry below the window, where subnormal entries could
//         matter and the split would misread them, or an inf or NaN entry)
//         the kernel falls back to native fp64.
struct SysClass {
  uint32_t ein, eo;   // exponent fields of the conversions in and out
  int d;              // rescaled systems: e - eo
  bool fast, zero, resc;
};
__device__ __forceinline__ SysClass classify(uint32_t smax, uint32_t emin, uint32_t emax) {
  SysClass r;
  const uint32_t e = smax >> 20;
  r.zero = smax == 0u;
  r.fast = e >= emin && e <= emax;
  r.resc = e > emax && e != 0x7FFu;
  r.ein = (r.fast || r.resc) ? e : 1023u;
  r.eo = r.fast ? e : (r.resc ? emax : 1023u);
  r.d = (int)r.ein - (int)r.eo;
  return r;
}

// One term of the magnitude word above for two entries: the larger high-word
// magnitude, and the OR of both low words folded into nz.
__device__ __forceinline__ uint32_t mag_pair(double u, double v, uint32_t& nz) {
  nz |= (uint32_t)__double2loint(u) | (uint32_t)__double2loint(v);
  return max(mag_bits(u), mag_bits(v));
}

// 2^(2s) as a float for the system exponent field e (s = e - 1023); zero when
// the cubic is below 2^-126 of the state and cannot matter
__device__ __forceinline__ float cubic_scale(uint32_t e) {
  const int t = 2 * ((int)e - 1023) + 127;
  return t >= 1 ? __uint_as_float((uint32_t)t << 23) : 0.f;
}

// 2^-s and 2^s as doubles (exact) for the system exponent field e
__device__ __forceinline__ double pow2_neg(uint32_t e) { return __hiloint2double((int)((2046u - e) << 20), 0); }
__device__ __forceinline__ double pow2_pos(uint32_t e) { return __hiloint2double((int)(e << 20), 0); }

}  // namespace fg
}  // namespace pent

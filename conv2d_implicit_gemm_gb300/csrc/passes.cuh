// Per-pixel steps of the output pass, shared by the output pass kernel and
// the final conv's fused epilogue so that both compute the same bits.
// Source: "oidn-webgpu 0.0.0-stage -> 0.6.0, src/native/denoise.ts",
// outputShader, with the readings of its imported helpers:
//  * sanitize(v, lo, hi): NaN becomes 0, then clamp by comparison;
//  * 'log' transfer: F^-1(y) = 2^y - 1.
// The HDR branch stores (2^d - 1) / inputScale correctly rounded to fp32:
// the quotient is evaluated as a float pair, and in double precision only
// when the pair lies too close to a rounding boundary to decide it.
#pragma once

#include <cfloat>
#include <cstdint>
#include <cuda_runtime.h>

namespace oidnx {

__device__ __forceinline__ float sanitize(float v, float lo, float hi) {
  if (isnan(v)) v = 0.0f;
  if (v < lo) v = lo;
  else if (v > hi) v = hi;
  return v;
}

// Knuth's two-sum: s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// (2^d - 1) / s in double precision, rounded once to fp32 (expm1 below
// d = 1, where 2^d - 1 cancels).  The fallback of hdr_inverse_rn.
static __device__ __noinline__ float hdr_inverse_double(float d, float s, bool div) {
  const double x = d;
  const double w = x < 1.0 ? expm1(x * 0.69314718055994530942) : exp2(x) - 1.0;
  return __double2float_rn(div ? w / static_cast<double>(s) : w);
}

// Fast two-sum: s + e == a + b exactly when a == 0 or |a| >= |b|.
__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  e = __fsub_rn(b, __fsub_rn(s, a));
}

// (2^d - 1) / s correctly rounded to fp32, for d in [0, FLT_MAX] (the
// sanitized network output) and s > 0 (div false: s is 1).
// tab: kExp2TabSize (32) entries {Th, Tl, Dh, Dl} with 2^(j/32) = Th + Tl
// and 2^(j/32) - 1 = Dh + Dl as float pairs (fill_exp2_table); 512 bytes, so
// a warp's lookups touch at most four 128-byte lines.
//  1. k = rint(32 d) splits d = n + j/32 + r (n = k >> 5, j = k & 31,
//     r = d - k/32 exact, |r| <= 1/64).
//  2. e = exp(r ln 2) - 1 by its Taylor series to the sixth power: t = r ln 2
//     (ln 2 split into a float and its remainder), t^2/2 and t^3/6 as pairs
//     (products split by FMA, 1/6 as a pair), t^4/24 .. t^6/720 in float.
//  3. u = 2^(j/32 + r) - 1 = D_j + T_j e; then
//     2^d - 1 = u + (2^n - 1) + (2^n - 1) u, with 2^n - 1 exact (n <= 24),
//     the product split by an FMA and the sums taken by exact two-sums (for
//     n = 0 the result is u itself: no cancellation for small d).
//  4. The division by s as a pair: the remainder z - q s is exact by FMA.
// The pair is within 2^-44 |F| of (2^d - 1) / s (an emulation of these
// steps against 120-bit arithmetic over d in [2^-60, 24.5): largest error
// 2^-44.8, for d in [2^-10, 2^-5] where D_j and T_j e partly cancel).  If
// the pair +- 2^-40 of its value rounds to one float, that float is the
// correctly rounded result; otherwise (about one value in 2^15), and for
// d < 2^-60, d >= 24.5 or a quotient outside [2^-100, 2^126], the double
// evaluation decides.
__device__ __forceinline__ float hdr_inverse_rn(float d, float s, bool div,
                                                const float4* __restrict__ tab) {
  if (d == 0.0f) return d;  // -0 stays -0, as expm1(-0) = -0
  if (!(d >= 0x1p-60f && d < 24.5f)) return hdr_inverse_double(d, s, div);
  const int k = __float2int_rn(__fmul_rn(d, 32.0f));
  const float r = __fsub_rn(d, __fmul_rn(__int2float_rn(k), 0.03125f));
  const int n = k >> 5;
  const float4 t = __ldg(tab + (k & 31));
  // t = r ln 2 = th + tl
  constexpr float kLn2Hi = 0x1.62e43p-1f;
  constexpr float kLn2Lo = -0x1.05c61p-29f;
  constexpr float kSixthHi = 0x1.555556p-3f;  // 1/6 = kSixthHi + kSixthLo
  constexpr float kSixthLo = -0x1.555556p-28f;
  const float th = __fmul_rn(r, kLn2Hi);
  const float tl = __fadd_rn(__fmaf_rn(r, kLn2Hi, -th), __fmul_rn(r, kLn2Lo));
  // th^2 = p2h + p2l, th^3 = c3h + c3l, th^3 / 6 = q3h + q3l
  const float p2h = __fmul_rn(th, th);
  const float p2l = __fmaf_rn(th, th, -p2h);
  const float c3h = __fmul_rn(th, p2h);
  const float c3l = __fadd_rn(__fmaf_rn(th, p2h, -c3h), __fmul_rn(th, p2l));
  const float q3h = __fmul_rn(c3h, kSixthHi);
  const float q3l = __fadd_rn(__fmaf_rn(c3h, kSixthHi, -q3h),
                              __fadd_rn(__fmul_rn(c3h, kSixthLo), __fmul_rn(c3l, kSixthHi)));
  // e = exp(t) - 1 = eh + el (|th| >= th^2 / 2 >= |th^3 / 6| ...)
  float eh, el;
  fast_two_sum(th, __fmul_rn(0.5f, p2h), eh, el);
  const float poly = __fmaf_rn(th, __fmaf_rn(th, 1.0f / 720.0f, 1.0f / 120.0f), 1.0f / 24.0f);
  const float tail = __fmul_rn(__fmul_rn(th, c3h), poly);
  // first-order terms of tl: tl (1 + th + th^2 / 2)
  el = __fadd_rn(el, __fadd_rn(__fadd_rn(__fadd_rn(__fmul_rn(0.5f, p2l), q3l), tail),
                               __fmaf_rn(tl, __fadd_rn(th, __fmul_rn(0.5f, p2h)), tl)));
  float e2;
  fast_two_sum(eh, q3h, eh, e2);
  el = __fadd_rn(el, e2);
  // u = D + T e = uh + ul (D_j > |T_j e| for j > 0; D_0 = 0)
  const float q = __fmul_rn(t.x, eh);
  const float ql = __fmaf_rn(t.x, eh, -q);
  float uh, ul;
  fast_two_sum(t.z, q, uh, ul);
  ul = __fadd_rn(ul, __fadd_rn(__fadd_rn(__fadd_rn(t.w, ql), __fmul_rn(t.x, el)), __fmul_rn(t.y, eh)));
  // w = (2^n - 1) + (2^n - 1) u + u = z + zl (|2^n - 1| > |(2^n - 1) u| and,
  // for n >= 1, the partial sum >= 0.98 > |u|)
  const float pm1 = __int2float_rn((1 << n) - 1);
  const float a = __fmul_rn(pm1, uh);
  const float al = __fmaf_rn(pm1, uh, -a);
  float s1, e1, s2, e3;
  fast_two_sum(pm1, a, s1, e1);
  fast_two_sum(s1, uh, s2, e3);
  const float low = __fadd_rn(__fadd_rn(e1, e3), __fadd_rn(al, __fmaf_rn(pm1, ul, ul)));
  float z = __fadd_rn(s2, low);
  float zl = __fsub_rn(low, __fsub_rn(z, s2));
  if (div) {
    const float qh = __fdiv_rn(z, s);
    if (!(fabsf(qh) >= 0x1p-100f && fabsf(qh) < 0x1p126f)) return hdr_inverse_double(d, s, div);
    const float rem = __fmaf_rn(-qh, s, z);
    const float qlo = __fdiv_rn(__fadd_rn(rem, zl), s);
    z = __fadd_rn(qh, qlo);
    zl = __fsub_rn(qlo, __fsub_rn(z, qh));
  }
  const float tol = __fmul_rn(fabsf(z), 0x1p-40f);
  const float r0 = __fadd_rn(z, __fsub_rn(zl, tol));
  const float r1 = __fadd_rn(z, __fadd_rn(zl, tol));
  if (r0 == r1) return r0;
  return hdr_inverse_double(d, s, div);
}

// One output pixel from the network's rgb and the input colour (whose
// alpha is copied bit for bit): sanitize to [0, hdr ? FLT_MAX : 1], then for
// HDR the inverse transfer divided by the input scale, correctly rounded
// (a division by an input scale of 1 is exact and skipped).
__device__ __forceinline__ float4 output_pixel(float nr, float ng, float nb, float4 col, int hdr,
                                               float scale, const float4* __restrict__ exp2_tab) {
  const float hi = hdr ? FLT_MAX : 1.0f;
  float r = sanitize(nr, 0.0f, hi);
  float g = sanitize(ng, 0.0f, hi);
  float b = sanitize(nb, 0.0f, hi);
  if (hdr) {
    const bool div = scale != 1.0f;
    r = hdr_inverse_rn(r, scale, div, exp2_tab);
    g = hdr_inverse_rn(g, scale, div, exp2_tab);
    b = hdr_inverse_rn(b, scale, div, exp2_tab);
  }
  return make_float4(r, g, b, __int_as_float(__float_as_int(col.w)));
}

}  // namespace oidnx

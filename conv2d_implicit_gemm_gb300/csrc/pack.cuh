// Per-pixel steps of the fp16 input pass, shared by the input pass kernel
// and the fused input pass + enc_conv0 kernel so that both compute the same
// bits.  Source: "oidn-webgpu 0.0.0-stage -> 0.6.0, src/native/denoise.ts",
// inputShader, with the channel order of "oidn-web 0.3.4 -> 0.4.0,
// nativeUNet.ts", createInputPackShader, and the readings of its imported
// helpers:
//  * sanitize(v, lo, hi): NaN becomes 0, then clamp by comparison;
//  * 'log' transfer: F(x) = log2(1 + x).
#pragma once

#include <cfloat>
#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "passes.cuh"

namespace oidnx {

// F(s) = log2(1 + s), s in [0, FLT_MAX], correctly rounded to fp16.
// The float estimate y is within 2^-22 (relative) of F(s): log1pf is within
// 1 ulp (2^-23), the rounded constant log2(e) and the product add 2^-24
// each.  y decides the code unless y(1 -+ 1.5 * 2^-22) round differently
// (the bracket also covers the rounding of those two products).  Then the
// rounding boundary b between the two candidate codes (exact in float) is
// compared through the monotone inverse instead: F(s) >= b <=> s >= 2^b - 1,
// with 2^b - 1 from exp2f/expm1f (a few ulp).  Only when s lies within
// 2^-18 (relative) of that value is F evaluated in double precision.  The
// bracket is kept tight because FP64 is slow on this GPU and one lane on
// the double path holds up its whole warp.
__device__ __forceinline__ __half hdr_forward_f16(float s) {
  const float y = log1pf(s) * 1.44269504088896341f;
  const __half lo = __float2half_rn(y * (1.0f - 0x1.8p-22f));
  const __half hi = __float2half_rn(y * (1.0f + 0x1.8p-22f));
  if (__half_as_ushort(lo) == __half_as_ushort(hi)) return lo;
  const float b = 0.5f * (__half2float(lo) + __half2float(hi));
  const float c = b < 1.0f ? expm1f(b * 0.693147180559945309f) : exp2f(b) - 1.0f;
  if (s > c * (1.0f + 0x1p-18f)) return hi;
  if (s < c * (1.0f - 0x1p-18f)) return lo;
  return __double2half(log1p(static_cast<double>(s)) / 0.69314718055994530942);
}

// The 3 * SOURCES input channels of one image pixel: colour (HDR: times
// the input scale, sanitized to [0, FLT_MAX]; LDR: to [0, 1]), albedo
// (sanitized to [0, 1]), normal (sanitized to [-1, 1], then * 0.5 + 0.5).
template <int SOURCES, bool HDR>
__device__ __forceinline__ void input_channels(float4 c, float4 a, float4 n, float scale,
                                               float (&ch)[3 * SOURCES]) {
  constexpr int kCh = 3 * SOURCES;
  if (HDR) {
    ch[0] = sanitize(__fmul_rn(c.x, scale), 0.0f, FLT_MAX);
    ch[1] = sanitize(__fmul_rn(c.y, scale), 0.0f, FLT_MAX);
    ch[2] = sanitize(__fmul_rn(c.z, scale), 0.0f, FLT_MAX);
  } else {
    ch[0] = sanitize(c.x, 0.0f, 1.0f);
    ch[1] = sanitize(c.y, 0.0f, 1.0f);
    ch[2] = sanitize(c.z, 0.0f, 1.0f);
  }
  if (SOURCES > 1) {
    ch[3 % kCh] = sanitize(a.x, 0.0f, 1.0f);
    ch[4 % kCh] = sanitize(a.y, 0.0f, 1.0f);
    ch[5 % kCh] = sanitize(a.z, 0.0f, 1.0f);
  }
  if (SOURCES > 2) {
    ch[6 % kCh] = __fadd_rn(__fmul_rn(sanitize(n.x, -1.0f, 1.0f), 0.5f), 0.5f);
    ch[7 % kCh] = __fadd_rn(__fmul_rn(sanitize(n.y, -1.0f, 1.0f), 0.5f), 0.5f);
    ch[8 % kCh] = __fadd_rn(__fmul_rn(sanitize(n.z, -1.0f, 1.0f), 0.5f), 0.5f);
  }
}

// fp16 storage: 16 lanes = 2 chunks of 8 halves (w[0..3], w[4..7]); the
// colour lanes take the HDR transfer; lanes past 3 * SOURCES are zero.
template <int SOURCES, bool HDR>
__device__ __forceinline__ void pack_f16(const float (&ch)[3 * SOURCES], uint32_t (&w)[8]) {
  constexpr int kCh = 3 * SOURCES;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    uint32_t pair = 0;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int lane = 2 * k + e;
      if (lane < kCh) {
        const __half hv = (HDR && lane < 3) ? hdr_forward_f16(ch[lane]) : __float2half_rn(ch[lane]);
        pair |= static_cast<uint32_t>(__half_as_ushort(hv)) << (16 * e);
      }
    }
    w[k] = pair;
  }
}

}  // namespace oidnx

// Per-pixel steps of the output pass, shared by the output pass kernel and
// the final conv's fused epilogue so that both compute the same bits.
// Source: "oidn-webgpu 0.0.0-stage -> 0.6.0, src/native/denoise.ts",
// outputShader, with the readings of its imported helpers:
//  * sanitize(v, lo, hi): NaN becomes 0, then clamp by comparison;
//  * 'log' transfer: F^-1(y) = 2^y - 1.
#pragma once

#include <cfloat>
#include <cuda_runtime.h>

namespace oidnx {

__device__ __forceinline__ float sanitize(float v, float lo, float hi) {
  if (isnan(v)) v = 0.0f;
  if (v < lo) v = lo;
  else if (v > hi) v = hi;
  return v;
}

// F^-1(d) = 2^d - 1 for d >= 0: expm1 where cancellation would hurt.
__device__ __forceinline__ float hdr_inverse(float d) {
  return d < 1.0f ? expm1f(d * 0.693147180559945309f) : exp2f(d) - 1.0f;
}

// One output pixel from the network's rgb and the input colour (whose
// alpha is copied bit for bit): sanitize to [0, hdr ? FLT_MAX : 1], then for
// HDR the inverse transfer divided by the input scale.
__device__ __forceinline__ float4 output_pixel(float nr, float ng, float nb, float4 col, int hdr,
                                               float scale) {
  const float hi = hdr ? FLT_MAX : 1.0f;
  float r = sanitize(nr, 0.0f, hi);
  float g = sanitize(ng, 0.0f, hi);
  float b = sanitize(nb, 0.0f, hi);
  if (hdr) {
    r = hdr_inverse(r);
    g = hdr_inverse(g);
    b = hdr_inverse(b);
    if (scale != 1.0f) {  // a division by 1 is exact: skipped
      r = __fdiv_rn(r, scale);
      g = __fdiv_rn(g, scale);
      b = __fdiv_rn(b, scale);
    }
  }
  return make_float4(r, g, b, __int_as_float(__float_as_int(col.w)));
}

}  // namespace oidnx

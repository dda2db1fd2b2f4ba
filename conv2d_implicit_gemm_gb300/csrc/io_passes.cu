// Per-tile input pass (pack) and output pass (unpack): elementwise, one
// thread per pixel, 16-byte loads and stores, coalesced along x.
//
// Source: "oidn-webgpu 0.0.0-stage -> 0.6.0, src/native/denoise.ts",
// inputShader / outputShader, with the channel order of "oidn-web 0.3.4 ->
// 0.4.0, nativeUNet.ts", createInputPackShader.
//
// Readings of the helpers the page imports without showing them:
//  * sanitize(v, lo, hi): NaN becomes 0, then clamp by comparison;
//  * 'log' transfer: F(x) = log2(1 + x), F^-1(y) = 2^y - 1.
// The fp16 input pass stores F correctly rounded: a float estimate decides
// the fp16 code unless it lies within 2^-19 (relative) of a rounding
// boundary, in which case the value is recomputed in double precision.
#include <cfloat>

#include "internal.h"

namespace oidnx {

namespace {

__device__ __forceinline__ float sanitize(float v, float lo, float hi) {
  if (isnan(v)) v = 0.0f;
  if (v < lo) v = lo;
  else if (v > hi) v = hi;
  return v;
}

constexpr double kLn2 = 0.69314718055994530942;

// F(s) = log2(1 + s), s in [0, FLT_MAX], correctly rounded to fp16.
__device__ __forceinline__ __half hdr_forward_f16(float s) {
  const float y = log1pf(s) * 1.44269504088896341f;  // within a few ulp
  const __half lo = __float2half_rn(y * (1.0f - 0x1p-19f));
  const __half hi = __float2half_rn(y * (1.0f + 0x1p-19f));
  if (__half_as_ushort(lo) == __half_as_ushort(hi)) return lo;
  return __double2half(log1p(static_cast<double>(s)) / kLn2);
}

// F(s) rounded to fp32 from a double-precision evaluation.
__device__ __forceinline__ float hdr_forward_f32(float s) {
  return __double2float_rn(log1p(static_cast<double>(s)) / kLn2);
}

// F^-1(d) = 2^d - 1 for d >= 0: expm1 where cancellation would hurt.
__device__ __forceinline__ float hdr_inverse(float d) {
  return d < 1.0f ? expm1f(d * 0.693147180559945309f) : exp2f(d) - 1.0f;
}

__global__ void pack_kernel(const PackParams p) {
  const int tx = blockIdx.x * blockDim.x + threadIdx.x;
  const int ty = blockIdx.y;
  if (tx >= p.tw) return;
  const int ix = min(max(p.tx + tx, 0), p.width - 1);
  const int iy = min(max(p.ty + ty, 0), p.height - 1);

  float ch[9];
  __half hch[9];
  const float4 c = p.img[0][static_cast<size_t>(iy) * p.stride[0] + ix];
  const float rgb[3] = {c.x, c.y, c.z};
  for (int k = 0; k < 3; ++k) {
    if (p.hdr) {
      const float s = sanitize(__fmul_rn(rgb[k], p.scale), 0.0f, FLT_MAX);
      if (p.fp16) hch[k] = hdr_forward_f16(s);
      else ch[k] = hdr_forward_f32(s);
    } else {
      ch[k] = sanitize(rgb[k], 0.0f, 1.0f);
      hch[k] = __float2half_rn(ch[k]);
    }
  }
  if (p.sources > 1) {
    const float4 a = p.img[1][static_cast<size_t>(iy) * p.stride[1] + ix];
    ch[3] = sanitize(a.x, 0.0f, 1.0f);
    ch[4] = sanitize(a.y, 0.0f, 1.0f);
    ch[5] = sanitize(a.z, 0.0f, 1.0f);
  }
  if (p.sources > 2) {
    const float4 n = p.img[2][static_cast<size_t>(iy) * p.stride[2] + ix];
    ch[6] = __fadd_rn(__fmul_rn(sanitize(n.x, -1.0f, 1.0f), 0.5f), 0.5f);
    ch[7] = __fadd_rn(__fmul_rn(sanitize(n.y, -1.0f, 1.0f), 0.5f), 0.5f);
    ch[8] = __fadd_rn(__fmul_rn(sanitize(n.z, -1.0f, 1.0f), 0.5f), 0.5f);
  }
  const int nch = 3 * p.sources;
  const size_t pixel = static_cast<size_t>(ty) * p.chunks * p.tw + tx;
  uint4* out = static_cast<uint4*>(p.out);
  if (p.fp16) {
    for (int k = 3; k < nch; ++k) hch[k] = __float2half_rn(ch[k]);
    unsigned short bits[16];
    for (int k = 0; k < 16; ++k) bits[k] = k < nch ? __half_as_ushort(hch[k]) : 0;
    for (int j = 0; j < p.chunks; ++j) {
      uint32_t w[4];
      for (int k = 0; k < 4; ++k)
        w[k] = static_cast<uint32_t>(bits[8 * j + 2 * k]) |
               (static_cast<uint32_t>(bits[8 * j + 2 * k + 1]) << 16);
      out[pixel + static_cast<size_t>(j) * p.tw] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
    float v[12];
    for (int k = 0; k < 12; ++k) v[k] = k < nch ? ch[k] : 0.0f;
    for (int j = 0; j < p.chunks; ++j)
      reinterpret_cast<float4*>(out)[pixel + static_cast<size_t>(j) * p.tw] =
          make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
  }
}

__global__ void unpack_kernel(const UnpackParams p) {
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  const int y = blockIdx.y;
  if (x >= p.ow) return;
  const float4 net = p.net[static_cast<size_t>(y + p.in_y) * p.tw + x + p.in_x];
  const float4 col = p.color[static_cast<size_t>(y + p.oy) * p.color_stride + x + p.ox];
  const float hi = p.hdr ? FLT_MAX : 1.0f;
  float r = sanitize(net.x, 0.0f, hi);
  float g = sanitize(net.y, 0.0f, hi);
  float b = sanitize(net.z, 0.0f, hi);
  if (p.hdr) {
    r = __fdiv_rn(hdr_inverse(r), p.scale);
    g = __fdiv_rn(hdr_inverse(g), p.scale);
    b = __fdiv_rn(hdr_inverse(b), p.scale);
  }
  const float a = __int_as_float(__float_as_int(col.w));
  p.out[static_cast<size_t>(y + p.oy) * p.out_stride + x + p.ox] = make_float4(r, g, b, a);
}

}  // namespace

cudaError_t launch_pack(const PackParams& p, cudaStream_t stream) {
  dim3 grid((p.tw + 127) / 128, p.th);
  pack_kernel<<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_unpack(const UnpackParams& p, cudaStream_t stream) {
  dim3 grid((p.ow + 127) / 128, p.oh);
  unpack_kernel<<<grid, 128, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace oidnx

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
// The input pass stores F correctly rounded to the storage precision
// (hdr_forward_f16: float estimate, exact decision near rounding boundaries
// through the inverse, double precision only when that decision is too
// close to call; hdr_forward_f32: a float-float evaluation of F that decides
// the fp32 rounding unless it is too close to call, then double precision).
// The output pass stores F^-1 / inputScale correctly rounded to fp32
// (hdr_inverse_rn, passes.cuh).
#include <cfloat>
#include <cmath>

#include "internal.h"
#include "pack.cuh"
#include "passes.cuh"
#include "ptx.cuh"

namespace oidnx {

namespace {

constexpr double kLn2 = 0.69314718055994530942;

__device__ __forceinline__ float pow2_neg(int k) {  // 2^-k, 0 <= k <= 126
  return __int_as_float((127 - k) << 23);
}

// F(s) = log2(1 + s), s in [0, FLT_MAX], correctly rounded to fp32.
//  1. 1 + s = uh + ul exactly (fast two-sum), uh = m 2^e with m in [1, 2);
//     ml = ul 2^-e exactly, so 1 + s = 2^e (m + ml).
//  2. A table entry r ~ 1/m (indexed by the top 9 mantissa bits) gives
//     w = (m + ml) r - 1 as a float pair: z = m r - 1 is exact (r is a
//     multiple of 2^-10 and |z| < 2^-9), ml r is split by an FMA.
//  3. ln(1 + w) by its Taylor series, |w| < 2^-9: w - w^2/2 kept exactly as
//     a pair, the terms from w^3/3 up to w^6/6 in float, plus the first-order
//     terms in the low part of w.
//  4. F = e + (-log2 r) + ln(1 + w) log2(e), summed as float pairs.
// The pair y + yl is within 2^-40.3 |F| of F for s < 2^-9 (the float error
// of the w^3/3 term dominates there) and within 2^-42.9 |F| otherwise.  If
// y + yl -+ tol (tol = 2^-38 resp. 2^-41 of |y|) round to the same float,
// that float is the correctly rounded F; else, and for 0 < s < 2^-60 where
// the result may be subnormal, F is evaluated in double precision.
__device__ __forceinline__ float hdr_forward_f32(float s, const float4* __restrict__ tab) {
  if (s < 0x1p-60f) {
    if (s == 0.0f) return 0.0f;
    return __double2float_rn(log1p(static_cast<double>(s)) / kLn2);
  }
  const float a = fmaxf(s, 1.0f), b = fminf(s, 1.0f);
  const float uh = __fadd_rn(a, b);
  const float ul = __fsub_rn(b, __fsub_rn(uh, a));
  const uint32_t bits = __float_as_uint(uh);
  const int e = static_cast<int>(bits >> 23) - 127;
  const float m = __uint_as_float((bits & 0x7FFFFFu) | 0x3F800000u);
  const float ml = __fmul_rn(__fmul_rn(ul, pow2_neg(e >> 1)), pow2_neg(e - (e >> 1)));
  const int j = static_cast<int>((bits >> 14) & 0x1FFu);
  const float4 t = __ldg(tab + j);  // {r, -log2 r hi, lo, 0}
  const float z = __fmaf_rn(m, t.x, -1.0f);
  const float q = __fmul_rn(ml, t.x);
  const float ql = __fmaf_rn(ml, t.x, -q);
  float wh, wl;
  two_sum(z, q, wh, wl);
  wl = __fadd_rn(wl, ql);
  // ln(1 + w) = Lh + Ll
  const float p = __fmul_rn(wh, wh);
  const float pl = __fmaf_rn(wh, wh, -p);
  float poly = __fmaf_rn(wh, -1.0f / 6.0f, 0.2f);
  poly = __fmaf_rn(wh, poly, -0.25f);
  poly = __fmaf_rn(wh, poly, 1.0f / 3.0f);
  const float tail = __fmul_rn(__fmul_rn(wh, p), poly);
  float Lh, Ll;
  two_sum(wh, -0.5f * p, Lh, Ll);
  // first-order terms of wl: wl (1 - w), and -pl/2 from w^2/2
  const float corr = __fsub_rn(__fmaf_rn(-0.5f, pl, wl), __fmul_rn(__fmul_rn(wh, wl), 1.0f - wh));
  Ll = __fadd_rn(Ll, __fadd_rn(tail, corr));
  // times log2(e) = Ch + Cl
  constexpr float Ch = 0x1.715476p+0f;
  constexpr float Cl = 0x1.4ae0cp-26f;
  const float Ph = __fmul_rn(Lh, Ch);
  const float Pl = __fadd_rn(__fmaf_rn(Lh, Ch, -Ph), __fadd_rn(__fmul_rn(Lh, Cl), __fmul_rn(Ll, Ch)));
  float s1h, s1l, s2h, s2l;
  two_sum(static_cast<float>(e), t.y, s1h, s1l);
  two_sum(s1h, Ph, s2h, s2l);
  const float lo = __fadd_rn(__fadd_rn(s1l, s2l), __fadd_rn(t.z, Pl));
  const float y = __fadd_rn(s2h, lo);
  const float yl = __fsub_rn(lo, __fsub_rn(y, s2h));
  const float tol = y * ((e == 0 && j == 0) ? 0x1p-38f : 0x1p-41f);
  const float y0 = __fadd_rn(y, __fsub_rn(yl, tol));
  const float y1 = __fadd_rn(y, __fadd_rn(yl, tol));
  if (y0 == y1) return y0;
  return __double2float_rn(log1p(static_cast<double>(s)) / kLn2);
}

template <int SOURCES, bool FP16, bool HDR>
__global__ void pack_kernel(const PackParams p) {
  griddep_wait();
  griddep_launch_dependents();
  const int tx = blockIdx.x * blockDim.x + threadIdx.x;
  const int ty = p.reverse ? gridDim.y - 1 - blockIdx.y : blockIdx.y;
  if (tx >= (p.out_split && p.split_pitch > p.pitch ? p.split_pitch : p.pitch)) return;
  const size_t pixel = static_cast<size_t>(ty) * p.chunks * p.pitch + tx;
  if (tx >= p.tw || ty >= p.th) {
    // row padding, and the gap rows below a stacked tile: zeros, so that
    // 8-pixel TMA rows read zero past the tile
    if (FP16) {
      uint4* out = static_cast<uint4*>(p.out);
      if (tx < p.pitch) {
        out[pixel] = make_uint4(0u, 0u, 0u, 0u);
        out[pixel + p.pitch] = make_uint4(0u, 0u, 0u, 0u);
      }
      if (p.out_split && tx < p.split_pitch) {
        uint4* o2 = static_cast<uint4*>(p.out_split);
        const size_t half = static_cast<size_t>(p.split_pitch) >> 1;
        const size_t s0 = (static_cast<size_t>(ty) * p.chunks * 2 + (tx & 1)) * half + (tx >> 1);
        o2[s0] = make_uint4(0u, 0u, 0u, 0u);
        o2[s0 + 2 * half] = make_uint4(0u, 0u, 0u, 0u);
      }
    } else {
      float4* out = static_cast<float4*>(p.out);
      const size_t half = static_cast<size_t>(p.split_pitch) >> 1;
      for (int j = 0; j < p.chunks; ++j) {
        if (tx < p.pitch) out[pixel + static_cast<size_t>(j) * p.pitch] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (p.out_split && tx < p.split_pitch)
          static_cast<float4*>(p.out_split)[((static_cast<size_t>(ty) * p.chunks + j) * 2 + (tx & 1)) * half +
                                            (tx >> 1)] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    return;
  }
  const int ix = min(max(p.tx + tx, 0), p.width - 1);
  const int iy = min(max(p.ty + ty, 0), p.height - 1);
  constexpr int kCh = 3 * SOURCES;
  float ch[kCh];
  const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
  // the images are read once per tile here (the output pass re-reads only the
  // colour, at the end of the step; the overlaps of neighbouring tiles read
  // the same rows again, measured no slower with this policy)
  const uint64_t pol = l2_evict_first();
  const float4 c = ld_global_hint(p.img[0] + static_cast<size_t>(iy) * p.stride[0] + ix, pol);
  const float4 a = SOURCES > 1 ? ld_global_hint(p.img[1] + static_cast<size_t>(iy) * p.stride[1] + ix, pol) : zero;
  const float4 n = SOURCES > 2 ? ld_global_hint(p.img[2] + static_cast<size_t>(iy) * p.stride[2] + ix, pol) : zero;
  input_channels<SOURCES, HDR>(c, a, n, p.scale, ch);
  if (FP16) {
    uint32_t w[8];
    pack_f16<SOURCES, HDR>(ch, w);
    uint4* out = static_cast<uint4*>(p.out);
    out[pixel] = make_uint4(w[0], w[1], w[2], w[3]);
    out[pixel + p.pitch] = make_uint4(w[4], w[5], w[6], w[7]);
    if (p.out_split) {
      // column-parity split copy: plane tx & 1, index tx >> 1 (read by the
      // last decoder only: evict-first)
      uint4* o2 = static_cast<uint4*>(p.out_split);
      const size_t half = static_cast<size_t>(p.split_pitch) >> 1;
      const size_t s0 = (static_cast<size_t>(ty) * p.chunks * 2 + (tx & 1)) * half + (tx >> 1);
      st_global_hint(o2 + s0, make_uint4(w[0], w[1], w[2], w[3]), pol);
      st_global_hint(o2 + s0 + 2 * half, make_uint4(w[4], w[5], w[6], w[7]), pol);
    }
  } else {
    float v[12];
#pragma unroll
    for (int k = 0; k < 12; ++k)
      v[k] = k < kCh ? ((HDR && k < 3) ? hdr_forward_f32(ch[k], p.log2_tab) : ch[k]) : 0.0f;
    float4* out = static_cast<float4*>(p.out);
    const size_t half = static_cast<size_t>(p.split_pitch) >> 1;
#pragma unroll
    for (int j = 0; j < (kCh + 3) / 4; ++j) {
      const float4 f = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      out[pixel + static_cast<size_t>(j) * p.pitch] = f;
      // column-parity split copy: plane tx & 1, index tx >> 1
      if (p.out_split)
        static_cast<float4*>(p.out_split)[((static_cast<size_t>(ty) * p.chunks + j) * 2 + (tx & 1)) * half +
                                          (tx >> 1)] = f;
    }
  }
}

__global__ void unpack_kernel(const UnpackParams p) {
  griddep_wait();
  griddep_launch_dependents();
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  const int y = blockIdx.y;
  if (x >= p.ow) return;
  const float4 net = p.net[static_cast<size_t>(y + p.in_y) * p.tw + x + p.in_x];
  const float4 col = p.color[static_cast<size_t>(y + p.oy) * p.color_stride + x + p.ox];
  p.out[static_cast<size_t>(y + p.oy) * p.out_stride + x + p.ox] =
      output_pixel(net.x, net.y, net.z, col, p.hdr, p.scale, p.exp2_tab);
}

__global__ void split_copy_kernel(const uint4* src, int src_pitch, uint4* dst, int dst_pitch,
                                  int w, int rows) {
  griddep_wait();
  griddep_launch_dependents();
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= dst_pitch) return;
  const size_t half = static_cast<size_t>(dst_pitch) >> 1;
  for (int row = blockIdx.y; row < rows; row += gridDim.y) {  // row = y * chunks + chunk
    const uint4 v = x < w ? src[static_cast<size_t>(row) * src_pitch + x] : make_uint4(0u, 0u, 0u, 0u);
    dst[(static_cast<size_t>(row) * 2 + (x & 1)) * half + (x >> 1)] = v;
  }
}

__global__ void pitch_copy_kernel(const uint4* src, int src_pitch, uint4* dst, int dst_pitch,
                                  int w, int rows) {
  griddep_wait();
  griddep_launch_dependents();
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= dst_pitch) return;
  for (int row = blockIdx.y; row < rows; row += gridDim.y) {
    const uint4 v = x < w ? src[static_cast<size_t>(row) * src_pitch + x] : make_uint4(0u, 0u, 0u, 0u);
    dst[static_cast<size_t>(row) * dst_pitch + x] = v;
  }
}

// Failure-detection probe: one thread waits on an mbarrier that nothing
// completes, with the given limit; the bounded wait must give up, record
// kErrTimeoutProbe in the status word and return.
__global__ void wait_probe_kernel(int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait_bounded(&bar, 0, status, kErrTimeoutProbe, limit_ns);
  __syncthreads();
}

}  // namespace

cudaError_t launch_wait_probe(int* status, unsigned long long limit_ns, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

cudaError_t launch_split_copy(const void* src, int src_pitch, void* dst, int dst_pitch, int w,
                              int h, int chunks, cudaStream_t stream) {
  const int rows = h * chunks;
  dim3 grid((dst_pitch + 127) / 128, rows < 65535 ? rows : 65535);
  return launch_pdl(split_copy_kernel, grid, dim3(128), 0, stream, static_cast<const uint4*>(src),
                    src_pitch, static_cast<uint4*>(dst), dst_pitch, w, rows);
}

cudaError_t launch_pitch_copy(const void* src, int src_pitch, void* dst, int dst_pitch, int w,
                              int rows, cudaStream_t stream) {
  dim3 grid((dst_pitch + 127) / 128, rows < 65535 ? rows : 65535);
  return launch_pdl(pitch_copy_kernel, grid, dim3(128), 0, stream, static_cast<const uint4*>(src),
                    src_pitch, static_cast<uint4*>(dst), dst_pitch, w, rows);
}

template <int S, bool F16, bool HDR>
cudaError_t launch_pack_t(const PackParams& p, cudaStream_t stream) {
  const int span = p.out_split && p.split_pitch > p.pitch ? p.split_pitch : p.pitch;
  dim3 grid((span + 127) / 128, p.th + p.gap_rows);
  return launch_pdl(pack_kernel<S, F16, HDR>, grid, dim3(128), 0, stream, p);
}

template <int S>
cudaError_t launch_pack_s(const PackParams& p, cudaStream_t stream) {
  if (p.fp16) return p.hdr ? launch_pack_t<S, true, true>(p, stream) : launch_pack_t<S, true, false>(p, stream);
  return p.hdr ? launch_pack_t<S, false, true>(p, stream) : launch_pack_t<S, false, false>(p, stream);
}

cudaError_t launch_pack(const PackParams& p, cudaStream_t stream) {
  if (!p.fp16 && p.hdr && !p.log2_tab) return cudaErrorInvalidValue;
  if (p.sources == 1) return launch_pack_s<1>(p, stream);
  if (p.sources == 2) return launch_pack_s<2>(p, stream);
  return launch_pack_s<3>(p, stream);
}

void fill_log2_table(float (*tab)[4]) {
  for (int j = 0; j < kLog2TabSize; ++j) {
    // r_j = 1 / (centre of the interval), rounded to a multiple of 2^-10;
    // then |m r_j - 1| < 2^-9 over the interval, and m r_j - 1 (a multiple
    // of 2^-33) fits in a float's 24 bits.  r_0 = 1 keeps F free of
    // cancellation for small s.
    const double r = j == 0 ? 1.0 : std::nearbyint(1024.0 / (1.0 + (j + 0.5) / kLog2TabSize)) / 1024.0;
    const double g = -std::log2(r);
    const float gh = static_cast<float>(g);
    tab[j][0] = static_cast<float>(r);
    tab[j][1] = gh;
    tab[j][2] = static_cast<float>(g - static_cast<double>(gh));
    tab[j][3] = 0.0f;
  }
}

void fill_exp2_table(float (*tab)[4]) {
  for (int j = 0; j < kExp2TabSize; ++j) {
    // 2^(j/32) and 2^(j/32) - 1 in double (expm1 keeps the small ones
    // accurate to their last bit), each split into a float and the float
    // nearest its remainder
    const double t = std::exp2(j / static_cast<double>(kExp2TabSize));
    const double d = std::expm1(j * 0.69314718055994530942 / kExp2TabSize);
    const float th = static_cast<float>(t);
    const float dh = static_cast<float>(d);
    tab[j][0] = th;
    tab[j][1] = static_cast<float>(t - static_cast<double>(th));
    tab[j][2] = dh;
    tab[j][3] = static_cast<float>(d - static_cast<double>(dh));
  }
}

cudaError_t launch_unpack(const UnpackParams& p, cudaStream_t stream) {
  if (p.hdr && !p.exp2_tab) return cudaErrorInvalidValue;
  dim3 grid((p.ow + 127) / 128, p.oh);
  return launch_pdl(unpack_kernel, grid, dim3(128), 0, stream, p);
}

}  // namespace oidnx

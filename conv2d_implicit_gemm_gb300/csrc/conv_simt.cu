// fp32 same-padded 3x3 conv + bias (+ReLU, +2x2 max-pool, or final output) on
// the CUDA cores, for the fp32 precision mode.  The fp32 tolerance (relative
// L2 1e-4 per layer) is below what the tf32 tensor-core path can reach, so
// this path multiplies in plain fp32.
//
// Semantics: "oidn-web 0.3.4 -> 0.4.0, package/src/nativeUNet.ts",
// createConvShader (one output pixel per thread, taps outside the image
// skipped, bias-initialised accumulator), createFusedConvPoolShader (max over
// the valid pixels of each 2x2 window of ReLU(conv)) and
// createFusedDecoderShader (concat of the upsampled source, read at
// (x/2, y/2), and the skip source).
//
// Layout: activations [H][C/4][W][4] floats; a block of 128 threads owns 128
// consecutive pixels of one row (or pooled pixels) and one group of 8 output
// channels, whose weights it stages in shared memory.
#include "internal.h"
#include "ptx.cuh"

namespace oidnx {

namespace {

template <bool UP>
__device__ __forceinline__ void accumulate_pixel(const SimtConvParams& p, const float* wsm,
                                                 int x, int y, float (&acc)[8]) {
  const int K4 = p.C40 + p.C41;
  const float4* s0 = reinterpret_cast<const float4*>(p.src0);
  const float4* s1 = reinterpret_cast<const float4*>(p.src1);
  for (int ky = 0; ky < 3; ++ky) {
    const int iy = y + ky - 1;
    if (iy < 0 || iy >= p.H) continue;
    for (int kx = 0; kx < 3; ++kx) {
      const int ix = x + kx - 1;
      if (ix < 0 || ix >= p.W) continue;
      const float* wt = wsm + (ky * 3 + kx) * K4 * 32;
      for (int k = 0; k < p.C40; ++k) {
        const float4 v = UP ? s0[(static_cast<size_t>(iy >> 1) * p.C40 + k) * p.W0 + (ix >> 1)]
                            : s0[(static_cast<size_t>(iy) * p.C40 + k) * p.W0 + ix];
        const float* w = wt + k * 32;
        const float lanes[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int l = 0; l < 4; ++l)
#pragma unroll
          for (int o = 0; o < 8; ++o) acc[o] = fmaf(lanes[l], w[l * 8 + o], acc[o]);
      }
      for (int k = 0; k < p.C41; ++k) {
        const float4 v = s1[(static_cast<size_t>(iy) * p.C41 + k) * p.W + ix];
        const float* w = wt + (p.C40 + k) * 32;
        const float lanes[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int l = 0; l < 4; ++l)
#pragma unroll
          for (int o = 0; o < 8; ++o) acc[o] = fmaf(lanes[l], w[l * 8 + o], acc[o]);
      }
    }
  }
}

template <int MODE, bool UP>
__global__ void __launch_bounds__(128) conv3x3_simt_kernel(const SimtConvParams p) {
  extern __shared__ float wsm[];
  const int g = blockIdx.z;
  const int K4 = p.C40 + p.C41;
  const int wcount = 9 * K4 * 32;
  const float* wsrc = p.weights + static_cast<size_t>(g) * wcount;
  for (int i = threadIdx.x; i < wcount; i += blockDim.x) wsm[i] = wsrc[i];
  __syncthreads();
  griddep_wait();  // activations come from the previous kernel in the stream
  griddep_launch_dependents();
  float bias[8];
#pragma unroll
  for (int o = 0; o < 8; ++o) bias[o] = p.bias[g * 8 + o];

  float4* out = reinterpret_cast<float4*>(p.out);
  if (MODE == kEpiReluPool) {
    const int Wp = (p.W + 1) >> 1, Hp = (p.H + 1) >> 1;
    const int xp = blockIdx.x * blockDim.x + threadIdx.x, yp = blockIdx.y;
    if (xp >= Wp || yp >= Hp) return;
    float best[8];
#pragma unroll
    for (int o = 0; o < 8; ++o) best[o] = -INFINITY;
    for (int py = 0; py < 2; ++py) {
      const int y = 2 * yp + py;
      if (y >= p.H) continue;
      for (int px = 0; px < 2; ++px) {
        const int x = 2 * xp + px;
        if (x >= p.W) continue;
        float acc[8];
#pragma unroll
        for (int o = 0; o < 8; ++o) acc[o] = bias[o];
        accumulate_pixel<UP>(p, wsm, x, y, acc);
#pragma unroll
        for (int o = 0; o < 8; ++o) best[o] = fmaxf(best[o], fmaxf(acc[o], 0.0f));
      }
    }
    for (int h = 0; h < 2; ++h) {
      const int c = 2 * g + h;
      if (c < p.cout4)
        out[(static_cast<size_t>(yp) * p.cout4 + c) * Wp + xp] =
            make_float4(best[4 * h], best[4 * h + 1], best[4 * h + 2], best[4 * h + 3]);
    }
  } else {
    const int x = blockIdx.x * blockDim.x + threadIdx.x, y = blockIdx.y;
    if (x >= p.W || y >= p.H) return;
    float acc[8];
#pragma unroll
    for (int o = 0; o < 8; ++o) acc[o] = bias[o];
    accumulate_pixel<UP>(p, wsm, x, y, acc);
    if (MODE == kEpiFinal) {
      out[static_cast<size_t>(y) * p.W + x] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    } else {
#pragma unroll
      for (int o = 0; o < 8; ++o) acc[o] = fmaxf(acc[o], 0.0f);
      for (int h = 0; h < 2; ++h) {
        const int c = 2 * g + h;
        if (c < p.cout4)
          out[(static_cast<size_t>(y) * p.cout4 + c) * p.W + x] =
              make_float4(acc[4 * h], acc[4 * h + 1], acc[4 * h + 2], acc[4 * h + 3]);
      }
    }
  }
}

template <int MODE, bool UP>
cudaError_t launch_variant(const SimtConvParams& p, cudaStream_t stream) {
  const size_t smem = static_cast<size_t>(9) * (p.C40 + p.C41) * 32 * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(conv3x3_simt_kernel<MODE, UP>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  const int wide = MODE == kEpiReluPool ? (p.W + 1) / 2 : p.W;
  const int rows = MODE == kEpiReluPool ? (p.H + 1) / 2 : p.H;
  dim3 grid((wide + 127) / 128, rows, p.groups);
  return launch_pdl(conv3x3_simt_kernel<MODE, UP>, grid, dim3(128), smem, stream, p);
}

}  // namespace

cudaError_t launch_conv_simt(const SimtConvParams& p, cudaStream_t stream) {
  if (p.mode == kEpiRelu)
    return p.upsample0 ? launch_variant<kEpiRelu, true>(p, stream)
                       : launch_variant<kEpiRelu, false>(p, stream);
  if (p.mode == kEpiReluPool) return launch_variant<kEpiReluPool, false>(p, stream);
  return launch_variant<kEpiFinal, false>(p, stream);
}

}  // namespace oidnx

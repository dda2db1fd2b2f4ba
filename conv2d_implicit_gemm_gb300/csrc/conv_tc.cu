// Same-padded 3x3 conv + bias (+ReLU, +2x2 max-pool, or fp32 final output) as
// an implicit GEMM on the 5th-generation tensor cores (tcgen05, fp16 operands,
// fp32 accumulators in tensor memory).
//
// Method: "oidn-web 0.4.0 -> 0.5.0, package/src/nativeUNet.ts",
// createTiledConvShader / createTiledDecoderShader: M = output pixels,
// N = output channels, K = 9 taps x input channels; the decoder's A operand
// is concat(upsample2x(source0), source1) with the upsampled source read at
// (x/2, y/2); the encoder's fused variant ("createFusedConvPoolShader") takes
// the 2x2 max of ReLU(conv) before the store.
//
// GB300 design (not the pages'):
//  * CTA = R output rows x 128 pixels; one M=128 UMMA tile per row, each
//    with its own fp32 accumulator of N columns in TMEM.
//  * K is walked in blocks of 16 input channels.  For one block the CTA
//    stages, by one TMA box, the whole input halo: (R+2) rows x 130 pixels x
//    16 channels, zero-filled outside the image (the same padding).  Stored
//    as [row][8-channel half][pixel][8], every 8-pixel x 8-channel core
//    matrix is a contiguous 128 B run, so the 9 taps of all R rows are just
//    9R shared-memory descriptors into the same halo: a kx shift is +16 B, a
//    ky shift selects the next halo row.  No im2col copy, no re-load per tap.
//  * Weights are pre-packed on the host into the exact shared-memory image
//    of the B operand ([tap][8-channel half][N][8] per K block) and fetched
//    with one bulk copy per stage.
//  * Warp roles: warp 0 issues TMA, warp 1 allocates TMEM and issues the
//    MMAs from one thread, warps 2-5 run the epilogue (and, for decoders,
//    build the upsampled halo in shared memory from a low-resolution TMA
//    box, since nearest upsampling is not an affine TMA box).
//  * Every wait is bounded: on timeout the kernel records a bit in the
//    status word, lets its in-flight copies land, frees TMEM and returns.
#include "internal.h"
#include "ptx.cuh"

namespace oidnx {

__global__ void __launch_bounds__(kTcThreads, 1)
    conv3x3_tc_kernel(const __grid_constant__ CUtensorMap map0,
                      const __grid_constant__ CUtensorMap map1, const TcConvParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;

  const int S = p.S, R = p.R, N = p.N, KB0 = p.KB0;
  const int KB = p.KB0 + p.KB1;
  uint8_t* A = smem;
  uint8_t* B = A + static_cast<size_t>(S) * p.a_stage;
  uint8_t* ST = B + static_cast<size_t>(S) * p.b_stage;
  uint64_t* full = reinterpret_cast<uint64_t*>(ST + static_cast<size_t>(S) * p.st_stage);
  uint64_t* empty = full + S;
  uint64_t* xdone = empty + S;
  uint64_t* accum = xdone + S;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int x0 = blockIdx.x * kTileM;
  const int y0 = blockIdx.y * R;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&xdone[s], 128);
    }
    mbar_init(accum, 1);
    fence_mbarrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&map0);
      if (p.KB1 > 0) prefetch_tmap(&map1);
      int issued = 0;
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % S;
        const uint32_t round = static_cast<uint32_t>(kb / S);
        if (!mbar_wait_bounded(&empty[s], (round & 1u) ^ 1u, p.status, kErrTimeoutProducer)) break;
        const bool low = p.upsample0 && kb < KB0;
        mbar_arrive_expect_tx(&full[s], (low ? p.st_tx : p.a_tx) + p.b_tx);
        if (kb < KB0) {
          if (low)
            tma_load_4d(ST + static_cast<size_t>(s) * p.st_stage, &map0, &full[s], 0,
                        (x0 >> 1) - 1, 2 * kb, (y0 >> 1) - 1);
          else
            tma_load_4d(A + static_cast<size_t>(s) * p.a_stage, &map0, &full[s], 0, x0 - 1,
                        2 * kb, y0 - 1);
        } else {
          tma_load_4d(A + static_cast<size_t>(s) * p.a_stage, &map1, &full[s], 0, x0 - 1,
                      2 * (kb - KB0), y0 - 1);
        }
        bulk_load(B + static_cast<size_t>(s) * p.b_stage,
                  reinterpret_cast<const uint8_t*>(p.weights) + static_cast<size_t>(kb) * p.b_tx,
                  p.b_tx, &full[s]);
        issued = kb + 1;
      }
      // Every copy issued must have landed before this CTA may exit.
      for (int kb = issued > S ? issued - S : 0; kb < issued; ++kb)
        mbar_wait_bounded(&full[kb % S], static_cast<uint32_t>(kb / S) & 1u, p.status,
                          kErrTimeoutDrain);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_f16_f32(kTileM, N);
      const uint32_t a_base = smem_u32(A);
      const uint32_t b_base = smem_u32(B);
      const uint32_t b_tap = 2u * N * kChunkBytes;
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % S;
        const uint32_t par = static_cast<uint32_t>(kb / S) & 1u;
        bool ok = mbar_wait_bounded(&full[s], par, p.status, kErrTimeoutMma);
        if (ok && p.upsample0 && kb < KB0)
          ok = mbar_wait_bounded(&xdone[s], par, p.status, kErrTimeoutMma);
        if (!ok) break;
        tc_fence_after();
        const uint32_t a_s = a_base + s * p.a_stage;
        const uint32_t b_s = b_base + s * p.b_stage;
#pragma unroll 1
        for (int t = 0; t < 9; ++t) {
          const int ky = t / 3, kx = t - 3 * (t / 3);
          const uint64_t bdesc =
              smem_desc_noswizzle(b_s + t * b_tap, static_cast<uint32_t>(N) * kChunkBytes, 128);
#pragma unroll 1
          for (int r = 0; r < R; ++r) {
            const uint32_t a_off = (static_cast<uint32_t>(r + ky) * 2u * kHaloPx + kx) * kChunkBytes;
            const uint64_t adesc = smem_desc_noswizzle(a_s + a_off, kHaloPx * kChunkBytes, 128);
            mma_f16_ss(tmem + static_cast<uint32_t>(r * N), adesc, bdesc, idesc,
                       (kb | t) != 0 ? 1u : 0u);
          }
        }
        mma_commit(&empty[s]);
      }
      mma_commit(accum);
      // TMEM is freed only after every MMA issued above has completed.
      mbar_wait_bounded(accum, 0, p.status, kErrTimeoutMma);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 64;  // 0..127
    if (p.upsample0) {
      // Build the full-resolution halo of the upsampled source in the A stage.
      const int ly0 = (y0 >> 1) - 1, lx0 = (x0 >> 1) - 1;
      const int total = (R + 2) * 2 * kHaloPx;
      for (int kb = 0; kb < KB0; ++kb) {
        const int s = kb % S;
        const uint32_t par = static_cast<uint32_t>(kb / S) & 1u;
        if (!mbar_wait_bounded(&full[s], par, p.status, kErrTimeoutEpilogue)) break;
        const uint4* src = reinterpret_cast<const uint4*>(ST + static_cast<size_t>(s) * p.st_stage);
        uint4* dst = reinterpret_cast<uint4*>(A + static_cast<size_t>(s) * p.a_stage);
        for (int i = et; i < total; i += 128) {
          const int px = i % kHaloPx;
          const int rc = i / kHaloPx;
          const int j = rc & 1, rr = rc >> 1;
          const int iy = y0 - 1 + rr, ix = x0 - 1 + px;
          uint4 v = make_uint4(0u, 0u, 0u, 0u);
          if (iy >= 0 && iy < p.H && ix >= 0 && ix < p.W) {
            const int sr = (iy >> 1) - ly0, sc = (ix >> 1) - lx0;
            v = src[(sr * 2 + j) * kLowPx + sc];
          }
          dst[i] = v;
        }
        fence_proxy_async_smem();
        mbar_arrive(&xdone[s]);
      }
    }

    mbar_wait_bounded(accum, 0, p.status, kErrTimeoutEpilogue);
    tc_fence_after();
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int m = q * 32 + lane;     // pixel in the M tile = TMEM lane
    const int x = x0 + m;
    const uint32_t tl = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const int nc = N / 16;

    if (p.mode == kEpiRelu) {
      __half* out = static_cast<__half*>(p.out);
      const int C8 = N / 8;
      for (int r = 0; r < R; ++r) {
        const int y = y0 + r;
        const bool valid = x < p.W && y < p.H;
        for (int c = 0; c < nc; ++c) {
          float v[16];
          tmem_ld16(tl + static_cast<uint32_t>(r * N + c * 16), v);
          uint32_t h[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float a = fmaxf(v[2 * k] + __ldg(&p.bias[c * 16 + 2 * k]), 0.0f);
            const float b = fmaxf(v[2 * k + 1] + __ldg(&p.bias[c * 16 + 2 * k + 1]), 0.0f);
            h[k] = pack_half2(a, b);
          }
          if (valid) {
            const size_t base0 = ((static_cast<size_t>(y) * C8 + 2 * c) * p.W + x) * 8;
            const size_t base1 = ((static_cast<size_t>(y) * C8 + 2 * c + 1) * p.W + x) * 8;
            *reinterpret_cast<uint4*>(out + base0) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(out + base1) = make_uint4(h[4], h[5], h[6], h[7]);
          }
        }
      }
    } else if (p.mode == kEpiReluPool) {
      __half* out = static_cast<__half*>(p.out);
      const int C8 = N / 8;
      const int Wp = (p.W + 1) >> 1, Hp = (p.H + 1) >> 1;
      for (int i = 0; i < R / 2; ++i) {
        const int ya = y0 + 2 * i;
        const bool va = x < p.W && ya < p.H;
        const bool vb = x < p.W && ya + 1 < p.H;
        const int yp = ya >> 1, xp = x >> 1;
        const bool store = ((lane & 1) == 0) && xp < Wp && yp < Hp;
        for (int c = 0; c < nc; ++c) {
          float va16[16], vb16[16];
          tmem_ld16(tl + static_cast<uint32_t>((2 * i) * N + c * 16), va16);
          tmem_ld16(tl + static_cast<uint32_t>((2 * i + 1) * N + c * 16), vb16);
          float mx[16];
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float bk = __ldg(&p.bias[c * 16 + k]);
            const float a = va ? fmaxf(va16[k] + bk, 0.0f) : -INFINITY;
            const float b = vb ? fmaxf(vb16[k] + bk, 0.0f) : -INFINITY;
            float t = fmaxf(a, b);
            t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 1));
            mx[k] = t;
          }
          if (store) {
            uint32_t h[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) h[k] = pack_half2(mx[2 * k], mx[2 * k + 1]);
            const size_t base0 = ((static_cast<size_t>(yp) * C8 + 2 * c) * Wp + xp) * 8;
            const size_t base1 = ((static_cast<size_t>(yp) * C8 + 2 * c + 1) * Wp + xp) * 8;
            *reinterpret_cast<uint4*>(out + base0) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(out + base1) = make_uint4(h[4], h[5], h[6], h[7]);
          }
        }
      }
    } else {
      float4* out = static_cast<float4*>(p.out);
      const float b0 = __ldg(&p.bias[0]), b1 = __ldg(&p.bias[1]);
      const float b2 = __ldg(&p.bias[2]), b3 = __ldg(&p.bias[3]);
      for (int r = 0; r < R; ++r) {
        const int y = y0 + r;
        float v[16];
        tmem_ld16(tl + static_cast<uint32_t>(r * N), v);
        if (x < p.W && y < p.H)
          out[static_cast<size_t>(y) * p.W + x] = make_float4(v[0] + b0, v[1] + b1, v[2] + b2, v[3] + b3);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

cudaError_t launch_conv_tc(const TcConvLaunch& L, cudaStream_t stream) {
  conv3x3_tc_kernel<<<L.grid, kTcThreads, L.smem, stream>>>(L.map0, L.map1, L.p);
  return cudaGetLastError();
}

cudaError_t conv_tc_set_smem_limit(size_t bytes) {
  return cudaFuncSetAttribute(conv3x3_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(bytes));
}

cudaError_t conv_tc_occupancy(size_t smem, int* blocks_per_sm) {
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, conv3x3_tc_kernel,
                                                       kTcThreads, smem);
}

}  // namespace oidnx

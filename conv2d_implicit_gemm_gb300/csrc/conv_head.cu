// The input pass and the U-Net's first layer in one kernel, fp16 storage:
// the packed input (9 channels in 16 lanes) of each conv tile's halo is
// computed from the source images straight into shared memory, in the
// layout enc_conv0's MMAs read, and never written in full to memory; only
// its column-parity copy, which dec_conv1a reads as its skip source, is
// stored.  What each step computes is the input pass of "oidn-webgpu
// 0.0.0-stage -> 0.6.0, src/native/denoise.ts" (inputShader, per-pixel code
// shared with the input pass kernel in pack.cuh) and the conv layer of
// "oidn-web 0.4.0 -> 0.5.0, package/src/nativeUNet.ts" (bias + ReLU).
//
// GB300 design (not the pages'):
//  * Persistent CTAs walk conv tiles of kHeadRows rows x 128 pixels (last
//    to first: the next layer then starts on the rows written last).
//  * One thread stages, per tile and source image, the kHeadRows + 2 halo
//    rows x 132 pixels from row min(ty + y0 - 1, height - 1) and column
//    min(tx + x0 - 1, width - 1), which hold every clamp-to-edge source
//    pixel of the halo: three TMA boxes of 44 pixels each, the image taken
//    as rows of floats so that a box row is 704 contiguous bytes (boxes of
//    16-byte rows load far slower).
//  * Sixteen pack warps turn the staged pixels into the packed input
//    [row][8-lane half][pixel][8 halves] (a pixel outside the tile's input
//    rectangle is zero: the conv's same padding) and store the tile's own
//    pixels into the column-parity copy.
//  * One warp issues the MMAs: one K block (16 lanes), ky stacked along N
//    (N <= 96), accumulators started from the bias, in the per-row order
//    (kx, ky) of the plain conv kernel, so the values equal that kernel's
//    bit for bit.  Two accumulator sets in tensor memory.
//  * Four epilogue warps apply ReLU, store fp16 and refill the bias.
//  Every wait is bounded.
#include "internal.h"
#include "pack.cuh"
#include "ptx.cuh"

namespace oidnx {

namespace {

constexpr int kHeadPackWarps = 16;
constexpr int kHeadEpiWarps = 4;                    // one per TMEM lane quarter
constexpr int kHeadThreads = 32 * (2 + kHeadPackWarps + kHeadEpiWarps);
constexpr int kHeadN = 32;                          // enc_conv0's output channels
constexpr int kHeadPx = kTileM + 2;                 // 130 staged pixels per halo row
constexpr uint32_t kHeadLbo = kHeadPx * kChunkBytes;                // 2080 B: one 8-lane half
constexpr uint32_t kHeadRowBytes = 2 * kHeadLbo;                    // 4160 B per halo row
constexpr uint32_t kHeadWBytes = 3u * 2u * 3u * kHeadN * kChunkBytes;  // [kx][half][ky][32][8]: 9216 B
constexpr int kHeadSubPx = 44;                                      // pixels per image box
constexpr uint32_t kHeadSubBox = (kHeadRows + 2) * kHeadSubPx * 16;   // 7040 B
constexpr uint32_t kHeadImgSlot = 3 * kHeadSubBox;                    // 21120 B: one image, 132 pixels

__device__ __forceinline__ void head_tile(const HeadParams& p, int t, int* x0, int* y0) {
  t = p.tiles_x * p.tiles_y - 1 - t;  // last to first
  const int ty = t / p.tiles_x;
  *x0 = (t - ty * p.tiles_x) * kTileM;
  *y0 = ty * kHeadRows;
}

// First image row and column of a tile's staged boxes.
__device__ __forceinline__ void head_box(const HeadParams& p, int x0, int y0, int* col0, int* row0) {
  *col0 = min(p.tx + x0 - 1, p.width - 1);
  *row0 = min(p.ty + y0 - 1, p.height - 1);
}

}  // namespace

template <int SOURCES, bool HDR>
__global__ void __launch_bounds__(kHeadThreads, 1)
    conv3x3_head_kernel(const __grid_constant__ CUtensorMap map0, const __grid_constant__ CUtensorMap map1,
                        const __grid_constant__ CUtensorMap map2, const HeadParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (128u - (smem_u32(smem_raw) & 127u)) & 127u;
  uint8_t* smem = smem_raw + pad;
  const int SI = p.SI, SA = p.SA;
  constexpr int R = kHeadRows;
  // shared memory: [image stages][packed stages][weights][bias][barriers]
  uint8_t* IMG = smem;
  uint8_t* A = IMG + static_cast<size_t>(SI) * p.img_stage;
  uint8_t* W = A + static_cast<size_t>(SA) * p.a_stage;
  float* bias_s = reinterpret_cast<float*>(W + kHeadWBytes);
  uint64_t* ifull = reinterpret_cast<uint64_t*>(bias_s + kHeadN);
  uint64_t* iempty = ifull + SI;
  uint64_t* full = iempty + SI;
  uint64_t* empty = full + SA;
  uint64_t* tfull = empty + SA;   // [set]: a tile's MMAs finished
  uint64_t* tempty = tfull + 2;   // [set]: accumulators read and refilled
  uint64_t* wbar = tempty + 2;
  uint64_t* done = wbar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_tiles = p.tiles_x * p.tiles_y;
  constexpr uint32_t kSetCols = R * kHeadN;  // 256

  if (threadIdx.x == 0) {
    for (int s = 0; s < SI; ++s) {
      mbar_init(&ifull[s], 1);
      mbar_init(&iempty[s], 32 * kHeadPackWarps);
    }
    for (int s = 0; s < SA; ++s) {
      mbar_init(&full[s], 32 * kHeadPackWarps);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 32 * kHeadEpiWarps);
    }
    mbar_init(wbar, 1);
    mbar_init(done, 1);
    fence_mbarrier_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, 2 * kSetCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      mbar_arrive_expect_tx(wbar, kHeadWBytes);
      bulk_load(W, p.weights, kHeadWBytes, wbar);
    }
    __syncwarp();
    const uint32_t idn[4] = {0u, idesc_f16_f32(kTileM, kHeadN), idesc_f16_f32(kTileM, 2 * kHeadN),
                             idesc_f16_f32(kTileM, 3 * kHeadN)};
    // A: halo row h at h * kHeadRowBytes, pixel x0 - 1 + i + kx at index
    // i + kx; B per kx: [8-lane half][ky stack][32][8]
    const uint64_t a0 = smem_desc_noswizzle(smem_u32(A), kHeadLbo, 128);
    const uint64_t b0 = smem_desc_noswizzle(smem_u32(W), 3u * kHeadN * kChunkBytes, 128);
    bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(wbar, 0, p.status, kErrTimeoutMma));
    uint32_t s = 0, ph = 0, tcount = 0;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++tcount) {
      const uint32_t b = tcount & 1u;
      ok = __all_sync(0xffffffffu,
                      mbar_wait_bounded(&tempty[b], (tcount >> 1) & 1u, p.status, kErrTimeoutMma) &&
                          mbar_wait_bounded(&full[s], ph, p.status, kErrTimeoutMma));
      if (!ok) break;
      tc_fence_after();
      const uint64_t ad = a0 + ((s * p.a_stage) >> 4);
      const uint32_t d = tmem + b * kSetCols;
      if (elect_one()) {
        // halo row h updates rows max(0, h - 2) .. min(R - 1, h) with the
        // ky-stacked B block (rows (2 - ky) * 32 ..)
#pragma unroll
        for (int kx = 0; kx < 3; ++kx)
#pragma unroll
          for (int h = 0; h < R + 2; ++h) {
            const int lo = h - 2 > 0 ? h - 2 : 0;
            const int hi = h < R - 1 ? h : R - 1;
            mma_f16_ss(d + static_cast<uint32_t>(lo * kHeadN),
                       ad + static_cast<uint32_t>(h * (kHeadRowBytes >> 4) + kx),
                       b0 + static_cast<uint32_t>(kx * 6 * kHeadN + (2 - h + lo) * kHeadN), idn[hi - lo + 1],
                       1u);
          }
        mma_commit(&empty[s]);
        mma_commit(&tfull[b]);
      }
      __syncwarp();
      if (++s == static_cast<uint32_t>(SA)) {
        s = 0;
        ph ^= 1u;
      }
    }
    // TMEM is freed only after every MMA issued above has completed.
    if (elect_one()) mma_commit(done);
    mbar_wait_bounded(done, 0, p.status, kErrTimeoutMma);
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ image staging
    if (lane == 0) {
      prefetch_tmap(&map0);
      if (SOURCES > 1) prefetch_tmap(&map1);
      if (SOURCES > 2) prefetch_tmap(&map2);
      uint32_t s = 0, ph = 0;
      for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
        int x0, y0, col0, row0;
        head_tile(p, tile, &x0, &y0);
        head_box(p, x0, y0, &col0, &row0);
        if (!mbar_wait_bounded(&iempty[s], ph ^ 1u, p.status, kErrTimeoutProducer)) break;
        mbar_arrive_expect_tx(&ifull[s], SOURCES * kHeadImgSlot);
        uint8_t* st = IMG + static_cast<size_t>(s) * p.img_stage;
        // x in floats: 4 per pixel (a multiple of 16 bytes)
#pragma unroll
        for (int b = 0; b < 3; ++b) {
          const int xf = 4 * (col0 + b * kHeadSubPx);
          // (one-tile frames only: the images read once, evict-first)
          tma_load_2d(st + b * kHeadSubBox, &map0, &ifull[s], xf, row0, l2_evict_first());
          if (SOURCES > 1)
            tma_load_2d(st + kHeadImgSlot + b * kHeadSubBox, &map1, &ifull[s], xf, row0, l2_evict_first());
          if (SOURCES > 2)
            tma_load_2d(st + 2 * kHeadImgSlot + b * kHeadSubBox, &map2, &ifull[s], xf, row0, l2_evict_first());
        }
        if (++s == static_cast<uint32_t>(SI)) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else if (warp < 2 + kHeadPackWarps) {
    // ------------------------------------------------------------ pack warps
    // Halo pixel i (row i / 130, column i % 130) = tile pixel (y0 - 1 +
    // row, x0 - 1 + column); consecutive threads take consecutive pixels.
    const int pt = threadIdx.x - 64;  // 0 .. 32 * kHeadPackWarps - 1
    // the buffers written here may still be read by the previous grid
    griddep_wait();
    uint32_t si = 0, phi = 0, sa = 0, pha = 0;
    const size_t half = static_cast<size_t>(p.split_pitch) >> 1;
    uint4* split = static_cast<uint4*>(p.split);
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      int x0, y0, col0, row0;
      head_tile(p, tile, &x0, &y0);
      head_box(p, x0, y0, &col0, &row0);
      if (!mbar_wait_bounded(&ifull[si], phi, p.status, kErrTimeoutEpilogue)) break;
      if (!mbar_wait_bounded(&empty[sa], pha ^ 1u, p.status, kErrTimeoutEpilogue)) break;
      const float4* img = reinterpret_cast<const float4*>(IMG + static_cast<size_t>(si) * p.img_stage);
      uint8_t* st = A + static_cast<size_t>(sa) * p.a_stage;
      for (int i = pt; i < (R + 2) * kHeadPx; i += 32 * kHeadPackWarps) {
        const int r = i / kHeadPx, c = i - r * kHeadPx;
        const int y = y0 - 1 + r, x = x0 - 1 + c;
        uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        if (x >= 0 && x < p.tw && y >= 0 && y < p.th) {
          // clamp-to-edge source pixel, inside the staged boxes: box bx / 44,
          // row by, pixel bx % 44
          const int bx = min(max(p.tx + x, 0), p.width - 1) - col0;
          const int by = min(max(p.ty + y, 0), p.height - 1) - row0;
          const int sub = bx / kHeadSubPx;
          const int e = sub * static_cast<int>(kHeadSubBox / 16) + by * kHeadSubPx + (bx - sub * kHeadSubPx);
          const float4 zero = make_float4(0.f, 0.f, 0.f, 0.f);
          const float4 cv = img[e];
          const float4 av = SOURCES > 1 ? img[kHeadImgSlot / 16 + e] : zero;
          const float4 nv = SOURCES > 2 ? img[2 * (kHeadImgSlot / 16) + e] : zero;
          float ch[3 * SOURCES];
          input_channels<SOURCES, HDR>(cv, av, nv, p.scale, ch);
          pack_f16<SOURCES, HDR>(ch, w);
        }
        uint4* sp = reinterpret_cast<uint4*>(st + r * kHeadRowBytes + c * kChunkBytes);
        sp[0] = make_uint4(w[0], w[1], w[2], w[3]);
        sp[kHeadPx] = make_uint4(w[4], w[5], w[6], w[7]);
        // the tile's own pixels into the column-parity copy (plane x & 1,
        // entry x >> 1; entries of columns >= tw are zero)
        if (r >= 1 && r <= R && c >= 1 && c <= kTileM && y < p.th && x < p.split_pitch) {
          const size_t s0 = (static_cast<size_t>(y) * 2 * 2 + (x & 1)) * half + (x >> 1);
          split[s0] = make_uint4(w[0], w[1], w[2], w[3]);
          split[s0 + 2 * half] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
      mbar_arrive(&iempty[si]);  // the image stage has been read
      fence_proxy_async_smem();  // the packed stage is read by the tensor cores
      mbar_arrive(&full[sa]);
      if (++si == static_cast<uint32_t>(SI)) {
        si = 0;
        phi ^= 1u;
      }
      if (++sa == static_cast<uint32_t>(SA)) {
        sa = 0;
        pha ^= 1u;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp w reads TMEM lane quarter w % 4 (pixel x0 + m of the tile), all
    // rows.
    const int q = warp & 3;
    constexpr int sub = 0, kRowStep = kHeadEpiWarps / 4;
    const int m = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int et = threadIdx.x - 32 * (2 + kHeadPackWarps);
    if (et < kHeadN) bias_s[et] = p.bias[et];
    named_barrier_sync(1, 32 * kHeadEpiWarps);
    uint32_t bz[2][16];
    bias16_regs(bias_s, bz[0]);
    bias16_regs(bias_s + 16, bz[1]);
    for (uint32_t b = 0; b < 2; ++b)
      for (int r = sub; r < R; r += kRowStep) {
        const uint32_t t0 = tmem + lane_off + b * kSetCols + static_cast<uint32_t>(r * kHeadN);
        tmem_st16(t0, bz[0]);
        tmem_st16(t0 + 16, bz[1]);
      }
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&tempty[0]);  // completion 0 of each: the first tiles start from the bias
    mbar_arrive(&tempty[1]);
    __half* out = p.out;
    uint32_t tcount = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++tcount) {
      const uint32_t buf = tcount & 1u;
      if (!mbar_wait_bounded(&tfull[buf], (tcount >> 1) & 1u, p.status, kErrTimeoutEpilogue)) break;
      tc_fence_after();
      int x0, y0;
      head_tile(p, tile, &x0, &y0);
      const int x = x0 + m;
      const uint32_t tl = tmem + lane_off + buf * kSetCols;
      for (int r = sub; r < R; r += kRowStep) {
        const int y = y0 + r;
        uint32_t v[2][16];
        const uint32_t t0 = tl + static_cast<uint32_t>(r * kHeadN);
        tmem_ld16_nowait(t0, v[0]);
        tmem_ld16_nowait(t0 + 16, v[1]);
        tmem_wait_ld();
        tmem_st16(t0, bz[0]);
        tmem_st16(t0 + 16, bz[1]);
        // columns [tw, pitch) are row padding: stored as zeros
        if (x < p.pitch && y < p.th) {
          const bool padc = x >= p.tw;
          __half* row = out + (static_cast<size_t>(y) * 4 * p.pitch + x) * 8;
#pragma unroll
          for (int b = 0; b < 2; ++b) {
            uint32_t h[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
              h[k] = padc ? 0u
                          : pack_half2(fmaxf(__uint_as_float(v[b][2 * k]), 0.0f),
                                       fmaxf(__uint_as_float(v[b][2 * k + 1]), 0.0f));
            const size_t c8 = 2 * b;
            *reinterpret_cast<uint4*>(row + c8 * p.pitch * 8) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4*>(row + (c8 + 1) * p.pitch * 8) = make_uint4(h[4], h[5], h[6], h[7]);
          }
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&tempty[buf]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kSetCols);
  }
}

namespace {

template <int S, bool HDR>
cudaError_t launch_head_t(const HeadLaunch& L, cudaStream_t stream) {
  return launch_pdl(conv3x3_head_kernel<S, HDR>, L.grid, dim3(kHeadThreads), L.smem, stream, L.map[0],
                    L.map[1], L.map[2], L.p);
}

template <int S, bool HDR>
cudaError_t head_limit_t(int bytes) {
  return cudaFuncSetAttribute(conv3x3_head_kernel<S, HDR>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

}  // namespace

cudaError_t launch_conv_head(const HeadLaunch& L, cudaStream_t stream) {
  const bool hdr = L.p.hdr != 0;
  switch (L.p.sources) {
    case 1: return hdr ? launch_head_t<1, true>(L, stream) : launch_head_t<1, false>(L, stream);
    case 2: return hdr ? launch_head_t<2, true>(L, stream) : launch_head_t<2, false>(L, stream);
    default: return hdr ? launch_head_t<3, true>(L, stream) : launch_head_t<3, false>(L, stream);
  }
}

cudaError_t conv_head_set_smem_limit(size_t bytes) {
  const int b = static_cast<int>(bytes);
  cudaError_t e = cudaSuccess;
  if (e == cudaSuccess) e = head_limit_t<1, true>(b);
  if (e == cudaSuccess) e = head_limit_t<1, false>(b);
  if (e == cudaSuccess) e = head_limit_t<2, true>(b);
  if (e == cudaSuccess) e = head_limit_t<2, false>(b);
  if (e == cudaSuccess) e = head_limit_t<3, true>(b);
  if (e == cudaSuccess) e = head_limit_t<3, false>(b);
  return e;
}

}  // namespace oidnx

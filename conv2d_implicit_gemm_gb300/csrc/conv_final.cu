// The U-Net's last layer, dec_conv0 (32 -> 3 channels, bias, no ReLU, fp32
// output), as its own tcgen05 kernel; optionally the output pass runs in
// its epilogue.  What it computes is the final conv of "oidn-web 0.4.0 ->
// 0.5.0, package/src/nativeUNet.ts" and, when fused, the output pass of
// "oidn-webgpu 0.0.0-stage -> 0.6.0, src/native/denoise.ts" (outputShader).
//
// GB300 design (not the pages'):
//  * With three output channels the generic kernel's MMAs (N = 3 ky x 16,
//    one per kx) are bound by their operand reads, not their math.  Here the
//    three kx taps are folded into N as well: B rows 16 (2 - ky) + 4 kx + co,
//    so one MMA per halo row and K block computes, for each pixel, the kx
//    partial sums of all three taps.  The epilogue adds the kx = 1 and 2
//    partials of pixels m + 1 and m + 2 (warp shuffles; shared memory across
//    warps) to pixel m's kx = 0 partial.  A tile is kFinalRows rows x 126 output
//    pixels, computed from 128 input pixels starting one left of it.
//  * Otherwise the structure of the generic kernel: persistent CTAs, one TMA
//    box per K block holding the halo (rows y0 - 1 .. y0 + kFinalRows, 144
//    pixels from the 8-pixel boundary at or left of x0 - 1), ky stacked
//    along N, two bias-started accumulator sets in TMEM, bounded waits.
//  * The fused output pass reads the tile's input colour and writes the
//    output image in place of the separate output pass kernel, which would
//    re-read the network output from HBM.
//  * fp32 storage (TF): K blocks of 8 channels, each product as three tf32
//    MMAs (A B_hi + A B_lo + A_lo B_hi) as in the generic kernel; four helper
//    warps split every staged box into A_hi (in place) and A_lo.
#include "internal.h"
#include "passes.cuh"
#include "ptx.cuh"

namespace oidnx {

namespace {

constexpr int kEpiWarps = 16;       // four per TMEM lane quarter
// TMA, MMA, epilogue warps, and for tf32 four helper warps
template <bool TF> constexpr int final_threads() { return 32 * (2 + kEpiWarps + (TF ? 4 : 0)); }
constexpr int kSubs = kEpiWarps / 4;  // epilogue warps per lane quarter
constexpr int kNc = 16;             // accumulator columns per output row (12 used)
constexpr int kR = kFinalRows;

__device__ __forceinline__ void final_tile(const FinalConvParams& p, int tile, int* x0, int* y0) {
  if (p.reverse) tile = p.tiles_x * p.tiles_y - 1 - tile;
  const int ty = tile / p.tiles_x;
  *x0 = (tile - ty * p.tiles_x) * kFinalSpan;
  *y0 = ty * kR;
}

// The MMAs of one K block: halo row h updates output rows
// max(0, h - 2) .. min(kR - 1, h) (ky stacked), one MMA each.
template <bool TF>
__device__ __forceinline__ void final_kblock(uint64_t ad, uint64_t bd, uint32_t dbase, uint32_t id1,
                                             uint32_t id2, uint32_t id3) {
  if (!elect_one()) return;  // one lane issues the K block's MMAs
#pragma unroll
  for (int h = 0; h < kR + 2; ++h) {
    const int lo = h - 2 > 0 ? h - 2 : 0;
    const int hi = h < kR - 1 ? h : kR - 1;
    const int n = hi - lo + 1;
    const uint32_t d = dbase + static_cast<uint32_t>(lo * kNc);
    const uint64_t a = ad + static_cast<uint32_t>(h * 2 * kHaloW);
    const uint64_t b = bd + static_cast<uint32_t>((2 - h + lo) * kNc);
    const uint32_t id = n == 1 ? id1 : (n == 2 ? id2 : id3);
    if (TF) mma_tf32_ss(d, a, b, id);
    else mma_f16_ss(d, a, b, id, 1u);
  }
}

}  // namespace

template <bool OUT, bool TF>
__global__ void __launch_bounds__(final_threads<TF>(), 1)
    conv3x3_final_kernel(const __grid_constant__ CUtensorMap map, const FinalConvParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;
  const int S = p.S;
  // 32 input channels: two K blocks of 16 (fp16) or four of 8 (tf32, each
  // with its B_hi then its B_lo)
  constexpr int kKB = TF ? 4 : 2;
  constexpr uint32_t kWkbBytes = (TF ? 2u : 1u) * 2u * 3u * kNc * kChunkBytes;
  constexpr uint32_t kWBytes = kKB * kWkbBytes;
  // shared memory: [stages][A_lo stages (tf32)][weights][boundary [sub][2
  // buf][4 quarter][rows][3]][bias][barriers]
  uint8_t* A = smem;
  uint8_t* ALO = A + static_cast<size_t>(S) * p.stage_bytes;
  uint8_t* Wsm = ALO + (TF ? static_cast<size_t>(S) * p.stage_bytes : 0u);
  float4* BND = reinterpret_cast<float4*>(Wsm + kWBytes);
  float* bias_s = reinterpret_cast<float*>(BND + kSubs * 2 * 4 * (kR / kSubs) * 3);
  uint64_t* full = reinterpret_cast<uint64_t*>(bias_s + kNc);
  uint64_t* empty = full + S;
  uint64_t* xdone = empty + S;   // [S] tf32: stage split by the helper warps
  uint64_t* tfull = xdone + (TF ? S : 0);   // [2]
  uint64_t* tempty = tfull + 2;  // [2]
  uint64_t* xbar = tempty + 2;   // [sub][2 buf] boundary values written
  uint64_t* wbar = xbar + 2 * kSubs;
  uint64_t* done = wbar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_tiles = p.tiles_x * p.tiles_y;
  constexpr uint32_t kSetCols = kR * kNc;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      if (TF) mbar_init(&xdone[s], 128);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 32 * kEpiWarps);
    }
    for (int k = 0; k < 2 * kSubs; ++k) mbar_init(&xbar[k], 128);
    mbar_init(wbar, 1);
    mbar_init(done, 1);
    fence_mbarrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 2 * kSetCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&map);
      mbar_arrive_expect_tx(wbar, kWBytes);
      bulk_load(Wsm, p.w, kWBytes, wbar);
      griddep_wait();
      const uint64_t pol = p.l2_first ? l2_evict_first() : l2_evict_normal();
      uint32_t it = 0, s = 0, ph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        int x0, y0;
        final_tile(p, tile, &x0, &y0);
        const int bx = (x0 - 1) & ~(kGroupPx - 1);
        for (int kb = 0; kb < kKB; ++kb, ++it) {
          if (!mbar_wait_bounded(&empty[s], ph ^ 1u, p.status, kErrTimeoutProducer)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], p.stage_tx);
          tma_load_4d(A + static_cast<size_t>(s) * p.stage_bytes, &map, &full[s], 0, bx >> p.xs, 2 * kb,
                      y0 - 1, pol);
          if (++s == static_cast<uint32_t>(S)) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      for (uint32_t k = it > static_cast<uint32_t>(S) ? it - S : 0u; k < it; ++k)
        mbar_wait_bounded(&full[k % S], (k / S) & 1u, p.status, kErrTimeoutDrain);
      mbar_wait_bounded(wbar, 0, p.status, kErrTimeoutDrain);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    const uint32_t id1 = TF ? idesc_tf32_f32(kTileM, kNc) : idesc_f16_f32(kTileM, kNc);
    const uint32_t id2 = TF ? idesc_tf32_f32(kTileM, 2 * kNc) : idesc_f16_f32(kTileM, 2 * kNc);
    const uint32_t id3 = TF ? idesc_tf32_f32(kTileM, 3 * kNc) : idesc_f16_f32(kTileM, 3 * kNc);
    const uint64_t a0 = smem_desc_noswizzle(smem_u32(A), kHaloW * kChunkBytes, 128);
    const uint64_t w0 = smem_desc_noswizzle(smem_u32(Wsm), 3u * kNc * kChunkBytes, 128);
    constexpr uint32_t kWkb = kWkbBytes >> 4;                       // one K block, 16 B units
    constexpr uint32_t kBlo = (2u * 3u * kNc * kChunkBytes) >> 4;   // tf32: B_lo after B_hi
    const uint32_t alo16 = TF ? (static_cast<uint32_t>(S) * p.stage_bytes) >> 4 : 0u;
    bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(wbar, 0, p.status, kErrTimeoutMma));
    uint32_t s = 0, ph = 0, tcount = 0;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++tcount) {
      const uint32_t buf = tcount & 1u;
      if (!__all_sync(0xffffffffu, mbar_wait_bounded(&tempty[buf], (tcount >> 1) & 1u, p.status,
                                                      kErrTimeoutMma))) {
        ok = false;
        break;
      }
      tc_fence_after();
      int x0, y0;
      final_tile(p, tile, &x0, &y0);
      // A row i is input pixel x0 - 1 + i: o pixels past the box start
      const uint32_t o = static_cast<uint32_t>((x0 - 1) - ((x0 - 1) & ~(kGroupPx - 1)));
      for (int kb = 0; kb < kKB; ++kb) {
        bool w = mbar_wait_bounded(&full[s], ph, p.status, kErrTimeoutMma);
        if (TF && w) w = mbar_wait_bounded(&xdone[s], ph, p.status, kErrTimeoutMma);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        const uint64_t ad = a0 + ((s * p.stage_bytes) >> 4) + o;
        const uint64_t bd = w0 + static_cast<uint32_t>(kb) * kWkb;
        // tf32: passes A_hi B_hi, A_hi B_lo, A_lo B_hi
#pragma unroll 1
        for (int pass = 0; pass < (TF ? 3 : 1); ++pass)
          final_kblock<TF>(ad + (pass == 2 ? alo16 : 0u), bd + (pass == 1 ? kBlo : 0u),
                           tmem + buf * kSetCols, id1, id2, id3);
        if (elect_one()) mma_commit(&empty[s]);
        if (++s == static_cast<uint32_t>(S)) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      if (elect_one()) mma_commit(&tfull[buf]);
    }
    if (elect_one()) mma_commit(done);
    mbar_wait_bounded(done, 0, p.status, kErrTimeoutMma);
    __syncwarp();
  } else if (TF && warp >= 2 + kEpiWarps) {
    // ------------------------------------------------------------ tf32 split
    // The 128 entries of every staged box row that the MMAs read (from the
    // tile's offset o): A_hi in place, A_lo into the A_lo stage.  Waiting on
    // every stage keeps these warps at most one use of a stage ahead of the
    // MMA warp, so the xdone phases stay paired.
    const int et = threadIdx.x - 32 * (2 + kEpiWarps);  // 0..127
    constexpr int kRows = (kR + 2) * 2;                 // halo rows x 2 chunks
    uint32_t s = 0, ph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
      int x0, y0;
      final_tile(p, tile, &x0, &y0);
      const int o = (x0 - 1) - ((x0 - 1) & ~(kGroupPx - 1));
      for (int kb = 0; kb < kKB; ++kb) {
        if (!mbar_wait_bounded(&full[s], ph, p.status, kErrTimeoutEpilogue)) {
          ok = false;
          break;
        }
        uint4* hi = reinterpret_cast<uint4*>(A + static_cast<size_t>(s) * p.stage_bytes);
        uint4* lo = reinterpret_cast<uint4*>(ALO + static_cast<size_t>(s) * p.stage_bytes);
        for (int i = et; i < kRows * kTileM; i += 128) {
          const int at = (i >> 7) * kHaloW + o + (i & (kTileM - 1));
          split_tf32(hi + at, lo + at);
        }
        fence_proxy_async_smem();
        mbar_arrive(&xdone[s]);
        if (++s == static_cast<uint32_t>(S)) {
          s = 0;
          ph ^= 1u;
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp w reads TMEM lane quarter w % 4 (pixel m of the 128-pixel row,
    // image column x0 - 1 + m); the kSubs warps of a quarter take every
    // kSubs-th row.  Output pixel m adds the kx = 1 partial of pixel m + 1 and the
    // kx = 2 partial of pixel m + 2: warp shuffles, except for the last two
    // lanes, which take them from the next quarter's first two lanes through
    // BND[sub][tile parity][quarter][row] (one barrier per tile).
    const int q = warp & 3;
    const int sub = (warp - 2) >> 2;
    const int m = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int et = threadIdx.x - 64;
    if (et < kNc) bias_s[et] = p.bias[et];
    named_barrier_sync(1, 32 * kEpiWarps);
    // every accumulator row restarts from the same 16 values: kept in registers
    uint32_t bz[16];
    bias16_regs(bias_s, bz);
    for (int b = 0; b < 2; ++b)
      for (int r = sub; r < kR; r += kSubs)
        tmem_st16(tmem + lane_off + b * kSetCols + static_cast<uint32_t>(r * kNc), bz);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&tempty[0]);
    mbar_arrive(&tempty[1]);
    uint32_t tcount = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++tcount) {
      const uint32_t buf = tcount & 1u;
      int x0, y0;
      final_tile(p, tile, &x0, &y0);
      // output pixel m of the tile is image column x0 + m
      const int x = x0 + m;
      constexpr int kJ = kR / kSubs;  // rows of this warp: sub + kSubs j
      // fused output pass: the input colour of this warp's pixels is loaded
      // before the accumulators are waited for, to overlap the tile's MMAs
      float4 col[kJ];
      if (OUT) {
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
          const int xo = x - p.in_x, yo = y0 + sub + kSubs * j - p.in_y;
          col[j] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (m < kFinalSpan && x < p.W && xo >= 0 && xo < p.ow && yo >= 0 && yo < p.oh)
            col[j] = p.color[static_cast<size_t>(p.oy + yo) * p.color_stride + p.ox + xo];
        }
      }
      if (!mbar_wait_bounded(&tfull[buf], (tcount >> 1) & 1u, p.status, kErrTimeoutEpilogue)) break;
      tc_fence_after();
      uint32_t d[kJ][16];
#pragma unroll
      for (int j = 0; j < kJ; ++j)
        tmem_ld16_nowait(tmem + lane_off + buf * kSetCols + static_cast<uint32_t>((sub + kSubs * j) * kNc), d[j]);
      tmem_wait_ld();
#pragma unroll
      for (int j = 0; j < kJ; ++j)
        tmem_st16(tmem + lane_off + buf * kSetCols + static_cast<uint32_t>((sub + kSubs * j) * kNc), bz);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&tempty[buf]);
      // the next quarter's first two lanes, for this quarter's last two
      float4* bnd = BND + ((sub * 2 + buf) * 4) * kJ * 3;
      if (lane < 2) {
#pragma unroll
        for (int j = 0; j < kJ; ++j) {
          float4* e = bnd + (q * kJ + j) * 3;
          if (lane == 0)
            e[0] = make_float4(__uint_as_float(d[j][4]), __uint_as_float(d[j][5]), __uint_as_float(d[j][6]), 0.f);
          e[1 + lane] = make_float4(__uint_as_float(d[j][8]), __uint_as_float(d[j][9]), __uint_as_float(d[j][10]), 0.f);
        }
      }
      mbar_arrive(&xbar[sub * 2 + buf]);
      if (!mbar_wait_bounded(&xbar[sub * 2 + buf], (tcount >> 1) & 1u, p.status, kErrTimeoutEpilogue)) break;
#pragma unroll
      for (int j = 0; j < kJ; ++j) {
        float n[3];
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          float k1 = __shfl_down_sync(0xffffffffu, __uint_as_float(d[j][4 + c]), 1);
          float k2 = __shfl_down_sync(0xffffffffu, __uint_as_float(d[j][8 + c]), 2);
          if (lane >= 30 && q < 3) {
            const float4* e = bnd + ((q + 1) * kJ + j) * 3;
            const float4 e1 = e[0], e2 = e[lane == 30 ? 1 : 2];
            if (lane == 31) k1 = c == 0 ? e1.x : (c == 1 ? e1.y : e1.z);
            k2 = c == 0 ? e2.x : (c == 1 ? e2.y : e2.z);
          }
          n[c] = __uint_as_float(d[j][c]) + k1 + k2;
        }
        const int y = y0 + sub + kSubs * j;
        if (m < kFinalSpan && x < p.W && y < p.H) {
          if (p.net) p.net[static_cast<size_t>(y) * p.W + x] = make_float4(n[0], n[1], n[2], 0.0f);
          if (OUT) {
            const int xo = x - p.in_x, yo = y - p.in_y;
            if (xo >= 0 && xo < p.ow && yo >= 0 && yo < p.oh) {
              const size_t oi = static_cast<size_t>(p.oy + yo) * p.out_stride + p.ox + xo;
              p.out[oi] = output_pixel(n[0], n[1], n[2], col[j], p.hdr, p.scale, p.exp2_tab);
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kSetCols);
  }
}

cudaError_t launch_conv_final(const FinalConvLaunch& L, cudaStream_t stream) {
  if (L.tf32) {
    const dim3 block(final_threads<true>());
    if (L.outpass)
      return launch_pdl(conv3x3_final_kernel<true, true>, L.grid, block, L.smem, stream, L.map, L.p);
    return launch_pdl(conv3x3_final_kernel<false, true>, L.grid, block, L.smem, stream, L.map, L.p);
  }
  const dim3 block(final_threads<false>());
  if (L.outpass)
    return launch_pdl(conv3x3_final_kernel<true, false>, L.grid, block, L.smem, stream, L.map, L.p);
  return launch_pdl(conv3x3_final_kernel<false, false>, L.grid, block, L.smem, stream, L.map, L.p);
}

cudaError_t conv_final_set_smem_limit(size_t bytes) {
  const int b = static_cast<int>(bytes);
  cudaError_t e = cudaFuncSetAttribute(conv3x3_final_kernel<true, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, b);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(conv3x3_final_kernel<false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, b);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(conv3x3_final_kernel<true, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, b);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(conv3x3_final_kernel<false, true>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, b);
  return e;
}

}  // namespace oidnx

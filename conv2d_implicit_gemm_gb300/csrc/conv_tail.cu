// The U-Net's last two layers in one kernel, fp16 storage: dec_conv1b
// (64 -> 32 channels, bias + ReLU, output rounded to fp16) and dec_conv0
// (32 -> 3, bias, fp32), optionally followed by the output pass.  What each
// step computes is the layer of "oidn-web 0.4.0 -> 0.5.0,
// package/src/nativeUNet.ts" (createTiledConvShader; the final conv) and the
// output pass of "oidn-webgpu 0.0.0-stage -> 0.6.0, src/native/denoise.ts"
// (outputShader).  dec_conv1b's 32-channel map, 134 MB at 1920x1088, is
// never written to memory: it goes from conv 1's accumulators to conv 2's A
// operand inside tensor memory.
//
// GB300 design (not the pages'):
//  * Persistent CTAs walk groups of up to p.run output tiles (kTailOut rows
//    x kFinalSpan pixels) that lie one above the other in a column strip:
//    group g covers row tiles band * run .. of strip g % tiles_x (band =
//    g / tiles_x), both counted from the bottom of the frame and walked
//    upwards (the previous layer's last rows are the ones still in L2), and
//    the CTAs take groups round robin, so the frame is read bottom to top.  A tile needs the kTailMid =
//    kTailOut + 2 conv-1 rows around it (one row above and below, 128
//    pixels from one pixel left of it); the two it shares with the previous
//    tile of its group are carried over in tensor memory, so conv 1
//    computes six new rows per tile and all eight only in a group's first.
//    One TMA box per 16-channel K block holds the input halo of the rows
//    computed (10 or 8 rows x 144 pixels); ky is stacked along N (N <= 96)
//    and the row accumulators start from the bias, in the per-row order (K
//    block, kx, ky) of the plain conv kernel, so the values equal that
//    kernel's bit for bit.
//  * Tensor memory holds two tile buffers of 256 columns.  Conv 1
//    accumulates row r in the 32 columns of slot r (slot r + 2 when rows 6
//    and 7 are carried).  The conversion warps read each row, apply ReLU,
//    round to fp16 and write it back as 16 columns of packed fp16 pairs
//    (zero for rows and pixels outside the image: conv 2's same padding):
//    rows 0..5 at columns 32 + 16 r, rows 6 and 7 at columns 0 and 16 (where
//    the previous tile of the group put its carried rows); then conv 2's
//    bias into columns 128..223.  Conv 2 takes the fp16 rows straight from
//    tensor memory as its A operand (tcgen05.mma with A in TMEM), with the
//    three kx taps folded into N = 16 as in the final-conv kernel and ky
//    stacked along N: output row r accumulates in columns 128 + 16 r, in the
//    final-conv kernel's order (K block, ky); the kx partial sums of pixels
//    m, m + 1, m + 2 are added in the epilogue.
//  * Overlap: while the epilogue turns tile t's conv-1 rows into fp16 and
//    later finishes its output, the tensor cores run conv 1 of tile t + 1
//    in the other buffer; conv 2 of tile t is issued between two K blocks
//    of that conv 1 as soon as its fp16 rows are ready.  The two carried
//    rows are written into the other buffer when they are converted.
//  * Warp 0 issues TMA, warp 1 allocates TMEM and issues the MMAs, warps
//    2-5 turn conv-1 rows into fp16, warps 6-13 read conv 2, refill the
//    bias and write the output, a tile behind.  Every wait is bounded.
#include "internal.h"
#include "passes.cuh"
#include "ptx.cuh"

namespace oidnx {

namespace {

constexpr int kTailMidWarps = 4;     // fp16 conversion: one per TMEM lane quarter
constexpr int kTailOutWarps = 8;     // output: two per lane quarter
constexpr int kTailSubs = 2;         // output warps per lane quarter
constexpr int kTailThreads = 32 * (2 + kTailMidWarps + kTailOutWarps);
constexpr int kMidC = 32;            // conv-1 output channels
constexpr int kC2 = 16;              // conv-2 accumulator columns per row (12 used)
constexpr uint32_t kSlot = 32;                  // columns per conv-1 row slot
constexpr uint32_t kBufCols = kTailMid * kSlot; // 256: one tile buffer
constexpr uint32_t kC2Col = 128;                // conv-2 accumulators: 6 rows x 16 columns

// Column of fp16 row r (of kTailMid) in a tile buffer.
__host__ __device__ constexpr uint32_t mid_col(int r) {
  return r < kTailOut ? 32u + 16u * static_cast<uint32_t>(r) : 16u * static_cast<uint32_t>(r - kTailOut);
}
constexpr uint32_t kTmemCols = 2 * kBufCols;
constexpr uint32_t kW1Block = 3u * 2u * 3u * kMidC * kChunkBytes;  // [kx][half][ky][32][8]: 9216 B
constexpr uint32_t kW2Block = 2u * 3u * kC2 * kChunkBytes;          // [half][ky][16][8]: 1536 B

// Row tile k (counted from the bottom) of strip sx, in the group of row
// tiles k0 .. k1 - 1: conv-1 rows 0 .. r1 - 1 are computed (all kTailMid in
// the group's first tile; else rows 6 and 7 are the previous tile's rows 0
// and 1); carry: the group's next tile, above this one, takes rows 0 and 1.
struct TailStep {
  int x0, y0, r1;
  bool carry;
};

// The output pass of one pixel, out of line: the output warps call it three
// times per tile row, and inlined copies crowded the instruction cache that
// the MMA warp shares.
__device__ __noinline__ float4 tail_output_pixel(float n0, float n1, float n2, float4 col, int hdr,
                                                 float scale, const float4* exp2_tab) {
  return output_pixel(n0, n1, n2, col, hdr, scale, exp2_tab);
}

__device__ __forceinline__ TailStep tail_step(const TailConvParams& p, int sx, int k, int k0, int k1) {
  TailStep st;
  st.x0 = sx * kFinalSpan;
  st.y0 = (p.tiles_y - 1 - k) * kTailOut;
  st.r1 = k == k0 ? kTailMid : kTailMid - 2;
  st.carry = k + 1 < k1;
  return st;
}

// A CTA's walk: groups blockIdx.x, blockIdx.x + gridDim.x, ..., each from
// row tile k0 to k1 - 1 of strip sx (band = g / tiles_x counted from the
// bottom of the frame).
struct TailWalk {
  int g, sx, k, k0, k1;
  __device__ __forceinline__ void set(const TailConvParams& p) {
    if (g < p.groups) {
      const int band = g / p.tiles_x;
      sx = g - band * p.tiles_x;
      k0 = band * p.run;
      k1 = k0 + p.run < p.tiles_y ? k0 + p.run : p.tiles_y;
      k = k0;
    }
  }
  __device__ __forceinline__ void begin(const TailConvParams& p) {
    g = blockIdx.x;
    set(p);
  }
  __device__ __forceinline__ bool valid(const TailConvParams& p) const { return g < p.groups; }
  __device__ __forceinline__ void next(const TailConvParams& p) {
    if (++k == k1) {
      g += gridDim.x;
      set(p);
    }
  }
  __device__ __forceinline__ TailStep step(const TailConvParams& p) const { return tail_step(p, sx, k, k0, k1); }
};


// Conv-1 MMAs of one K block and kx for rows 0 .. R1 - 1: box row h (image
// row y0 - 2 + h) updates rows max(0, h - 2) .. min(R1 - 1, h) with the
// ky-stacked B block.
template <int R1>
__device__ __forceinline__ void conv1_kx(uint32_t d1, uint64_t adk, uint64_t bdk, const uint32_t (&i1)[4]) {
  if (!elect_one()) return;  // one lane issues the MMAs
#pragma unroll
  for (int h = 0; h < R1 + 2; ++h) {
    const int lo = h - 2 > 0 ? h - 2 : 0;
    const int hi = h < R1 - 1 ? h : R1 - 1;
    mma_f16_ss(d1 + static_cast<uint32_t>(lo) * kSlot, adk + static_cast<uint32_t>(h * 2 * kHaloW),
               bdk + static_cast<uint32_t>((2 - h + lo) * kMidC), i1[hi - lo + 1], 1u);
  }
}

}  // namespace

template <bool OUT>
__global__ void __launch_bounds__(kTailThreads, 1)
    conv3x3_tail_kernel(const __grid_constant__ CUtensorMap map10, const __grid_constant__ CUtensorMap map8,
                        const TailConvParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (128u - (smem_u32(smem_raw) & 127u)) & 127u;
  uint8_t* smem = smem_raw + pad;
  const int S = p.S, KB = p.KB1;
  constexpr int kJ2 = kTailOut / kTailSubs;  // output rows per output warp
  // shared memory: [stages][conv-1 weights][conv-2 weights][boundary
  // [sub][2][quarter][kJ2][3]][bias1][bias2][barriers]
  uint8_t* A = smem;
  uint8_t* W1 = A + static_cast<size_t>(S) * p.stage_bytes;
  uint8_t* W2 = W1 + static_cast<size_t>(KB) * kW1Block;
  float4* BND = reinterpret_cast<float4*>(W2 + 2 * kW2Block);
  float* bias1_s = reinterpret_cast<float*>(BND + kTailSubs * 2 * 4 * kJ2 * 3);
  float* bias2_s = bias1_s + kMidC;
  uint64_t* full = reinterpret_cast<uint64_t*>(bias2_s + kC2);
  uint64_t* empty = full + S;
  uint64_t* c1full = empty + S;     // [buffer]: conv 1 of a tile (and conv 2 before it) finished
  uint64_t* midready = c1full + 2;  // [buffer]: fp16 rows and conv-2 bias written
  uint64_t* c2full = midready + 2;  // [buffer]: conv 2 finished
  uint64_t* c1empty = c2full + 2;   // [buffer]: conv 2 read, conv-1 bias written
  uint64_t* xbar = c1empty + 2;     // [sub][2]: boundary values written
  uint64_t* wbar = xbar + 2 * kTailSubs;
  uint64_t* done = wbar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&c1full[b], 1);
      mbar_init(&midready[b], 32 * kTailMidWarps);
      mbar_init(&c2full[b], 1);
      mbar_init(&c1empty[b], 32 * kTailOutWarps);
    }
    for (int k = 0; k < 2 * kTailSubs; ++k) mbar_init(&xbar[k], 128);
    mbar_init(wbar, 1);
    mbar_init(done, 1);
    fence_mbarrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&map10);
      prefetch_tmap(&map8);
      const uint32_t wbytes = static_cast<uint32_t>(KB) * kW1Block + 2u * kW2Block;
      mbar_arrive_expect_tx(wbar, wbytes);
      bulk_load(W1, p.w1, static_cast<uint32_t>(KB) * kW1Block, wbar);
      bulk_load(W2, p.w2, 2u * kW2Block, wbar);
      // weights and bias are constants; the input comes from the previous kernel
      griddep_wait();
      const uint64_t pol = p.l2_first ? l2_evict_first() : l2_evict_normal();
      uint32_t it = 0, s = 0, ph = 0;
      bool ok = true;
      TailWalk w;
      for (w.begin(p); w.valid(p) && ok; w.next(p)) {
        const TailStep st = w.step(p);
        // the box starts at the 8-pixel boundary at or left of x0 - 2
        const int bx = (st.x0 - 2) & ~(kGroupPx - 1);
        const bool all = st.r1 == kTailMid;
        for (int kb = 0; kb < KB; ++kb, ++it) {
          if (!mbar_wait_bounded(&empty[s], ph ^ 1u, p.status, kErrTimeoutProducer)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], all ? p.stage_tx : p.stage_tx8);
          tma_load_4d(A + static_cast<size_t>(s) * p.stage_bytes, all ? &map10 : &map8, &full[s], 0,
                      bx >> p.xs, 2 * kb, st.y0 - 2, pol);
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
    const uint32_t i1[4] = {0u, idesc_f16_f32(kTileM, kMidC), idesc_f16_f32(kTileM, 2 * kMidC),
                            idesc_f16_f32(kTileM, 3 * kMidC)};
    const uint32_t i2[4] = {0u, idesc_f16_f32(kTileM, kC2), idesc_f16_f32(kTileM, 2 * kC2),
                            idesc_f16_f32(kTileM, 3 * kC2)};
    // stage box rows are kHaloW pixels; A row i of conv 1 is image pixel
    // x0 - 2 + i + kx, o pixels past the box start
    const uint64_t a0 = smem_desc_noswizzle(smem_u32(A), kHaloW * kChunkBytes, 128);
    // conv-1 B: per K block [kx][8-lane half][ky stack][32][8]; conv-2 B:
    // per K block [8-lane half][ky stack][16][8] (kx folded into the 16)
    const uint64_t w1d = smem_desc_noswizzle(smem_u32(W1), 3u * kMidC * kChunkBytes, 128);
    const uint64_t w2d = smem_desc_noswizzle(smem_u32(W2), 3u * kC2 * kChunkBytes, 128);
    // conv 2 of the tile in buffer b: fp16 row h (A, K block kb = its
    // columns kb * 8 .. + 7) updates output rows max(0, h - 2) .. min(5, h)
    // with the ky-stacked B block
    auto conv2 = [&](uint32_t b) {
      const uint32_t base = tmem + b * kBufCols;
      if (elect_one()) {
#pragma unroll
        for (int kb = 0; kb < 2; ++kb)
#pragma unroll
          for (int h = 0; h < kTailMid; ++h) {
            const int lo = h - 2 > 0 ? h - 2 : 0;
            const int hi = h < kTailOut - 1 ? h : kTailOut - 1;
            mma_f16_ts(base + kC2Col + static_cast<uint32_t>(lo * kC2),
                       base + mid_col(h) + static_cast<uint32_t>(kb * 8),
                       w2d + static_cast<uint32_t>(kb) * (kW2Block >> 4) +
                           static_cast<uint32_t>((2 - h + lo) * kC2),
                       i2[hi - lo + 1]);
          }
        mma_commit(&c2full[b]);
      }
      __syncwarp();
    };
    bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(wbar, 0, p.status, kErrTimeoutMma));
    uint32_t s = 0, ph = 0, tcount = 0;
    bool pend = false;        // conv 2 of the previous tile not yet issued
    uint32_t pb = 0, pph = 0; // its buffer and midready parity
    TailWalk w;
    for (w.begin(p); w.valid(p) && ok; w.next(p), ++tcount) {
      const uint32_t b = tcount & 1u;
      // conv 1 writes buffer b once the tile two back has left it (the
      // output warps' first bias fill for the first two tiles)
      ok = __all_sync(0xffffffffu,
                      mbar_wait_bounded(&c1empty[b], (tcount >> 1) & 1u, p.status, kErrTimeoutMma));
      if (!ok) break;
      tc_fence_after();
      const TailStep st = w.step(p);
      const uint32_t o = static_cast<uint32_t>((st.x0 - 2) - ((st.x0 - 2) & ~(kGroupPx - 1)));
      const uint32_t d1 = tmem + b * kBufCols;
      for (int kb = 0; kb < KB; ++kb) {
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&full[s], ph, p.status, kErrTimeoutMma));
        if (!ok) break;
        // conv 2 of the previous tile goes in as soon as its fp16 rows are
        // ready, and at the latest before this tile's last K block, so that
        // c1full also covers it
        if (pend) {
          const bool ready = kb == KB - 1
                                 ? mbar_wait_bounded(&midready[pb], pph, p.status, kErrTimeoutMma)
                                 : mbar_test_wait(&midready[pb], pph);
          if (__all_sync(0xffffffffu, ready)) {
            tc_fence_after();
            conv2(pb);
            pend = false;
          } else if (kb == KB - 1) {
            ok = false;
            break;
          }
        }
        const uint64_t ad = a0 + ((s * p.stage_bytes) >> 4) + o;
        const uint64_t bd = w1d + static_cast<uint32_t>(kb) * (kW1Block >> 4);
        // (not unrolled: the kernel's four warp roles run different code,
        // and a smaller MMA loop stays in the instruction cache)
        if (st.r1 == kTailMid) {
#pragma unroll 1
          for (int kx = 0; kx < 3; ++kx)
            conv1_kx<kTailMid>(d1, ad + static_cast<uint32_t>(kx), bd + static_cast<uint32_t>(kx * 6 * kMidC), i1);
        } else {
#pragma unroll
          for (int kx = 0; kx < 3; ++kx)
            conv1_kx<kTailMid - 2>(d1 + 2 * kSlot, ad + static_cast<uint32_t>(kx),
                                   bd + static_cast<uint32_t>(kx * 6 * kMidC), i1);
        }
        if (elect_one()) mma_commit(&empty[s]);
        if (++s == static_cast<uint32_t>(S)) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) break;
      if (elect_one()) mma_commit(&c1full[b]);
      pend = true;
      pb = b;
      pph = (tcount >> 1) & 1u;
    }
    if (ok && pend &&
        __all_sync(0xffffffffu, mbar_wait_bounded(&midready[pb], pph, p.status, kErrTimeoutMma))) {
      tc_fence_after();
      conv2(pb);
    }
    // TMEM is freed only after every MMA issued above has completed.
    if (elect_one()) mma_commit(done);
    mbar_wait_bounded(done, 0, p.status, kErrTimeoutMma);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogues
    // Warp w reads TMEM lane quarter w % 4: pixel m of the 128-pixel rows
    // (conv-1 image column x0 - 1 + m; output image column x0 + m).
    const int q = warp & 3;
    const int m = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int et = threadIdx.x - 64;
    if (et < kMidC) bias1_s[et] = p.bias1[et];
    if (et < kC2) bias2_s[et] = p.bias2[et];
    named_barrier_sync(1, 32 * (kTailMidWarps + kTailOutWarps));
    if (warp < 2 + kTailMidWarps) {
      // -------- conversion warps: conv-1 row r (image row y0 - 1 + r) ->
      // ReLU -> fp16 pairs at mid_col(r) (channel 2c in the low half of
      // column c), each row written over columns already read; rows 0 and 1
      // also go to the next tile's buffer as its rows 6 and 7; then conv 2's
      // bias
      uint32_t tcount = 0;
      TailWalk w;
      for (w.begin(p); w.valid(p); w.next(p), ++tcount) {
        const uint32_t buf = tcount & 1u;
        const uint32_t tb = tmem + lane_off + buf * kBufCols;
        const uint32_t nb = tmem + lane_off + (buf ^ 1u) * kBufCols;
        const TailStep st = w.step(p);
        const int xm = st.x0 - 1 + m;
        const int sb = st.r1 == kTailMid ? 0 : 2;  // slot of conv-1 row 0
        if (!mbar_wait_bounded(&c1full[buf], (tcount >> 1) & 1u, p.status, kErrTimeoutEpilogue)) break;
        tc_fence_after();
        for (int r2 = 0; r2 < st.r1; r2 += 2) {
          uint32_t v[2][2][16];
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const uint32_t t0 = tb + static_cast<uint32_t>(sb + r2 + i) * kSlot;
            tmem_ld16_nowait(t0, v[i][0]);
            tmem_ld16_nowait(t0 + 16, v[i][1]);
          }
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int r = r2 + i;
            const int ym = st.y0 - 1 + r;
            const bool inside = xm >= 0 && xm < p.W && ym >= 0 && ym < p.H;
            uint32_t h[16];
#pragma unroll
            for (int k = 0; k < 16; ++k)
              h[k] = inside ? pack_half2(fmaxf(__uint_as_float(v[i][k >> 3][2 * (k & 7)]), 0.0f),
                                         fmaxf(__uint_as_float(v[i][k >> 3][2 * (k & 7) + 1]), 0.0f))
                            : 0u;
            tmem_st16(tb + mid_col(r), h);
            if (st.carry && r < 2) tmem_st16(nb + mid_col(r + kTailOut), h);
          }
        }
        uint32_t b2[16];
        bias16_regs(bias2_s, b2);
#pragma unroll
        for (int r = 0; r < kTailOut; ++r) tmem_st16(tb + kC2Col + static_cast<uint32_t>(r * kC2), b2);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&midready[buf]);
      }
    } else {
      // -------- output warps: the two of a lane quarter take every other
      // output row.  Output pixel m adds the kx = 1 partial of pixel m + 1
      // and the kx = 2 partial of pixel m + 2 (warp shuffles; the last two
      // lanes take the next quarter's first two through BND, one barrier per
      // tile).  After reading conv 2 they refill the buffer's conv-1 rows
      // with the bias for the tile after next (its six new rows, or all
      // eight when it starts a group).
      const int sub = (warp - 2 - kTailMidWarps) >> 2;
      // conv-1 bias into slots first .. 7 of a buffer, this warp taking
      // columns 16 sub .. 16 sub + 15 of each slot (channels 16 sub ..): in
      // columns 128..223 those hold exactly the conv-2 rows it has read, so
      // it never overwrites a row the other warp of its quarter still reads
      auto fill_bias1 = [&](uint32_t tb, int first) {
        uint32_t b1[16];
        bias16_regs(bias1_s + 16 * sub, b1);
        for (int r = first; r < kTailMid; ++r) tmem_st16(tb + static_cast<uint32_t>(r) * kSlot + 16u * sub, b1);
      };
      fill_bias1(tmem + lane_off, 0);
      fill_bias1(tmem + lane_off + kBufCols, 0);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&c1empty[0]);  // completion 0 of each: conv 1 starts from the bias
      mbar_arrive(&c1empty[1]);
      uint32_t tcount = 0;
      TailWalk w, w2;  // w2: two tiles ahead (the buffer's next user)
      w2.begin(p);
      w2.next(p);
      w2.next(p);
      bool ok = true;
      for (w.begin(p); w.valid(p) && ok; w.next(p), w2.next(p), ++tcount) {
        const uint32_t buf = tcount & 1u;
        const uint32_t par = (tcount >> 1) & 1u;
        const uint32_t tb = tmem + lane_off + buf * kBufCols;
        const TailStep st = w.step(p);
        const int x0 = st.x0, y0 = st.y0;
        // the buffer's next tile accumulates in slots 0..7, or 2..7 when it
        // takes two carried rows (slots 0 and 1 then hold them)
        const int refill = !w2.valid(p) ? kTailMid : (w2.step(p).r1 == kTailMid ? 0 : 2);
        // fused output pass: the input colour of this warp's output pixels is
        // loaded before the accumulators are waited for
        const int x = x0 + m;
        float4 col[kJ2];
        if (OUT) {
#pragma unroll
          for (int j = 0; j < kJ2; ++j) {
            const int xo = x - p.in_x, yo = y0 + sub + kTailSubs * j - p.in_y;
            col[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (m < kFinalSpan && x < p.W && xo >= 0 && xo < p.ow && yo >= 0 && yo < p.oh)
              col[j] = p.color[static_cast<size_t>(p.oy + yo) * p.color_stride + p.ox + xo];
          }
        }
        if (!(ok = mbar_wait_bounded(&c2full[buf], par, p.status, kErrTimeoutEpilogue))) break;
        tc_fence_after();
        uint32_t d[kJ2][16];
#pragma unroll
        for (int j = 0; j < kJ2; ++j)
          tmem_ld16_nowait(tb + kC2Col + static_cast<uint32_t>((sub + kTailSubs * j) * kC2), d[j]);
        tmem_wait_ld();
        fill_bias1(tb, refill);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&c1empty[buf]);
        // the next quarter's first two lanes, for this quarter's last two
        float4* bnd = BND + ((sub * 2 + buf) * 4) * kJ2 * 3;
        if (lane < 2) {
#pragma unroll
          for (int j = 0; j < kJ2; ++j) {
            float4* e = bnd + (q * kJ2 + j) * 3;
            if (lane == 0)
              e[0] = make_float4(__uint_as_float(d[j][4]), __uint_as_float(d[j][5]), __uint_as_float(d[j][6]), 0.f);
            e[1 + lane] = make_float4(__uint_as_float(d[j][8]), __uint_as_float(d[j][9]), __uint_as_float(d[j][10]), 0.f);
          }
        }
        mbar_arrive(&xbar[sub * 2 + buf]);
        if (!(ok = mbar_wait_bounded(&xbar[sub * 2 + buf], par, p.status, kErrTimeoutEpilogue))) break;
#pragma unroll
        for (int j = 0; j < kJ2; ++j) {
          float n[3];
#pragma unroll
          for (int c = 0; c < 3; ++c) {
            float k1 = __shfl_down_sync(0xffffffffu, __uint_as_float(d[j][4 + c]), 1);
            float k2 = __shfl_down_sync(0xffffffffu, __uint_as_float(d[j][8 + c]), 2);
            if (lane >= 30 && q < 3) {
              const float4* e = bnd + ((q + 1) * kJ2 + j) * 3;
              const float4 e1 = e[0], e2 = e[lane == 30 ? 1 : 2];
              if (lane == 31) k1 = c == 0 ? e1.x : (c == 1 ? e1.y : e1.z);
              k2 = c == 0 ? e2.x : (c == 1 ? e2.y : e2.z);
            }
            n[c] = __uint_as_float(d[j][c]) + k1 + k2;
          }
          const int y = y0 + sub + kTailSubs * j;
          if (m < kFinalSpan && x < p.W && y < p.H) {
            if (p.net) p.net[static_cast<size_t>(y) * p.W + x] = make_float4(n[0], n[1], n[2], 0.0f);
            if (OUT) {
              const int xo = x - p.in_x, yo = y - p.in_y;
              if (xo >= 0 && xo < p.ow && yo >= 0 && yo < p.oh) {
                const size_t oi = static_cast<size_t>(p.oy + yo) * p.out_stride + p.ox + xo;
                p.out[oi] = tail_output_pixel(n[0], n[1], n[2], col[j], p.hdr, p.scale, p.exp2_tab);
              }
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
    tmem_dealloc(tmem, kTmemCols);
  }
}

cudaError_t launch_conv_tail(const TailConvLaunch& L, cudaStream_t stream) {
  const dim3 block(kTailThreads);
  if (L.outpass)
    return launch_pdl(conv3x3_tail_kernel<true>, L.grid, block, L.smem, stream, L.map10, L.map8, L.p);
  return launch_pdl(conv3x3_tail_kernel<false>, L.grid, block, L.smem, stream, L.map10, L.map8, L.p);
}

cudaError_t conv_tail_set_smem_limit(size_t bytes) {
  const int b = static_cast<int>(bytes);
  cudaError_t e = cudaFuncSetAttribute(conv3x3_tail_kernel<true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, b);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(conv3x3_tail_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, b);
  return e;
}

}  // namespace oidnx

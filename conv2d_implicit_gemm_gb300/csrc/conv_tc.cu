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
//  * Persistent CTAs (one per SM) walk the output tiles of R rows x 128
//    pixels.  One M=128 UMMA tile per output row; the R accumulators of a
//    tile (N fp32 columns each) live in tensor memory, double-buffered so the
//    epilogue of one tile runs while the MMAs of the next are issued.
//  * K is walked in blocks of 16 input channels.  For one block the CTA
//    stages, by one TMA box, the whole input halo: (R+2) rows x 130 pixels x
//    16 channels, zero-filled outside the image (the same padding).  Stored
//    as [row][8-channel half][pixel][8], every 8-pixel x 8-channel core
//    matrix is a contiguous 128 B run, so the 9 taps of all R rows are just
//    9R shared-memory descriptors into the same halo: a kx shift is +16 B, a
//    ky shift selects the next halo row.  No im2col copy, no re-load per tap.
//  * The box is widened to 144 pixels starting 8 left of the tile, so that
//    with activation rows padded to a multiple of 8 pixels the tensor map's
//    innermost box dimension is 8 pixels x 8 lanes (128 B).  With a 16-byte
//    innermost dimension the TMA unit moves one pixel per request and
//    delivered ~4.6 TB/s from L2 over the whole GPU; 128-byte rows deliver
//    ~21 TB/s, which takes the loads off the critical path.
//  * The three ky taps are stacked along N: halo row h feeds output rows h,
//    h-1 and h-2 through ky = 0, 1, 2, so one MMA with B = [W(ky=2); W(ky=1);
//    W(ky=0)] (N = 3 x Cout <= 256) updates three row accumulators that sit
//    next to each other in TMEM.  An M=128, K=16 MMA costs at least ~46
//    cycles of operand fetch whatever N is, so small-Cout layers reach the
//    tensor rate only with N stacked this way; it also cuts the MMA count
//    per K block from 9R to 3(R+2).
//  * Weights are pre-packed on the host into the exact shared-memory image
//    of the B operand ([kx][8-channel half][ky stack][Cout][8] per K block).
//    When they fit they are loaded once per CTA and stay resident; otherwise
//    one block per pipeline stage is streamed with the A halo.
//  * Warp roles: warp 0 issues TMA, warp 1 allocates TMEM and issues the
//    MMAs from one thread, warps 2-9 run the epilogue (bias, ReLU, pool,
//    fp16/fp32 stores), warps 10-13 (expansion decoders and fp32 kinds)
//    build the upsampled halo in shared memory from a low-resolution TMA
//    box, since nearest upsampling is not an affine TMA box, and split fp32
//    operands into their tf32 parts.
//  * Every wait is bounded: on timeout the kernel records a bit in the
//    status word, lets its in-flight copies land, frees TMEM and returns.
#include "internal.h"
#include "ptx.cuh"

namespace oidnx {

// 3xTF32 kinds (fp32 storage), expansion and sub-pixel decoder kinds, and the
// kinds with the four helper warps
template <int KIND> __host__ __device__ constexpr bool kind_tf32() {
  return KIND == kTcPlain32 || KIND == kTcExpand32 || KIND == kTcSubpixel32;
}
template <int KIND> __host__ __device__ constexpr bool kind_expand() { return KIND == kTcExpand || KIND == kTcExpand32; }
template <int KIND> __host__ __device__ constexpr bool kind_subpixel() { return KIND == kTcSubpixel || KIND == kTcSubpixel32; }
template <int KIND> __host__ __device__ constexpr bool kind_helpers() { return kind_tf32<KIND>() || kind_expand<KIND>(); }

namespace {

// Tile index in walking order -> tile index in the image: last to first
// when p.reverse is set.  A layer that walks its tiles in the opposite
// order to the layer that wrote its input starts on the rows written last,
// which are still in L2.  (Sub-pixel tiles alternate column parity and
// their count is even, so reversing flips every CTA's parity.)
__device__ __forceinline__ int tile_at(const TcConvParams& p, int tile) {
  return p.reverse ? p.tiles_x * p.tiles_y - 1 - tile : tile;
}

// Step t of the walk -> origin and row count of its tile: a full tile of
// p.R rows, or in the last wave a sub-tile (rows R / tail_split further down
// per sub-index) of the walk step's parent tile.  Sub-pixel decoder tiles
// span 256 columns and hold one column parity px (tile index = 2 * 256-column
// block + px).
template <int KIND>
__device__ __forceinline__ int tile_origin_k(const TcConvParams& p, int t, int* x0, int* y0,
                                             int* px) {
  int rows = p.R, dy = 0;
  if (t >= p.tail_first) {
    const int u = t - p.tail_first;
    rows = p.R / p.tail_split;
    dy = (u % p.tail_split) * rows;
    t = p.tail_first + u / p.tail_split;
  }
  const int tile = tile_at(p, t);
  const int ty = tile / p.tiles_x;
  const int tx = tile - ty * p.tiles_x;
  *y0 = ty * p.R + dy;
  if (kind_subpixel<KIND>()) {
    *x0 = (tx >> 1) * (2 * kTileM);
    *px = tx & 1;
  } else {
    *x0 = tx * kTileM;
    *px = 0;
  }
  return rows;
}

// Advance a pipeline position (stage s of S, phase parity ph) by one item.
__device__ __forceinline__ void next_stage(uint32_t& s, uint32_t& ph, uint32_t S) {
  if (++s == S) {
    s = 0;
    ph ^= 1u;
  }
}

// One fp16 (kind::f16) or tf32 (kind::tf32) MMA, issued by the thread that
// runs it: the issue functions below elect one lane of the (converged) MMA
// warp once and let it issue a whole K block, with no branch per MMA.
// Every MMA accumulates: the epilogue refills each accumulator with the
// bias after reading it (and before the first tile), so no MMA has to
// overwrite one.  An overwriting MMA issued amid accumulating ones stalled
// the tensor pipe (~200 cycles each in a microbenchmark of this issue
// sequence).
template <bool TF>
__device__ __forceinline__ void umma_k(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc) {
  if (!TF) mma_f16_ss(d, a, b, idesc, 1u);
  else mma_tf32_ss(d, a, b, idesc);
}

// All MMAs of one K block for a tile of R rows, fully unrolled so that the
// issuing warp spends a handful of instructions per MMA (its instruction
// stream, not the tensor core, is otherwise the bottleneck).  Halo row h
// updates output rows lo..hi = max(0,h-2)..min(R-1,h) with the ky-stacked B
// block; rows are grouped G at a time (N = rows x Cout <= 256).
template <int R, int G, bool TF>
__device__ __forceinline__ void issue_kblock(uint64_t ad, uint64_t bd, uint32_t dbase, uint32_t N,
                                             uint32_t kx_b16, uint32_t id1, uint32_t id2,
                                             uint32_t id3) {
  if (!elect_one()) return;
  const uint32_t idn[4] = {0u, id1, id2, id3};
#pragma unroll
  for (int kx = 0; kx < 3; ++kx) {
    const uint64_t adk = ad + kx;
    const uint64_t bdk = bd + kx * kx_b16;
#pragma unroll
    for (int h = 0; h < R + 2; ++h) {
      const int lo = h - 2 > 0 ? h - 2 : 0;
      const int hi = h < R - 1 ? h : R - 1;
      const uint64_t a = adk + static_cast<uint32_t>(h * 2 * kHaloW);
#pragma unroll
      for (int c = lo; c <= hi; c += G) {
        const int e = c + G - 1 < hi ? c + G - 1 : hi;
        umma_k<TF>(dbase + c * N, a, bdk + (2 - h + c) * N, idn[e - c + 1]);
      }
    }
  }
}

template <int G, bool TF>
__device__ __forceinline__ void issue_kblock_r1(int R, uint64_t ad, uint64_t bd, uint32_t dbase,
                                                uint32_t N, uint32_t kx_b16, uint32_t id1,
                                                uint32_t id2, uint32_t id3) {
  switch (R) {
    case 1: issue_kblock<1, G, TF>(ad, bd, dbase, N, kx_b16, id1, id2, id3); break;
    case 2: issue_kblock<2, G, TF>(ad, bd, dbase, N, kx_b16, id1, id2, id3); break;
    case 4: issue_kblock<4, G, TF>(ad, bd, dbase, N, kx_b16, id1, id2, id3); break;
    default: issue_kblock<8, G, TF>(ad, bd, dbase, N, kx_b16, id1, id2, id3); break;
  }
}

// One K block.  fp32 storage (TF): each product A * B as three tf32 MMAs,
// A*B_hi + A*B_lo + A_lo*B_hi, issued as three passes over the K block.  The
// stage holds A_hi (A rounded to the nearest tf32 value) and, alo16 units
// further, A_lo = A - A_hi; the weights hold B_hi and, blo16 units further,
// B_lo.  The omitted A_lo*B_lo term and the tf32 precision of the lo parts
// leave a relative error near 2^-21 per product.
template <int G, bool TF>
__device__ __forceinline__ void issue_kblock_r(int R, uint64_t ad, uint64_t bd, uint32_t dbase,
                                               uint32_t N, uint32_t kx_b16, uint32_t id1,
                                               uint32_t id2, uint32_t id3, uint32_t alo16,
                                               uint32_t blo16) {
  if constexpr (!TF) {
    issue_kblock_r1<G, TF>(R, ad, bd, dbase, N, kx_b16, id1, id2, id3);
  } else {
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
      const uint64_t a = ad + (pass == 2 ? alo16 : 0u);
      const uint64_t b = bd + (pass == 1 ? blo16 : 0u);
      issue_kblock_r1<G, TF>(R, a, b, dbase, N, kx_b16, id1, id2, id3);
    }
  }
}

// Sub-pixel decoder, upsampled part: the tile holds 128 outputs of column
// parity px (x = xb + 2m + px) in R rows.  Nearest upsampling folds the 3x3
// taps over the upsampled source into 2x2 taps over the low-resolution halo:
// low-res row hl feeds output rows 2hl-3 .. 2hl of the tile (parity classes
// (1,+1), (0,0), (1,0), (0,-1) in (row parity, row offset)), whose summed
// weights are stacked along N in that order; the column offset dx runs over
// two values selected by px (A shifted by d + px pixels).
template <int R, int G, bool TF>
__device__ __forceinline__ void issue_up(uint64_t ad, uint64_t bd, uint32_t dbase, uint32_t N,
                                         int px, int pxb, uint32_t row16, uint32_t id1,
                                         uint32_t id2, uint32_t id3, uint32_t id4) {
  if (!elect_one()) return;
#pragma unroll
  for (int d = 0; d < 2; ++d) {
    const uint64_t adk = ad + static_cast<uint32_t>(d + px);
    const uint64_t bdk = bd + static_cast<uint32_t>(pxb * 2 + d) * 8u * N;
#pragma unroll
    for (int hl = 0; hl < R / 2 + 2; ++hl) {
      const int lo = 2 * hl - 3 > 0 ? 2 * hl - 3 : 0;
      const int hi = 2 * hl < R - 1 ? 2 * hl : R - 1;
      const uint64_t a = adk + static_cast<uint32_t>(hl) * row16;
#pragma unroll
      for (int c = lo; c <= hi; c += G) {
        const int e = c + G - 1 < hi ? c + G - 1 : hi;
        const int n = e - c + 1;
        umma_k<TF>(dbase + c * N, a, bdk + static_cast<uint32_t>(c - 2 * hl + 3) * N,
                   n == 1 ? id1 : n == 2 ? id2 : n == 3 ? id3 : id4);
      }
    }
  }
}

// Sub-pixel decoder, skip part for one kx: the halo box of one column-parity
// plane of the skip source holds the skip pixels xb + px + kx - 1 + 2m (A
// shifted by one element for kx = 2 in the outer plane); ky stacked along N
// as in issue_kblock.
template <int R, int G, bool TF>
__device__ __forceinline__ void issue_skip(uint64_t ad, uint64_t bd, uint32_t dbase, uint32_t N,
                                           uint32_t row16, uint32_t id1, uint32_t id2, uint32_t id3) {
  if (!elect_one()) return;
#pragma unroll
  for (int h = 0; h < R + 2; ++h) {
    const int lo = h - 2 > 0 ? h - 2 : 0;
    const int hi = h < R - 1 ? h : R - 1;
    const uint64_t a = ad + static_cast<uint32_t>(h) * row16;
#pragma unroll
    for (int c = lo; c <= hi; c += G) {
      const int e = c + G - 1 < hi ? c + G - 1 : hi;
      const int n = e - c + 1;
      umma_k<TF>(dbase + c * N, a, bd + static_cast<uint32_t>(2 - h + c) * N,
                 n == 1 ? id1 : n == 2 ? id2 : id3);
    }
  }
}

template <int R, int G4, int G3, bool TF>
__device__ __forceinline__ void issue_subpixel_r(bool up, uint64_t ad, uint64_t bd,
                                                 uint32_t dbase, uint32_t N, int px, int pxb,
                                                 uint32_t row16, uint32_t id1, uint32_t id2,
                                                 uint32_t id3, uint32_t id4) {
  if (!up) {
    // bd: first kx slice; pxb (reused): 16-byte units to the second slice, 0 if none
    issue_skip<R, G3, TF>(ad, bd, dbase, N, row16, id1, id2, id3);
    if (pxb) issue_skip<R, G3, TF>(ad + 1, bd + static_cast<uint32_t>(pxb), dbase, N, row16, id1, id2, id3);
  } else {
    issue_up<R, G4, TF>(ad, bd, dbase, N, px, pxb, row16, id1, id2, id3, id4);
  }
}

template <int G4, int G3, bool TF>
__device__ __forceinline__ void issue_subpixel_item(int R, bool up, uint64_t ad, uint64_t bd,
                                                    uint32_t dbase, uint32_t N, int px, int pxb,
                                                    uint32_t row16, uint32_t id1, uint32_t id2,
                                                    uint32_t id3, uint32_t id4) {
  switch (R) {
    case 2: issue_subpixel_r<2, G4, G3, TF>(up, ad, bd, dbase, N, px, pxb, row16, id1, id2, id3, id4); break;
    case 4: issue_subpixel_r<4, G4, G3, TF>(up, ad, bd, dbase, N, px, pxb, row16, id1, id2, id3, id4); break;
    default: issue_subpixel_r<8, G4, G3, TF>(up, ad, bd, dbase, N, px, pxb, row16, id1, id2, id3, id4); break;
  }
}

// One sub-pixel item of a compile-time shape SPEC = 100 + 10 R + G4 (every
// walk step a whole tile of R rows).
template <int SPEC, bool TF>
__device__ __forceinline__ void issue_subpixel_spec(bool up, uint64_t ad, uint64_t bd, uint32_t dbase,
                                                    uint32_t N, int px, int pxb, uint32_t row16,
                                                    uint32_t id1, uint32_t id2, uint32_t id3,
                                                    uint32_t id4) {
  constexpr int SR = (SPEC - 100) / 10, SG4 = SPEC % 10, SG3 = SG4 < 3 ? SG4 : 3;
  issue_subpixel_r<SR, SG4, SG3, TF>(up, ad, bd, dbase, N, px, pxb, row16, id1, id2, id3, id4);
}

// One sub-pixel item with the row grouping G4 = min(4, 256 / N) (upsampled
// part; the skip part groups min(3, G4) rows).
template <bool TF>
__device__ __forceinline__ void issue_subpixel_g(int g4, int R, bool up, uint64_t ad, uint64_t bd,
                                                 uint32_t dbase, uint32_t N, int px, int pxb,
                                                 uint32_t row16, uint32_t id1, uint32_t id2,
                                                 uint32_t id3, uint32_t id4) {
  if (g4 == 4) issue_subpixel_item<4, 3, TF>(R, up, ad, bd, dbase, N, px, pxb, row16, id1, id2, id3, id4);
  else if (g4 == 2) issue_subpixel_item<2, 2, TF>(R, up, ad, bd, dbase, N, px, pxb, row16, id1, id2, id3, id4);
  else issue_subpixel_item<1, 1, TF>(R, up, ad, bd, dbase, N, px, pxb, row16, id1, id2, id3, id4);
}

}  // namespace

// SPEC fixes the issue sequence at compile time for the common shapes, so
// that the MMA warp's loop holds one or two unrolled sequences instead of one
// per (rows, grouping) pair: 0 = chosen at run time; 10 R + G = plain tiles
// of R rows (R / 2 in a last wave split in two), G rows stacked per MMA;
// 100 + 10 R + G = sub-pixel tiles of R rows (no split), G row classes
// stacked.  Plain shapes also fix the epilogue mode: + 1000 (mode + 1).
// (A smaller MMA loop is an instruction-cache matter: the 1080p step went
// from 494 to 478 us.)
constexpr int kSpecAny = 0;
constexpr int spec_plain(int r, int g, int mode) { return 1000 * (mode + 1) + 10 * r + g; }
constexpr int spec_sub(int r, int g) { return 100 + 10 * r + g; }

template <int KIND, int SPEC>
__global__ void __launch_bounds__(kind_helpers<KIND>() ? kTcThreadsDecoder : kTcThreads, 1)
    conv3x3_tc_kernel(const __grid_constant__ CUtensorMap map0,
                      const __grid_constant__ CUtensorMap map1, const TcConvParams p) {
  extern __shared__ uint8_t smem_raw[];
  // 128-byte alignment suffices: TMA tile destinations need 128 B, the
  // unswizzled UMMA operands 16 B (every region below is a 1 KB multiple)
  const uint32_t pad = (128u - (smem_u32(smem_raw) & 127u)) & 127u;
  uint8_t* smem = smem_raw + pad;

  const int S = p.S, R = p.R, N = p.N, KB0 = p.KB0;
  const int KB = p.KB0 + p.KB1;
  const int num_tiles = p.walk_tiles;  // walk steps (tiles and tail sub-tiles)
  constexpr bool SP = kind_subpixel<KIND>();
  constexpr bool TF = kind_tf32<KIND>();
  constexpr bool EXP = kind_expand<KIND>();
  constexpr bool HELP = kind_helpers<KIND>();
  constexpr int SRG = SPEC % 1000;                         // the shape part of SPEC
  constexpr int SMODE = SPEC >= 1000 ? SPEC / 1000 - 1 : -1;  // the epilogue mode, or -1
  // pipeline items per tile: K blocks, or (sub-pixel) upsampled K blocks plus
  // one item per (skip K block, kx)
  // sub-pixel: items are groups of up_pair upsampled K blocks (one TMA box
  // of 2 * up_pair chunks), then one item per (skip K block, plane)
  const int n_up = SP ? (KB0 + p.up_pair - 1) / p.up_pair : KB0;
  const int items = SP ? n_up + 2 * p.KB1 : KB;
  // shared memory: [resident weights][A stages][A_lo stages (tf32)][B stages]
  // [staging][bias][barriers]
  uint8_t* Wres = smem;
  uint8_t* A = Wres + (p.resident ? ((p.wres_bytes + 1023u) & ~1023u) : 0u);
  uint8_t* ALO = A + static_cast<size_t>(S) * p.a_stage;
  uint8_t* B = ALO + (TF ? static_cast<size_t>(S) * p.a_stage : 0u);
  uint8_t* ST = B + (p.resident ? 0 : static_cast<size_t>(S) * p.b_stage);
  float* bias_s = reinterpret_cast<float*>(ST + static_cast<size_t>(S) * p.st_stage);
  uint64_t* full = reinterpret_cast<uint64_t*>(bias_s + ((N + 31) / 32) * 32);
  uint64_t* empty = full + S;
  uint64_t* xdone = empty + S;
  uint64_t* tfull = xdone + S;   // [2] accumulator set ready
  uint64_t* tempty = tfull + 2;  // [2] accumulator set drained
  uint64_t* wbar = tempty + 2;   // resident weights landed
  uint64_t* done = wbar + 1;     // every MMA finished
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&xdone[s], 128);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 32 * kTcEpilogueWarps);
    }
    mbar_init(wbar, 1);
    mbar_init(done, 1);
    fence_mbarrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Every CTA of this persistent grid is resident: the next layer's kernel
  // may start its prologue on SMs as they free up.
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&map0);
      if (p.KB1 > 0) prefetch_tmap(&map1);
      if (p.resident) {
        if (SP) {
          // This CTA's tiles all have column parity blockIdx.x & 1 (even
          // grid; flipped when the tiles are walked in reverse): only that
          // parity's half of each upsampled block stays resident, followed
          // by the skip blocks.
          const uint8_t* w = reinterpret_cast<const uint8_t*>(p.weights);
          const uint32_t half = p.b_tx / 2;
          const uint32_t cpx = (blockIdx.x ^ static_cast<uint32_t>(p.reverse)) & 1u;
          mbar_arrive_expect_tx(wbar, p.wres_bytes);
          for (int kb = 0; kb < KB0; ++kb)
            bulk_load(Wres + static_cast<size_t>(kb) * half,
                      w + static_cast<size_t>(kb) * p.b_tx + cpx * half, half, wbar);
          const uint32_t skip = p.wres_bytes - static_cast<uint32_t>(KB0) * half;
          for (uint32_t off = 0; off < skip; off += 65536u)
            bulk_load(Wres + static_cast<size_t>(KB0) * half + off,
                      w + static_cast<size_t>(KB0) * p.b_tx + off, min(65536u, skip - off), wbar);
        } else {
          mbar_arrive_expect_tx(wbar, static_cast<uint32_t>(KB) * p.b_tx);
          for (int kb = 0; kb < KB; ++kb)
            bulk_load(Wres + static_cast<size_t>(kb) * p.b_stage,
                      reinterpret_cast<const uint8_t*>(p.weights) + static_cast<size_t>(kb) * p.b_tx,
                      p.b_tx, wbar);
        }
      }
      // Weights and bias are constants; the activations come from the
      // previous kernel in the stream.
      griddep_wait();
      const uint64_t pol = p.l2_first ? l2_evict_first() : l2_evict_normal();
      uint32_t it = 0, s = 0, ph = 0;  // item count, its stage and phase
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        int x0, y0, px;
        tile_origin_k<KIND>(p, tile, &x0, &y0, &px);
        for (int kb = 0; kb < items; ++kb, ++it, next_stage(s, ph, S)) {
          if (!mbar_wait_bounded(&empty[s], ph ^ 1u, p.status, kErrTimeoutProducer)) {
            ok = false;
            break;
          }
          if (SP) {
            const uint8_t* wsrc = reinterpret_cast<const uint8_t*>(p.weights);
            if (kb < n_up) {
              const uint32_t half = p.b_tx / 2;  // one column parity of the block
              mbar_arrive_expect_tx(&full[s], p.a_tx + (p.resident ? 0u : half));
              // low-resolution box from kGroupPx left of the block's first
              // pixel (up_pair K blocks; a box reaching past the last chunk
              // reads zeros there, and no MMA uses them)
              tma_load_4d(A + static_cast<size_t>(s) * p.a_stage, &map0, &full[s], 0,
                          ((x0 >> 1) - kGroupPx) >> p.xs0, 2 * p.up_pair * kb, (y0 >> 1) - 1, pol);
              if (!p.resident)
                bulk_load(B + static_cast<size_t>(s) * p.b_stage,
                          wsrc + static_cast<size_t>(kb) * p.b_tx + static_cast<size_t>(px) * half,
                          half, &full[s]);
            } else {
              // skip source, column-parity split: the outer plane (parity
              // px ^ 1, serving kx = 0 and kx = 2) or the centre plane
              // (parity px, kx = 1) of one 16-channel block, from kGroupPx
              // entries left of the block's first entry
              const int j = (kb - n_up) >> 1, part = (kb - n_up) & 1;
              const int plane = part ? px : (px ^ 1);
              const int i0 = ((x0 >> 1) - kGroupPx) >> p.xs1;
              const uint32_t wb = part ? p.b_tx2 : 2u * p.b_tx2;
              mbar_arrive_expect_tx(&full[s], p.st_tx + (p.resident ? 0u : wb));
              tma_load_5d(A + static_cast<size_t>(s) * p.a_stage, &map1, &full[s], 0, i0, plane,
                          2 * j, y0 - 1, pol);
              if (!p.resident) {
                const size_t kb_off = static_cast<size_t>(KB0) * p.b_tx + static_cast<size_t>(3 * j) * p.b_tx2;
                if (part) {
                  bulk_load(B + static_cast<size_t>(s) * p.b_stage, wsrc + kb_off + p.b_tx2, p.b_tx2,
                            &full[s]);
                } else {  // kx = 0 and kx = 2 slices, one after the other
                  bulk_load(B + static_cast<size_t>(s) * p.b_stage, wsrc + kb_off, p.b_tx2, &full[s]);
                  bulk_load(B + static_cast<size_t>(s) * p.b_stage + p.b_tx2,
                            wsrc + kb_off + 2 * static_cast<size_t>(p.b_tx2), p.b_tx2, &full[s]);
                }
              }
            }
            continue;
          }
          const bool low = p.upsample0 && kb < KB0;
          mbar_arrive_expect_tx(&full[s], (low ? p.st_tx : p.a_tx) + (p.resident ? 0u : p.b_tx));
          if (kb < KB0) {
            // boxes start kGroupPx pixels left of the tile (a multiple of 8,
            // so 128-byte-row maps address it in 8-pixel units)
            if (low)
              tma_load_4d(ST + static_cast<size_t>(s) * p.st_stage, &map0, &full[s], 0,
                          ((x0 >> 1) - kGroupPx) >> p.xs0, 2 * kb, (y0 >> 1) - 1, pol);
            else
              tma_load_4d(A + static_cast<size_t>(s) * p.a_stage, &map0, &full[s], 0,
                          (x0 - kGroupPx) >> p.xs0, 2 * kb, y0 - 1, pol);
          } else {
            tma_load_4d(A + static_cast<size_t>(s) * p.a_stage, &map1, &full[s], 0,
                        (x0 - kGroupPx) >> p.xs1, 2 * (kb - KB0), y0 - 1, pol);
          }
          if (!p.resident)
            bulk_load(B + static_cast<size_t>(s) * p.b_stage,
                      reinterpret_cast<const uint8_t*>(p.weights) + static_cast<size_t>(kb) * p.b_tx,
                      p.b_tx, &full[s]);
        }
      }
      // Every copy issued must have landed before this CTA may exit.
      for (uint32_t k = it > static_cast<uint32_t>(S) ? it - S : 0u; k < it; ++k)
        mbar_wait_bounded(&full[k % S], (k / S) & 1u, p.status, kErrTimeoutDrain);
      if (p.resident) mbar_wait_bounded(wbar, 0, p.status, kErrTimeoutDrain);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp walks the loop (descriptor arithmetic stays warp-uniform);
    // one elected lane issues each MMA and commit.  Waits are taken by every
    // lane and their outcome agreed on, so the warp never diverges.
    {
      const int g = min(3, 256 / N);
      const int g4 = min(4, 256 / N);
      const uint32_t id1 = TF ? idesc_tf32_f32(kTileM, N) : idesc_f16_f32(kTileM, N);
      const uint32_t id2 = TF ? idesc_tf32_f32(kTileM, min(2 * N, 256))
                              : idesc_f16_f32(kTileM, min(2 * N, 256));
      const uint32_t id3 = TF ? idesc_tf32_f32(kTileM, min(3 * N, 256))
                              : idesc_f16_f32(kTileM, min(3 * N, 256));
      const uint32_t id4 = TF ? idesc_tf32_f32(kTileM, min(4 * N, 256))
                              : idesc_f16_f32(kTileM, min(4 * N, 256));
      // tf32: the A_lo stages follow the A stages; each K block's B_lo
      // follows its B_hi (half of the block).  Sub-pixel: B_lo follows B_hi
      // within each column parity's half of an upsampled block and within
      // each kx slice of a skip block.
      const uint32_t alo16 = TF ? (static_cast<uint32_t>(S) * p.a_stage) >> 4 : 0u;
      const uint32_t blo16 = TF ? (p.b_tx / 2) >> 4 : 0u;
      const uint32_t blo_up16 = TF ? (p.b_tx / 4) >> 4 : 0u;
      const uint32_t blo_sk16 = TF ? (p.b_tx2 / 2) >> 4 : 0u;
      constexpr int kPasses = TF ? 3 : 1;
      // sub-pixel boxes: rows of kHaloW entries starting kGroupPx left of the
      // block (low-resolution x0/2 - 1 at kHaloOff)
      const uint64_t a_up0 = smem_desc_noswizzle(smem_u32(A), kHaloW * kChunkBytes, 128);
      const uint32_t wbase = smem_u32(p.resident ? Wres : B);
      const uint64_t b_up0 = smem_desc_noswizzle(wbase, 4u * N * kChunkBytes, 128);
      const uint64_t b_sk0 = smem_desc_noswizzle(wbase, 3u * N * kChunkBytes, 128);
      // plain / expansion halo rows are kHaloW pixels, x0 - 1 at kHaloOff
      const uint64_t a_desc0 =
          smem_desc_noswizzle(smem_u32(A), kHaloW * kChunkBytes, 128) + kHaloOff;
      const uint64_t b_desc0 =
          smem_desc_noswizzle(smem_u32(p.resident ? Wres : B), 3u * N * kChunkBytes, 128);
      const uint32_t kx_b16 = 6u * N;  // one kx block of B = 2 x 3N rows x 16 B
      const uint32_t set_cols = static_cast<uint32_t>(R * N);
      bool ok = __all_sync(0xffffffffu,
                           !p.resident || mbar_wait_bounded(wbar, 0, p.status, kErrTimeoutMma));
      uint32_t it = 0, s = 0, ph = 0, tcount = 0;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++tcount) {
        const uint32_t buf = tcount & 1u;
        // use k of a set needs phase k of tempty: the epilogue's initial
        // bias fill (k = 0), then its drain of use k - 1
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&tempty[buf], (tcount >> 1) & 1u, p.status,
                                                        kErrTimeoutMma))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_base = tmem + buf * set_cols;
        int tx0, ty0, tpx;
        const int R = tile_origin_k<KIND>(p, tile, &tx0, &ty0, &tpx);  // this tile's rows
        for (int kb = 0; kb < items; ++kb, ++it, next_stage(s, ph, S)) {
          bool w = mbar_wait_bounded(&full[s], ph, p.status, kErrTimeoutMma);
          if (HELP && w) w = mbar_wait_bounded(&xdone[s], ph, p.status, kErrTimeoutMma);
          ok = __all_sync(0xffffffffu, w);
          if (!ok) break;
          // (no tcgen05 fence: the stage barrier orders the TMA / expansion
          // writes before these MMA reads; the accumulator release below is
          // the one that orders TMEM accesses of other threads)
          if (SP) {
            const bool up = kb < n_up;
            const uint32_t soff = (s * p.a_stage) >> 4;
            uint32_t woff;
            int pxb;
            if (up) {
              // resident weights and streamed stages both hold only this
              // tile's parity half of an upsampled block
              const uint32_t half = p.b_tx / 2;
              const int kb0 = kb * p.up_pair;
              woff = p.resident ? static_cast<uint32_t>(kb0) * half : s * p.b_stage;
              // one item covers up_pair K blocks: their chunks sit 2 * kHaloW
              // entries apart in each box row, their weights one half apart
              const uint64_t ad = a_up0 + soff + static_cast<uint32_t>(kHaloOff);
              const uint64_t bd = b_up0 + (woff >> 4);
              const uint32_t row16 = static_cast<uint32_t>(2 * p.up_pair * kHaloW);
              const int nkb = min(p.up_pair, KB0 - kb0);
              // tf32: passes A_hi B_hi, A_hi B_lo, A_lo B_hi
#pragma unroll 1
              for (int pass = 0; pass < kPasses; ++pass) {
                const uint64_t ap = ad + (pass == 2 ? alo16 : 0u);
                const uint64_t bp = bd + (pass == 1 ? blo_up16 : 0u);
                for (int jj = 0; jj < nkb; ++jj) {
                  const uint64_t adj = ap + static_cast<uint32_t>(jj * 2 * kHaloW);
                  const uint64_t bdj = bp + static_cast<uint32_t>(jj) * (half >> 4);
                  if constexpr (SRG >= 100)
                    issue_subpixel_spec<SRG, TF>(true, adj, bdj, d_base, N, tpx, 0, row16, id1, id2, id3, id4);
                  else
                    issue_subpixel_g<TF>(g4, R, true, adj, bdj, d_base, N, tpx, 0, row16, id1, id2, id3, id4);
                }
              }
              if (elect_one()) mma_commit(&empty[s]);
              continue;
            } else {
              const int j = (kb - n_up) >> 1, part = (kb - n_up) & 1;
              if (p.resident)
                woff = static_cast<uint32_t>(KB0) * (p.b_tx / 2) + static_cast<uint32_t>(3 * j + part) * p.b_tx2;
              else
                woff = s * p.b_stage;
              // outer plane: kx = 0 then kx = 2 (two slices apart when resident,
              // adjacent when streamed); centre plane: kx = 1 only
              pxb = part ? 0 : static_cast<int>((p.resident ? 2u * p.b_tx2 : p.b_tx2) >> 4);
            }
            // upsampled: x0/2 - 1 at kHaloOff; skip: the centre plane's first
            // entry at kGroupPx, the outer plane's x0/2 + px - 1 at kHaloOff + px
            const int aoff = (kb - n_up) & 1 ? kGroupPx : kHaloOff + tpx;
            const uint64_t ad = a_up0 + soff + static_cast<uint32_t>(aoff);
            const uint64_t bd = b_sk0 + (woff >> 4);
            const uint32_t row16 = static_cast<uint32_t>(2 * kHaloW);
#pragma unroll 1
            for (int pass = 0; pass < kPasses; ++pass) {
              if constexpr (SRG >= 100)
                issue_subpixel_spec<SRG, TF>(false, ad + (pass == 2 ? alo16 : 0u),
                                              bd + (pass == 1 ? blo_sk16 : 0u), d_base, N, tpx, pxb,
                                              row16, id1, id2, id3, id4);
              else
                issue_subpixel_g<TF>(g4, R, false, ad + (pass == 2 ? alo16 : 0u),
                                     bd + (pass == 1 ? blo_sk16 : 0u), d_base, N, tpx, pxb, row16, id1,
                                     id2, id3, id4);
            }
            if (elect_one()) mma_commit(&empty[s]);
            continue;
          }
          const uint64_t ad = a_desc0 + ((s * p.a_stage) >> 4);
          const uint64_t bd = b_desc0 + ((static_cast<uint32_t>(p.resident ? kb : s) * p.b_stage) >> 4);
          if constexpr (SRG > 0 && SRG < 100) {
            constexpr int SR = SRG / 10, SG = SRG % 10;
            // tf32: passes A_hi B_hi, A_hi B_lo, A_lo B_hi
#pragma unroll 1
            for (int pass = 0; pass < kPasses; ++pass) {
              const uint64_t ap = ad + (pass == 2 ? alo16 : 0u);
              const uint64_t bp = bd + (pass == 1 ? blo16 : 0u);
              if (R == SR) issue_kblock<SR, SG, TF>(ap, bp, d_base, N, kx_b16, id1, id2, id3);
              else issue_kblock<(SR > 1 ? SR / 2 : 1), SG, TF>(ap, bp, d_base, N, kx_b16, id1, id2, id3);
            }
          } else if (g == 3) {
            issue_kblock_r<3, TF>(R, ad, bd, d_base, N, kx_b16, id1, id2, id3, alo16, blo16);
          } else if (g == 2) {
            issue_kblock_r<2, TF>(R, ad, bd, d_base, N, kx_b16, id1, id2, id3, alo16, blo16);
          } else {
            issue_kblock_r<1, TF>(R, ad, bd, d_base, N, kx_b16, id1, id2, id3, alo16, blo16);
          }
          if (elect_one()) mma_commit(&empty[s]);
        }
        if (!ok) break;
        if (elect_one()) mma_commit(&tfull[buf]);
      }
      // TMEM is freed only after every MMA issued above has completed.
      if (elect_one()) mma_commit(done);
      mbar_wait_bounded(done, 0, p.status, kErrTimeoutMma);
    }
    __syncwarp();
  } else if (warp >= 2 + kTcEpilogueWarps) {
    // (only launched with these warps for the expansion and tf32 kinds)
    // ------------------------------------------------------------ helpers
    // Expansion kinds: build the upsampled halo of each upsampled K block
    // from its low-resolution staging box.  tf32 kinds: split every stage's
    // A into A_hi (rounded to tf32, in place) and A_lo = A - A_hi (the A_lo
    // stage).  Only the kHaloPx pixels the MMAs read (x0 - 1
    // .. x0 + 128) of each row are touched.
    const int et = threadIdx.x - 32 * (2 + kTcEpilogueWarps);  // 0..127
    const int total = (R + 2) * 2 * kHaloPx;
    uint32_t it = 0, s = 0, ph = 0;
    bool ok = true;
    // sub-pixel (tf32 only): every staged box is split whole, the upsampled
    // items' low-resolution box or the skip items' plane box.  (Splitting
    // only the 130 entries per row the MMAs read was not faster.)
    for (int tile = blockIdx.x; SP && tile < num_tiles && ok; tile += gridDim.x) {
      for (int kb = 0; kb < items; ++kb, ++it, next_stage(s, ph, S)) {
        if (!mbar_wait_bounded(&full[s], ph, p.status, kErrTimeoutEpilogue)) {
          ok = false;
          break;
        }
        uint4* hi = reinterpret_cast<uint4*>(A + static_cast<size_t>(s) * p.a_stage);
        uint4* lo = reinterpret_cast<uint4*>(ALO + static_cast<size_t>(s) * p.a_stage);
        const int n16 = static_cast<int>((kb < n_up ? p.a_tx : p.st_tx) >> 4);
        for (int i = et; i < n16; i += 128) split_tf32(hi + i, lo + i);
        fence_proxy_async_smem();
        mbar_arrive(&xdone[s]);
      }
    }
    for (int tile = blockIdx.x; !SP && tile < num_tiles && ok; tile += gridDim.x) {
      int x0, y0, px;
      tile_origin_k<KIND>(p, tile, &x0, &y0, &px);
      const int ly0 = (y0 >> 1) - 1, lx0 = (x0 >> 1) - kGroupPx;
      for (int kb = 0; kb < KB; ++kb, ++it, next_stage(s, ph, S)) {
        // Waiting on every stage keeps this warp group at most one use of a
        // stage ahead of the MMA issuer, so the xdone phases stay paired.
        if (!mbar_wait_bounded(&full[s], ph, p.status, kErrTimeoutEpilogue)) {
          ok = false;
          break;
        }
        uint4* dst = reinterpret_cast<uint4*>(A + static_cast<size_t>(s) * p.a_stage);
        uint4* lo = reinterpret_cast<uint4*>(ALO + static_cast<size_t>(s) * p.a_stage);
        const bool expand = EXP && kb < KB0;
        if (expand || TF) {
          const uint4* src = reinterpret_cast<const uint4*>(ST + static_cast<size_t>(s) * p.st_stage);
          for (int i = et; i < total; i += 128) {
            const int px = i % kHaloPx;
            const int rc = i / kHaloPx;
            const int at = rc * kHaloW + kHaloOff + px;
            uint4 v;
            if (expand) {
              const int j = rc & 1, rr = rc >> 1;
              const int iy = y0 - 1 + rr, ix = x0 - 1 + px;
              v = make_uint4(0u, 0u, 0u, 0u);
              if (iy >= 0 && iy < p.H && ix >= 0 && ix < p.W) {
                const int sr = (iy >> 1) - ly0, sc = (ix >> 1) - lx0;
                v = src[(sr * 2 + j) * kLowW + sc];
              }
            } else {
              v = dst[at];
            }
            if (TF) {
              // hi: rounded to the nearest tf32 value, so |lo| <= 2^-11 |A|
              const uint4 h = make_uint4((v.x + 0x1000u) & 0xFFFFE000u, (v.y + 0x1000u) & 0xFFFFE000u,
                                         (v.z + 0x1000u) & 0xFFFFE000u, (v.w + 0x1000u) & 0xFFFFE000u);
              lo[at] = make_uint4(__float_as_uint(__uint_as_float(v.x) - __uint_as_float(h.x)),
                                  __float_as_uint(__uint_as_float(v.y) - __uint_as_float(h.y)),
                                  __float_as_uint(__uint_as_float(v.z) - __uint_as_float(h.z)),
                                  __float_as_uint(__uint_as_float(v.w) - __uint_as_float(h.w)));
              v = h;
            }
            dst[at] = v;
          }
          fence_proxy_async_smem();
        }
        mbar_arrive(&xdone[s]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Eight warps: warp w reads TMEM lane quarter w % 4 (pixels 32q..32q+31
    // of the M tile); the two warps of a quarter split the tile's rows.
    const int et = threadIdx.x - 64;  // 0..255
    for (int i = et; i < N; i += 32 * kTcEpilogueWarps) bias_s[i] = p.bias[i];
    named_barrier_sync(1, 32 * kTcEpilogueWarps);
    const int q = warp & 3;
    const int sub = (warp - 2) >> 2;  // 0 or 1
    const int m = q * 32 + lane;      // pixel in the M tile = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const int nc = N / 16;
    const int C8 = N / 8;
    const uint32_t set_cols = static_cast<uint32_t>(R * N);
    // The accumulators start from the bias: both sets are filled before the
    // first tile (rows sub, sub + 2, ... of this lane quarter), and every
    // accumulator is refilled right after it has been read.
    for (int b = 0; b < 2; ++b)
      for (int r = sub; r < R; r += 2)
        for (int c = 0; c < nc; ++c)
          tmem_fill_bias(tmem + lane_off + b * set_cols + static_cast<uint32_t>(r * N + c * 16),
                         bias_s + c * 16);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&tempty[0]);
    mbar_arrive(&tempty[1]);
    uint32_t tcount = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++tcount) {
      const uint32_t buf = tcount & 1u;
      if (!mbar_wait_bounded(&tfull[buf], (tcount >> 1) & 1u, p.status, kErrTimeoutEpilogue)) break;
      tc_fence_after();
      int x0, y0, px;
      const int R = tile_origin_k<KIND>(p, tile, &x0, &y0, &px);  // this tile's rows
      // sub-pixel tiles hold every other output column
      const int x = SP ? x0 + 2 * m + px : x0 + m;
      const uint32_t tl = tmem + lane_off + buf * set_cols;

      // decoders (expansion, sub-pixel) always take the ReLU epilogue
      const int mode = SMODE >= 0 ? SMODE : p.mode;
      if (EXP || SP || mode == kEpiRelu) {
        __half* out = static_cast<__half*>(p.out);
        for (int c0 = 0; c0 < nc; c0 += 2) {
          const bool two = c0 + 1 < nc;
          // the refill values of these 32 columns, read once for all rows
          // (per row in the fp32 kinds, whose helper warps leave no
          // registers to spare for them)
          constexpr bool kHoist = !TF;
          uint32_t bz[2][16];
          if (kHoist) {
            bias16_regs(bias_s + c0 * 16, bz[0]);
            if (two) bias16_regs(bias_s + c0 * 16 + 16, bz[1]);
          }
          for (int r = sub; r < R; r += 2) {
            const int y = y0 + r;
            uint32_t v[2][16];
            const uint32_t t0 = tl + static_cast<uint32_t>(r * N + c0 * 16);
            tmem_ld16_nowait(t0, v[0]);
            if (two) tmem_ld16_nowait(t0 + 16, v[1]);
            tmem_wait_ld();
            if (!kHoist) {
              bias16_regs(bias_s + c0 * 16, bz[0]);
              if (two) bias16_regs(bias_s + c0 * 16 + 16, bz[1]);
            }
            tmem_st16(t0, bz[0]);
            if (two) tmem_st16(t0 + 16, bz[1]);
            // columns [W, pitch) are row padding: stored as zeros
            if (TF && x < p.pitch && y < p.H) {
              const bool pad = x >= p.W || (p.period && y % p.period >= p.rows);
              float* row = static_cast<float*>(p.out) + (static_cast<size_t>(y) * p.out_c4 * p.pitch + x) * 4;
#pragma unroll
              for (int b = 0; b < 2; ++b) {
                if (b == 1 && !two) break;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                  float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
                  if (!pad)
                    f = make_float4(fmaxf(__uint_as_float(v[b][4 * q4]), 0.0f),
                                    fmaxf(__uint_as_float(v[b][4 * q4 + 1]), 0.0f),
                                    fmaxf(__uint_as_float(v[b][4 * q4 + 2]), 0.0f),
                                    fmaxf(__uint_as_float(v[b][4 * q4 + 3]), 0.0f));
                  const int c4 = 4 * (c0 + b) + q4;
                  if (c4 < p.out_c4)
                    *reinterpret_cast<float4*>(row + static_cast<size_t>(c4) * p.pitch * 4) = f;
                }
              }
            } else if (!TF && x < p.pitch && y < p.H) {
              const bool pad = x >= p.W || (p.period && y % p.period >= p.rows);
              __half* row = out + (static_cast<size_t>(y) * C8 * p.pitch + x) * 8;
#pragma unroll
              for (int b = 0; b < 2; ++b) {
                if (b == 1 && !two) break;
                uint32_t h[8];
#pragma unroll
                for (int k = 0; k < 8; ++k)
                  h[k] = pad ? 0u
                             : pack_half2(fmaxf(__uint_as_float(v[b][2 * k]), 0.0f),
                                          fmaxf(__uint_as_float(v[b][2 * k + 1]), 0.0f));
                const size_t c8 = 2 * (c0 + b);
                *reinterpret_cast<uint4*>(row + c8 * p.pitch * 8) = make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4*>(row + (c8 + 1) * p.pitch * 8) = make_uint4(h[4], h[5], h[6], h[7]);
              }
            }
          }
        }
      } else if (mode == kEpiReluPool) {
        __half* out = static_cast<__half*>(p.out);
        const int Wp = (p.W + 1) >> 1, Hp = (p.H + 1) >> 1;
        const int xp = x >> 1;
        for (int c = 0; c < nc; ++c) {
          uint32_t bz[16];  // refill values of these 16 columns, read once
          bias16_regs(bias_s + c * 16, bz);
          for (int i = sub; i < R / 2; i += 2) {
            const int ya = y0 + 2 * i;
            const bool va = x < p.W && ya < p.H;
            const bool vb = x < p.W && ya + 1 < p.H;
            // stacked tiles: a pooled gap row (rows and period are even) is zero
            const bool gap = p.period && ya % p.period >= p.rows;
            const int yp = ya >> 1;
            uint32_t v[2][16];
            const uint32_t t0 = tl + static_cast<uint32_t>((2 * i) * N + c * 16);
            tmem_ld16_nowait(t0, v[0]);
            tmem_ld16_nowait(t0 + static_cast<uint32_t>(N), v[1]);
            tmem_wait_ld();
            tmem_st16(t0, bz);
            tmem_st16(t0 + static_cast<uint32_t>(N), bz);
            float mx[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const float a = va ? fmaxf(__uint_as_float(v[0][k]), 0.0f) : -INFINITY;
              const float b2 = vb ? fmaxf(__uint_as_float(v[1][k]), 0.0f) : -INFINITY;
              float t = fmaxf(a, b2);
              t = fmaxf(t, __shfl_xor_sync(0xffffffffu, t, 1));
              mx[k] = t;
            }
            // pooled columns [Wp, pitch) are row padding: stored as zeros
            if (TF && ((lane & 1) == 0) && yp < Hp) {
              const bool pad = xp >= Wp || gap;
              float* base = static_cast<float*>(p.out) + (static_cast<size_t>(yp) * p.out_c4 * p.pitch + xp) * 4;
              // split copy: plane xp & 1, index xp >> 1 (the split pitch is even)
              float* base2 = p.out_split == nullptr ? nullptr
                             : static_cast<float*>(p.out_split) +
                                   ((static_cast<size_t>(yp) * p.out_c4 * 2 + (xp & 1)) * (p.split_pitch >> 1) + (xp >> 1)) * 4;
#pragma unroll
              for (int q4 = 0; q4 < 4; ++q4) {
                const float4 f = pad ? make_float4(0.f, 0.f, 0.f, 0.f)
                                     : make_float4(mx[4 * q4], mx[4 * q4 + 1], mx[4 * q4 + 2], mx[4 * q4 + 3]);
                const int c4 = 4 * c + q4;
                if (c4 < p.out_c4 && xp < p.pitch)
                  *reinterpret_cast<float4*>(base + c4 * static_cast<size_t>(p.pitch) * 4) = f;
                if (c4 < p.out_c4 && p.out_split && xp < p.split_pitch)
                  *reinterpret_cast<float4*>(base2 + c4 * static_cast<size_t>(p.split_pitch) * 4) = f;
              }
            } else if (!TF && ((lane & 1) == 0) && yp < Hp) {
              const bool pad = xp >= Wp || gap;
              uint32_t h[8];
#pragma unroll
              for (int k = 0; k < 8; ++k) h[k] = pad ? 0u : pack_half2(mx[2 * k], mx[2 * k + 1]);
              if (xp < p.pitch) {
                const size_t base0 = ((static_cast<size_t>(yp) * C8 + 2 * c) * p.pitch + xp) * 8;
                const size_t base1 = base0 + static_cast<size_t>(p.pitch) * 8;
                *reinterpret_cast<uint4*>(out + base0) = make_uint4(h[0], h[1], h[2], h[3]);
                *reinterpret_cast<uint4*>(out + base1) = make_uint4(h[4], h[5], h[6], h[7]);
              }
              if (p.out_split && xp < p.split_pitch) {
                // plane xp & 1, index xp >> 1 (the split pitch is even)
                // (read by a decoder only: evict-first)
                __half* o2 = static_cast<__half*>(p.out_split);
                const size_t s0 =
                    ((((static_cast<size_t>(yp) * C8 + 2 * c) * 2 + (xp & 1)) * (p.split_pitch >> 1)) + (xp >> 1)) * 8;
                const size_t s1 = s0 + static_cast<size_t>(p.split_pitch) * 8;
                const uint64_t pol = l2_evict_first();
                st_global_hint(o2 + s0, make_uint4(h[0], h[1], h[2], h[3]), pol);
                st_global_hint(o2 + s1, make_uint4(h[4], h[5], h[6], h[7]), pol);
              }
            }
          }
        }
      } else {
        float4* out = static_cast<float4*>(p.out);
        for (int r0 = sub; r0 < R; r0 += 8) {
          uint32_t v[4][4];  // the 3 output channels and the zero lane
#pragma unroll
          for (int b = 0; b < 4; ++b)
            if (r0 + 2 * b < R) tmem_ld4_nowait(tl + static_cast<uint32_t>((r0 + 2 * b) * N), v[b]);
          tmem_wait_ld();
#pragma unroll
          for (int b = 0; b < 4; ++b)
            if (r0 + 2 * b < R) tmem_fill_bias(tl + static_cast<uint32_t>((r0 + 2 * b) * N), bias_s);
#pragma unroll
          for (int b = 0; b < 4; ++b) {
            const int y = y0 + r0 + 2 * b;
            if (r0 + 2 * b < R && x < p.W && y < p.H)
              out[static_cast<size_t>(y) * p.W + x] =
                  make_float4(__uint_as_float(v[b][0]), __uint_as_float(v[b][1]),
                              __uint_as_float(v[b][2]), __uint_as_float(v[b][3]));
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
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, p.tmem_cols);
  }
}

namespace {

// The compile-time shapes instantiated for the plain and sub-pixel kinds,
// fp16 and fp32 (the shapes of the 1080p and 4K U-Net layers); other
// shapes, and the expansion kinds, run the run-time form.
template <int KIND, int SPEC>
cudaError_t launch_tc(const TcConvLaunch& L, cudaStream_t stream) {
  return launch_pdl(conv3x3_tc_kernel<KIND, SPEC>, L.grid,
                    dim3(kind_helpers<KIND>() ? kTcThreadsDecoder : kTcThreads), L.smem, stream, L.map0,
                    L.map1, L.p);
}

// (rows, stacking, epilogue mode); the fp32 kind's 8-row form spills, so it
// keeps the run-time form
#define OIDNX_PLAIN_SPECS(X) \
  X(8, 3, 0) X(4, 3, 0) X(2, 3, 0) X(2, 2, 0) X(1, 2, 0) X(1, 3, 0) X(8, 3, 1) X(4, 3, 1) X(2, 3, 1)
#define OIDNX_PLAIN32_SPECS(X) \
  X(4, 3, 0) X(2, 3, 0) X(2, 2, 0) X(1, 2, 0) X(1, 3, 0) X(4, 3, 1) X(2, 3, 1)
#define OIDNX_SUB_SPECS(X) X(4, 4) X(2, 2)

// The spec of a launch: its tile rows, stacking factor and (plain kinds)
// epilogue mode, when every walk step has those rows (plain kinds: or half
// of them); kSpecAny otherwise, or when the filter asks for the run-time
// form ("shapeKernels" 0).
int tc_spec(const TcConvLaunch& L) {
  const TcConvParams& p = L.p;
  if (L.any_shape) return kSpecAny;
  if (L.kind == kTcSubpixel || L.kind == kTcSubpixel32) {
    const int g4 = std::min(4, 256 / p.N);
    // (a split last wave runs the run-time form: dec_conv2a at 1080p, whose
    // split tiles took 54.9 us specialised against 53.0)
    const bool steps = p.tail_split == 1;
#define X(r, g) if (steps && p.R == r && g4 == g) return spec_sub(r, g);
    OIDNX_SUB_SPECS(X)
#undef X
    return kSpecAny;
  }
  if (L.kind == kTcPlain || L.kind == kTcPlain32) {
    const int g = std::min(3, 256 / p.N);
    if (p.tail_split > 2) return kSpecAny;
#define X(r, gg, m) if (p.R == r && g == gg && p.mode == m) return spec_plain(r, gg, m);
    if (L.kind == kTcPlain) {
      OIDNX_PLAIN_SPECS(X)
    } else {
      OIDNX_PLAIN32_SPECS(X)
    }
#undef X
  }
  return kSpecAny;
}

}  // namespace

int conv_tc_shape(const TcConvLaunch& L) { return tc_spec(L); }

cudaError_t launch_conv_tc(const TcConvLaunch& L, cudaStream_t stream) {
  const int spec = tc_spec(L);
  switch (L.kind) {
    case kTcPlain32:
#define X(r, g, m) if (spec == spec_plain(r, g, m)) return launch_tc<kTcPlain32, spec_plain(r, g, m)>(L, stream);
      OIDNX_PLAIN32_SPECS(X)
#undef X
      return launch_tc<kTcPlain32, kSpecAny>(L, stream);
    case kTcExpand32: return launch_tc<kTcExpand32, kSpecAny>(L, stream);
    case kTcExpand: return launch_tc<kTcExpand, kSpecAny>(L, stream);
    case kTcSubpixel32:
#define X(r, g) if (spec == spec_sub(r, g)) return launch_tc<kTcSubpixel32, spec_sub(r, g)>(L, stream);
      OIDNX_SUB_SPECS(X)
#undef X
      return launch_tc<kTcSubpixel32, kSpecAny>(L, stream);
    case kTcSubpixel:
#define X(r, g) if (spec == spec_sub(r, g)) return launch_tc<kTcSubpixel, spec_sub(r, g)>(L, stream);
      OIDNX_SUB_SPECS(X)
#undef X
      return launch_tc<kTcSubpixel, kSpecAny>(L, stream);
    default:
#define X(r, g, m) if (spec == spec_plain(r, g, m)) return launch_tc<kTcPlain, spec_plain(r, g, m)>(L, stream);
      OIDNX_PLAIN_SPECS(X)
#undef X
      return launch_tc<kTcPlain, kSpecAny>(L, stream);
  }
}

cudaError_t conv_tc_set_smem_limit(size_t bytes) {
  const int b = static_cast<int>(bytes);
  const void* fns[] = {
      reinterpret_cast<const void*>(conv3x3_tc_kernel<kTcExpand, kSpecAny>),
      reinterpret_cast<const void*>(conv3x3_tc_kernel<kTcSubpixel, kSpecAny>),
      reinterpret_cast<const void*>(conv3x3_tc_kernel<kTcPlain32, kSpecAny>),
      reinterpret_cast<const void*>(conv3x3_tc_kernel<kTcExpand32, kSpecAny>),
      reinterpret_cast<const void*>(conv3x3_tc_kernel<kTcSubpixel32, kSpecAny>),
      reinterpret_cast<const void*>(conv3x3_tc_kernel<kTcPlain, kSpecAny>),
#define X(r, g, m) reinterpret_cast<const void*>(conv3x3_tc_kernel<kTcPlain, spec_plain(r, g, m)>),
      OIDNX_PLAIN_SPECS(X)
#undef X
#define X(r, g) reinterpret_cast<const void*>(conv3x3_tc_kernel<kTcSubpixel, spec_sub(r, g)>),
      OIDNX_SUB_SPECS(X)
#undef X
#define X(r, g, m) reinterpret_cast<const void*>(conv3x3_tc_kernel<kTcPlain32, spec_plain(r, g, m)>),
      OIDNX_PLAIN32_SPECS(X)
#undef X
#define X(r, g) reinterpret_cast<const void*>(conv3x3_tc_kernel<kTcSubpixel32, spec_sub(r, g)>),
      OIDNX_SUB_SPECS(X)
#undef X
  };
  for (const void* fn : fns) {
    const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, b);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t conv_tc_occupancy(size_t smem, int* blocks_per_sm) {
  // the plain variant has fewer threads and so the higher occupancy bound
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, conv3x3_tc_kernel<kTcPlain, kSpecAny>,
                                                       kTcThreads, smem);
}

}  // namespace oidnx

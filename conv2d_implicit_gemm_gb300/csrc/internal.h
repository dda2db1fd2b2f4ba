// Internal interfaces between the host runtime (oidnx.cpp) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace oidnx {

// Pixels of one output row per tensor-core M tile and halo geometry.
constexpr int kTileM = 128;
constexpr int kHaloPx = kTileM + 2;        // input pixels of one halo row
constexpr int kLowPx = kTileM / 2 + 2;     // low-resolution pixels for one M tile
// Plain and expansion kernels stage each halo row 8-pixel aligned: the box
// starts 8 pixels left of the tile, so that a TMA row can be 8 pixels x 16
// bytes (128 B) wide instead of one 16-byte pixel; the first pixel the MMA
// reads (x0 - 1) sits at index kHaloOff.
constexpr int kGroupPx = 8;                      // pixels per 128-byte TMA row
constexpr int kHaloW = kTileM + 2 * kGroupPx;    // 144 staged pixels per halo row
constexpr int kLowW = kTileM / 2 + 2 * kGroupPx; // 80 staged low-resolution pixels
constexpr int kHaloOff = kGroupPx - 1;           // 7
constexpr int kChunkBytes = 16;            // one 16-byte channel block
constexpr int kTcEpilogueWarps = 8;        // two per TMEM lane quarter
constexpr int kTcThreads = 320;            // 10 warps: TMA, MMA, 8 x epilogue
constexpr int kTcThreadsDecoder = 448;     // + 4 helper warps (upsampled halo, tf32 split)

enum EpilogueMode : int {
  kEpiRelu = 0,      // bias + ReLU, fp16 store
  kEpiReluPool = 1,  // bias + ReLU + 2x2 max-pool, fp16 store
  kEpiFinal = 2,     // bias only, fp32 [H][W][4] store
};

// Parameters of one tensor-core conv launch (one layer).
struct TcConvParams {
  const __half* weights;   // packed B operand, [kb][tap][2][N][8] halves (fp32 kinds:
                           // [kb][hi, lo][tap][2][N][4] floats)
  const float* bias;       // [N] (zero padded)
  void* out;               // fp16 [Ho][N/8][Wo][8] or f32 [H][W][4]
  int* status;             // device error word
  int W, H;                // conv (full-resolution) extent of this layer
  int N;                   // Cout rounded up to 16
  int KB0, KB1;            // 16-lane K blocks from source 0 / source 1
  int R;                   // output rows per CTA
  int S;                   // pipeline stages
  int mode;                // EpilogueMode
  int upsample0;           // source 0 is at half resolution (decoder)
  int tiles_x, tiles_y;    // output tiles of 128 pixels x R rows
  int resident;            // all weights held in shared memory for the CTA's life
  uint32_t tmem_cols;      // power of two >= max(32, 2*R*N): two accumulator sets
  uint32_t a_stage;        // bytes per A stage (1024-aligned)
  uint32_t b_stage;        // bytes per B block (1024-aligned)
  uint32_t st_stage;       // bytes per low-res staging stage (0 if none)
  uint32_t a_tx, b_tx, st_tx;  // transaction bytes per stage
  // sub-pixel decoder: b_tx = upsampled B block (512 N; tf32 1024 N), b_tx2 =
  // skip B kx slice (96 N; tf32 192 N), st_tx = strided skip box; wres_bytes =
  // resident weights
  uint32_t b_tx2;
  uint32_t wres_bytes;
  // pool epilogue: optional second copy of the output, column-parity split
  // [Ho][N/8][2][split_pitch/2][8] (fp32: [Ho][out_c4][2][split_pitch/2][4])
  // read by the sub-pixel decoder as its skip source; entries past the output
  // width are written as zeros
  void* out_split;
  int split_pitch;
  int pitch;               // fp16 output row pitch in pixels (>= output width);
                           // columns [width, pitch) are written as zeros
  int up_pair;             // sub-pixel: upsampled K blocks per pipeline item (1 or 2)
  // stacked tiles: rows y with y % period >= rows are the zero gap rows
  // between tiles (stored as zeros); period 0: a single image
  int period, rows;
  int out_c4;              // fp32 storage: 4-channel chunks of the output value
                           // (Cout rounded up to 4; may be fewer than N / 4)
  int xs0, xs1;            // log2 pixels per x unit of map0 / map1: 3 for
                           // 128-byte rows (pitch % 8 == 0), 0 for 16-byte rows
  int reverse;             // walk the tiles last to first (see tile_at)
  // Last wave: the walk's last (tiles_x * tiles_y - tail_first) tiles are
  // split into tail_split sub-tiles of R / tail_split rows each, so that a
  // short last wave spreads over more CTAs; walk_tiles counts the walk's
  // steps (tail_first = tiles, tail_split = 1: no split)
  int tail_first, tail_split, walk_tiles;
  int l2_first;            // activation loads evict-first in L2 (one-tile frames)
};

enum TcKind : int {
  kTcPlain = 0,     // plain conv (also pool / final epilogues)
  kTcExpand = 1,    // decoder, upsampled halo built in shared memory
  kTcSubpixel = 2,  // decoder, upsampled part as parity-class 2x2 taps
  kTcPlain32 = 3,   // fp32 storage, 3xTF32 products: plain conv
  kTcExpand32 = 4,  // fp32 storage, 3xTF32 products: decoder with expansion
  kTcSubpixel32 = 5,  // fp32 storage, 3xTF32 products: sub-pixel decoder
};

// Two same-padded 3x3 convs fused in one kernel (fp16 storage): conv 1
// (Cin -> 32, bias + ReLU, fp16-rounded) streams its output rows through
// tensor memory into shared memory, where conv 2 reads them; the 32-channel
// map between the two never reaches global memory.
enum PairMode : int {
  kPairFinal = 0,  // conv 2: 32 -> 3 final conv, fp32 [H][W][4] output
  kPairPool = 1,   // conv 2: 32 -> 32, bias + ReLU + 2x2 max-pool, fp16 output
};

constexpr int kPairSlots = 8;      // TMEM row accumulators per conv (ring)
constexpr int kPairBatch = 3;      // source rows whose MMAs are issued interleaved
constexpr int kPairMid = 2 * kPairBatch;  // conv-1 output rows held in shared memory
constexpr int kPairSpan = kTileM - 2;  // output pixels per strip at most

struct PairConvParams {
  const __half* w1;        // conv 1 B operand, [kb][kx][2][3 x 32][8] halves
  const __half* w2;        // conv 2 B operand: final [kb][2][3 x 16][8] (kx folded:
                           // row 16 * (2 - ky) + 4 * kx + co), pool as w1
  const float* bias1;      // [32]
  const float* bias2;      // final: [16] = {b0, b1, b2, 0, ...}; pool: [32]
  void* out;               // final: f32 [H][W][4]; pool: fp16 [Hp][4][pitch][8]
  void* out_split;         // pool: optional column-parity split copy, or null
  int* status;
  int W, H;                // conv extent (both convs)
  int KB1;                 // 16-channel K blocks of conv 1's input
  int C8;                  // 16-byte chunks per input pixel (2 * KB1)
  int strips, sw;          // column strips of sw output pixels (sw even, <= kPairSpan)
  int row_unit;            // 1 (final) or 2 (pool: rows in pairs)
  int units;               // strips * ceil(H / row_unit)
  int pitch, split_pitch;  // pool output pitches (pooled pixels)
  int S;                   // input row stages
  uint32_t stage_tx;       // one input row: kHaloW pixels x C8 chunks x 16 B
  uint32_t stage_bytes;    // its shared-memory stride (a multiple of 1024)
  uint32_t w1_bytes, w2_bytes;
  int xs;                  // log2 pixels per x unit of the input map
};

struct PairConvLaunch {
  CUtensorMap map;         // conv 1 input: boxes of one row, kHaloW pixels, C8 chunks
  PairConvParams p;
  int mode;                // PairMode
  dim3 grid;
  size_t smem;
};

cudaError_t launch_conv_pair(const PairConvLaunch& L, cudaStream_t stream);
cudaError_t conv_pair_set_smem_limit(size_t bytes);
cudaError_t conv_pair_occupancy(int mode, size_t smem, int* blocks_per_sm);

// The final conv (32 -> 3, bias, no ReLU; fp16 operands, or for fp32
// storage 3xTF32 products) with the three kx taps folded into N: tiles of
// kFinalRows rows x kFinalSpan output pixels.
// Optionally the output pass runs in its epilogue (denoise path), writing
// the output image directly.
constexpr int kFinalRows = 8;
constexpr int kFinalSpan = kTileM - 2;

struct FinalConvParams {
  const __half* w;         // folded B operand: [kb][2][3 x 16][8], row 16 (2 - ky) + 4 kx + co
                           // (tf32: floats, [kb][hi, lo][2][3 x 16][4] over 8-channel blocks)
  const float* bias;       // [16]: b0, b1, b2, zeros
  float4* net;             // [H][W] network output (lane 3 zero), or null
  int* status;
  int W, H;                // conv extent
  int tiles_x, tiles_y;    // tiles of kFinalRows rows x kFinalSpan pixels
  int S;                   // stages (one per K block)
  uint32_t stage_tx, stage_bytes;
  int xs;                  // log2 pixels per x unit of the input map
  // output pass (when fused): the tile's output rectangle, as UnpackParams
  const float4* color;
  size_t color_stride;
  float4* out;
  size_t out_stride;
  int in_x, in_y, ox, oy, ow, oh;
  int hdr;
  float scale;
  const float4* exp2_tab;  // HDR: kExp2TabSize entries from fill_exp2_table
  int reverse;             // walk the tiles last to first
  int l2_first;            // activation loads evict-first in L2 (one-tile frames)
};

struct FinalConvLaunch {
  CUtensorMap map;         // input: boxes of kFinalRows + 2 rows x kHaloW pixels x 2 chunks
  FinalConvParams p;
  int outpass;             // epilogue also runs the output pass
  int tf32;                // fp32 storage: 3xTF32 products
  dim3 grid;
  size_t smem;
};

cudaError_t launch_conv_final(const FinalConvLaunch& L, cudaStream_t stream);
cudaError_t conv_final_set_smem_limit(size_t bytes);

// dec_conv1b (64 -> 32, ReLU, fp16) and dec_conv0 (32 -> 3, folded) in one
// kernel, fp16 storage: output tiles of kTailOut rows x kFinalSpan pixels,
// conv 1 over the kTailMid rows x 128 pixels around each, its output kept in
// tensor memory as conv 2's A operand; CTAs take groups of `run` row tiles
// of one column strip round robin, carrying two conv-1 rows from tile to
// tile of a group; optionally the output pass in the epilogue (as
// FinalConvParams).
constexpr int kTailOut = 6;
constexpr int kTailMid = kTailOut + 2;

struct TailConvParams {
  const __half* w1;        // conv-1 B operand, [kb][kx][2][3 x 32][8] (the plain packing)
  const __half* w2;        // conv-2 B operand, kx folded: [kb][2][3 x 16][8]
  const float* bias1;      // [32]
  const float* bias2;      // [16]: b0, b1, b2, zeros
  float4* net;             // [H][W] network output (lane 3 zero), or null
  int* status;
  int W, H;                // conv extent
  int KB1;                 // 16-channel K blocks of conv 1's input
  int tiles_x, tiles_y;    // tiles of kTailOut rows x kFinalSpan pixels
  int S;                   // input stages (one K block's halo box each)
  uint32_t stage_tx, stage_bytes;  // bytes of a kTailMid + 2 row box; stage size
  uint32_t stage_tx8;      // bytes of a kTailMid row box (six new conv-1 rows)
  int xs;                  // log2 pixels per x unit of the input maps
  int run, groups;         // row tiles per group; groups (ceil(tiles_y / run) x tiles_x)
  // output pass (when fused): as FinalConvParams
  const float4* color;
  size_t color_stride;
  float4* out;
  size_t out_stride;
  int in_x, in_y, ox, oy, ow, oh;
  int hdr;
  float scale;
  const float4* exp2_tab;
  int l2_first;            // activation loads evict-first in L2 (one-tile frames)
};

struct TailConvLaunch {
  CUtensorMap map10;       // conv-1 input: boxes of kTailMid + 2 rows x kHaloW pixels x 2 chunks
  CUtensorMap map8;        // the same with boxes of kTailMid rows
  TailConvParams p;
  int outpass;
  dim3 grid;
  size_t smem;
};

cudaError_t launch_conv_tail(const TailConvLaunch& L, cudaStream_t stream);
cudaError_t conv_tail_set_smem_limit(size_t bytes);

// The input pass and enc_conv0 (16 input lanes -> 32, bias + ReLU) in one
// kernel, fp16 storage: conv tiles of kHeadRows rows x 128 pixels whose
// packed input halo is computed in shared memory from TMA-staged boxes of
// the source images.  Writes enc_conv0's output and the packed input's
// column-parity copy (not the plain packed input).
constexpr int kHeadRows = 8;

struct HeadParams {
  // input pass (as PackParams)
  int sources;             // 1..3
  int width, height;       // image extent
  int tx, ty, tw, th;      // tile input rect (= enc_conv0's extent)
  int hdr;
  float scale;
  // outputs
  void* split;             // packed input, column-parity copy [th][2][2][split_pitch/2][8]
  int split_pitch;
  __half* out;             // enc_conv0 output [th][4][pitch][8]; columns [tw, pitch) zero
  int pitch;
  // enc_conv0
  const __half* weights;   // B operand, one K block: [kx][2][3 x 32][8]
  const float* bias;       // [32]
  int* status;
  int tiles_x, tiles_y;    // tiles of kHeadRows rows x 128 pixels
  int SI, SA;              // image stages, packed-input stages
  uint32_t img_stage, a_stage;  // their bytes
};

struct HeadLaunch {
  CUtensorMap map[3];      // colour, albedo, normal: float4 pixels, boxes of kHeadRows + 2 rows x 130
  HeadParams p;
  dim3 grid;
  size_t smem;
};

cudaError_t launch_conv_head(const HeadLaunch& L, cudaStream_t stream);
cudaError_t conv_head_set_smem_limit(size_t bytes);

struct TcConvLaunch {
  CUtensorMap map0;        // source 0 (full-res halo box, or low-res box)
  CUtensorMap map1;        // source 1 (full-res halo box, or stride-2 box); unused if KB1 == 0
  TcConvParams p;
  int kind;                // TcKind
  int any_shape;           // 1: the run-time issue form even for a compile-time shape
  dim3 grid;
  size_t smem;
};

// Launch with programmatic stream serialization, so that the kernel's
// prologue overlaps the previous kernel in the stream (each kernel calls
// griddepcontrol.wait before touching data the previous one produced).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

cudaError_t launch_conv_tc(const TcConvLaunch& L, cudaStream_t stream);
// The compile-time shape the launch runs (0: the run-time issue form).
int conv_tc_shape(const TcConvLaunch& L);
cudaError_t conv_tc_set_smem_limit(size_t bytes);
cudaError_t conv_tc_occupancy(size_t smem, int* blocks_per_sm);


// Input pass of one tile.
struct PackParams {
  const float4* img[3];    // colour, albedo, normal (device)
  size_t stride[3];        // row stride in float4 elements
  int sources;             // 1..3
  int width, height;       // image extent
  int tx, ty, tw, th;      // tile input rect
  int hdr;
  float scale;             // effective inputScale (HDR)
  int fp16;                // storage precision
  void* out;               // [th][chunks][pitch][lanes]; columns >= tw are zeros
  int pitch;               // row pitch in pixels (fp16: tw rounded up to 8; fp32: tw)
  int chunks;              // 16-byte chunks per pixel
  void* out_split;         // optional parity-split copy [th][chunks][2][split_pitch/2][lanes]
  int split_pitch;         // its pitch (a multiple of 16), columns >= tw zero
  const float4* log2_tab;  // fp32 HDR: kLog2TabSize entries from fill_log2_table
  int gap_rows;            // stacked tiles: rows th .. th + gap_rows - 1 of out and
                           // out_split are written as zeros
  int reverse;             // row blocks in reverse order
};
cudaError_t launch_pack(const PackParams& p, cudaStream_t stream);

// Reduction table of the fp32 log transfer: entry j covers mantissas
// m in [1 + j/512, 1 + (j+1)/512) and holds {r_j, -log2(r_j) as a float
// pair (hi, lo), 0}; r_j (a multiple of 2^-10, r_0 = 1) is close enough to
// 1/m that m * r_j - 1 is exact in float.
constexpr int kLog2TabSize = 512;
void fill_log2_table(float (*tab)[4]);

// Table of the output pass's inverse transfer: entry j holds 2^(j/32) and
// 2^(j/32) - 1, each as a float pair (hi, lo): {Th, Tl, Dh, Dl}.
constexpr int kExp2TabSize = 32;
void fill_exp2_table(float (*tab)[4]);

// Output pass of one tile.
struct UnpackParams {
  const float4* net;       // [th][tw] network output of the tile
  int tw;                  // tile input width (row stride of net)
  int in_x, in_y;          // output rect offset inside the tile
  const float4* color;     // input colour image
  size_t color_stride;     // in float4
  float4* out;             // output image
  size_t out_stride;       // in float4
  int ox, oy, ow, oh;      // output rect in the image
  int hdr;
  float scale;
  const float4* exp2_tab;  // HDR: kExp2TabSize entries from fill_exp2_table
};
cudaError_t launch_unpack(const UnpackParams& p, cudaStream_t stream);

// Failure-detection probe: a wait that nothing completes, bounded by limit_ns.
cudaError_t launch_wait_probe(int* status, unsigned long long limit_ns, cudaStream_t stream);

// Column-parity split copy of an fp16 activation: [h][chunks][src_pitch][8]
// -> [h][chunks][2][dst_pitch/2][8] (dst_pitch even); columns >= w are zeros.
cudaError_t launch_split_copy(const void* src, int src_pitch, void* dst, int dst_pitch, int w,
                              int h, int chunks, cudaStream_t stream);

// Re-pitch an activation: rows of w 16-byte elements at src_pitch into rows
// at dst_pitch >= w, columns [w, dst_pitch) written as zeros.
cudaError_t launch_pitch_copy(const void* src, int src_pitch, void* dst, int dst_pitch, int w,
                              int rows, cudaStream_t stream);

}  // namespace oidnx

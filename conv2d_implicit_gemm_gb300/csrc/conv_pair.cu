// Two consecutive same-padded 3x3 convs of the U-Net fused into one kernel,
// so that the 32-channel map between them never reaches global memory:
//  * dec_conv1b (64 -> 32, ReLU) + dec_conv0 (32 -> 3, final fp32 output),
//  * enc_conv0 (input -> 32, ReLU) + enc_conv1 (32 -> 32, ReLU, 2x2 max-pool).
// What each conv computes is the layer of "oidn-web 0.4.0 -> 0.5.0,
// package/src/nativeUNet.ts" (createTiledConvShader, createFusedConvPoolShader
// for the pooled variant), with conv 1's output rounded to fp16 storage as
// the unfused network stores it.
//
// GB300 design (not the pages'):
//  * A CTA owns segments of a column strip (at most 126 output pixels) and
//    streams its rows top to bottom.  Conv 1 runs on 128 pixels starting one
//    left of the strip, which is the whole neighbourhood conv 2 needs.
//  * One input row (all channels, kHaloW pixels) per pipeline stage, by one
//    TMA box.  Input row r feeds conv-1 output rows r+1, r, r-1 through
//    ky = 0, 1, 2 stacked along N, into a ring of eight TMEM row
//    accumulators (an MMA is split in two where its rows wrap the ring).
//  * A conv-1 row is complete once the input row below it is in: four
//    epilogue warps read it, add ReLU, round to fp16 and write it into a
//    ring of four shared-memory rows laid out as the next MMA's A operand.
//  * Conv 2 streams over those rows the same way into a second TMEM ring.
//    For the final 32 -> 3 conv the three kx taps are folded into N as well
//    (N = 3 ky x 16, of which 3 kx x 3 channels used): one MMA per K block
//    instead of three, and its epilogue sums the kx partial results of
//    pixels m, m+1, m+2 (exchanged through shared memory).
//  * Warp 0 issues TMA, warp 1 allocates TMEM and issues every MMA, warps
//    2-5 run conv 1's epilogue and warps 6-9 conv 2's.  Every wait is
//    bounded as in the single-conv kernel.
#include "internal.h"
#include "ptx.cuh"

namespace oidnx {

namespace {

constexpr int kPairThreads = 320;
constexpr int kMidC = 32;                  // conv-1 output channels
constexpr uint32_t kRing2 = 256;           // TMEM column of conv 2's ring

template <int MODE> __host__ __device__ constexpr int pair_c2() { return MODE == kPairFinal ? 16 : 32; }
// pixels per shared-memory row of conv-1 output: the folded final conv reads
// pixels 0..127 only; the pooled conv reads A shifted by kx (up to 129)
template <int MODE> __host__ __device__ constexpr int pair_mid_px() { return MODE == kPairFinal ? kTileM : kTileM + 8; }
template <int MODE> __host__ __device__ constexpr uint32_t pair_mid_bytes() {
  return static_cast<uint32_t>(4 * pair_mid_px<MODE>() * kChunkBytes);
}

// The CTA's work: row units [k, kend) in strip-major order, walked as
// segments that stay within one strip.
struct Seg {
  int strip, ya, yb;
};

__device__ __forceinline__ void cta_units(const PairConvParams& p, int* k, int* kend) {
  *k = static_cast<int>((static_cast<long long>(blockIdx.x) * p.units) / gridDim.x);
  *kend = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * p.units) / gridDim.x);
}

__device__ __forceinline__ Seg next_seg(const PairConvParams& p, int* k, int kend) {
  const int hu = (p.H + p.row_unit - 1) / p.row_unit;
  const int strip = *k / hu;
  const int r0 = *k - strip * hu;
  const int r1 = min(hu, r0 + (kend - *k));
  *k += r1 - r0;
  Seg s;
  s.strip = strip;
  s.ya = r0 * p.row_unit;
  s.yb = min(p.H, r1 * p.row_unit);
  return s;
}

__device__ __forceinline__ void advance(uint32_t& s, uint32_t& ph, uint32_t S) {
  if (++s == S) {
    s = 0;
    ph ^= 1u;
  }
}

// Rows of batch j of a segment with nO output rows (nI = nO + 2 conv-1
// rows, nO + 4 input rows): conv 1 takes input rows [t0, t1); that completes
// conv-1 rows [r0, r1); conv 2 takes the rows completed two batches earlier,
// [c0, c1), which completes output rows [v0, v1).  Empty ranges are [0, 0).
struct Batch {
  int t0, t1, r0, r1, c0, c1, v0, v1;
};

__host__ __device__ __forceinline__ int pair_batches(int nO) {
  return (nO + 4 + kPairBatch - 1) / kPairBatch + 2;
}

__device__ __forceinline__ void batch_rows(int k, int nO, int* a, int* b) {
  const int J = (nO + 4 + kPairBatch - 1) / kPairBatch;
  if (k < 0 || k >= J) {
    *a = *b = 0;
    return;
  }
  *a = max(0, kPairBatch * k - 2);
  *b = min(nO + 2, kPairBatch * k + kPairBatch - 2);
}

__device__ __forceinline__ Batch batch_of(int j, int nO) {
  Batch q;
  const int n_in = nO + 4;
  q.t0 = min(kPairBatch * j, n_in);
  q.t1 = min(kPairBatch * j + kPairBatch, n_in);
  batch_rows(j, nO, &q.r0, &q.r1);
  batch_rows(j - 2, nO, &q.c0, &q.c1);
  q.v0 = 0;
  q.v1 = 0;
  if (q.c0 < q.c1) {
    q.v0 = max(0, q.c0 - 2);
    q.v1 = max(q.v0, min(nO, q.c1 - 2));
  }
  return q;
}

// MMAs of one source row t into target rows lo..hi of a ring of eight row
// accumulators of `cols` columns (target u in slot (g + u) & 7).  B holds
// the three ky blocks stacked (stack position u - t + 2 for target u), each
// `nb` rows of 16 bytes.  At most two MMAs: the run is split where it wraps.
__device__ __forceinline__ void issue_rows(uint32_t ring, uint32_t cols, uint32_t g, int t, int lo,
                                           int hi, uint64_t a, uint64_t b, uint32_t nb,
                                           uint32_t id1, uint32_t id2, uint32_t id3) {
  int u = lo;
  while (u <= hi) {
    const uint32_t slot = (g + static_cast<uint32_t>(u)) & 7u;
    const int e = min(hi, u + static_cast<int>(7u - slot));
    const int n = e - u + 1;
    const uint32_t id = n == 1 ? id1 : (n == 2 ? id2 : id3);
    if (elect_one())
      mma_f16_ss(ring + slot * cols, a, b + static_cast<uint32_t>(u - t + 2) * nb, id, 1u);
    u = e + 1;
  }
}

// The same for a batch of three source rows t0 + j (A descriptors a0, a1,
// a2) whose three targets t-2 .. t all exist, the ring slot of target
// t0 - 2 being P: every slot and split is a compile-time constant, so the
// issuing warp spends a few instructions per MMA.  b: B at stack position 0.
template <int P>
__device__ __forceinline__ void issue_batch(uint32_t ring, uint32_t cols, uint64_t a0, uint64_t a1,
                                            uint64_t a2, uint64_t b, uint32_t nb, uint32_t id1,
                                            uint32_t id2, uint32_t id3, bool leader) {
  static_assert(kPairBatch == 3, "three source rows per batch");
  if (!leader) return;
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const uint64_t a = j == 0 ? a0 : (j == 1 ? a1 : a2);
    const int s0 = (P + j) & 7;  // slot of target t0 + j - 2 (stack position 0)
    if (s0 <= 5) {
      mma_f16_ss(ring + s0 * cols, a, b, id3, 1u);
    } else if (s0 == 6) {
      mma_f16_ss(ring + 6 * cols, a, b, id2, 1u);
      mma_f16_ss(ring, a, b + 2 * nb, id1, 1u);
    } else {
      mma_f16_ss(ring + 7 * cols, a, b, id1, 1u);
      mma_f16_ss(ring, a, b + nb, id2, 1u);
    }
  }
}

// Dispatch on the ring position of the batch.
__device__ __forceinline__ void issue_batch_at(uint32_t P, uint32_t ring, uint32_t cols,
                                               uint64_t a0, uint64_t a1, uint64_t a2, uint64_t b,
                                               uint32_t nb, uint32_t id1, uint32_t id2,
                                               uint32_t id3, bool leader) {
  switch (P & 7u) {
    case 0: issue_batch<0>(ring, cols, a0, a1, a2, b, nb, id1, id2, id3, leader); break;
    case 1: issue_batch<1>(ring, cols, a0, a1, a2, b, nb, id1, id2, id3, leader); break;
    case 2: issue_batch<2>(ring, cols, a0, a1, a2, b, nb, id1, id2, id3, leader); break;
    case 3: issue_batch<3>(ring, cols, a0, a1, a2, b, nb, id1, id2, id3, leader); break;
    case 4: issue_batch<4>(ring, cols, a0, a1, a2, b, nb, id1, id2, id3, leader); break;
    case 5: issue_batch<5>(ring, cols, a0, a1, a2, b, nb, id1, id2, id3, leader); break;
    case 6: issue_batch<6>(ring, cols, a0, a1, a2, b, nb, id1, id2, id3, leader); break;
    default: issue_batch<7>(ring, cols, a0, a1, a2, b, nb, id1, id2, id3, leader); break;
  }
}

}  // namespace

template <int MODE>
__global__ void __launch_bounds__(kPairThreads, 1)
    conv3x3_pair_kernel(const __grid_constant__ CUtensorMap map, const PairConvParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t pad = (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
  uint8_t* smem = smem_raw + pad;

  constexpr int C2 = pair_c2<MODE>();
  constexpr int MIDPX = pair_mid_px<MODE>();
  constexpr uint32_t MIDB = pair_mid_bytes<MODE>();
  const int S = p.S;
  // shared memory: [input stages][w1][w2][conv-1 rows][exchange][bias][barriers]
  uint8_t* IN = smem;
  uint8_t* W1 = IN + static_cast<size_t>(S) * p.stage_bytes;
  uint8_t* W2 = W1 + p.w1_bytes;
  uint8_t* MID = W2 + ((p.w2_bytes + 1023u) & ~1023u);
  float4* XB = reinterpret_cast<float4*>(MID + kPairMid * MIDB);  // [2][2][128] (final)
  float* b1s = reinterpret_cast<float*>(XB + (MODE == kPairFinal ? 4 * kTileM : 0));
  float* b2s = b1s + kMidC;
  uint64_t* full = reinterpret_cast<uint64_t*>(b2s + 32);
  uint64_t* empty = full + S;
  uint64_t* bdone = empty + S;   // [4] every MMA of batch b finished
  uint64_t* e1done = bdone + 4;  // [4] conv-1 rows completed by batch b drained
  uint64_t* e2done = e1done + 4; // [4] conv-2 rows completed by batch b drained
  uint64_t* xbar = e2done + 4;   // [2] final epilogue exchange
  uint64_t* filled = xbar + 2;   // accumulators hold the bias
  uint64_t* wbar = filled + 1;
  uint64_t* done = wbar + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int k = 0; k < 4; ++k) {
      mbar_init(&bdone[k], 1);
      mbar_init(&e1done[k], 128);
      mbar_init(&e2done[k], 128);
    }
    mbar_init(&xbar[0], 128);
    mbar_init(&xbar[1], 128);
    mbar_init(filled, 256);
    mbar_init(wbar, 1);
    mbar_init(done, 1);
    fence_mbarrier_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch_dependents();

  int k0, kend;
  cta_units(p, &k0, &kend);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // One stage per conv-1 batch: kPairBatch input rows by one TMA box.
    if (lane == 0) {
      prefetch_tmap(&map);
      mbar_arrive_expect_tx(wbar, p.w1_bytes + p.w2_bytes);
      bulk_load(W1, p.w1, p.w1_bytes, wbar);
      bulk_load(W2, p.w2, p.w2_bytes, wbar);
      griddep_wait();
      uint32_t it = 0, s = 0, ph = 0;
      bool ok = true;
      for (int k = k0; k < kend && ok;) {
        const Seg g = next_seg(p, &k, kend);
        const int x0 = g.strip * p.sw;
        // conv 1 reads input pixels x0 - 2 .. x0 + 127: the box starts at the
        // 8-pixel boundary at or left of x0 - 2
        const int bx = (x0 - 2) & ~(kGroupPx - 1);
        const int n_in = g.yb - g.ya + 4;
        for (int t0 = 0; t0 < n_in; t0 += kPairBatch, ++it, advance(s, ph, S)) {
          if (!mbar_wait_bounded(&empty[s], ph ^ 1u, p.status, kErrTimeoutProducer)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], p.stage_tx);
          tma_load_4d(IN + static_cast<size_t>(s) * p.stage_bytes, &map, &full[s], 0, bx >> p.xs, 0,
                      g.ya - 2 + t0, l2_evict_first());  // (fused pairs: one-tile frames)
        }
      }
      for (uint32_t j = it > static_cast<uint32_t>(S) ? it - S : 0u; j < it; ++j)
        mbar_wait_bounded(&full[j % S], (j / S) & 1u, p.status, kErrTimeoutDrain);
      mbar_wait_bounded(wbar, 0, p.status, kErrTimeoutDrain);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The MMAs of one source row all accumulate into the same TMEM columns;
    // an MMA into columns the previous one writes waits for it.  So source
    // rows are taken kPairBatch at a time (one pipeline stage), and within a
    // batch the MMAs of its rows, and those of conv 2 over the rows conv 1
    // completed two batches earlier, are interleaved.  Per batch the warp
    // takes three waits and makes one commit besides the stage release.
    const uint32_t ia1 = idesc_f16_f32(kTileM, kMidC), ia2 = idesc_f16_f32(kTileM, 2 * kMidC),
                   ia3 = idesc_f16_f32(kTileM, 3 * kMidC);
    const uint32_t ib1 = idesc_f16_f32(kTileM, C2), ib2 = idesc_f16_f32(kTileM, 2 * C2),
                   ib3 = idesc_f16_f32(kTileM, 3 * C2);
    const uint64_t a0 = smem_desc_noswizzle(smem_u32(IN), kHaloW * kChunkBytes, 128);
    const uint64_t w1d = smem_desc_noswizzle(smem_u32(W1), 3u * kMidC * kChunkBytes, 128);
    const uint64_t w2d = smem_desc_noswizzle(smem_u32(W2), 3u * C2 * kChunkBytes, 128);
    const uint64_t md = smem_desc_noswizzle(smem_u32(MID), MIDPX * kChunkBytes, 128);
    const uint32_t w1kb = (9u * 2u * kMidC * kChunkBytes) >> 4;  // one K block of w1, 16 B units
    const uint32_t w2kb = (MODE == kPairFinal ? 2u * 3u * C2 * kChunkBytes
                                              : 9u * 2u * C2 * kChunkBytes) >> 4;
    const uint32_t row16 = static_cast<uint32_t>(p.C8 * kHaloW);  // one staged row, 16 B units
    constexpr int KX2 = MODE == kPairFinal ? 1 : 3;               // conv-2 kx groups
    const uint32_t ring1 = tmem, ring2 = tmem + kRing2;
    bool ok = __all_sync(0xffffffffu, mbar_wait_bounded(wbar, 0, p.status, kErrTimeoutMma) &&
                                          mbar_wait_bounded(filled, 0, p.status, kErrTimeoutMma));
    const bool leader = elect_one();
    uint32_t s = 0, ph = 0, g1 = 0, g2 = 0, b = 0;
    for (int k = k0; k < kend && ok;) {
      const Seg g = next_seg(p, &k, kend);
      const int x0 = g.strip * p.sw;
      const uint32_t o = static_cast<uint32_t>((x0 - 2) - ((x0 - 2) & ~(kGroupPx - 1)));
      const int nO = g.yb - g.ya, nI = nO + 2;
      const int nb = pair_batches(nO);
      for (int j = 0; j < nb && ok; ++j, ++b) {
        const Batch q = batch_of(j, nO);
        const bool has1 = q.t0 < q.t1, has2 = q.c0 < q.c1;
        // the batch's new conv-1 rows reuse ring slots of rows drained with
        // batch b - 2, and its conv-2 rows were written to shared memory then
        bool w = true;
        if (has1) w = mbar_wait_bounded(&full[s], ph, p.status, kErrTimeoutMma);
        if (w && b >= 2) {
          w = mbar_wait_bounded(&e1done[(b - 2) & 3u], ((b - 2) >> 2) & 1u, p.status, kErrTimeoutMma);
          if (w && has2)
            w = mbar_wait_bounded(&e2done[(b - 2) & 3u], ((b - 2) >> 2) & 1u, p.status, kErrTimeoutMma);
        }
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        tc_fence_after();
        const uint64_t as = a0 + ((s * p.stage_bytes) >> 4) + o;
        const bool fast1 = has1 && q.t1 - q.t0 == kPairBatch && q.t0 >= 2 && q.t1 <= nI;
        const bool fast2 = has2 && q.c1 - q.c0 == kPairBatch && q.c0 >= 2 && q.c1 <= nO;
        // conv-1 rows c0 .. c0 + 2 in shared memory (slots G % kPairMid)
        auto mid_desc = [&](int u) -> uint64_t {
          return md + ((((g1 + static_cast<uint32_t>(u)) % kPairMid) * MIDB) >> 4);
        };
        const uint64_t m0 = mid_desc(q.c0), m1 = mid_desc(q.c0 + 1), m2 = mid_desc(q.c0 + 2);
        const uint32_t P1 = g1 + static_cast<uint32_t>(q.t0 - 2);
        const uint32_t P2 = g2 + static_cast<uint32_t>(q.c0 - 2);
        // conv-1 groups (kb, kx) and conv-2 groups (kb, kx) merged in
        // proportion, so that the two rings alternate
        const int n1 = fast1 ? p.KB1 * 3 : 0, n2 = fast2 ? 2 * KX2 : 0;
        int i1 = 0, i2 = 0;
        while (i1 < n1 || i2 < n2) {
          if (i2 >= n2 || (i1 < n1 && i1 * n2 <= i2 * n1)) {
            const int kb = i1 / 3, kx = i1 - 3 * kb;
            const uint64_t a = as + static_cast<uint32_t>(kb * 2 * kHaloW + kx);
            issue_batch_at(P1, ring1, kMidC, a, a + row16, a + 2 * row16,
                           w1d + static_cast<uint32_t>(kb) * w1kb + static_cast<uint32_t>(kx * 6 * kMidC),
                           kMidC, ia1, ia2, ia3, leader);
            ++i1;
          } else {
            const int kb = i2 / KX2, kx = i2 - KX2 * kb;
            const uint32_t off = static_cast<uint32_t>(kb * 2 * MIDPX + kx);
            issue_batch_at(P2, ring2, C2, m0 + off, m1 + off, m2 + off,
                           w2d + static_cast<uint32_t>(kb) * w2kb + static_cast<uint32_t>(kx * 6 * C2), C2,
                           ib1, ib2, ib3, leader);
            ++i2;
          }
        }
        // batches at the segment's edges (targets missing): one row at a time
        if (has1 && !fast1) {
          for (int kb = 0; kb < p.KB1; ++kb)
            for (int kx = 0; kx < 3; ++kx)
              for (int t = q.t0; t < q.t1; ++t)
                issue_rows(ring1, kMidC, g1, t, max(0, t - 2), min(nI - 1, t),
                           as + static_cast<uint32_t>(t - q.t0) * row16 +
                               static_cast<uint32_t>(kb * 2 * kHaloW + kx),
                           w1d + static_cast<uint32_t>(kb) * w1kb + static_cast<uint32_t>(kx * 6 * kMidC),
                           kMidC, ia1, ia2, ia3);
        }
        if (has2 && !fast2) {
          for (int kb = 0; kb < 2; ++kb)
            for (int kx = 0; kx < KX2; ++kx)
              for (int u = q.c0; u < q.c1; ++u) {
                const int lo = max(0, u - 2), hi = min(nO - 1, u);
                if (lo > hi) continue;
                issue_rows(ring2, C2, g2, u, lo, hi,
                           mid_desc(u) + static_cast<uint32_t>(kb * 2 * MIDPX + kx),
                           w2d + static_cast<uint32_t>(kb) * w2kb + static_cast<uint32_t>(kx * 6 * C2), C2,
                           ib1, ib2, ib3);
              }
        }
        if (leader) {
          if (has1) mma_commit(&empty[s]);
          mma_commit(&bdone[b & 3u]);
        }
        __syncwarp();
        if (has1) advance(s, ph, S);
      }
      g1 += static_cast<uint32_t>(nI);
      g2 += static_cast<uint32_t>(nO);
    }
    if (leader) mma_commit(done);
    __syncwarp();
    mbar_wait_bounded(done, 0, p.status, kErrTimeoutMma);
    __syncwarp();
  } else if (warp < 6) {
    // ------------------------------------------------------------ conv-1 epilogue
    // Warp w reads TMEM lane quarter w % 4: pixel i of the 128-pixel conv-1
    // row (image column x0 - 1 + i).
    const int q4 = warp & 3;
    const int i = q4 * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const int et = threadIdx.x - 64;  // 0..127
    if (et < kMidC) b1s[et] = p.bias1[et];
    named_barrier_sync(1, 128);
    for (int sl = 0; sl < 8; ++sl)
      for (int c = 0; c < kMidC / 16; ++c)
        tmem_fill_bias(tmem + lane_off + static_cast<uint32_t>(sl * kMidC + c * 16), b1s + c * 16);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(filled);
    uint32_t g1 = 0, b = 0;
    bool ok = true;
    for (int k = k0; k < kend && ok;) {
      const Seg g = next_seg(p, &k, kend);
      const int x = g.strip * p.sw - 1 + i;
      const int nO = g.yb - g.ya;
      const int nb = pair_batches(nO);
      for (int j = 0; j < nb; ++j, ++b) {
        const Batch q = batch_of(j, nO);
        if (q.r0 < q.r1) {
          if (!mbar_wait_bounded(&bdone[b & 3u], (b >> 2) & 1u, p.status, kErrTimeoutEpilogue)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int u = q.r0; u < q.r1; ++u) {
            const uint32_t G = g1 + static_cast<uint32_t>(u);
            uint32_t v[2][16];
            const uint32_t t0 = tmem + lane_off + (G & 7u) * kMidC;
            tmem_ld16_nowait(t0, v[0]);
            tmem_ld16_nowait(t0 + 16, v[1]);
            tmem_wait_ld();
            tmem_fill_bias(t0, b1s);
            tmem_fill_bias(t0 + 16, b1s + 16);
            // conv 2 pads its input with zeros: rows and columns outside the
            // image; the shared-memory row's previous contents were read by
            // conv 2 in this batch or earlier
            const int y = g.ya - 1 + u;
            const bool valid = y >= 0 && y < p.H && x >= 0 && x < p.W;
            uint4* row = reinterpret_cast<uint4*>(MID + (G % kPairMid) * MIDB);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t h[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int ch = 8 * c + 2 * e;
                h[e] = valid ? pack_half2(fmaxf(__uint_as_float(v[ch >> 4][ch & 15]), 0.0f),
                                          fmaxf(__uint_as_float(v[ch >> 4][(ch & 15) + 1]), 0.0f))
                             : 0u;
              }
              row[c * MIDPX + i] = make_uint4(h[0], h[1], h[2], h[3]);
            }
          }
          fence_proxy_async_smem();
          tmem_wait_st();
          tc_fence_before();
        }
        mbar_arrive(&e1done[b & 3u]);
      }
      g1 += static_cast<uint32_t>(nO + 2);
    }
  } else {
    // ------------------------------------------------------------ conv-2 epilogue
    const int q4 = warp & 3;
    const int m = q4 * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q4 * 32) << 16;
    const int et = threadIdx.x - 192;  // 0..127
    if (et < 32) b2s[et] = et < C2 ? p.bias2[et] : 0.0f;
    named_barrier_sync(2, 128);
    for (int sl = 0; sl < 8; ++sl)
      for (int c = 0; c < C2 / 16; ++c)
        tmem_fill_bias(tmem + kRing2 + lane_off + static_cast<uint32_t>(sl * C2 + c * 16), b2s + c * 16);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(filled);
    uint32_t g2 = 0, b = 0, xr = 0;
    bool ok = true;
    float pend[32];  // pool: the first row of a pair whose second row is not complete yet
    for (int k = k0; k < kend && ok;) {
      const Seg g = next_seg(p, &k, kend);
      const int x0 = g.strip * p.sw;
      const int x = x0 + m;
      // the last strip also writes the padding columns of a pitched output
      const int span = g.strip == p.strips - 1 ? kPairSpan : p.sw;
      const int nO = g.yb - g.ya;
      const int nb = pair_batches(nO);
      for (int j = 0; j < nb && ok; ++j, ++b) {
        const Batch q = batch_of(j, nO);
        if (q.v0 < q.v1) {
          if (!mbar_wait_bounded(&bdone[b & 3u], (b >> 2) & 1u, p.status, kErrTimeoutEpilogue)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int v = q.v0; v < q.v1 && ok; ++v) {
            const uint32_t t0 = tmem + kRing2 + lane_off + ((g2 + static_cast<uint32_t>(v)) & 7u) * C2;
            if (MODE == kPairFinal) {
              uint32_t d[16];
              tmem_ld16_nowait(t0, d);
              tmem_wait_ld();
              tmem_fill_bias(t0, b2s);
              // columns 4 kx + c hold the kx partial sums of this pixel; the
              // output at pixel m takes kx from pixel m + kx (bias in kx = 0)
              const uint32_t xb_i = xr & 1u;
              float4* xb = XB + xb_i * 2 * kTileM;
              xb[m] = make_float4(__uint_as_float(d[4]), __uint_as_float(d[5]), __uint_as_float(d[6]),
                                  __uint_as_float(d[7]));
              xb[kTileM + m] = make_float4(__uint_as_float(d[8]), __uint_as_float(d[9]),
                                           __uint_as_float(d[10]), __uint_as_float(d[11]));
              mbar_arrive(&xbar[xb_i]);
              if (!mbar_wait_bounded(&xbar[xb_i], (xr >> 1) & 1u, p.status, kErrTimeoutEpilogue)) {
                ok = false;
                break;
              }
              ++xr;
              const int y = g.ya + v;
              if (m < span && x < p.W) {
                const float4 f1 = xb[m + 1];
                const float4 f2 = xb[kTileM + m + 2];
                static_cast<float4*>(p.out)[static_cast<size_t>(y) * p.W + x] =
                    make_float4(__uint_as_float(d[0]) + f1.x + f2.x, __uint_as_float(d[1]) + f1.y + f2.y,
                                __uint_as_float(d[2]) + f1.z + f2.z, 0.0f);
              }
            } else {
              // ReLU, then the 2x2 max: rows v (even) and v + 1 of the segment
              // (g.ya is even), pixels m and m ^ 1 (x0 is even)
              uint32_t r[2][16];
              tmem_ld16_nowait(t0, r[0]);
              tmem_ld16_nowait(t0 + 16, r[1]);
              tmem_wait_ld();
              tmem_fill_bias(t0, b2s);
              tmem_fill_bias(t0 + 16, b2s + 16);
              float cur[32];
#pragma unroll
              for (int e = 0; e < 32; ++e)
                cur[e] = x < p.W ? fmaxf(__uint_as_float(r[e >> 4][e & 15]), 0.0f) : -INFINITY;
              const bool second = (v & 1) != 0;
              if (!second && v + 1 < nO) {
#pragma unroll
                for (int e = 0; e < 32; ++e) pend[e] = cur[e];
                continue;
              }
              if (second) {
#pragma unroll
                for (int e = 0; e < 32; ++e) cur[e] = fmaxf(cur[e], pend[e]);
              }
#pragma unroll
              for (int e = 0; e < 32; ++e) cur[e] = fmaxf(cur[e], __shfl_xor_sync(0xffffffffu, cur[e], 1));
              const int Wp = (p.W + 1) >> 1, Hp = (p.H + 1) >> 1;
              const int xp = x >> 1, yp = (g.ya + v) >> 1;
              // even pixels store the pooled value; pooled columns [Wp, pitch)
              // are row padding, stored as zeros
              if ((m & 1) == 0 && m < span && yp < Hp) {
                const bool padc = xp >= Wp;
                __half* out = static_cast<__half*>(p.out);
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                  uint32_t h[8];
#pragma unroll
                  for (int e = 0; e < 8; ++e)
                    h[e] = padc ? 0u : pack_half2(cur[16 * c + 2 * e], cur[16 * c + 2 * e + 1]);
                  if (xp < p.pitch) {
                    const size_t b0 = ((static_cast<size_t>(yp) * 4 + 2 * c) * p.pitch + xp) * 8;
                    const size_t b1 = b0 + static_cast<size_t>(p.pitch) * 8;
                    *reinterpret_cast<uint4*>(out + b0) = make_uint4(h[0], h[1], h[2], h[3]);
                    *reinterpret_cast<uint4*>(out + b1) = make_uint4(h[4], h[5], h[6], h[7]);
                  }
                  if (p.out_split && xp < p.split_pitch) {
                    __half* o2 = static_cast<__half*>(p.out_split);
                    const size_t s0 =
                        ((((static_cast<size_t>(yp) * 4 + 2 * c) * 2 + (xp & 1)) * (p.split_pitch >> 1)) + (xp >> 1)) * 8;
                    const size_t s1 = s0 + static_cast<size_t>(p.split_pitch) * 8;
                    *reinterpret_cast<uint4*>(o2 + s0) = make_uint4(h[0], h[1], h[2], h[3]);
                    *reinterpret_cast<uint4*>(o2 + s1) = make_uint4(h[4], h[5], h[6], h[7]);
                  }
                }
              }
            }
          }
          tmem_wait_st();
          tc_fence_before();
        }
        mbar_arrive(&e2done[b & 3u]);
      }
      g2 += static_cast<uint32_t>(nO);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

cudaError_t launch_conv_pair(const PairConvLaunch& L, cudaStream_t stream) {
  if (L.mode == kPairFinal)
    return launch_pdl(conv3x3_pair_kernel<kPairFinal>, L.grid, dim3(kPairThreads), L.smem, stream,
                      L.map, L.p);
  return launch_pdl(conv3x3_pair_kernel<kPairPool>, L.grid, dim3(kPairThreads), L.smem, stream,
                    L.map, L.p);
}

cudaError_t conv_pair_set_smem_limit(size_t bytes) {
  cudaError_t e = cudaFuncSetAttribute(conv3x3_pair_kernel<kPairFinal>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(bytes));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(conv3x3_pair_kernel<kPairPool>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

cudaError_t conv_pair_occupancy(int mode, size_t smem, int* blocks_per_sm) {
  if (mode == kPairFinal)
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, conv3x3_pair_kernel<kPairFinal>,
                                                         kPairThreads, smem);
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, conv3x3_pair_kernel<kPairPool>,
                                                       kPairThreads, smem);
}

}  // namespace oidnx

// Host runtime of the oidnx C ABI: weight blob parsing and packing, the tile
// planner, per-tile-shape network plans (activation arena from value
// liveness, tensor maps, launch parameters), CUDA-graph replay, profiling and
// the extern "C" entry points declared in include/oidnx.h.
//
// Structure follows "oidn-web 0.3.4 -> 0.4.0, package/src/nativeUNet.ts"
// (NativeUNetExecutor: constructor validation and weight packing,
// _createExecution liveness + best-fit slot reuse, _execution LRU shape cache
// with deferred destruction of evicted plans, profileNextExecution) and
// "oidn-webgpu 0.0.0-stage -> 0.6.0, src/native/denoise.ts"
// (recordDenoiseExecution: overlap, tile grid, per-tile input pass ->
// network -> output pass in order on one queue).
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <list>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/oidnx.h"
#include "internal.h"

using namespace oidnx;

// ======================================================================
// errors
// ======================================================================
namespace {

thread_local std::string g_last_error;

oidnx_status fail(oidnx_status s, const char* fmt, ...) {
  char buf[1024];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

oidnx_status ok() {
  g_last_error.clear();
  return OIDNX_OK;
}

#define OIDNX_CUDA(call)                                                               \
  do {                                                                                 \
    cudaError_t e_ = (call);                                                           \
    if (e_ != cudaSuccess) {                                                           \
      if (e_ == cudaErrorMemoryAllocation)                                             \
        return fail(OIDNX_ERR_OUT_OF_MEMORY, "%s: %s", #call, cudaGetErrorString(e_)); \
      return fail(OIDNX_ERR_CUDA, "%s: %s", #call, cudaGetErrorString(e_));            \
    }                                                                                  \
  } while (0)

#define OIDNX_TRY(expr)               \
  do {                                \
    oidnx_status s_ = (expr);         \
    if (s_ != OIDNX_OK) return s_;    \
  } while (0)

// ======================================================================
// model
// ======================================================================
constexpr int kLayers = 16;
const char* const kLayerNames[kLayers] = {
    "enc_conv0",  "enc_conv1",  "enc_conv2",  "enc_conv3",  "enc_conv4",  "enc_conv5a",
    "enc_conv5b", "dec_conv4a", "dec_conv4b", "dec_conv3a", "dec_conv3b", "dec_conv2a",
    "dec_conv2b", "dec_conv1a", "dec_conv1b", "dec_conv0"};

struct ConvTensors {
  int cout = 0, cin = 0;
  std::vector<float> w;  // OIHW
  std::vector<float> b;  // [cout]
};

enum Kind { kPlain, kPool, kDecoder, kFinal };

// Values of the network dataflow.
enum Val {
  V_IN, V_E0, V_P1, V_P2, V_P3, V_P4, V_E5A, V_E5B, V_D4A, V_D4B,
  V_D3A, V_D3B, V_D2A, V_D2B, V_D1A, V_D1B, V_OUT,
  // column-parity split copies of the decoders' skip sources
  V_INS, V_P1S, V_P2S, V_P3S, V_COUNT
};

// A split copy is written by the producer of `base` (layer index, -1 for the
// input pass) next to the normal copy and read by decoder `consumer` when
// that decoder runs in sub-pixel mode.
struct SplitCopy {
  int split, base, producer, consumer;
};
const SplitCopy kSplits[4] = {
    {V_INS, V_IN, -1, 13}, {V_P1S, V_P1, 1, 11}, {V_P2S, V_P2, 2, 9}, {V_P3S, V_P3, 3, 7}};

struct LayerDef {
  int src0, src1, dst, kind, level;  // level of the conv (full-resolution) extent
};

// enc_conv0 -> enc_conv1+pool -> (enc_convK+pool)x3 -> enc_conv5a/5b ->
// per decoder level up+concat(skip) conv, conv -> dec_conv0 (no ReLU, fp32).
const LayerDef kDefs[kLayers] = {
    {V_IN, -1, V_E0, kPlain, 0},     {V_E0, -1, V_P1, kPool, 0},
    {V_P1, -1, V_P2, kPool, 1},      {V_P2, -1, V_P3, kPool, 2},
    {V_P3, -1, V_P4, kPool, 3},      {V_P4, -1, V_E5A, kPlain, 4},
    {V_E5A, -1, V_E5B, kPlain, 4},   {V_E5B, V_P3, V_D4A, kDecoder, 3},
    {V_D4A, -1, V_D4B, kPlain, 3},   {V_D4B, V_P2, V_D3A, kDecoder, 2},
    {V_D3A, -1, V_D3B, kPlain, 2},   {V_D3B, V_P1, V_D2A, kDecoder, 1},
    {V_D2A, -1, V_D2B, kPlain, 1},   {V_D2B, V_IN, V_D1A, kDecoder, 0},
    {V_D1A, -1, V_D1B, kPlain, 0},   {V_D1B, -1, V_OUT, kFinal, 0},
};

int round_up(int v, int a) { return (v + a - 1) / a * a; }
size_t round_up_sz(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Half-precision bits of a float, round to nearest even (host side).
uint16_t to_half_bits(float f) {
  __half h = __float2half_rn(f);
  uint16_t b;
  std::memcpy(&b, &h, 2);
  return b;
}

float half_bits_to_float(uint16_t bits) {
  __half h;
  std::memcpy(&h, &bits, 2);
  return __half2float(h);
}

// ---------------------------------------------------------------- blob
struct BlobReader {
  const uint8_t* p;
  size_t n, off = 0;
  bool u32(uint32_t* v) {
    if (off + 4 > n) return false;
    std::memcpy(v, p + off, 4);
    off += 4;
    return true;
  }
  bool bytes(const uint8_t** v, size_t len) {
    if (len > n || off + len > n) return false;
    *v = p + off;
    off += len;
    return true;
  }
};

oidnx_status parse_blob(const void* blob, size_t bytes, ConvTensors (&layers)[kLayers],
                        int* in_channels) {
  BlobReader r{static_cast<const uint8_t*>(blob), bytes};
  const uint8_t* magic;
  uint32_t version, count;
  if (!r.bytes(&magic, 4) || std::memcmp(magic, "OXW1", 4) != 0)
    return fail(OIDNX_ERR_INVALID_MODEL, "weight blob: bad magic (expected OXW1)");
  if (!r.u32(&version) || version != 1)
    return fail(OIDNX_ERR_INVALID_MODEL, "weight blob: unsupported version");
  if (!r.u32(&count) || count > 4096)
    return fail(OIDNX_ERR_INVALID_MODEL, "weight blob: bad tensor count");
  bool have_w[kLayers] = {}, have_b[kLayers] = {};
  for (uint32_t t = 0; t < count; ++t) {
    uint32_t name_len, ndim, dtype;
    const uint8_t* name_p;
    if (!r.u32(&name_len) || name_len > 256 || !r.bytes(&name_p, name_len) ||
        !r.bytes(&name_p, 0))
      return fail(OIDNX_ERR_INVALID_MODEL, "weight blob: truncated tensor name");
    std::string name(reinterpret_cast<const char*>(r.p + r.off - name_len), name_len);
    const uint8_t* skip;
    if (!r.bytes(&skip, (4 - name_len % 4) % 4))
      return fail(OIDNX_ERR_INVALID_MODEL, "weight blob: truncated");
    if (!r.u32(&ndim) || ndim < 1 || ndim > 4)
      return fail(OIDNX_ERR_INVALID_MODEL, "weight blob: tensor %s: bad rank", name.c_str());
    uint32_t dims[4] = {1, 1, 1, 1};
    uint64_t elems = 1;
    for (uint32_t d = 0; d < ndim; ++d) {
      if (!r.u32(&dims[d]) || dims[d] == 0 || dims[d] > 65536)
        return fail(OIDNX_ERR_INVALID_MODEL, "weight blob: tensor %s: bad dims", name.c_str());
      elems *= dims[d];
    }
    if (!r.u32(&dtype) || dtype > 1)
      return fail(OIDNX_ERR_INVALID_MODEL, "weight blob: tensor %s: bad dtype", name.c_str());
    const size_t data_bytes = elems * (dtype == 0 ? 4 : 2);
    const uint8_t* data;
    if (!r.bytes(&data, data_bytes) || !r.bytes(&skip, (4 - data_bytes % 4) % 4))
      return fail(OIDNX_ERR_INVALID_MODEL, "weight blob: tensor %s: truncated data",
                  name.c_str());
    std::vector<float> vals(elems);
    for (uint64_t i = 0; i < elems; ++i) {
      if (dtype == 0) {
        std::memcpy(&vals[i], data + 4 * i, 4);
      } else {
        uint16_t b;
        std::memcpy(&b, data + 2 * i, 2);
        vals[i] = half_bits_to_float(b);
      }
    }
    int layer = -1;
    bool is_weight = false;
    for (int l = 0; l < kLayers; ++l) {
      if (name == std::string(kLayerNames[l]) + ".weight") { layer = l; is_weight = true; }
      if (name == std::string(kLayerNames[l]) + ".bias") { layer = l; is_weight = false; }
    }
    if (layer < 0) continue;  // unknown tensors are ignored
    ConvTensors& L = layers[layer];
    if (is_weight) {
      if (ndim != 4 || dims[2] != 3 || dims[3] != 3)
        return fail(OIDNX_ERR_INVALID_MODEL, "%s: expected a 3x3 OIHW weight", name.c_str());
      L.cout = static_cast<int>(dims[0]);
      L.cin = static_cast<int>(dims[1]);
      L.w = std::move(vals);
      have_w[layer] = true;
    } else {
      if (ndim != 1)
        return fail(OIDNX_ERR_INVALID_MODEL, "%s: expected a 1-D bias", name.c_str());
      L.b = std::move(vals);
      have_b[layer] = true;
    }
  }
  for (int l = 0; l < kLayers; ++l) {
    if (!have_w[l] || !have_b[l])
      return fail(OIDNX_ERR_INVALID_MODEL, "weight blob: missing %s weight or bias",
                  kLayerNames[l]);
    if (static_cast<int>(layers[l].b.size()) != layers[l].cout)
      return fail(OIDNX_ERR_INVALID_MODEL, "%s: bias size %zu != %d outputs", kLayerNames[l],
                  layers[l].b.size(), layers[l].cout);
  }
  // Topology checks (channel counts must chain as the U-Net's dataflow).
  const int cin = layers[0].cin;
  if (cin != 3 && cin != 6 && cin != 9)
    return fail(OIDNX_ERR_INVALID_MODEL, "expects 3, 6, or 9 input channels, got %d", cin);
  auto out_ch = [&](int v) -> int {
    if (v == V_IN) return cin;
    for (int l = 0; l < kLayers; ++l)
      if (kDefs[l].dst == v) return layers[l].cout;
    return -1;
  };
  for (int l = 0; l < kLayers; ++l) {
    int need = out_ch(kDefs[l].src0) + (kDefs[l].src1 >= 0 ? out_ch(kDefs[l].src1) : 0);
    if (layers[l].cin != need)
      return fail(OIDNX_ERR_INVALID_MODEL, "%s: %d input channels, the U-Net needs %d",
                  kLayerNames[l], layers[l].cin, need);
    if (layers[l].cout > 256)
      return fail(OIDNX_ERR_UNSUPPORTED, "%s: more than 256 output channels", kLayerNames[l]);
  }
  if (layers[15].cout != 3)
    return fail(OIDNX_ERR_INVALID_MODEL, "dec_conv0 must have 3 outputs");
  *in_channels = cin;
  return ok();
}

// ---------------------------------------------------------------- packing
// fp16 tensor-core B operand: per 16-lane K block kb, per tap, per 8-lane
// half j, N rows of 8 halves ([kb][tap][j][n][8]).  K lanes enumerate the
// concatenated sources, each padded to a multiple of 16 lanes; padded rows
// and lanes are zero.
// fp16 tensor-core B operand, per 16-lane K block kb: [kx][8-lane half j]
// [ky stack pos][N][8] halves with pos = 2 - ky, so that rows pos*N .. of one
// (kx, j) slice are W(ky=2), W(ky=1), W(ky=0) one after the other.  K lanes
// enumerate the concatenated sources, each padded to a multiple of 16 lanes;
// padded rows and lanes are zero.
std::vector<uint16_t> pack_weights_tc(const ConvTensors& L, int c0, int c1, int* KB0,
                                      int* KB1, int* N) {
  const int p0 = round_up(c0, 16), p1 = c1 > 0 ? round_up(c1, 16) : 0;
  *KB0 = p0 / 16;
  *KB1 = p1 / 16;
  *N = round_up(L.cout, 16);
  const int KB = *KB0 + *KB1;
  std::vector<uint16_t> out(static_cast<size_t>(KB) * 9 * 2 * (*N) * 8, 0);
  for (int kb = 0; kb < KB; ++kb)
    for (int kx = 0; kx < 3; ++kx)
      for (int j = 0; j < 2; ++j)
        for (int pos = 0; pos < 3; ++pos)
          for (int n = 0; n < L.cout; ++n)
            for (int l = 0; l < 8; ++l) {
              const int v = kb * 16 + j * 8 + l;
              int ch = -1;
              if (v < p0) ch = v < c0 ? v : -1;
              else ch = (v - p0) < c1 ? c0 + (v - p0) : -1;
              if (ch < 0) continue;
              const int ky = 2 - pos;
              const float w = L.w[(static_cast<size_t>(n) * L.cin + ch) * 9 + ky * 3 + kx];
              const size_t idx =
                  (((((static_cast<size_t>(kb) * 3 + kx) * 2 + j) * 3 + pos) * (*N) + n) * 8) + l;
              out[idx] = to_half_bits(w);
            }
  return out;
}

// The final 32 -> 3 conv's B operand for the fused pair kernel, kx folded
// into N: per K block [j][pos][16][8] halves, row pos * 16 + 4 * kx + co
// (pos = 2 - ky); rows 4 kx + 3 and 12..15 are zero.
std::vector<uint16_t> pack_weights_folded(const ConvTensors& L) {
  const int KB = round_up(L.cin, 16) / 16;
  std::vector<uint16_t> out(static_cast<size_t>(KB) * 2 * 48 * 8, 0);
  for (int kb = 0; kb < KB; ++kb)
    for (int j = 0; j < 2; ++j)
      for (int pos = 0; pos < 3; ++pos)
        for (int kx = 0; kx < 3; ++kx)
          for (int co = 0; co < L.cout; ++co)
            for (int l = 0; l < 8; ++l) {
              const int ch = kb * 16 + j * 8 + l;
              if (ch >= L.cin) continue;
              const int ky = 2 - pos;
              const float w = L.w[(static_cast<size_t>(co) * L.cin + ch) * 9 + ky * 3 + kx];
              const size_t row = static_cast<size_t>(pos) * 16 + 4 * kx + co;
              out[((static_cast<size_t>(kb) * 2 + j) * 48 + row) * 8 + l] = to_half_bits(w);
            }
  return out;
}

// tf32 split of an fp32 weight: hi = w rounded to the nearest tf32 value,
// lo = w - hi (exact).
void split_tf32(float w, float* hi, float* lo) {
  uint32_t bits;
  std::memcpy(&bits, &w, 4);
  bits = (bits + 0x1000u) & 0xFFFFE000u;
  std::memcpy(hi, &bits, 4);
  *lo = w - *hi;
}

// fp32 storage: the B operand for 3xTF32 products.  K blocks of 8 channels
// (two 16-byte chunks of 4 lanes) over each source padded to 4 lanes; per
// block [hi, lo][kx][j][pos][N][4] floats with pos = 2 - ky, where hi is the
// weight rounded to the nearest tf32 value and lo = w - hi (exact).
std::vector<float> pack_weights_tf32(const ConvTensors& L, int c0, int c1, int* KB0, int* KB1,
                                     int* N) {
  const int q0 = round_up(c0, 4) / 4, q1 = c1 > 0 ? round_up(c1, 4) / 4 : 0;  // chunks
  *KB0 = (q0 + 1) / 2;
  *KB1 = (q1 + 1) / 2;
  *N = round_up(L.cout, 16);
  const int KB = *KB0 + *KB1;
  std::vector<float> out(static_cast<size_t>(KB) * 2 * 9 * 2 * (*N) * 4, 0.0f);
  for (int kb = 0; kb < KB; ++kb)
    for (int kx = 0; kx < 3; ++kx)
      for (int j = 0; j < 2; ++j)
        for (int pos = 0; pos < 3; ++pos)
          for (int n = 0; n < L.cout; ++n)
            for (int l = 0; l < 4; ++l) {
              const bool first = kb < *KB0;
              const int ci = ((first ? kb : kb - *KB0) * 2 + j) * 4 + l;  // within the source
              if (ci >= (first ? c0 : c1)) continue;
              const int ch = first ? ci : c0 + ci;
              const int ky = 2 - pos;
              const float w = L.w[(static_cast<size_t>(n) * L.cin + ch) * 9 + ky * 3 + kx];
              float hl[2];
              split_tf32(w, &hl[0], &hl[1]);
              for (int part = 0; part < 2; ++part) {
                const size_t idx =
                    ((((((static_cast<size_t>(kb) * 2 + part) * 3 + kx) * 2 + j) * 3 + pos) * (*N) + n) * 4) + l;
                out[idx] = hl[part];
              }
            }
  return out;
}

// Sub-pixel decoder B operand.  Upsampled K blocks (source 0): per block
// [px][d][j][pos][N][8] where, for output column parity px, d selects the
// low-resolution column offset dx = d - 1 + px and pos the (row parity py,
// row offset dy) class (1,+1), (0,0), (1,0), (0,-1); each entry is the sum of
// the fp16-rounded 3x3 weights whose taps land on that low-resolution pixel
// (ky in Ky(py,dy), kx in Kx(px,dx)), rounded once more to fp16.  Skip K
// blocks follow in the plain layout.  Returns bytes of the upsampled part per
// K block in *ub.
// Taps of a 3x3 kernel row (or column) that fall on low-resolution offset
// `off` for output parity `parity` under nearest 2x upsampling: the output at
// 2i + parity reads the upsampled source at 2i + parity + k - 1, i.e. the
// low-resolution pixel i + floor((parity + k - 1) / 2).
int subpixel_taps(int parity, int off, int* t) {
  if (parity == 0) {
    if (off == -1) { t[0] = 0; return 1; }
    t[0] = 1; t[1] = 2; return 2;       // off 0
  }
  if (off == 0) { t[0] = 0; t[1] = 1; return 2; }
  t[0] = 2; return 1;                    // off +1
}

// (row parity, row offset) of the four row classes stacked along N
const int kPosPy[4] = {1, 0, 1, 0}, kPosDy[4] = {1, 0, 0, -1};

std::vector<uint16_t> pack_weights_subpixel(const ConvTensors& L, int c0, int c1, int N,
                                            size_t* ub) {
  const int p0 = round_up(c0, 16), p1 = round_up(c1, 16);
  const int KB0 = p0 / 16, KB1 = p1 / 16;
  auto taps = subpixel_taps;
  const int* pos_py = kPosPy;
  const int* pos_dy = kPosDy;
  const size_t up_halves = static_cast<size_t>(2) * 2 * 2 * 4 * N * 8;   // per K block
  const size_t sk_halves = static_cast<size_t>(3) * 2 * 3 * N * 8;
  *ub = up_halves * 2;
  std::vector<uint16_t> out(KB0 * up_halves + KB1 * sk_halves, 0);
  auto q = [](float w) { return half_bits_to_float(to_half_bits(w)); };
  for (int kb = 0; kb < KB0; ++kb)
    for (int px = 0; px < 2; ++px)
      for (int d = 0; d < 2; ++d)
        for (int j = 0; j < 2; ++j)
          for (int pos = 0; pos < 4; ++pos) {
            int kys[2], kxs[2];
            const int nky = taps(pos_py[pos], pos_dy[pos], kys);
            const int nkx = taps(px, d - 1 + px, kxs);
            for (int n = 0; n < L.cout; ++n)
              for (int l = 0; l < 8; ++l) {
                const int ch = kb * 16 + j * 8 + l;
                if (ch >= c0) continue;
                float sum = 0.0f;
                for (int a = 0; a < nky; ++a)
                  for (int b = 0; b < nkx; ++b)
                    sum += q(L.w[(static_cast<size_t>(n) * L.cin + ch) * 9 + kys[a] * 3 + kxs[b]]);
                const size_t idx = kb * up_halves +
                                   ((((static_cast<size_t>(px) * 2 + d) * 2 + j) * 4 + pos) * N + n) * 8 + l;
                out[idx] = to_half_bits(sum);
              }
          }
  for (int kb = 0; kb < KB1; ++kb)
    for (int kx = 0; kx < 3; ++kx)
      for (int j = 0; j < 2; ++j)
        for (int pos = 0; pos < 3; ++pos)
          for (int n = 0; n < L.cout; ++n)
            for (int l = 0; l < 8; ++l) {
              const int v = kb * 16 + j * 8 + l;
              if (v >= c1) continue;
              const int ky = 2 - pos;
              const float w = L.w[(static_cast<size_t>(n) * L.cin + c0 + v) * 9 + ky * 3 + kx];
              const size_t idx = KB0 * up_halves +
                                 ((((static_cast<size_t>(kb) * 3 + kx) * 2 + j) * 3 + pos) * N + n) * 8 + l;
              out[idx] = to_half_bits(w);
            }
  return out;
}


// Sub-pixel decoder B operand for fp32 storage (3xTF32 products): the same
// per-class sums, taken in double over the fp32 weights and rounded once to
// fp32, then split into tf32 hi and lo parts.  K blocks of 8 channels (two
// 4-lane chunks j).  Upsampled blocks: [px][hi, lo][d][j][pos][N][4] floats
// (1024 N bytes, so each column parity's half holds its hi and lo parts);
// skip blocks, per kx slice: [hi, lo][j][pos][N][4] floats (192 N bytes),
// pos = 2 - ky.  Returns bytes of the upsampled part per K block in *ub.
std::vector<float> pack_weights_subpixel_tf32(const ConvTensors& L, int c0, int c1, int N,
                                              size_t* ub) {
  const int KB0 = (round_up(c0, 4) / 4 + 1) / 2, KB1 = (round_up(c1, 4) / 4 + 1) / 2;
  const size_t up_f = static_cast<size_t>(2) * 2 * 2 * 2 * 4 * N * 4;  // floats per block
  const size_t sl_f = static_cast<size_t>(2) * 2 * 3 * N * 4;          // floats per kx slice
  *ub = up_f * 4;
  std::vector<float> out(KB0 * up_f + static_cast<size_t>(KB1) * 3 * sl_f, 0.0f);
  for (int kb = 0; kb < KB0; ++kb)
    for (int px = 0; px < 2; ++px)
      for (int d = 0; d < 2; ++d)
        for (int j = 0; j < 2; ++j)
          for (int pos = 0; pos < 4; ++pos) {
            int kys[2], kxs[2];
            const int nky = subpixel_taps(kPosPy[pos], kPosDy[pos], kys);
            const int nkx = subpixel_taps(px, d - 1 + px, kxs);
            for (int n = 0; n < L.cout; ++n)
              for (int l = 0; l < 4; ++l) {
                const int ch = kb * 8 + j * 4 + l;
                if (ch >= c0) continue;
                double sum = 0.0;
                for (int a = 0; a < nky; ++a)
                  for (int b = 0; b < nkx; ++b)
                    sum += L.w[(static_cast<size_t>(n) * L.cin + ch) * 9 + kys[a] * 3 + kxs[b]];
                float hl[2];
                split_tf32(static_cast<float>(sum), &hl[0], &hl[1]);
                for (int part = 0; part < 2; ++part)
                  out[kb * up_f +
                      ((((((static_cast<size_t>(px) * 2 + part) * 2 + d) * 2 + j) * 4 + pos) * N + n) * 4) + l] =
                      hl[part];
              }
          }
  for (int kb = 0; kb < KB1; ++kb)
    for (int kx = 0; kx < 3; ++kx)
      for (int j = 0; j < 2; ++j)
        for (int pos = 0; pos < 3; ++pos)
          for (int n = 0; n < L.cout; ++n)
            for (int l = 0; l < 4; ++l) {
              const int v = kb * 8 + j * 4 + l;
              if (v >= c1) continue;
              const int ky = 2 - pos;
              float hl[2];
              split_tf32(L.w[(static_cast<size_t>(n) * L.cin + c0 + v) * 9 + ky * 3 + kx], &hl[0], &hl[1]);
              for (int part = 0; part < 2; ++part)
                out[KB0 * up_f + (static_cast<size_t>(kb) * 3 + kx) * sl_f +
                    (((static_cast<size_t>(part) * 2 + j) * 3 + pos) * N + n) * 4 + l] = hl[part];
            }
  return out;
}


// The folded final-conv B operand for fp32 storage: per K block of 8
// channels [hi, lo][j][pos][16][4] floats, row pos * 16 + 4 * kx + co
// (pos = 2 - ky), each weight split into its tf32 hi and lo parts.
std::vector<float> pack_weights_folded_tf32(const ConvTensors& L) {
  const int KB = round_up(L.cin, 8) / 8;
  std::vector<float> out(static_cast<size_t>(KB) * 2 * 2 * 48 * 4, 0.0f);
  for (int kb = 0; kb < KB; ++kb)
    for (int j = 0; j < 2; ++j)
      for (int pos = 0; pos < 3; ++pos)
        for (int kx = 0; kx < 3; ++kx)
          for (int co = 0; co < L.cout; ++co)
            for (int l = 0; l < 4; ++l) {
              const int ch = kb * 8 + j * 4 + l;
              if (ch >= L.cin) continue;
              const int ky = 2 - pos;
              float hl[2];
              split_tf32(L.w[(static_cast<size_t>(co) * L.cin + ch) * 9 + ky * 3 + kx], &hl[0], &hl[1]);
              const size_t row = static_cast<size_t>(pos) * 16 + 4 * kx + co;
              for (int part = 0; part < 2; ++part)
                out[(((static_cast<size_t>(kb) * 2 + part) * 2 + j) * 48 + row) * 4 + l] = hl[part];
            }
  return out;
}

// ---------------------------------------------------------------- tiles
struct AxisTile {
  int in_start, in_size, out_start, out_size;
};

// Per-axis tile plan on the 16-aligned extent; see oidnx_plan_tiles.
bool plan_axis(int extent, int limit, int overlap, std::vector<AxisTile>* tiles) {
  tiles->clear();
  if (extent <= 0 || overlap < 0 || overlap % 16) return false;
  const int ea = round_up(extent, 16);
  const int tmax = limit / 16 * 16;
  if (ea <= tmax) {
    tiles->push_back({0, ea, 0, extent});
    return true;
  }
  int n = 2, c = 0;
  for (;; ++n) {
    c = round_up((ea + n - 1) / n, 16);
    if (c + 2 * overlap <= tmax) break;
    if (c <= 16) return false;
  }
  const int size = c + 2 * overlap;
  for (int i = 0; i < n; ++i) {
    const int o = i * c;
    const int o_next = i + 1 < n ? (i + 1) * c : ea;
    const int s = std::min(std::max(o - overlap, 0), ea - size);
    const int osz = std::min(o_next, extent) - o;
    if (osz > 0) tiles->push_back({s, size, o, osz});
  }
  return true;
}

// One-sided dependency radius of the 4-level U-Net output on its input,
// by interval propagation (conv: +-1, pool source: [2a, 2b+1], nearest
// upsample source: [a>>1, b>>1], concat: union), worst over residues mod 16.
int dependency_radius() {
  struct Iv { long a, b; };
  auto conv = [](Iv v) { return Iv{v.a - 1, v.b + 1}; };
  auto pool_src = [](Iv v) { return Iv{2 * v.a, 2 * v.b + 1}; };
  auto up_src = [](Iv v) { return Iv{v.a >> 1, v.b >> 1}; };
  const int levels = 4;
  // input interval of a pooled value at `level` (0 = the input itself)
  auto pooled = [&](Iv v, int level) {
    while (level > 0) {
      v = conv(pool_src(v));
      if (level == 1) v = conv(v);
      --level;
    }
    return v;
  };
  // input interval of the decoder output at `level`
  std::function<Iv(Iv, int)> decoded;
  decoded = [&](Iv v, int level) -> Iv {
    if (level == levels) return pooled(conv(conv(v)), levels);
    Iv cat = conv(conv(v));
    Iv low = decoded(up_src(cat), level + 1);
    Iv skip = pooled(cat, level);
    return Iv{std::min(low.a, skip.a), std::max(low.b, skip.b)};
  };
  long r = 0;
  for (int res = 0; res < 16; ++res) {
    const long p = 16L * 64 * 10 + res;
    Iv d = decoded(conv(Iv{p, p}), 0);
    r = std::max(r, std::max(p - d.a, d.b - p));
  }
  return static_cast<int>(r);
}

int default_overlap_value() { return round_up(dependency_radius(), 16); }

// ---------------------------------------------------------------- tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  }
  return fn;
}

// fp16 activation [H][C8][pitch][8] (columns [W, pitch) zero) as a 4-D
// tensor.  When the pitch is a multiple of 8 pixels the innermost dimension
// is one 8-pixel group (64 halves = 128 B) and x counts groups (*xs = 3);
// otherwise it is one pixel (16 B, *xs = 0).  The box is box_w pixels (a
// multiple of 8 for the 8-pixel form) x 2 channel chunks x box_h rows.
oidnx_status encode_act_map(CUtensorMap* map, const void* base, int W, int pitch, int H, int C8,
                            int box_w, int box_h, bool allow_groups, int* xs, int box_c = 2) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return fail(OIDNX_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const bool groups = allow_groups && pitch % kGroupPx == 0 && box_w % kGroupPx == 0;
  const cuuint64_t row = static_cast<cuuint64_t>(pitch) * 16;
  cuuint64_t dims[4], strides[3] = {0, row, row * C8};
  cuuint32_t box[4];
  if (groups) {
    dims[0] = 8 * kGroupPx;
    dims[1] = static_cast<cuuint64_t>(pitch / kGroupPx);
    strides[0] = 16 * kGroupPx;
    box[0] = 8 * kGroupPx;
    box[1] = static_cast<cuuint32_t>(box_w / kGroupPx);
  } else {
    dims[0] = 8;
    dims[1] = static_cast<cuuint64_t>(W);
    strides[0] = 16;
    box[0] = 8;
    box[1] = static_cast<cuuint32_t>(box_w);
  }
  dims[2] = static_cast<cuuint64_t>(C8);
  dims[3] = static_cast<cuuint64_t>(H);
  box[2] = static_cast<cuuint32_t>(box_c);
  box[3] = static_cast<cuuint32_t>(box_h);
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(OIDNX_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for %dx%dx%d (pitch %d)",
                int(r), W, H, C8, pitch);
  if (xs) *xs = groups ? 3 : 0;
  return ok();
}

// fp16 column-parity split activation [H][C8][2][pitch/2][8] (entries
// [W/2, pitch/2) of each plane zero) as a 5-D tensor {lanes, x, plane, C8, H}.
// With pitch % 16 == 0 the innermost dimension is 8 entries (128 B) and x
// counts 8-entry groups (*xs = 3), else one entry (16 B, *xs = 0); the box
// is box_w entries (a multiple of 8 for the first form) x 1 plane x 2 chunks
// x box_h rows.
oidnx_status encode_split_map(CUtensorMap* map, const void* base, int W, int pitch, int H, int C8,
                              int box_w, int box_h, int* xs) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return fail(OIDNX_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  const cuuint64_t half = static_cast<cuuint64_t>(pitch / 2);
  const bool groups = half % kGroupPx == 0 && box_w % kGroupPx == 0;
  cuuint64_t dims[5], strides[4] = {0, half * 16, half * 32, half * 32 * C8};
  cuuint32_t box[5];
  if (groups) {
    dims[0] = 8 * kGroupPx;
    dims[1] = half / kGroupPx;
    strides[0] = 16 * kGroupPx;
    box[0] = 8 * kGroupPx;
    box[1] = static_cast<cuuint32_t>(box_w / kGroupPx);
  } else {
    dims[0] = 8;
    dims[1] = static_cast<cuuint64_t>(W / 2);
    strides[0] = 16;
    box[0] = 8;
    box[1] = static_cast<cuuint32_t>(box_w);
  }
  dims[2] = 2;
  dims[3] = static_cast<cuuint64_t>(C8);
  dims[4] = static_cast<cuuint64_t>(H);
  box[2] = 1;
  box[3] = 2;
  box[4] = static_cast<cuuint32_t>(box_h);
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(OIDNX_ERR_CUDA, "cuTensorMapEncodeTiled (split) failed (%d)", int(r));
  if (xs) *xs = groups ? 3 : 0;
  return ok();
}

// ======================================================================
// device-side model and plans
// ======================================================================
// A float4 image [height][width] with row stride `stride` bytes as a 2-D
// tensor {4 * width floats, height}; boxes of kHeadRows + 2 rows x 176
// floats (44 pixels): the fused input pass stages 132 pixels as three.
oidnx_status encode_image_map(CUtensorMap* map, const void* base, int width, int height, size_t stride) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return fail(OIDNX_ERR_CUDA, "cuTensorMapEncodeTiled is not available");
  cuuint64_t dims[2] = {4 * static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(height)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(stride)};
  cuuint32_t box[2] = {4 * 44, static_cast<cuuint32_t>(kHeadRows + 2)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    return fail(OIDNX_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d) for a %dx%d image", int(r), width, height);
  return ok();
}

struct DeviceLayer {
  int cout = 0, cin = 0, c0 = 0, c1 = 0;
  // B operands, each fp16 or (fp32 storage) tf32 hi/lo
  void* wtc = nullptr;  // packed tensor-core B operand of the generic kinds
  bool tf32 = false;    // fp32 storage: 3xTF32 products
  int KB0 = 0, KB1 = 0, N = 0;
  void* wsub = nullptr;  // sub-pixel decoder B operand (decoders only)
  size_t sub_bytes = 0, sub_ub = 0;
  void* wfold = nullptr;    // fused final conv: B operand with kx folded into N
  size_t fold_bytes = 0;
  float* bias = nullptr;  // [N]
  size_t weight_bytes = 0;
};

// Extent of an activation; pitch = row stride in pixels (fp16 values of the
// network: w rounded up to 8, padding columns zero; otherwise w).
struct Extent {
  int w, h, pitch;
};

int fp16_pitch(int w) { return (w + kGroupPx - 1) / kGroupPx * kGroupPx; }

// Zero rows below each tile of a stacked frame at level 0 (one row at level
// 4): the same padding for every conv as an image border gives.
constexpr int kStackGap = 16;
// Activation bytes a stacked group of tiles may take; frames with more
// tiles run in several groups.  (Groups of 8 + 7 tiles of a 3840 x 2160
// frame ran 9% slower than one stack of 15: 4.4 GB of fp16 activations.)
constexpr size_t kStackBudget = size_t(16) << 30;

// Pitch of a column-parity split copy: 16-pixel multiple, so that each
// parity plane (pitch / 2 entries) is a whole number of 8-entry TMA rows.
int split_pitch(int w) { return (w + 2 * kGroupPx - 1) / (2 * kGroupPx) * (2 * kGroupPx); }

struct LayerLaunch {
  int layer;               // first layer of the launch
  int pair;                // 1: layers `layer` and `layer + 1` fused (pcl)
  int final;               // 1: the final conv with kx folded (fcl)
  int tail;                // 1: the last two layers in one kernel (tlcl)
  const char* name;
  TcConvLaunch tcl;
  PairConvLaunch pcl;
  FinalConvLaunch fcl;
  TailConvLaunch tlcl;
  double flop;   // logical conv FLOPs
  double bytes;  // algorithmic bytes: inputs read once, output written once
};

struct Plan {
  int w = 0, h = 0;
  Extent lvl[5];
  size_t value_off[V_COUNT] = {};
  size_t value_bytes[V_COUNT] = {};
  Extent value_ext[V_COUNT];
  int value_ch[V_COUNT] = {};
  void* arena = nullptr;
  size_t arena_bytes = 0;
  std::vector<LayerLaunch> launches;
  bool split_on[4] = {};  // kSplits[i] in use (its decoder runs in sub-pixel mode)
  bool fused[2] = {};     // kPairs[i] runs as one fused kernel
  // stacked tiles: the frame's `stack` tiles (h rows each) sit one above the
  // other in every value, each followed by kStackGap zero rows at level 0
  // (kStackGap >> L at level L); the convs run once over the stack, the
  // input pass and the final conv (final_tiles) once per tile
  int stack = 1;
  std::vector<LayerLaunch> final_tiles;
  // the last execution stored the network output (not so when the output
  // pass ran in the final conv's epilogue without keepActivations)
  bool out_stored = true;
  // the last execution ran the output pass in the last conv's epilogue
  bool outpass_fused = false;
  // one-tile-at-a-time frames: the input pass and enc_conv0 as one kernel
  // (head: built when the plan allows it; head_used: the last execution
  // ran it)
  bool head_on = false, head_used = false;
  HeadLaunch head;
  uint64_t last_used = 0;
  cudaEvent_t done = nullptr;  // recorded after each use
  bool used = false;
  void* ptr(int v) const { return static_cast<uint8_t*>(arena) + value_off[v]; }
};

// Per-kernel timing events of one execution.
struct Profile {
  std::vector<cudaEvent_t> ev;        // ev[0] = start, one per launch after it
  std::vector<int> label;             // layer id per launch: -1 pack, 0..15, 16 unpack
  int used = 0;
  bool valid = false;
};

}  // namespace

struct oidnx_filter {
  bool released = false;
  int precision = OIDNX_PRECISION_FP16;  // resolved: 1 or 2
  int in_channels = 9;
  DeviceLayer layers[kLayers];
  size_t weight_bytes = 0;
  int* status = nullptr;  // device error word
  void* log2_tab = nullptr;  // fp32 log-transfer table (kLog2TabSize float4)
  void* exp2_tab = nullptr;  // output pass's inverse-transfer table (kExp2TabSize float4)
  // parameters
  int width = 0, height = 0, hdr = 0, transfer = OIDNX_TRANSFER_LOG, max_tile = 0,
      overlap = -1, shape_cache = 2, keep_acts = 0, profile_always = 0, subpixel = 1,
      fuse = 0, fuse_output = 1, fuse_tail = 1, fuse_input = 0, stack_tiles = 0,
      shape_kernels = 1;
  float input_scale = 1.0f;
  void* img[4] = {};
  size_t img_stride[4] = {};
  // committed state
  bool committed = false;
  std::vector<AxisTile> tx, ty;
  Plan* current = nullptr;
  std::list<std::unique_ptr<Plan>> plans;    // LRU cache
  std::list<std::unique_ptr<Plan>> retired;  // evicted, maybe still in flight
  uint64_t clock = 0;
  // graphs of the committed denoise, one per image set (the host path
  // alternates two device staging sets), least recently used replaced
  struct GraphEntry {
    cudaGraphExec_t exec = nullptr;
    bool profiled = false;
    void* img[4] = {};
    uint64_t used = 0;
  } graphs[2];
  uint64_t graph_clock = 0;
  cudaStream_t capture_stream = nullptr;
  // profiling
  bool profile_next = false;
  Profile prof;
  // host path: two device staging sets (colour, albedo, normal, output), an
  // upload and a download stream, and per set the events that order them
  // with the denoise: inputs uploaded, denoise done, output downloaded
  void* host_img[2][4] = {};
  size_t host_img_bytes = 0;
  cudaStream_t host_in = nullptr, host_out = nullptr;
  cudaEvent_t ev_in[2] = {}, ev_comp[2] = {}, ev_out[2] = {};
  bool host_used[2] = {};
  int host_next = 0;
  // last network run (for debug reads)
  Plan* last_plan = nullptr;
};

static void drop_graphs(oidnx_filter* f) {
  for (auto& g : f->graphs) {
    if (g.exec) cudaGraphExecDestroy(g.exec);
    g = oidnx_filter::GraphEntry();
  }
}

struct oidnx_conv {
  DeviceLayer L;
  int precision = OIDNX_PRECISION_FP16;
  int* status = nullptr;
};

namespace {

oidnx_status upload(const void* host, size_t bytes, void** dev) {
  OIDNX_CUDA(cudaMalloc(dev, bytes));
  OIDNX_CUDA(cudaMemcpy(*dev, host, bytes, cudaMemcpyHostToDevice));
  return ok();
}

void free_layer(DeviceLayer& L) {
  cudaFree(L.wsub);
  L.wsub = nullptr;
  cudaFree(L.wfold);
  L.wfold = nullptr;
  cudaFree(L.wtc);
  cudaFree(L.bias);
  L.wtc = nullptr;
  L.bias = nullptr;
}

oidnx_status make_device_layer(const ConvTensors& T, int c0, int c1, int precision,
                               DeviceLayer* L) {
  L->cout = T.cout;
  L->cin = T.cin;
  L->c0 = c0;
  L->c1 = c1;
  if (precision == OIDNX_PRECISION_FP16) {
    std::vector<uint16_t> w = pack_weights_tc(T, c0, c1, &L->KB0, &L->KB1, &L->N);
    if (L->N > 256) return fail(OIDNX_ERR_UNSUPPORTED, "more than 256 output channels");
    OIDNX_TRY(upload(w.data(), w.size() * 2, &L->wtc));
    if (c1 > 0) {
      std::vector<uint16_t> ws = pack_weights_subpixel(T, c0, c1, L->N, &L->sub_ub);
      L->sub_bytes = ws.size() * 2;
      OIDNX_TRY(upload(ws.data(), L->sub_bytes, &L->wsub));
    }
    if (T.cout == 3 && T.cin == 32 && c1 == 0) {
      std::vector<uint16_t> wf = pack_weights_folded(T);
      L->fold_bytes = wf.size() * 2;
      OIDNX_TRY(upload(wf.data(), L->fold_bytes, &L->wfold));
    }
    std::vector<float> b(L->N, 0.0f);
    std::copy(T.b.begin(), T.b.end(), b.begin());
    OIDNX_TRY(upload(b.data(), b.size() * 4, reinterpret_cast<void**>(&L->bias)));
    L->weight_bytes = w.size() * 2 + b.size() * 4 + L->sub_bytes + L->fold_bytes;
  } else {
    std::vector<float> w = pack_weights_tf32(T, c0, c1, &L->KB0, &L->KB1, &L->N);
    if (L->N > 256) return fail(OIDNX_ERR_UNSUPPORTED, "more than 256 output channels");
    OIDNX_TRY(upload(w.data(), w.size() * 4, &L->wtc));
    L->tf32 = true;
    if (c1 > 0) {
      std::vector<float> ws = pack_weights_subpixel_tf32(T, c0, c1, L->N, &L->sub_ub);
      L->sub_bytes = ws.size() * 4;
      OIDNX_TRY(upload(ws.data(), L->sub_bytes, &L->wsub));
    }
    if (T.cout == 3 && T.cin == 32 && c1 == 0) {
      std::vector<float> wf = pack_weights_folded_tf32(T);
      L->fold_bytes = wf.size() * 4;
      OIDNX_TRY(upload(wf.data(), L->fold_bytes, &L->wfold));
    }
    std::vector<float> b(L->N, 0.0f);
    std::copy(T.b.begin(), T.b.end(), b.begin());
    OIDNX_TRY(upload(b.data(), b.size() * 4, reinterpret_cast<void**>(&L->bias)));
    L->weight_bytes = w.size() * 4 + b.size() * 4 + L->sub_bytes + L->fold_bytes;
  }
  return ok();
}

// Bytes of one stored activation: fp16 rounds channels up to 16 lanes, fp32
// to 4; the network output is [h][w][4] floats.
size_t act_bytes(int precision, Extent e, int c, bool final_out) {
  if (final_out) return static_cast<size_t>(e.w) * e.h * 16;
  if (precision == OIDNX_PRECISION_FP16) return static_cast<size_t>(e.pitch) * e.h * round_up(c, 16) * 2;
  return static_cast<size_t>(e.pitch) * e.h * round_up(c, 4) * 4;
}

// Extent of a stored value of conv extent e.
Extent value_extent(int precision, Extent e, bool final_out) {
  const bool padded = precision == OIDNX_PRECISION_FP16 && !final_out;
  return Extent{e.w, e.h, padded ? fp16_pitch(e.w) : e.w};
}

int act_chunks(int precision, int c) {
  return precision == OIDNX_PRECISION_FP16 ? round_up(c, 16) / 8 : round_up(c, 4) / 4;
}

// Per-device facts and settings.  Kernel attributes (the raised shared-memory
// limit) belong to the current device's context, so each is set once per
// device, under a mutex, for up to kMaxDevices devices (beyond that on every
// call).
constexpr int kMaxDevices = 64;
std::mutex g_device_mutex;
int g_num_sms[kMaxDevices] = {};
uint64_t g_smem_limit_set[5] = {};  // per kernel family: bit d for device d

int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  return dev;
}

int num_sms() {
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(g_device_mutex);
  if (dev < kMaxDevices && g_num_sms[dev] > 0) return g_num_sms[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    n = 148;
  if (dev < kMaxDevices) g_num_sms[dev] = n;
  return n;
}

enum KernelFamily { kFamilyTc = 0, kFamilyPair = 1, kFamilyFinal = 2, kFamilyTail = 3, kFamilyHead = 4 };

// Raise a kernel family's dynamic shared-memory limit to the 227 KB an SM
// offers, on the current device.
oidnx_status ensure_smem_limit(int family) {
  const int dev = current_device();
  std::lock_guard<std::mutex> lock(g_device_mutex);
  const uint64_t bit = dev < kMaxDevices ? (uint64_t(1) << dev) : 0;
  if (bit && (g_smem_limit_set[family] & bit)) return ok();
  const size_t max_smem = 227 * 1024;
  const cudaError_t e = family == kFamilyTc      ? conv_tc_set_smem_limit(max_smem)
                        : family == kFamilyPair  ? conv_pair_set_smem_limit(max_smem)
                        : family == kFamilyFinal ? conv_final_set_smem_limit(max_smem)
                        : family == kFamilyTail  ? conv_tail_set_smem_limit(max_smem)
                                                 : conv_head_set_smem_limit(max_smem);
  if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "smem limit: %s", cudaGetErrorString(e));
  g_smem_limit_set[family] |= bit;
  return ok();
}

// Last wave of a persistent conv grid: when the tiles do not fill the
// final wave and at most half of the grid would work in it, its tiles are
// split into sub-tiles of fewer rows (a power of two, at least min_rows
// rows each: even rows for pools and decoders), as many as the grid takes.
// A sub-tile loads its parent tile's boxes and issues only its own rows.
void plan_tail(TcConvParams* p, long grid, int min_rows, bool allowed) {
  const long tiles = static_cast<long>(p->tiles_x) * p->tiles_y;
  const long r = tiles % grid;
  int split = 1;
  if (allowed && r > 0 && 2 * r <= grid)
    while (p->R % (2 * split) == 0 && p->R / (2 * split) >= min_rows && r * 2 * split <= grid)
      split *= 2;
  p->tail_first = static_cast<int>(split > 1 ? tiles - r : tiles);
  p->tail_split = split;
  p->walk_tiles = static_cast<int>(p->tail_first + (tiles - p->tail_first) * split);
}

// Build the tensor-core launch of one conv.  src0/src1: device pointers of the
// sources (fp16 layout), ext0: extent of source 0, (W, H): conv extent.
// Pad the shared-memory request until at most `allowed` CTAs fit one SM, so
// that CTAs sharing an SM never wait for tensor memory.
oidnx_status bound_ctas_per_sm(size_t* smem, uint32_t tmem_cols, int* blocks) {
  const size_t max_smem = 227 * 1024;
  OIDNX_TRY(ensure_smem_limit(kFamilyTc));
  const int allowed = static_cast<int>(512 / tmem_cols);
  for (;;) {
    cudaError_t e = conv_tc_occupancy(*smem, blocks);
    if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "occupancy: %s", cudaGetErrorString(e));
    if (*blocks <= allowed) return ok();
    *smem += 4096;
    if (*smem > max_smem) return fail(OIDNX_ERR_UNSUPPORTED, "cannot bound CTAs per SM");
  }
}

// Sub-pixel decoder launch (even W and H): tiles of R rows x 128 outputs of
// one column parity; the upsampled source is read as a low-resolution halo
// box, the skip source (src1) from its column-parity split copy.  fp16
// layers, or fp32 layers (L.tf32: 3xTF32 products, every A stage followed by
// its A_lo stage).
oidnx_status build_tc_launch_subpixel(const DeviceLayer& L, const void* src0, Extent ext0,
                                      const void* src1, Extent ext1, int W, int H, void* out,
                                      int out_pitch, int* status, TcConvLaunch* T) {
  const int N = L.N;
  int R = 8;
  while (R > 2 && R * N > 256) R /= 2;
  if (2 * R * N > 512) return fail(OIDNX_ERR_UNSUPPORTED, "accumulators exceed tensor memory");
  const int tiles_x = 2 * ((W + 2 * kTileM - 1) / (2 * kTileM));
  while (R > 2 && static_cast<long>(tiles_x) * ((H + R - 1) / R) < num_sms()) R /= 2;
  uint32_t tmem_cols = 32;
  while (tmem_cols < static_cast<uint32_t>(2 * R * N)) tmem_cols *= 2;
  TcConvParams& p = T->p;
  std::memset(&p, 0, sizeof(p));
  T->kind = L.tf32 ? kTcSubpixel32 : kTcSubpixel;
  p.weights = static_cast<const __half*>(L.wsub);
  p.bias = L.bias;
  p.out = out;
  p.pitch = out_pitch;
  p.status = status;
  p.W = W;
  p.H = H;
  p.N = N;
  p.KB0 = L.KB0;
  p.KB1 = L.KB1;
  p.R = R;
  p.mode = kEpiRelu;
  p.upsample0 = 1;
  p.out_c4 = round_up(L.cout, 4) / 4;
  p.tiles_x = tiles_x;
  p.tiles_y = (H + R - 1) / R;
  p.tmem_cols = tmem_cols;
  p.up_pair = 1;
  p.a_tx = static_cast<uint32_t>((R / 2 + 2) * 2 * kHaloW * kChunkBytes);    // low-res box
  p.st_tx = static_cast<uint32_t>((R + 2) * 2 * kHaloW * kChunkBytes);       // skip plane box
  p.b_tx = static_cast<uint32_t>(L.sub_ub);                                  // 512 N (tf32 1024 N)
  p.b_tx2 = static_cast<uint32_t>((L.tf32 ? 12 : 6) * N * kChunkBytes);      // 96 N (tf32 192 N)
  p.a_stage = static_cast<uint32_t>(round_up_sz(std::max(p.a_tx, p.st_tx), 1024));
  p.b_stage = static_cast<uint32_t>(round_up_sz(std::max(p.b_tx / 2, 2 * p.b_tx2), 1024));
  p.st_stage = 0;
  const int items = L.KB0 + 2 * L.KB1;
  const size_t max_smem = 227 * 1024;
  const size_t fixed = 128 + static_cast<size_t>((N + 31) / 32) * 32 * 4 + 256;
  // resident: one column parity's half of every upsampled block + the skip blocks
  const size_t wres = static_cast<size_t>(L.KB0) * (L.sub_ub / 2) +
                      (L.sub_bytes - static_cast<size_t>(L.KB0) * L.sub_ub);
  const size_t wbytes = round_up_sz(wres, 1024);
  const int min_stages = std::max(2, std::min(items, 4));
  const size_t a_mul = L.tf32 ? 2 : 1;  // A (and A_lo) stages
  size_t smem;
  // resident weights: pairs of upsampled K blocks per item (one wait and one
  // commit per pair) when at least three stages of the wider box still fit
  const uint32_t a_tx_pair = static_cast<uint32_t>((R / 2 + 2) * 4 * kHaloW * kChunkBytes);
  const uint32_t a_stage_pair = static_cast<uint32_t>(round_up_sz(std::max(a_tx_pair, p.st_tx), 1024));
  if (L.KB0 >= 2 && fixed + wbytes + 3 * a_mul * a_stage_pair <= max_smem) {
    p.up_pair = 2;
    p.a_tx = a_tx_pair;
    p.a_stage = a_stage_pair;
  }
  // resident weights only with at least four stages beside them; otherwise
  // streaming them (one K block per stage) keeps a deeper ring, which
  // measured faster (dec_conv2a: 3 resident stages 59.4 us, 5 streamed 57.1)
  if (fixed + wbytes + min_stages * a_mul * p.a_stage <= max_smem) {
    p.resident = 1;
    p.wres_bytes = static_cast<uint32_t>(wres);  // bytes loaded; the layout rounds up to 1 KB
    p.S = static_cast<int>(std::min<size_t>(8, (max_smem - fixed - wbytes) / (a_mul * p.a_stage)));
    smem = fixed + wbytes + p.S * a_mul * p.a_stage;
  } else {
    // streamed weights: each stage holds one upsampled K block's weights,
    // so an item is one K block
    if (p.up_pair != 1) {
      p.up_pair = 1;
      p.a_tx = static_cast<uint32_t>((R / 2 + 2) * 2 * kHaloW * kChunkBytes);
      p.a_stage = static_cast<uint32_t>(round_up_sz(std::max(p.a_tx, p.st_tx), 1024));
    }
    p.resident = 0;
    const size_t stage = a_mul * p.a_stage + p.b_stage;
    p.S = static_cast<int>(std::min<size_t>(8, (max_smem - fixed) / stage));
    if (p.S < 2) return fail(OIDNX_ERR_UNSUPPORTED, "conv stage does not fit shared memory");
    smem = fixed + p.S * stage;
  }
  int blocks = 0;
  OIDNX_TRY(bound_ctas_per_sm(&smem, tmem_cols, &blocks));
  T->smem = smem;
  const long tiles = static_cast<long>(p.tiles_x) * p.tiles_y;
  long grid = std::min<long>(tiles, static_cast<long>(num_sms()) * blocks);
  // an even grid keeps each CTA on one column parity (tiles alternate parity)
  if (grid > 1 && grid % 2) --grid;
  T->grid = dim3(static_cast<unsigned>(grid), 1, 1);
  // (CTAs that keep one column parity's weights resident stay on their
  // parity: no split for them)
  plan_tail(&p, grid, 2, !p.resident);
  // 16-byte chunks per pixel of each source: 8 halves, or 4 floats
  auto chunks = [&](int c) { return L.tf32 ? round_up(c, 4) / 4 : round_up(c, 16) / 8; };
  const int c8_0 = chunks(L.c0);
  const int c8_1 = chunks(L.c1);
  OIDNX_TRY(encode_act_map(&T->map0, src0, ext0.w, ext0.pitch, ext0.h, c8_0, kHaloW, R / 2 + 2,
                           true, &p.xs0, 2 * p.up_pair));
  OIDNX_TRY(encode_split_map(&T->map1, src1, W, ext1.pitch, H, c8_1, kHaloW, R + 2, &p.xs1));
  return ok();
}

// Whether a decoder with conv extent (W, H) and low-resolution source ext0
// runs in sub-pixel mode (then its skip source must be the split copy).
bool use_subpixel(int W, int H, Extent ext0) {
  return W % 2 == 0 && H % 2 == 0 && ext0.w * 2 == W && ext0.h * 2 == H;
}

// src0/src1: sources with their extents (pitch included); (W, H): conv
// extent; out: destination with row pitch out_pitch.  fp16 layers, or fp32
// layers (L.tf32) whose products are formed as three tf32 MMAs.
oidnx_status build_tc_launch(const DeviceLayer& L, int kind, const void* src0, Extent ext0,
                             const void* src1, Extent ext1, int W, int H, void* out,
                             int out_pitch, int* status, TcConvLaunch* T, bool subpixel = false,
                             void* out_split = nullptr, int out_split_pitch = 0) {
  if (kind == kDecoder && subpixel && L.wsub)
    return build_tc_launch_subpixel(L, src0, ext0, src1, ext1, W, H, out, out_pitch, status, T);
  const bool up = kind == kDecoder;
  T->kind = up ? (L.tf32 ? kTcExpand32 : kTcExpand) : (L.tf32 ? kTcPlain32 : kTcPlain);
  const int N = L.N;
  const int minR = (kind == kPool || kind == kDecoder) ? 2 : 1;
  // Two accumulator sets of R x N fp32 columns must fit the 512 TMEM columns.
  int R = 8;
  while (R > minR && R * N > 256) R /= 2;
  if (2 * R * N > 512) return fail(OIDNX_ERR_UNSUPPORTED, "accumulators exceed tensor memory");
  const int tiles_x = (W + kTileM - 1) / kTileM;
  // Fewer tiles than SMs: the tile height that finishes first, by rounds of
  // tiles x estimated cycles per tile (K blocks x (~600 cycles of per-item
  // synchronisation + the MMAs of the cost model: max(45.7, N / 2, operand
  // bytes / 128 B per clock) each)).  dec_conv4b at 1080p: 2 rows, one
  // round of 136 tiles, not 1 row in two rounds (14.4 against 15.0 us).
  if (static_cast<long>(tiles_x) * ((H + R - 1) / R) < num_sms()) {
    auto mma = [](int n) { return std::max(45.7, std::max(n / 2.0, (4096.0 + 32.0 * n) / 128.0)); };
    const int G = std::min(3, 256 / N);
    double best = 0.0;
    int best_r = R;
    for (int r = R; r >= minR; r /= 2) {
      double kx = 0.0;  // cycles of the MMAs of one kx over the halo rows
      for (int h = 0; h < r + 2; ++h) {
        const int lo = std::max(0, h - 2), hi = std::min(r - 1, h);
        for (int c = lo; c <= hi; c += G) kx += mma(N * (std::min(hi, c + G - 1) - c + 1));
      }
      const long tiles = static_cast<long>(tiles_x) * ((H + r - 1) / r);
      const double est = static_cast<double>((tiles + num_sms() - 1) / num_sms()) *
                         (L.KB0 + L.KB1) * (600.0 + 3.0 * kx);
      if (r == R || est < best) {
        best = est;
        best_r = r;
      }
      if (r == 1) break;
    }
    R = best_r;
  }
  uint32_t tmem_cols = 32;
  while (tmem_cols < static_cast<uint32_t>(2 * R * N)) tmem_cols *= 2;

  TcConvParams& p = T->p;
  std::memset(&p, 0, sizeof(p));
  p.weights = static_cast<const __half*>(L.wtc);
  p.bias = L.bias;
  p.out = out;
  p.pitch = out_pitch;
  p.status = status;
  p.W = W;
  p.H = H;
  p.N = N;
  p.KB0 = L.KB0;
  p.KB1 = L.KB1;
  p.R = R;
  p.mode = kind == kPool ? kEpiReluPool : (kind == kFinal ? kEpiFinal : kEpiRelu);
  p.upsample0 = up ? 1 : 0;
  p.out_c4 = round_up(L.cout, 4) / 4;
  p.out_split = kind == kPool ? out_split : nullptr;
  p.split_pitch = out_split_pitch;
  p.tiles_x = tiles_x;
  p.tiles_y = (H + R - 1) / R;
  p.tmem_cols = tmem_cols;
  p.a_tx = static_cast<uint32_t>((R + 2) * 2 * kHaloW * kChunkBytes);
  // a K block of B: 9 taps x 2 chunks x N rows of 16 bytes (tf32: hi, then lo)
  p.b_tx = static_cast<uint32_t>((L.tf32 ? 2 : 1) * 9 * 2 * N * kChunkBytes);
  p.st_tx = up ? static_cast<uint32_t>((R / 2 + 2) * 2 * kLowW * kChunkBytes) : 0u;
  p.a_stage = static_cast<uint32_t>(round_up_sz(p.a_tx, 1024));
  p.b_stage = static_cast<uint32_t>(round_up_sz(p.b_tx, 1024));
  p.st_stage = static_cast<uint32_t>(round_up_sz(p.st_tx, 1024));
  const int KB = L.KB0 + L.KB1;
  const size_t max_smem = 227 * 1024;
  // alignment slack (128 B) + bias + barriers
  const size_t fixed = 128 + static_cast<size_t>((N + 31) / 32) * 32 * 4 + 256;
  const size_t wbytes = static_cast<size_t>(KB) * p.b_stage;
  // per stage: A (and for tf32 its A_lo split), low-resolution staging
  const size_t a_st = static_cast<size_t>(p.a_stage) * (L.tf32 ? 2 : 1) + p.st_stage;
  // resident weights need up to four stages beside them (see the sub-pixel
  // builder); with fewer the weights are streamed
  const int min_stages = std::min(KB, 4) < 2 ? 2 : std::min(KB, 4);
  size_t smem;
  if (fixed + wbytes + min_stages * a_st <= max_smem) {
    p.resident = 1;
    p.wres_bytes = static_cast<uint32_t>(wbytes);
    p.S = static_cast<int>(std::min<size_t>(8, (max_smem - fixed - wbytes) / a_st));
    smem = fixed + wbytes + p.S * a_st;
  } else {
    p.resident = 0;
    const size_t stage = a_st + p.b_stage;
    p.S = static_cast<int>(std::min<size_t>(8, (max_smem - fixed) / stage));
    if (p.S < 2) return fail(OIDNX_ERR_UNSUPPORTED, "conv stage does not fit shared memory");
    smem = fixed + p.S * stage;
  }
  OIDNX_TRY(ensure_smem_limit(kFamilyTc));
  // CTAs resident on one SM must share the 512 TMEM columns without waiting:
  // pad the shared-memory request until the occupancy allows no more.
  const int allowed = static_cast<int>(512 / tmem_cols);
  int blocks = 0;
  for (;;) {
    cudaError_t e = conv_tc_occupancy(smem, &blocks);
    if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "occupancy: %s", cudaGetErrorString(e));
    if (blocks <= allowed) break;
    smem += 4096;
    if (smem > max_smem) return fail(OIDNX_ERR_UNSUPPORTED, "cannot bound CTAs per SM");
  }
  T->smem = smem;
  const long tiles = static_cast<long>(p.tiles_x) * p.tiles_y;
  T->grid = dim3(static_cast<unsigned>(std::min<long>(tiles, static_cast<long>(num_sms()) * blocks)), 1, 1);
  plan_tail(&p, T->grid.x, minR, true);

  // 16-byte chunks per pixel of each source: 8 halves, or 4 floats
  auto chunks = [&](int c) { return L.tf32 ? round_up(c, 4) / 4 : round_up(c, 16) / 8; };
  const int c8_0 = chunks(L.c0);
  OIDNX_TRY(encode_act_map(&T->map0, src0, ext0.w, ext0.pitch, ext0.h, c8_0,
                           up ? kLowW : kHaloW, up ? R / 2 + 2 : R + 2, true, &p.xs0));
  if (L.KB1 > 0) {
    const int c8_1 = chunks(L.c1);
    OIDNX_TRY(encode_act_map(&T->map1, src1, ext1.w, ext1.pitch, ext1.h, c8_1, kHaloW, R + 2, true,
                             &p.xs1));
  } else {
    T->map1 = T->map0;
    p.xs1 = p.xs0;
  }
  return ok();
}

// Layer pairs that run as one fused kernel when the filter allows it (fp16
// storage, "fuseLayers"): the first layer's output is never stored.
struct PairDef {
  int first, mode;
  const char* name;
};
const PairDef kPairs[2] = {{0, kPairPool, "enc_conv0+enc_conv1"},
                           {14, kPairFinal, "dec_conv1b+dec_conv0"}};

bool pair_fusable(const oidnx_filter* f, const PairDef& d) {
  if (!f->fuse || f->precision != OIDNX_PRECISION_FP16) return false;
  const DeviceLayer& a = f->layers[d.first];
  const DeviceLayer& b = f->layers[d.first + 1];
  if (a.c1 != 0 || a.cout != 32 || a.KB0 < 1 || a.KB0 > 4 || b.c0 != 32 || b.c1 != 0) return false;
  return d.mode == kPairFinal ? b.cout == 3 && b.wfold != nullptr : b.cout == 32;
}

// Launch of a fused pair over a W x H conv extent: conv 1 reads `src`
// (fp16, one source), conv 2 writes `out` (final: f32 [H][W][4]; pool:
// fp16 pooled with pitch out_pitch, plus the optional split copy).
oidnx_status build_pair_launch(const DeviceLayer& A, const DeviceLayer& B, int mode,
                               const void* src, Extent ext, int W, int H, void* out,
                               int out_pitch, void* out_split, int out_split_pitch, int* status,
                               PairConvLaunch* T) {
  T->mode = mode;
  PairConvParams& p = T->p;
  std::memset(&p, 0, sizeof(p));
  p.w1 = static_cast<const __half*>(A.wtc);
  p.w2 = static_cast<const __half*>(mode == kPairFinal ? B.wfold : B.wtc);
  p.bias1 = A.bias;
  p.bias2 = B.bias;
  p.out = out;
  p.out_split = out_split;
  p.status = status;
  p.W = W;
  p.H = H;
  p.KB1 = A.KB0;
  p.C8 = 2 * A.KB0;
  p.row_unit = mode == kPairPool ? 2 : 1;
  p.pitch = out_pitch;
  p.split_pitch = out_split ? out_split_pitch : 0;
  // Strips of sw output columns (even, at most kPairSpan); the last strip's
  // lanes reach kPairSpan columns past its start, which must cover every
  // column to be written (pooled: the zero padding of both pitched copies).
  const int need = mode == kPairPool ? 2 * std::max(p.pitch, p.split_pitch) : W;
  for (int n = std::max(1, (W + kPairSpan - 1) / kPairSpan);; ++n) {
    const int sw = round_up((W + n - 1) / n, 2);
    if (sw <= kPairSpan && (n - 1) * sw + kPairSpan >= need) {
      p.strips = n;
      p.sw = sw;
      break;
    }
  }
  p.units = p.strips * ((H + p.row_unit - 1) / p.row_unit);
  // one stage: the kPairBatch input rows of one batch
  p.stage_tx = static_cast<uint32_t>(kPairBatch * kHaloW * p.C8 * kChunkBytes);
  p.stage_bytes = static_cast<uint32_t>(round_up_sz(p.stage_tx, 1024));
  p.w1_bytes = static_cast<uint32_t>(A.KB0 * 9 * 2 * 32 * kChunkBytes);
  p.w2_bytes = static_cast<uint32_t>(mode == kPairFinal ? B.fold_bytes : 2 * 9 * 2 * 32 * kChunkBytes);
  const size_t mid_row = static_cast<size_t>(4) * (mode == kPairFinal ? kTileM : kTileM + 8) * kChunkBytes;
  const size_t xb = mode == kPairFinal ? static_cast<size_t>(4) * kTileM * 16 : 0;
  // alignment slack, weights, conv-1 rows, exchange, bias, 17 barriers + 2
  // per stage, the TMEM address
  const size_t fixed = 1024 + p.w1_bytes + round_up_sz(p.w2_bytes, 1024) + kPairMid * mid_row + xb +
                       64 * 4 + 17 * 8 + 16;
  const size_t max_smem = 227 * 1024;
  // the MMA issuer holds one batch of input rows while the next one loads
  if (fixed + 2 * (16 + static_cast<size_t>(p.stage_bytes)) > max_smem)
    return fail(OIDNX_ERR_UNSUPPORTED, "fused conv does not fit shared memory");
  p.S = static_cast<int>(std::min<size_t>(4, (max_smem - fixed) / (16 + p.stage_bytes)));
  size_t smem = fixed + 16 * static_cast<size_t>(p.S) + static_cast<size_t>(p.S) * p.stage_bytes;
  OIDNX_TRY(ensure_smem_limit(kFamilyPair));
  // one CTA per SM: it allocates all 512 TMEM columns
  for (;;) {
    int blocks = 0;
    cudaError_t e = conv_pair_occupancy(mode, smem, &blocks);
    if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "occupancy: %s", cudaGetErrorString(e));
    if (blocks <= 1) break;
    smem += 4096;
    if (smem > max_smem) return fail(OIDNX_ERR_UNSUPPORTED, "cannot bound CTAs per SM");
  }
  T->smem = smem;
  T->grid = dim3(static_cast<unsigned>(std::min(p.units, num_sms())), 1, 1);
  return encode_act_map(&T->map, src, ext.w, ext.pitch, ext.h, p.C8, kHaloW, kPairBatch, true, &p.xs,
                        p.C8);
}

// The final conv with kx folded (fp16, 32 -> 3): tiles of kFinalRows rows x
// kFinalSpan pixels over the W x H extent, writing the network output to
// `net` (may be null when the output pass runs in the epilogue).
bool final_foldable(const DeviceLayer& L) {
  return L.wfold && L.cin == 32 && L.cout == 3 && L.c1 == 0;
}

oidnx_status build_final_launch(const DeviceLayer& L, const void* src, Extent ext, int W, int H,
                                void* net, int* status, FinalConvLaunch* T) {
  T->outpass = 0;
  T->tf32 = L.tf32 ? 1 : 0;
  FinalConvParams& p = T->p;
  std::memset(&p, 0, sizeof(p));
  p.w = static_cast<const __half*>(L.wfold);
  p.bias = L.bias;
  p.net = static_cast<float4*>(net);
  p.status = status;
  p.W = W;
  p.H = H;
  p.tiles_x = (W + kFinalSpan - 1) / kFinalSpan;
  p.tiles_y = (H + kFinalRows - 1) / kFinalRows;
  p.stage_tx = static_cast<uint32_t>((kFinalRows + 2) * 2 * kHaloW * kChunkBytes);
  p.stage_bytes = static_cast<uint32_t>(round_up_sz(p.stage_tx, 1024));
  // alignment slack, weights (fp16: 2 K blocks; tf32: 4 K blocks, hi and
  // lo), boundary exchange (4 sub x 2 x 4 quarters x 2 rows x 3 float4),
  // bias, barriers (14 + 2 per stage, 3 for tf32)
  const size_t wbytes = static_cast<size_t>(L.tf32 ? 4 * 2 : 2) * 2 * 3 * 16 * kChunkBytes;
  const size_t fixed = 1024 + wbytes + 4 * 2 * 4 * 2 * 3 * 16 + 16 * 4 + 14 * 8 + 16;
  // per stage: the halo box (tf32: and its A_lo split) and its barriers
  const size_t per_stage = static_cast<size_t>(p.stage_bytes) * (L.tf32 ? 2 : 1) + 24;
  const size_t max_smem = 227 * 1024;
  p.S = static_cast<int>(std::min<size_t>(4, (max_smem - fixed) / per_stage));
  if (p.S < 2) return fail(OIDNX_ERR_UNSUPPORTED, "final conv stages do not fit");
  T->smem = fixed + static_cast<size_t>(p.S) * per_stage;
  OIDNX_TRY(ensure_smem_limit(kFamilyFinal));
  const long tiles = static_cast<long>(p.tiles_x) * p.tiles_y;
  T->grid = dim3(static_cast<unsigned>(std::min<long>(tiles, num_sms())), 1, 1);
  return encode_act_map(&T->map, src, ext.w, ext.pitch, ext.h,
                        act_chunks(L.tf32 ? OIDNX_PRECISION_FP32 : OIDNX_PRECISION_FP16, L.cin), kHaloW,
                        kFinalRows + 2, true, &p.xs);
}

// dec_conv1b and dec_conv0 as one kernel ("fuseTail", fp16, activations not
// kept): dec_conv1b's 32-channel map stays in tensor memory.  Stacked tiles
// run it once per tile.  Not with the fused pairs ("fuseLayers"), which take
// these layers.
bool tail_fusable(const oidnx_filter* f) {
  if (!f->fuse_tail || f->fuse || f->keep_acts || f->precision != OIDNX_PRECISION_FP16)
    return false;
  const DeviceLayer& a = f->layers[kLayers - 2];
  return a.c1 == 0 && a.cout == 32 && a.N == 32 && a.KB0 >= 1 && a.KB0 <= 4 &&
         final_foldable(f->layers[kLayers - 1]);
}

// Launch of the fused last two layers over a W x H extent: A = dec_conv1b
// reading `src` (fp16, extent ext), B = dec_conv0 writing `net` (f32
// [H][W][4]; may be null when the output pass runs in the epilogue).
oidnx_status build_tail_launch(const DeviceLayer& A, const DeviceLayer& B, const void* src, Extent ext,
                               int W, int H, void* net, int* status, TailConvLaunch* T) {
  T->outpass = 0;
  TailConvParams& p = T->p;
  std::memset(&p, 0, sizeof(p));
  p.w1 = static_cast<const __half*>(A.wtc);
  p.w2 = static_cast<const __half*>(B.wfold);
  p.bias1 = A.bias;
  p.bias2 = B.bias;
  p.net = static_cast<float4*>(net);
  p.status = status;
  p.W = W;
  p.H = H;
  p.KB1 = A.KB0;
  p.tiles_x = (W + kFinalSpan - 1) / kFinalSpan;
  p.tiles_y = (H + kTailOut - 1) / kTailOut;
  // one stage: one K block's halo box, kTailMid + 2 rows x kHaloW pixels x 2
  // chunks (kTailMid rows when six conv-1 rows are computed)
  p.stage_tx = static_cast<uint32_t>((kTailMid + 2) * 2 * kHaloW * kChunkBytes);
  p.stage_tx8 = static_cast<uint32_t>(kTailMid * 2 * kHaloW * kChunkBytes);
  p.stage_bytes = static_cast<uint32_t>(round_up_sz(p.stage_tx, 1024));
  // alignment slack, weights of both convs, boundary exchange (2 sub x 2 x 4
  // quarters x 3 rows x 3 float4), both biases, 14 barriers + 2 per stage,
  // the TMEM address
  const size_t fixed = 128 + static_cast<size_t>(p.KB1) * 3 * 2 * 3 * 32 * kChunkBytes + B.fold_bytes +
                       2 * 2 * 4 * (kTailOut / 2) * 3 * 16 + (32 + 16) * 4 + 14 * 8 + 16;
  const size_t per_stage = static_cast<size_t>(p.stage_bytes) + 16;
  const size_t max_smem = 227 * 1024;
  if (fixed + 2 * per_stage > max_smem) return fail(OIDNX_ERR_UNSUPPORTED, "tail conv does not fit");
  p.S = static_cast<int>(std::min<size_t>(4, (max_smem - fixed) / per_stage));
  // one CTA per SM (it allocates all 512 TMEM columns): more than half the
  // shared memory of an SM
  T->smem = std::max<size_t>(fixed + static_cast<size_t>(p.S) * per_stage, 120 * 1024);
  OIDNX_TRY(ensure_smem_limit(kFamilyTail));
  // Groups of `run` row tiles of one strip, taken round robin: the run that
  // gives the busiest CTA the fewest conv-1 rows (rounds of groups x
  // (6 run + 2)), the shortest among equals (the frame is then read closest
  // to the walk's order).
  const long sms = num_sms();
  long best = LONG_MAX;
  for (int run = 1; run <= p.tiles_y; ++run) {
    const long groups = static_cast<long>((p.tiles_y + run - 1) / run) * p.tiles_x;
    const long cost = (groups + sms - 1) / sms * ((kTailMid - 2) * static_cast<long>(run) + 2);
    if (cost < best) {
      best = cost;
      p.run = run;
      p.groups = static_cast<int>(groups);
    }
  }
  T->grid = dim3(static_cast<unsigned>(std::min<long>(p.groups, sms)), 1, 1);
  OIDNX_TRY(encode_act_map(&T->map8, src, ext.w, ext.pitch, ext.h, 2 * p.KB1, kHaloW, kTailMid, true,
                           &p.xs));
  return encode_act_map(&T->map10, src, ext.w, ext.pitch, ext.h, 2 * p.KB1, kHaloW, kTailMid + 2, true,
                        &p.xs);
}

// The input pass and enc_conv0 as one kernel ("fuseInput", off by default:
// inside the replayed graph it is not faster; fp16, frames run
// one tile at a time, activations not kept, the sub-pixel dec_conv1a
// reading the packed input's column-parity copy): the plain packed input is
// then neither written nor read.
bool head_fusable(const oidnx_filter* f) {
  if (!f->fuse_input || f->keep_acts || f->precision != OIDNX_PRECISION_FP16) return false;
  const DeviceLayer& L = f->layers[0];
  return L.c1 == 0 && L.KB0 == 1 && L.N == 32 && L.cout == 32 && L.wtc != nullptr;
}

// The head launch over a W x H tile: enc_conv0's weights and the value
// buffers; the tile's image fields are filled per tile when it is enqueued.
oidnx_status build_head_launch(const DeviceLayer& L, int W, int H, void* out, int pitch, void* split,
                               int split_pitch, int* status, HeadLaunch* T) {
  HeadParams& p = T->p;
  std::memset(&p, 0, sizeof(p));
  p.weights = static_cast<const __half*>(L.wtc);
  p.bias = L.bias;
  p.status = status;
  p.out = static_cast<__half*>(out);
  p.pitch = pitch;
  p.split = split;
  p.split_pitch = split_pitch;
  p.tw = W;
  p.th = H;
  p.tiles_x = (W + kTileM - 1) / kTileM;
  p.tiles_y = (H + kHeadRows - 1) / kHeadRows;
  // image stage: per image kHeadRows + 2 rows x 132 float4 pixels (three
  // boxes of 44); packed stage: kHeadRows + 2 halo rows x 2 halves
  // x 130 pixels x 16 bytes
  const size_t img_box = static_cast<size_t>(kHeadRows + 2) * 3 * 44 * 16;  // 132 pixels
  p.img_stage = static_cast<uint32_t>(3 * img_box);
  p.a_stage = static_cast<uint32_t>(round_up_sz((kHeadRows + 2) * 2 * (kTileM + 2) * kChunkBytes, 128));
  p.SI = 2;
  p.SA = 2;
  // alignment slack, stages, weights (one K block), bias, 6 barriers + 2
  // per stage, the TMEM address
  const size_t smem = 128 + static_cast<size_t>(p.SI) * p.img_stage + static_cast<size_t>(p.SA) * p.a_stage +
                      3 * 2 * 3 * 32 * kChunkBytes + 32 * 4 + (6 + 2 * p.SI + 2 * p.SA) * 8 + 16;
  if (smem > 227 * 1024) return fail(OIDNX_ERR_UNSUPPORTED, "input conv stages do not fit");
  // one CTA per SM (it allocates all 512 TMEM columns): more than half the
  // shared memory of an SM
  T->smem = std::max<size_t>(smem, 120 * 1024);
  OIDNX_TRY(ensure_smem_limit(kFamilyHead));
  const long tiles = static_cast<long>(p.tiles_x) * p.tiles_y;
  T->grid = dim3(static_cast<unsigned>(std::min<long>(tiles, num_sms())), 1, 1);
  return ok();
}

oidnx_status run_launch(const LayerLaunch& L, cudaStream_t s) {
  (void)cudaGetLastError();  // drop a stale, non-sticky error of an earlier call
  if (L.final) {
    cudaError_t e = launch_conv_final(L.fcl, s);
    if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "%s launch: %s", L.name, cudaGetErrorString(e));
    return ok();
  }
  if (L.tail) {
    cudaError_t e = launch_conv_tail(L.tlcl, s);
    if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "%s launch: %s", L.name, cudaGetErrorString(e));
    return ok();
  }
  if (L.pair) {
    cudaError_t e = launch_conv_pair(L.pcl, s);
    if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "%s launch: %s", L.name, cudaGetErrorString(e));
    return ok();
  }
  cudaError_t e = launch_conv_tc(L.tcl, s);
  if (e != cudaSuccess)
    return fail(OIDNX_ERR_CUDA, "%s launch: %s", kLayerNames[L.layer], cudaGetErrorString(e));
  return ok();
}

void destroy_plan(Plan* p) {
  if (!p) return;
  if (p->done) {
    cudaEventSynchronize(p->done);
    cudaEventDestroy(p->done);
  }
  cudaFree(p->arena);
  p->arena = nullptr;
}

// Tensor-core FLOPs one launch issues (2 M N K summed over its MMAs; tile
// rows and channels padded as the kernels run them): per tile, K blocks x
// taps x R rows x N x 128 pixels x K x 2, with 4 taps on the upsampled
// channels of a sub-pixel decoder, three passes for 3xTF32, and for the
// folded final conv 3 R rows of N = 16 (three kx taps) per K block.  The
// fused tail: conv 1 over the rows each tile computes (kTailMid in a
// group's first tile, else kTailMid - 2; 3 ky each) of N = 32 per
// K block and kx, conv 2 over kTailOut rows of N = 16 per K block and ky.
// 0 for fused pairs.
double mma_flop(const LayerLaunch& LL) {
  if (LL.pair) return 0;
  if (LL.tail) {
    const TailConvParams& p = LL.tlcl.p;
    const double T = static_cast<double>(p.tiles_x) * p.tiles_y;
    const double rows = (kTailMid - 2) * T + 2.0 * p.groups;  // 8 rows in a group's first tile
    return 128.0 * 16 * 2 * (rows * p.KB1 * 3 * 3 * 32 + T * 2 * 3 * kTailOut * 16);
  }
  if (LL.final) {  // 32 input channels: 2 K blocks of 16, or 4 of 8 x 3 tf32 passes
    const FinalConvParams& p = LL.fcl.p;
    return static_cast<double>(p.tiles_x) * p.tiles_y * 3 * kFinalRows * 16 * 128.0 * 32 * 2 *
           (LL.fcl.tf32 ? 3 : 1);
  }
  const TcConvParams& p = LL.tcl.p;
  const int kind = LL.tcl.kind;
  const bool tf = kind == kTcPlain32 || kind == kTcExpand32 || kind == kTcSubpixel32;
  const bool sp = kind == kTcSubpixel || kind == kTcSubpixel32;
  const double per_tap = static_cast<double>(p.R) * p.N * 128.0 * (tf ? 8 : 16) * 2 * (tf ? 3 : 1);
  const double taps = sp ? 4.0 * p.KB0 + 9.0 * p.KB1 : 9.0 * (p.KB0 + p.KB1);
  return static_cast<double>(p.tiles_x) * p.tiles_y * taps * per_tap;
}

// Shapes, liveness and arena placement of the network's values for a w x h
// input, shared by the plan cache and the allocation-free path.  Memory is
// reused by liveness, the rule of "nativeUNet.ts" (_createExecution): a
// value's memory is free again once its last reader has run.  Here every
// value is an interval in time (from the launch that writes it through its
// last reader) and in address; values are placed in the order they are
// written, each at the lowest offset where it overlaps, in address, no
// placed value that is still live when it is written.  io_external: the
// network input (rows of w pixels) and output are the caller's buffers and
// are not placed; keep: nothing is reused.  Fixed-size arrays only: no
// allocation.
struct ValueLayout {
  Extent lvl[5];
  Extent ext[V_COUNT];
  int ch[V_COUNT];
  int last_use[V_COUNT];
  bool split_on[4];       // kSplits[i] in use (its decoder runs in sub-pixel mode)
  bool fused[2];          // kPairs[i] runs as one fused kernel
  bool tail;              // the last two layers run as one kernel
  bool stored[kLayers];   // layer l's output is stored (not fused away)
  size_t off[V_COUNT];    // arena offset of each placed value
  size_t bytes[V_COUNT];  // its bytes; 0 if not placed
  size_t total;           // arena bytes
};

void layout_values(const oidnx_filter* f, int w, int h, bool io_external, bool keep,
                   ValueLayout* V, int stack = 1) {
  std::memset(V, 0, sizeof(*V));
  V->lvl[0] = {w, stack > 1 ? stack * (h + kStackGap) : h, w};
  for (int l = 1; l < 5; ++l) {
    const int lw = (V->lvl[l - 1].w + 1) / 2;
    V->lvl[l] = {lw, (V->lvl[l - 1].h + 1) / 2, lw};
  }
  V->ext[V_IN] = io_external ? V->lvl[0] : value_extent(f->precision, V->lvl[0], false);
  V->ch[V_IN] = f->in_channels;
  for (int l = 0; l < kLayers; ++l) {
    const LayerDef& d = kDefs[l];
    V->ext[d.dst] = value_extent(f->precision, V->lvl[d.kind == kPool ? d.level + 1 : d.level],
                                 d.dst == V_OUT);
    V->ch[d.dst] = f->layers[l].cout;
  }
  for (int v = 0; v < V_COUNT; ++v) V->last_use[v] = -1;
  for (int l = 0; l < kLayers; ++l) {
    V->last_use[kDefs[l].src0] = l;
    if (kDefs[l].src1 >= 0) V->last_use[kDefs[l].src1] = l;
  }
  V->last_use[V_OUT] = kLayers;
  for (int i = 0; i < 4; ++i) {
    const SplitCopy& sc = kSplits[i];
    const LayerDef& d = kDefs[sc.consumer];
    V->split_on[i] = f->subpixel && use_subpixel(V->lvl[d.level].w, V->lvl[d.level].h, V->ext[d.src0]);
    V->ext[sc.split] = V->ext[sc.base];
    V->ext[sc.split].pitch = split_pitch(V->ext[sc.base].w);
    V->ch[sc.split] = V->ch[sc.base];
    V->last_use[sc.split] = sc.consumer;
  }
  // a fused pair's intermediate map is never stored
  for (int l = 0; l < kLayers; ++l) V->stored[l] = true;
  for (int i = 0; i < 2; ++i) {
    V->fused[i] = pair_fusable(f, kPairs[i]);
    if (V->fused[i]) V->stored[kPairs[i].first] = false;
  }
  V->tail = !keep && tail_fusable(f);
  if (V->tail) V->stored[kLayers - 2] = false;
  struct Placed {
    size_t lo, hi;  // byte range (1 KB multiples)
    int until;      // index of the last launch that reads it
  } placed[V_COUNT];
  int nplaced = 0;
  // v is written by launch `index`
  auto place = [&](int v, int index) {
    const size_t need = act_bytes(f->precision, V->ext[v], V->ch[v], v == V_OUT);
    const size_t span = round_up_sz(need, 1024);
    // lowest offset clear of every value still read at or after `index`: a
    // candidate that overlaps one moves past its end (no clear offset lies
    // in between), until none overlaps
    size_t off = 0;
    for (bool moved = true; moved;) {
      moved = false;
      for (int i = 0; i < nplaced; ++i)
        if (placed[i].until >= index && placed[i].lo < off + span && off < placed[i].hi) {
          off = placed[i].hi;
          moved = true;
        }
    }
    placed[nplaced++] = {off, off + span, keep ? INT_MAX : V->last_use[v]};
    V->off[v] = off;
    V->bytes[v] = need;
    V->total = std::max(V->total, off + span);
  };
  if (!io_external) place(V_IN, -1);
  if (V->split_on[0]) place(V_INS, -1);
  for (int l = 0; l < kLayers; ++l) {
    // a fused pair reads the first layer's inputs while it writes the second
    // layer's outputs: place those as if the first layer wrote them
    const int at = l > 0 && !V->stored[l - 1] ? l - 1 : l;
    if (V->stored[l] && !(io_external && kDefs[l].dst == V_OUT)) place(kDefs[l].dst, at);
    for (int i = 0; i < 4; ++i)
      if (V->split_on[i] && kSplits[i].producer == l) place(kSplits[i].split, at);
  }
}

// The launches of one network pass over the values of V, in order, with
// device pointers from ptr(value); emit(LayerLaunch&) receives each launch
// (with its logical FLOPs and algorithmic bytes) and returns a status.
// stack_rows: tile rows of a stacked layout (0: one image): every conv
// gets its level's gap period, the final conv is left to the caller (one
// launch per tile), and FLOPs and bytes count the tiles' rows only.
// Launch k of a network pass (k = layer index + 1; the input pass is 0)
// walks its tiles in reverse when k is odd: each layer then starts on the
// rows its input's producer wrote last, which are still in L2.
int walk_reverse(int layer) { return (layer + 1) & 1; }

template <class Ptr, class Emit>
oidnx_status build_network_launches(const oidnx_filter* f, const ValueLayout& V, Ptr ptr, Emit emit,
                                    int stack_rows = 0) {
  const int bpe = f->precision == OIDNX_PRECISION_FP16 ? 2 : 4;
  // share of the stacked rows that are tile rows (the same at every level)
  const double tile_share =
      stack_rows ? static_cast<double>(stack_rows) / (stack_rows + kStackGap) : 1.0;
  auto logical_bytes = [&](int v) {
    return static_cast<double>(V.ext[v].w) * V.ext[v].h * V.ch[v] * bpe * tile_share;
  };
  for (int l = 0; l < kLayers; ++l) {
    const LayerDef& d = kDefs[l];
    const DeviceLayer& L = f->layers[l];
    LayerLaunch LL;
    std::memset(&LL, 0, sizeof(LL));
    LL.layer = l;
    LL.name = kLayerNames[l];
    const Extent conv = V.lvl[d.level];
    const double px = static_cast<double>(conv.w) * conv.h * tile_share;
    const int pi = l == kPairs[0].first ? 0 : (l == kPairs[1].first ? 1 : -1);
    if (pi >= 0 && V.fused[pi]) {
      const LayerDef& d2 = kDefs[l + 1];
      const DeviceLayer& L2 = f->layers[l + 1];
      void* out_split = nullptr;
      int out_split_pitch = 0;
      for (int i = 0; i < 4; ++i)
        if (V.split_on[i] && kSplits[i].producer == l + 1) {
          out_split = ptr(kSplits[i].split);
          out_split_pitch = V.ext[kSplits[i].split].pitch;
        }
      LL.pair = 1;
      LL.name = kPairs[pi].name;
      OIDNX_TRY(build_pair_launch(L, L2, kPairs[pi].mode, ptr(d.src0), V.ext[d.src0], conv.w, conv.h,
                                  ptr(d2.dst), V.ext[d2.dst].pitch, out_split, out_split_pitch,
                                  f->status, &LL.pcl));
      LL.flop = 2.0 * 9.0 * (L.cin * L.cout + L2.cin * L2.cout) * px;
      const Extent oe = V.ext[d2.dst];
      LL.bytes = logical_bytes(d.src0) +
                 (d2.kind == kFinal ? static_cast<double>(oe.w) * oe.h * 16 : logical_bytes(d2.dst)) +
                 static_cast<double>(L.weight_bytes + L2.weight_bytes);
      OIDNX_TRY(emit(LL));
      ++l;
      continue;
    }
    if (l == kLayers - 2 && V.tail) {
      if (stack_rows) break;  // one launch per tile, built by the caller
      const LayerDef& d2 = kDefs[l + 1];
      const DeviceLayer& L2 = f->layers[l + 1];
      LL.tail = 1;
      LL.name = "dec_conv1b+dec_conv0";
      OIDNX_TRY(build_tail_launch(L, L2, ptr(d.src0), V.ext[d.src0], conv.w, conv.h, ptr(d2.dst),
                                  f->status, &LL.tlcl));
      LL.tlcl.p.l2_first = 1;  // one image: evict-first activation loads
      LL.flop = 2.0 * 9.0 * (L.cin * L.cout + L2.cin * L2.cout) * px;
      LL.bytes = logical_bytes(d.src0) + static_cast<double>(V.ext[d2.dst].w) * V.ext[d2.dst].h * 16 +
                 static_cast<double>(L.weight_bytes + L2.weight_bytes);
      OIDNX_TRY(emit(LL));
      ++l;
      continue;
    }
    if (d.kind == kFinal && final_foldable(L)) {
      if (stack_rows) continue;  // one launch per tile, built by the caller
      LL.final = 1;
      OIDNX_TRY(build_final_launch(L, ptr(d.src0), V.ext[d.src0], conv.w, conv.h, ptr(d.dst),
                                   f->status, &LL.fcl));
      LL.fcl.p.reverse = walk_reverse(l);
      LL.fcl.p.l2_first = 1;  // one image: evict-first activation loads
      LL.flop = 2.0 * 9.0 * L.cin * L.cout * px;
      LL.bytes = logical_bytes(d.src0) + static_cast<double>(V.ext[d.dst].w) * V.ext[d.dst].h * 16 +
                 static_cast<double>(L.weight_bytes);
      OIDNX_TRY(emit(LL));
      continue;
    }
    const void* s1 = d.src1 >= 0 ? ptr(d.src1) : nullptr;
    Extent e1 = d.src1 >= 0 ? V.ext[d.src1] : Extent{0, 0, 0};
    bool subpixel = false;
    void* out_split = nullptr;
    int out_split_pitch = 0;
    for (int i = 0; i < 4; ++i) {
      if (!V.split_on[i]) continue;
      if (kSplits[i].consumer == l) {
        subpixel = true;
        s1 = ptr(kSplits[i].split);
        e1 = V.ext[kSplits[i].split];
      }
      if (kSplits[i].producer == l) {
        out_split = ptr(kSplits[i].split);
        out_split_pitch = V.ext[kSplits[i].split].pitch;
      }
    }
    OIDNX_TRY(build_tc_launch(L, d.kind, ptr(d.src0), V.ext[d.src0], s1, e1, conv.w, conv.h,
                              ptr(d.dst), V.ext[d.dst].pitch, f->status, &LL.tcl, subpixel,
                              out_split, out_split_pitch));
    LL.tcl.any_shape = f->shape_kernels ? 0 : 1;
    if (stack_rows) {
      LL.tcl.p.period = (stack_rows + kStackGap) >> d.level;
      LL.tcl.p.rows = stack_rows >> d.level;
    }
    // Evict-first activation loads pay in one image, not in a stack of tiles,
    // whose neighbouring tiles' shared halo rows they pushed out to DRAM
    // (3840x2160 in 15 tiles: 3.25 ms with them, 2.86 without).
    LL.tcl.p.l2_first = stack_rows ? 0 : 1;
    LL.tcl.p.reverse = walk_reverse(l);
    LL.flop = 2.0 * 9.0 * L.cin * L.cout * px;
    const Extent oe = V.ext[d.dst];
    const double out_bytes = (d.kind == kFinal ? static_cast<double>(oe.w) * oe.h * 16
                                               : static_cast<double>(oe.w) * oe.h * L.cout * bpe) *
                             tile_share;
    LL.bytes = logical_bytes(d.src0) + (d.src1 >= 0 ? logical_bytes(d.src1) : 0.0) + out_bytes +
               static_cast<double>(L.weight_bytes);
    OIDNX_TRY(emit(LL));
  }
  return ok();
}

// The cached plan for a w x h network input: its arena (zeroed once) and
// its launch descriptors.
oidnx_status create_plan(oidnx_filter* f, int w, int h, int stack, std::unique_ptr<Plan>* out) {
  std::unique_ptr<Plan> P(new Plan());
  // on any failure below, free what was already created (arena, event)
  struct Release {
    Plan* p;
    ~Release() { destroy_plan(p); }
  } release{P.get()};
  P->w = w;
  P->h = h;
  P->stack = stack;
  ValueLayout V;
  layout_values(f, w, h, false, f->keep_acts != 0, &V, stack);
  for (int l = 0; l < 5; ++l) P->lvl[l] = V.lvl[l];
  for (int v = 0; v < V_COUNT; ++v) {
    P->value_ext[v] = V.ext[v];
    P->value_ch[v] = V.ch[v];
    P->value_off[v] = V.off[v];
    P->value_bytes[v] = V.bytes[v];
  }
  for (int i = 0; i < 4; ++i) P->split_on[i] = V.split_on[i];
  for (int i = 0; i < 2; ++i) P->fused[i] = V.fused[i];
  P->arena_bytes = V.total;
  cudaError_t e = cudaMalloc(&P->arena, V.total);
  if (e != cudaSuccess)
    return fail(OIDNX_ERR_OUT_OF_MEMORY, "activation arena of %zu bytes: %s", V.total,
                cudaGetErrorString(e));
  // Zero once so that padded lanes read as zero before any write.
  e = cudaMemset(P->arena, 0, V.total);
  if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "arena memset: %s", cudaGetErrorString(e));
  e = cudaEventCreateWithFlags(&P->done, cudaEventDisableTiming);
  if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "event: %s", cudaGetErrorString(e));
  Plan* plan = P.get();
  OIDNX_TRY(build_network_launches(
      f, V, [plan](int v) { return plan->ptr(v); },
      [plan](const LayerLaunch& LL) {
        plan->launches.push_back(LL);
        return ok();
      },
      stack > 1 ? h : 0));
  if (stack == 1 && V.split_on[0] && head_fusable(f)) {
    const LayerDef& d = kDefs[0];
    OIDNX_TRY(build_head_launch(f->layers[0], V.lvl[0].w, V.lvl[0].h, plan->ptr(d.dst), V.ext[d.dst].pitch,
                                plan->ptr(V_INS), V.ext[V_INS].pitch, f->status, &plan->head));
    plan->head_on = true;
  }
  if (stack > 1) {
    // the final conv of each tile (or the fused tail) reads that tile's rows
    // of its source (its own halo rows beyond them read as zeros, as the
    // gap rows give the stacked layers)
    const int l = V.tail ? kLayers - 2 : kLayers - 1;
    const LayerDef& d = kDefs[l];
    const DeviceLayer& L = f->layers[l];
    const DeviceLayer& L2 = f->layers[kLayers - 1];
    const Extent se = V.ext[d.src0];
    const size_t row_bytes = static_cast<size_t>(act_chunks(f->precision, V.ch[d.src0])) * se.pitch * 16;
    const int bpe = f->precision == OIDNX_PRECISION_FP16 ? 2 : 4;
    for (int t = 0; t < stack; ++t) {
      LayerLaunch LL;
      std::memset(&LL, 0, sizeof(LL));
      LL.layer = l;
      const uint8_t* src = static_cast<const uint8_t*>(plan->ptr(d.src0)) +
                           static_cast<size_t>(t) * (h + kStackGap) * row_bytes;
      if (V.tail) {
        LL.tail = 1;
        LL.name = "dec_conv1b+dec_conv0";
        OIDNX_TRY(build_tail_launch(L, L2, src, Extent{w, h, se.pitch}, w, h, nullptr, f->status, &LL.tlcl));
        LL.flop = 2.0 * 9.0 * (L.cin * L.cout + L2.cin * L2.cout) * w * h;
        LL.bytes = static_cast<double>(w) * h * (V.ch[d.src0] * bpe + 16) +
                   static_cast<double>(L.weight_bytes + L2.weight_bytes);
      } else {
        LL.name = kLayerNames[l];
        LL.final = 1;
        OIDNX_TRY(build_final_launch(L, src, Extent{w, h, se.pitch}, w, h, nullptr, f->status, &LL.fcl));
        LL.fcl.p.reverse = walk_reverse(l);
        LL.flop = 2.0 * 9.0 * L.cin * L.cout * w * h;
        LL.bytes = static_cast<double>(w) * h * (V.ch[d.src0] * bpe + 16) + static_cast<double>(L.weight_bytes);
      }
      plan->final_tiles.push_back(LL);
    }
  }
  release.p = nullptr;
  *out = std::move(P);
  return ok();
}

// LRU lookup/creation of the plan for a w x h network input ("nativeUNet.ts",
// _execution): evicted plans are destroyed once their last use has finished.
oidnx_status get_plan(oidnx_filter* f, int w, int h, Plan** out, int stack = 1) {
  for (auto it = f->retired.begin(); it != f->retired.end();) {
    if (cudaEventQuery((*it)->done) == cudaSuccess) {
      destroy_plan(it->get());
      it = f->retired.erase(it);
    } else {
      ++it;
    }
  }
  for (auto& p : f->plans)
    if (p->w == w && p->h == h && p->stack == stack) {
      p->last_used = ++f->clock;
      *out = p.get();
      return ok();
    }
  std::unique_ptr<Plan> P;
  OIDNX_TRY(create_plan(f, w, h, stack, &P));
  P->last_used = ++f->clock;
  Plan* raw = P.get();
  f->plans.push_back(std::move(P));
  while (static_cast<int>(f->plans.size()) > f->shape_cache) {
    auto oldest = f->plans.end();
    for (auto it = f->plans.begin(); it != f->plans.end(); ++it)
      if (it->get() != raw && (oldest == f->plans.end() || (*it)->last_used < (*oldest)->last_used))
        oldest = it;
    if (oldest == f->plans.end()) break;
    if (f->current == oldest->get()) {
      f->current = nullptr;
      drop_graphs(f);
    }
    if (f->last_plan == oldest->get()) f->last_plan = nullptr;
    f->retired.push_back(std::move(*oldest));
    f->plans.erase(oldest);
  }
  *out = raw;
  return ok();
}

// ---------------------------------------------------------------- profiling
oidnx_status prof_begin(oidnx_filter* f, size_t launches) {
  Profile& P = f->prof;
  while (P.ev.size() < launches + 1) {
    cudaEvent_t e;
    OIDNX_CUDA(cudaEventCreate(&e));
    P.ev.push_back(e);
  }
  P.label.assign(launches, 0);
  P.used = 0;
  P.valid = true;
  return ok();
}

oidnx_status prof_mark(oidnx_filter* f, bool on, int label, cudaStream_t s) {
  if (!on) return ok();
  Profile& P = f->prof;
  if (P.used > 0) P.label[P.used - 1] = label;
  // Inside stream capture an event becomes a graph node only when recorded
  // as an external event; otherwise it would only order captured work.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  OIDNX_CUDA(cudaStreamIsCapturing(s, &cap));
  if (cap == cudaStreamCaptureStatusActive)
    OIDNX_CUDA(cudaEventRecordWithFlags(P.ev[P.used], s, cudaEventRecordExternal));
  else
    OIDNX_CUDA(cudaEventRecord(P.ev[P.used], s));
  P.used++;
  return ok();
}

// ---------------------------------------------------------------- enqueue
oidnx_status enqueue_network(oidnx_filter* f, Plan* P, bool prof, cudaStream_t s) {
  for (const LayerLaunch& L : P->launches) {
    OIDNX_TRY(run_launch(L, s));
    OIDNX_TRY(prof_mark(f, prof, L.layer, s));
  }
  return ok();
}

// The output pass runs in the final conv's epilogue (kx-folded final conv
// or the fused tail, "fuseOutput" on).
bool output_fused(const oidnx_filter* f, const Plan* P) {
  return P && f->fuse_output && !P->launches.empty() &&
         (P->launches.back().final || P->launches.back().tail);
}

// Output-pass parameters of one tile in a final-conv or tail epilogue.
template <class Params>
void set_output_pass(const oidnx_filter* f, void* const img[4], const size_t stride[4],
                     const AxisTile& tx, const AxisTile& ty, float scale, Params* fp) {
  fp->color = static_cast<const float4*>(img[0]);
  fp->color_stride = stride[0] / 16;
  fp->out = static_cast<float4*>(img[3]);
  fp->out_stride = stride[3] / 16;
  fp->in_x = tx.out_start - tx.in_start;
  fp->in_y = ty.out_start - ty.in_start;
  fp->ox = tx.out_start;
  fp->oy = ty.out_start;
  fp->ow = tx.out_size;
  fp->oh = ty.out_size;
  fp->hdr = f->hdr;
  fp->scale = scale;
  fp->exp2_tab = static_cast<const float4*>(f->exp2_tab);
}

// Input-pass parameters of one tile; out / out_split: where its packed
// input and parity-split copy go (split null when unused).
PackParams tile_pack_params(const oidnx_filter* f, const Plan* P, void* const img[4],
                            const size_t stride[4], const AxisTile& tx, const AxisTile& ty,
                            float scale, void* out, void* out_split) {
  PackParams pp;
  std::memset(&pp, 0, sizeof(pp));
  for (int i = 0; i < 3; ++i) {
    pp.img[i] = static_cast<const float4*>(img[i]);
    pp.stride[i] = stride[i] / 16;
  }
  pp.sources = f->in_channels / 3;
  pp.width = f->width;
  pp.height = f->height;
  pp.tx = tx.in_start;
  pp.ty = ty.in_start;
  pp.tw = tx.in_size;
  pp.th = ty.in_size;
  pp.hdr = f->hdr;
  pp.scale = scale;
  pp.fp16 = f->precision == OIDNX_PRECISION_FP16;
  pp.out = out;
  pp.out_split = out_split;
  pp.split_pitch = out_split ? P->value_ext[V_INS].pitch : 0;
  pp.chunks = act_chunks(f->precision, f->in_channels);
  pp.pitch = P->value_ext[V_IN].pitch;
  pp.log2_tab = static_cast<const float4*>(f->log2_tab);
  return pp;
}

// Stacked frame, in groups of up to P->stack tiles: each tile's input pass
// into its block of the stack (gap rows zeroed), the convs once over the
// stack, then each tile's final conv with the output pass in its epilogue.
oidnx_status enqueue_stacked(oidnx_filter* f, Plan* P, void* const img[4], const size_t stride[4],
                             float scale, bool prof, cudaStream_t s) {
  const int period = P->h + kStackGap;
  const int chunks = act_chunks(f->precision, f->in_channels);
  const size_t in_row = static_cast<size_t>(chunks) * P->value_ext[V_IN].pitch * 16;
  const size_t split_row = static_cast<size_t>(chunks) * P->value_ext[V_INS].pitch * 16;
  const int nx = static_cast<int>(f->tx.size());
  const int tiles = nx * static_cast<int>(f->ty.size());
  // groups of up to P->stack tiles; a short last group leaves the blocks it
  // does not fill with stale (finite) values, which no tile of it reads
  for (int g0 = 0; g0 < tiles; g0 += P->stack) {
    const int n = std::min(P->stack, tiles - g0);
    for (int b = 0; b < n; ++b) {
      const AxisTile& tx = f->tx[(g0 + b) % nx];
      const AxisTile& ty = f->ty[(g0 + b) / nx];
      PackParams pp = tile_pack_params(
          f, P, img, stride, tx, ty, scale,
          static_cast<uint8_t*>(P->ptr(V_IN)) + static_cast<size_t>(b) * period * in_row,
          P->split_on[0] ? static_cast<uint8_t*>(P->ptr(V_INS)) + static_cast<size_t>(b) * period * split_row
                         : nullptr);
      pp.gap_rows = kStackGap;
      (void)cudaGetLastError();
      cudaError_t e = launch_pack(pp, s);
      if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "input pass: %s", cudaGetErrorString(e));
      OIDNX_TRY(prof_mark(f, prof, -1, s));
    }
    for (const LayerLaunch& L : P->launches) {
      OIDNX_TRY(run_launch(L, s));
      OIDNX_TRY(prof_mark(f, prof, L.layer, s));
    }
    for (int b = 0; b < n; ++b) {
      const AxisTile& tx = f->tx[(g0 + b) % nx];
      const AxisTile& ty = f->ty[(g0 + b) / nx];
      LayerLaunch L = P->final_tiles[b];
      if (L.tail) {
        L.tlcl.outpass = 1;
        L.name = "dec_conv1b+dec_conv0+output";
        set_output_pass(f, img, stride, tx, ty, scale, &L.tlcl.p);
      } else {
        L.fcl.outpass = 1;
        L.name = "dec_conv0+output";
        L.fcl.p.net = nullptr;
        set_output_pass(f, img, stride, tx, ty, scale, &L.fcl.p);
      }
      OIDNX_TRY(run_launch(L, s));
      OIDNX_TRY(prof_mark(f, prof, L.layer, s));
    }
  }
  P->out_stored = false;
  P->outpass_fused = true;
  P->head_used = false;
  return ok();
}

// All tiles: input pass -> network -> output pass, on stream s.
oidnx_status enqueue_denoise(oidnx_filter* f, void* const img[4], const size_t stride[4],
                             bool prof, cudaStream_t s) {
  Plan* P = f->current;
  const float scale = f->input_scale == 0.0f ? 1.0f : f->input_scale;
  OIDNX_TRY(prof_mark(f, prof, -2, s));
  if (P->stack > 1) return enqueue_stacked(f, P, img, stride, scale, prof, s);
  P->outpass_fused = output_fused(f, P);
  P->head_used = P->head_on;
  // with the head kernel the plan's enc_conv0 launch is skipped
  const size_t first = P->head_used ? 1 : 0;
  for (const AxisTile& ty : f->ty)
    for (const AxisTile& tx : f->tx) {
      PackParams pp = tile_pack_params(f, P, img, stride, tx, ty, scale, P->ptr(V_IN),
                                       P->split_on[0] ? P->ptr(V_INS) : nullptr);
      (void)cudaGetLastError();
      if (P->head_used) {
        HeadLaunch H = P->head;
        for (int i = 0; i < 3; ++i)
          OIDNX_TRY(encode_image_map(&H.map[i], img[i < pp.sources ? i : 0], f->width, f->height,
                                     stride[i < pp.sources ? i : 0]));
        H.p.sources = pp.sources;
        H.p.width = pp.width;
        H.p.height = pp.height;
        H.p.tx = pp.tx;
        H.p.ty = pp.ty;
        H.p.hdr = pp.hdr;
        H.p.scale = pp.scale;
        cudaError_t e = launch_conv_head(H, s);
        if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "input pass + enc_conv0: %s", cudaGetErrorString(e));
        OIDNX_TRY(prof_mark(f, prof, 0, s));
      } else {
        cudaError_t e = launch_pack(pp, s);
        if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "input pass: %s", cudaGetErrorString(e));
        OIDNX_TRY(prof_mark(f, prof, -1, s));
      }
      if (output_fused(f, P)) {
        // the final conv's epilogue runs the output pass for this tile
        for (size_t i = first; i + 1 < P->launches.size(); ++i) {
          OIDNX_TRY(run_launch(P->launches[i], s));
          OIDNX_TRY(prof_mark(f, prof, P->launches[i].layer, s));
        }
        LayerLaunch L = P->launches.back();
        float4* net = f->keep_acts ? static_cast<float4*>(P->ptr(V_OUT)) : nullptr;
        P->out_stored = f->keep_acts != 0;
        if (L.tail) {
          L.tlcl.outpass = 1;
          L.name = "dec_conv1b+dec_conv0+output";
          L.tlcl.p.net = net;
          set_output_pass(f, img, stride, tx, ty, scale, &L.tlcl.p);
        } else {
          L.fcl.outpass = 1;
          L.name = "dec_conv0+output";
          L.fcl.p.net = net;
          set_output_pass(f, img, stride, tx, ty, scale, &L.fcl.p);
        }
        OIDNX_TRY(run_launch(L, s));
        OIDNX_TRY(prof_mark(f, prof, L.layer, s));
        continue;
      }
      for (size_t i = first; i < P->launches.size(); ++i) {
        OIDNX_TRY(run_launch(P->launches[i], s));
        OIDNX_TRY(prof_mark(f, prof, P->launches[i].layer, s));
      }
      P->out_stored = true;
      UnpackParams up;
      std::memset(&up, 0, sizeof(up));
      up.net = static_cast<const float4*>(P->ptr(V_OUT));
      up.tw = tx.in_size;
      up.in_x = tx.out_start - tx.in_start;
      up.in_y = ty.out_start - ty.in_start;
      up.color = static_cast<const float4*>(img[0]);
      up.color_stride = stride[0] / 16;
      up.out = static_cast<float4*>(img[3]);
      up.out_stride = stride[3] / 16;
      up.ox = tx.out_start;
      up.oy = ty.out_start;
      up.ow = tx.out_size;
      up.oh = ty.out_size;
      up.hdr = f->hdr;
      up.scale = scale;
      up.exp2_tab = static_cast<const float4*>(f->exp2_tab);
      cudaError_t e = launch_unpack(up, s);
      if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "output pass: %s", cudaGetErrorString(e));
      OIDNX_TRY(prof_mark(f, prof, kLayers, s));
    }
  return ok();
}

size_t denoise_launches(const oidnx_filter* f) {
  // input pass, the plan's conv launches, output pass (folded into the final
  // conv when fused); stacked: per tile the input pass and the final conv,
  // once each of the other convs
  const Plan* P = f->current;
  if (P && P->stack > 1) {
    const size_t tiles = f->tx.size() * f->ty.size();
    const size_t groups = (tiles + P->stack - 1) / P->stack;
    return 2 * tiles + groups * P->launches.size();
  }
  const size_t convs = P ? P->launches.size() : kLayers;
  return f->tx.size() * f->ty.size() * (convs + (output_fused(f, P) ? 1 : 2));
}

bool filter_alive(oidnx_filter* f, oidnx_status* st) {
  if (!f) {
    *st = fail(OIDNX_ERR_INVALID_ARGUMENT, "filter is NULL");
    return false;
  }
  if (f->released) {
    *st = fail(OIDNX_ERR_RELEASED, "filter was released");
    return false;
  }
  return true;
}

void invalidate(oidnx_filter* f) {
  f->committed = false;
  drop_graphs(f);
}

oidnx_status execute_images(oidnx_filter* f, void* const img[4], const size_t stride[4],
                            cudaStream_t s) {
  if (!f->committed) return fail(OIDNX_ERR_NOT_COMMITTED, "execute before a successful commit");
  const bool prof = f->profile_next || f->profile_always;
  if (f->profile_next) {
    // One-shot profile: a plain (eager) run with events between the kernels.
    f->profile_next = false;
    OIDNX_TRY(prof_begin(f, denoise_launches(f)));
    OIDNX_TRY(enqueue_denoise(f, img, stride, true, s));
  } else {
    oidnx_filter::GraphEntry* ge = nullptr;
    for (auto& g : f->graphs) {
      bool same = g.exec && g.profiled == prof;
      for (int i = 0; i < 4 && same; ++i) same = g.img[i] == img[i];
      if (same) ge = &g;
    }
    if (!ge) {
      ge = f->graphs[0].used <= f->graphs[1].used ? &f->graphs[0] : &f->graphs[1];
      if (ge->exec) {
        cudaGraphExecDestroy(ge->exec);
        *ge = oidnx_filter::GraphEntry();
      }
      if (!f->capture_stream)
        OIDNX_CUDA(cudaStreamCreateWithFlags(&f->capture_stream, cudaStreamNonBlocking));
      if (prof) OIDNX_TRY(prof_begin(f, denoise_launches(f)));
      OIDNX_CUDA(cudaStreamBeginCapture(f->capture_stream, cudaStreamCaptureModeThreadLocal));
      oidnx_status st = enqueue_denoise(f, img, stride, prof, f->capture_stream);
      cudaGraph_t g = nullptr;
      cudaError_t e = cudaStreamEndCapture(f->capture_stream, &g);
      if (st != OIDNX_OK) {
        if (g) cudaGraphDestroy(g);
        return st;
      }
      if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "graph capture: %s", cudaGetErrorString(e));
      e = cudaGraphInstantiate(&ge->exec, g, 0);
      cudaGraphDestroy(g);
      if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "graph instantiate: %s", cudaGetErrorString(e));
      ge->profiled = prof;
      for (int i = 0; i < 4; ++i) ge->img[i] = img[i];
    }
    ge->used = ++f->graph_clock;
    OIDNX_CUDA(cudaGraphLaunch(ge->exec, s));
  }
  OIDNX_CUDA(cudaEventRecord(f->current->done, s));
  f->last_plan = f->current;
  return ok();
}

}  // namespace

// ======================================================================
// network in caller-given scratch (no device allocation)
// ======================================================================
namespace oidnx {

oidnx_status noalloc_scratch_address(void** out);

oidnx_status report_error(oidnx_status status, const char* message) {
  return fail(status, "%s", message);
}

// Plan the network for a w x h input with every intermediate activation
// placed in `arena` (cap bytes) by the same liveness best-fit rule as the
// plan cache, the input read from `in` and the output written to `out`, then
// enqueue the 16 conv kernels on `s`.  No device memory is allocated and no
// plan is cached; the launch descriptors live on the stack.
oidnx_status network_enqueue_in_arena(oidnx_filter* f, const void* in, int w, int h, void* out,
                                      void* arena, size_t cap, cudaStream_t s) {
  if (!f) return fail(OIDNX_ERR_INVALID_ARGUMENT, "filter is NULL");
  if (f->released) return fail(OIDNX_ERR_RELEASED, "filter was released");
  if (!in || !out || w <= 0 || h <= 0)
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "network_execute_noalloc: bad arguments");
  if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) % 16)
    return fail(OIDNX_ERR_INVALID_ARGUMENT,
                "network_execute_noalloc: pointers must be 16-byte aligned");
  ValueLayout V;
  layout_values(f, w, h, true, false, &V);
  if (V.total > cap)
    return fail(OIDNX_ERR_INVALID_ARGUMENT,
                "network_execute_noalloc: a %dx%d input needs %zu bytes of activation scratch; "
                "the static arena holds %zu bytes",
                w, h, V.total, cap);
  auto ptr = [&](int v) -> void* {
    if (v == V_IN) return const_cast<void*>(in);
    if (v == V_OUT) return out;
    return static_cast<uint8_t*>(arena) + V.off[v];
  };
  if (V.split_on[0]) {
    cudaError_t e = launch_split_copy(in, w, ptr(V_INS), V.ext[V_INS].pitch, w, h,
                                      act_chunks(f->precision, f->in_channels), s);
    if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "split copy: %s", cudaGetErrorString(e));
  }
  OIDNX_TRY(build_network_launches(f, V, ptr, [s](const LayerLaunch& LL) { return run_launch(LL, s); }));
  return ok();
}

}  // namespace oidnx

// ======================================================================
// C ABI
// ======================================================================
extern "C" {

const char* oidnx_last_error(void) { return g_last_error.c_str(); }

const char* oidnx_version(void) { return "oidnx 0.1 (sm_103a)"; }

int oidnx_default_overlap(void) { return default_overlap_value(); }

oidnx_status oidnx_plan_tiles(int width, int height, int max_tile_size, int overlap, int* rects,
                              int cap, int* count) {
  if (width <= 0 || height <= 0 || !count || cap < 0 || (cap > 0 && !rects))
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "plan_tiles: bad arguments");
  if (overlap < 0) overlap = default_overlap_value();
  const int limit = max_tile_size > 0 ? max_tile_size : round_up(std::max(width, height), 16);
  std::vector<AxisTile> xs, ys;
  if (!plan_axis(width, limit, overlap, &xs) || !plan_axis(height, limit, overlap, &ys))
    return fail(OIDNX_ERR_INVALID_ARGUMENT,
                "maxTileSize %d too small for overlap %d (or bad overlap)", max_tile_size, overlap);
  *count = static_cast<int>(xs.size() * ys.size());
  int i = 0;
  for (const AxisTile& y : ys)
    for (const AxisTile& x : xs) {
      if (i < cap) {
        int* r = rects + 8 * i;
        r[0] = x.in_start; r[1] = y.in_start; r[2] = x.in_size; r[3] = y.in_size;
        r[4] = x.out_start; r[5] = y.out_start; r[6] = x.out_size; r[7] = y.out_size;
      }
      ++i;
    }
  return ok();
}

oidnx_status oidnx_filter_create(const void* blob, size_t bytes, int precision,
                                 oidnx_filter** out) {
  if (!blob || !out) return fail(OIDNX_ERR_INVALID_ARGUMENT, "filter_create: NULL argument");
  *out = nullptr;
  if (precision < 0 || precision > 2)
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "precision must be 0 (auto), 1 (fp32) or 2 (fp16)");
  ConvTensors T[kLayers];
  int cin = 0;
  OIDNX_TRY(parse_blob(blob, bytes, T, &cin));
  std::unique_ptr<oidnx_filter> f(new oidnx_filter());
  f->precision = precision == OIDNX_PRECISION_FP32 ? OIDNX_PRECISION_FP32 : OIDNX_PRECISION_FP16;
  f->in_channels = cin;
  auto out_ch = [&](int v) -> int {
    if (v == V_IN) return cin;
    for (int l = 0; l < kLayers; ++l)
      if (kDefs[l].dst == v) return T[l].cout;
    return 0;
  };
  oidnx_status st = OIDNX_OK;
  for (int l = 0; l < kLayers && st == OIDNX_OK; ++l) {
    const int c0 = out_ch(kDefs[l].src0);
    const int c1 = kDefs[l].src1 >= 0 ? out_ch(kDefs[l].src1) : 0;
    st = make_device_layer(T[l], c0, c1, f->precision, &f->layers[l]);
    f->weight_bytes += f->layers[l].weight_bytes;
  }
  if (st == OIDNX_OK) {
    cudaError_t e = cudaMalloc(&f->status, 256);
    if (e == cudaSuccess) e = cudaMemset(f->status, 0, 256);
    if (e != cudaSuccess) st = fail(OIDNX_ERR_CUDA, "status word: %s", cudaGetErrorString(e));
  }
  if (st == OIDNX_OK && f->precision == OIDNX_PRECISION_FP32) {
    float tab[kLog2TabSize][4];
    fill_log2_table(tab);
    st = upload(tab, sizeof(tab), &f->log2_tab);
  }
  if (st == OIDNX_OK) {
    float tab[kExp2TabSize][4];
    fill_exp2_table(tab);
    st = upload(tab, sizeof(tab), &f->exp2_tab);
  }
  if (st == OIDNX_OK) {
    // set-up of the allocation-free entry point on this device: the array
    // it uses is placed here, not by its first call
    void* scratch = nullptr;
    st = noalloc_scratch_address(&scratch);
  }
  if (st != OIDNX_OK) {
    std::string msg = g_last_error;
    for (DeviceLayer& L : f->layers) free_layer(L);
    cudaFree(f->status);
    cudaFree(f->log2_tab);
    cudaFree(f->exp2_tab);
    g_last_error = msg;
    return st;
  }
  *out = f.release();
  return ok();
}

oidnx_status oidnx_filter_set_image(oidnx_filter* f, int which, void* device_ptr,
                                    size_t row_stride_bytes) {
  oidnx_status st;
  if (!filter_alive(f, &st)) return st;
  if (which < 0 || which > 3) return fail(OIDNX_ERR_INVALID_ARGUMENT, "bad image slot %d", which);
  if (reinterpret_cast<uintptr_t>(device_ptr) % 16)
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "image pointer must be 16-byte aligned");
  if (row_stride_bytes % 16)
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "row stride must be a multiple of 16 bytes");
  f->img[which] = device_ptr;
  f->img_stride[which] = row_stride_bytes;
  invalidate(f);
  return ok();
}

oidnx_status oidnx_filter_set_int(oidnx_filter* f, const char* name, int value) {
  oidnx_status st;
  if (!filter_alive(f, &st)) return st;
  if (!name) return fail(OIDNX_ERR_INVALID_ARGUMENT, "NULL parameter name");
  const std::string n(name);
  if (n == "width" || n == "height") {
    if (value <= 0) return fail(OIDNX_ERR_INVALID_ARGUMENT, "Image dimensions must be positive");
    (n == "width" ? f->width : f->height) = value;
  } else if (n == "hdr") {
    if (value != 0 && value != 1) return fail(OIDNX_ERR_INVALID_ARGUMENT, "hdr must be 0 or 1");
    f->hdr = value;
  } else if (n == "transfer") {
    if (value != OIDNX_TRANSFER_PU && value != OIDNX_TRANSFER_LOG)
      return fail(OIDNX_ERR_INVALID_ARGUMENT, "transfer must be 0 (pu) or 1 (log)");
    f->transfer = value;
  } else if (n == "maxTileSize") {
    if (value < 0) return fail(OIDNX_ERR_INVALID_ARGUMENT, "maxTileSize must be >= 0");
    f->max_tile = value;
  } else if (n == "overlap") {
    if (value < -1 || (value >= 0 && value % 16))
      return fail(OIDNX_ERR_INVALID_ARGUMENT, "overlap must be -1 or a multiple of 16");
    f->overlap = value;
  } else if (n == "shapeCacheSize") {
    if (value < 1) return fail(OIDNX_ERR_INVALID_ARGUMENT, "shapeCacheSize must be >= 1");
    f->shape_cache = value;
  } else if (n == "fuseOutput") {
    f->fuse_output = value ? 1 : 0;  // the graph is re-recorded on commit
  } else if (n == "stackTiles") {
    if (value < 0) return fail(OIDNX_ERR_INVALID_ARGUMENT, "stackTiles must be >= 0");
    f->stack_tiles = value;
  } else if (n == "keepActivations" || n == "subpixelDecoder" || n == "fuseLayers" ||
             n == "fuseTail" || n == "fuseInput" || n == "shapeKernels") {
    (n == "keepActivations"   ? f->keep_acts
     : n == "subpixelDecoder" ? f->subpixel
     : n == "fuseLayers"      ? f->fuse
     : n == "fuseTail"        ? f->fuse_tail
     : n == "fuseInput"       ? f->fuse_input
                              : f->shape_kernels) = value ? 1 : 0;
    for (auto& p : f->plans) f->retired.push_back(std::move(p));
    f->plans.clear();
    f->current = nullptr;
    f->last_plan = nullptr;
  } else if (n == "profile") {
    f->profile_always = value ? 1 : 0;  // the graph is re-recorded on demand
    return ok();
  } else {
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "unknown integer parameter '%s'", name);
  }
  invalidate(f);
  return ok();
}

oidnx_status oidnx_filter_get_int(oidnx_filter* f, const char* name, int* value) {
  oidnx_status st;
  if (!filter_alive(f, &st)) return st;
  if (!name || !value) return fail(OIDNX_ERR_INVALID_ARGUMENT, "NULL argument");
  const std::string n(name);
  if (n == "width") *value = f->width;
  else if (n == "height") *value = f->height;
  else if (n == "hdr") *value = f->hdr;
  else if (n == "transfer") *value = f->transfer;
  else if (n == "maxTileSize") *value = f->max_tile;
  else if (n == "overlap") *value = f->overlap < 0 ? default_overlap_value() : f->overlap;
  else if (n == "shapeCacheSize") *value = f->shape_cache;
  else if (n == "keepActivations") *value = f->keep_acts;
  else if (n == "subpixelDecoder") *value = f->subpixel;
  else if (n == "fuseLayers") *value = f->fuse;
  else if (n == "fuseOutput") *value = f->fuse_output;
  else if (n == "fuseTail") *value = f->fuse_tail;
  else if (n == "fuseInput") *value = f->fuse_input;
  else if (n == "shapeKernels") *value = f->shape_kernels;
  else if (n == "stackTiles") *value = f->stack_tiles;
  else if (n == "stackedTiles") *value = f->committed && f->current ? f->current->stack : 0;
  else if (n == "profile") *value = f->profile_always;
  else if (n == "inputChannels") *value = f->in_channels;
  else if (n == "precision") *value = f->precision;
  else if (n == "tiles") *value = f->committed ? static_cast<int>(f->tx.size() * f->ty.size()) : 0;
  else return fail(OIDNX_ERR_INVALID_ARGUMENT, "unknown integer parameter '%s'", name);
  return ok();
}

oidnx_status oidnx_filter_set_float(oidnx_filter* f, const char* name, float value) {
  oidnx_status st;
  if (!filter_alive(f, &st)) return st;
  if (!name) return fail(OIDNX_ERR_INVALID_ARGUMENT, "NULL parameter name");
  if (std::string(name) != "inputScale")
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "unknown float parameter '%s'", name);
  if (!std::isfinite(value) || value < 0.0f)
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "inputScale must be finite and >= 0");
  f->input_scale = value;
  invalidate(f);
  return ok();
}

oidnx_status oidnx_filter_commit(oidnx_filter* f) {
  oidnx_status st;
  if (!filter_alive(f, &st)) return st;
  invalidate(f);
  if (f->width <= 0 || f->height <= 0)
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "Image dimensions must be positive");
  if (f->hdr && f->transfer == OIDNX_TRANSFER_PU)
    return fail(OIDNX_ERR_UNSUPPORTED, "the 'pu' transfer is not defined by this build");
  const int sources = f->in_channels / 3;
  if (!f->img[OIDNX_IMAGE_COLOR] || !f->img[OIDNX_IMAGE_OUTPUT] ||
      (sources > 1 && !f->img[OIDNX_IMAGE_ALBEDO]) || (sources > 2 && !f->img[OIDNX_IMAGE_NORMAL]))
    return fail(OIDNX_ERR_INVALID_ARGUMENT,
                "expected %d input image(s) (colour%s) and an output image", sources,
                sources == 3 ? ", albedo, normal" : sources == 2 ? ", albedo" : "");
  for (int i = 0; i < 4; ++i)
    if (f->img[i] && f->img_stride[i] != 0 && f->img_stride[i] < static_cast<size_t>(f->width) * 16)
      return fail(OIDNX_ERR_INVALID_ARGUMENT, "row stride of image %d below width*16", i);
  const int overlap = f->overlap < 0 ? default_overlap_value() : f->overlap;
  const int limit = f->max_tile > 0 ? f->max_tile : round_up(std::max(f->width, f->height), 16);
  if (!plan_axis(f->width, limit, overlap, &f->tx) || !plan_axis(f->height, limit, overlap, &f->ty))
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "maxTileSize %d too small for overlap %d",
                f->max_tile, overlap);
  // Frames of several (equal) tiles are stacked: each conv layer runs once
  // over all tiles.  Not with kept activations (per-tile debug reads), fused
  // layer pairs, or a separate output pass.
  const int tiles = static_cast<int>(f->tx.size() * f->ty.size());
  int stack = 1;
  if (tiles > 1 && f->fuse_output && !f->keep_acts && !f->fuse &&
      final_foldable(f->layers[kLayers - 1])) {
    // groups of tiles whose stacked arena fits kStackBudget (tiles bound the
    // memory a frame needs), as even as the group count allows
    ValueLayout one;
    layout_values(f, f->tx[0].in_size, f->ty[0].in_size, false, false, &one);
    const size_t per_tile = std::max<size_t>(one.total, 1);
    const int fit = f->stack_tiles > 0
                        ? std::min(f->stack_tiles, tiles)
                        : static_cast<int>(std::max<size_t>(1, std::min<size_t>(tiles, kStackBudget / per_tile)));
    const int groups = (tiles + fit - 1) / fit;
    stack = (tiles + groups - 1) / groups;
  }
  Plan* P = nullptr;
  OIDNX_TRY(get_plan(f, f->tx[0].in_size, f->ty[0].in_size, &P, stack));
  f->current = P;
  f->committed = true;
  return ok();
}

oidnx_status oidnx_filter_execute(oidnx_filter* f, void* stream) {
  oidnx_status st;
  if (!filter_alive(f, &st)) return st;
  void* img[4];
  size_t stride[4];
  for (int i = 0; i < 4; ++i) {
    img[i] = f->img[i];
    stride[i] = f->img_stride[i] ? f->img_stride[i] : static_cast<size_t>(f->width) * 16;
  }
  return execute_images(f, img, stride, static_cast<cudaStream_t>(stream));
}

oidnx_status oidnx_filter_execute_host_async(oidnx_filter* f, const float* color,
                                             const float* albedo, const float* normal,
                                             float* output, void* stream) {
  oidnx_status st;
  if (!filter_alive(f, &st)) return st;
  if (!f->committed) return fail(OIDNX_ERR_NOT_COMMITTED, "execute before a successful commit");
  const int sources = f->in_channels / 3;
  if (!color || !output || (sources > 1 && !albedo) || (sources > 2 && !normal))
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "missing host image");
  const size_t bytes = static_cast<size_t>(f->width) * f->height * 16;
  if (f->host_img_bytes != bytes) {
    // the staging sets are resized only with nothing in flight
    if (f->host_out) OIDNX_CUDA(cudaStreamSynchronize(f->host_out));
    for (int b = 0; b < 2; ++b)
      for (int i = 0; i < 4; ++i) {
        cudaFree(f->host_img[b][i]);
        f->host_img[b][i] = nullptr;
      }
    f->host_img_bytes = 0;
    f->host_used[0] = f->host_used[1] = false;
    for (int b = 0; b < 2; ++b)
      for (int i = 0; i < 4; ++i) OIDNX_CUDA(cudaMalloc(&f->host_img[b][i], bytes));
    f->host_img_bytes = bytes;
  }
  if (!f->host_in) {
    OIDNX_CUDA(cudaStreamCreateWithFlags(&f->host_in, cudaStreamNonBlocking));
    OIDNX_CUDA(cudaStreamCreateWithFlags(&f->host_out, cudaStreamNonBlocking));
    for (int b = 0; b < 2; ++b) {
      OIDNX_CUDA(cudaEventCreateWithFlags(&f->ev_in[b], cudaEventDisableTiming));
      OIDNX_CUDA(cudaEventCreateWithFlags(&f->ev_comp[b], cudaEventDisableTiming));
      OIDNX_CUDA(cudaEventCreateWithFlags(&f->ev_out[b], cudaEventDisableTiming));
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int b = f->host_next;
  f->host_next ^= 1;
  void** img = f->host_img[b];
  // upload: the set's inputs were last read by the denoise two calls ago
  if (f->host_used[b]) OIDNX_CUDA(cudaStreamWaitEvent(f->host_in, f->ev_comp[b], 0));
  const float* src[3] = {color, albedo, normal};
  for (int i = 0; i < sources; ++i)
    OIDNX_CUDA(cudaMemcpyAsync(img[i], src[i], bytes, cudaMemcpyHostToDevice, f->host_in));
  OIDNX_CUDA(cudaEventRecord(f->ev_in[b], f->host_in));
  // denoise on the caller's stream once the inputs are in and the set's
  // output buffer has been downloaded
  OIDNX_CUDA(cudaStreamWaitEvent(s, f->ev_in[b], 0));
  if (f->host_used[b]) OIDNX_CUDA(cudaStreamWaitEvent(s, f->ev_out[b], 0));
  size_t stride[4];
  for (int i = 0; i < 4; ++i) stride[i] = static_cast<size_t>(f->width) * 16;
  OIDNX_TRY(execute_images(f, img, stride, s));
  OIDNX_CUDA(cudaEventRecord(f->ev_comp[b], s));
  // download
  OIDNX_CUDA(cudaStreamWaitEvent(f->host_out, f->ev_comp[b], 0));
  OIDNX_CUDA(cudaMemcpyAsync(output, img[3], bytes, cudaMemcpyDeviceToHost, f->host_out));
  OIDNX_CUDA(cudaEventRecord(f->ev_out[b], f->host_out));
  f->host_used[b] = true;
  return ok();
}

oidnx_status oidnx_filter_wait_host(oidnx_filter* f) {
  oidnx_status st;
  if (!filter_alive(f, &st)) return st;
  if (f->host_out) OIDNX_CUDA(cudaStreamSynchronize(f->host_out));
  return ok();
}

oidnx_status oidnx_filter_execute_host(oidnx_filter* f, const float* color, const float* albedo,
                                       const float* normal, float* output, void* stream) {
  OIDNX_TRY(oidnx_filter_execute_host_async(f, color, albedo, normal, output, stream));
  return oidnx_filter_wait_host(f);
}

oidnx_status oidnx_network_execute(oidnx_filter* f, const void* packed_in, int w, int h,
                                   void* out, void* stream) {
  oidnx_status st;
  if (!filter_alive(f, &st)) return st;
  if (!packed_in || !out || w <= 0 || h <= 0)
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "network_execute: bad arguments");
  if ((reinterpret_cast<uintptr_t>(packed_in) | reinterpret_cast<uintptr_t>(out)) % 16)
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "network_execute: pointers must be 16-byte aligned");
  Plan* P = nullptr;
  OIDNX_TRY(get_plan(f, w, h, &P));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool prof = f->profile_next || f->profile_always;
  f->profile_next = false;
  if (prof) OIDNX_TRY(prof_begin(f, kLayers));
  const Extent ein = P->value_ext[V_IN];
  const int in_chunks = act_chunks(f->precision, f->in_channels);
  if (ein.pitch == w) {
    OIDNX_CUDA(cudaMemcpyAsync(P->ptr(V_IN), packed_in, P->value_bytes[V_IN],
                               cudaMemcpyDeviceToDevice, s));
  } else {
    cudaError_t e = launch_pitch_copy(packed_in, w, P->ptr(V_IN), ein.pitch, w, h * in_chunks, s);
    if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "input copy: %s", cudaGetErrorString(e));
  }
  if (P->split_on[0]) {
    cudaError_t e = launch_split_copy(P->ptr(V_IN), ein.pitch, P->ptr(V_INS),
                                      P->value_ext[V_INS].pitch, w, h, in_chunks, s);
    if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "split copy: %s", cudaGetErrorString(e));
  }
  P->out_stored = true;
  P->outpass_fused = false;
  P->head_used = false;
  OIDNX_TRY(prof_mark(f, prof, -2, s));
  OIDNX_TRY(enqueue_network(f, P, prof, s));
  OIDNX_CUDA(cudaMemcpyAsync(out, P->ptr(V_OUT), P->value_bytes[V_OUT], cudaMemcpyDeviceToDevice, s));
  OIDNX_CUDA(cudaEventRecord(P->done, s));
  f->last_plan = P;
  return ok();
}

oidnx_status oidnx_output_pass(oidnx_filter* f, const void* net, int w, int h, const void* color,
                               size_t color_stride, void* output, size_t output_stride, int hdr,
                               float input_scale, void* stream) {
  oidnx_status st;
  if (!filter_alive(f, &st)) return st;
  if (!net || !color || !output || w <= 0 || h <= 0 || h > 65535)
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "output_pass: bad arguments");
  if (hdr != 0 && hdr != 1) return fail(OIDNX_ERR_INVALID_ARGUMENT, "output_pass: hdr must be 0 or 1");
  if (!std::isfinite(input_scale) || input_scale < 0.0f)
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "output_pass: inputScale must be finite and >= 0");
  if ((reinterpret_cast<uintptr_t>(net) | reinterpret_cast<uintptr_t>(color) |
       reinterpret_cast<uintptr_t>(output)) % 16 || color_stride % 16 || output_stride % 16)
    return fail(OIDNX_ERR_INVALID_ARGUMENT,
                "output_pass: pointers and row strides must be 16-byte aligned");
  const size_t row = static_cast<size_t>(w) * 16;
  if ((color_stride && color_stride < row) || (output_stride && output_stride < row))
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "output_pass: row stride below width*16");
  UnpackParams up;
  std::memset(&up, 0, sizeof(up));
  up.net = static_cast<const float4*>(net);
  up.tw = w;
  up.color = static_cast<const float4*>(color);
  up.color_stride = (color_stride ? color_stride : row) / 16;
  up.out = static_cast<float4*>(output);
  up.out_stride = (output_stride ? output_stride : row) / 16;
  up.ow = w;
  up.oh = h;
  up.hdr = hdr;
  up.scale = input_scale == 0.0f ? 1.0f : input_scale;
  up.exp2_tab = static_cast<const float4*>(f->exp2_tab);
  (void)cudaGetLastError();
  cudaError_t e = launch_unpack(up, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "output pass: %s", cudaGetErrorString(e));
  return ok();
}

oidnx_status oidnx_filter_sync_status(oidnx_filter* f) {
  oidnx_status st;
  if (!filter_alive(f, &st)) return st;
  OIDNX_CUDA(cudaDeviceSynchronize());
  int word = 0;
  OIDNX_CUDA(cudaMemcpy(&word, f->status, sizeof(int), cudaMemcpyDeviceToHost));
  if (word) {
    OIDNX_CUDA(cudaMemset(f->status, 0, sizeof(int)));
    return fail(OIDNX_ERR_TIMEOUT, "a device-side wait gave up (status bits 0x%x)", word);
  }
  return ok();
}

oidnx_status oidnx_debug_wait_probe(oidnx_filter* f, unsigned int limit_us, void* stream) {
  oidnx_status st;
  if (!filter_alive(f, &st)) return st;
  if (limit_us == 0 || limit_us > 1000000)
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "wait probe limit must be 1 us .. 1 s");
  cudaError_t e = launch_wait_probe(f->status, 1000ull * limit_us, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(OIDNX_ERR_CUDA, "wait probe: %s", cudaGetErrorString(e));
  return ok();
}

oidnx_status oidnx_profile_next(oidnx_filter* f) {
  oidnx_status st;
  if (!filter_alive(f, &st)) return st;
  f->profile_next = true;
  return ok();
}

oidnx_status oidnx_get_profile(oidnx_filter* f, char* json, size_t cap) {
  oidnx_status st;
  if (!filter_alive(f, &st)) return st;
  Profile& P = f->prof;
  if (!P.valid || P.used < 2 || !json)
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "nothing profiled");
  OIDNX_CUDA(cudaEventSynchronize(P.ev[P.used - 1]));
  double ms[kLayers + 3] = {};  // index label + 2: -2 unused, -1 pack, 0..15, 16 unpack
  int count[kLayers + 3] = {};
  for (int i = 1; i < P.used; ++i) {
    float t = 0;
    OIDNX_CUDA(cudaEventElapsedTime(&t, P.ev[i - 1], P.ev[i]));
    const int idx = P.label[i - 1] + 2;
    if (idx >= 0 && idx < kLayers + 3) {
      ms[idx] += t;
      count[idx] += 1;
    }
  }
  float total = 0;
  OIDNX_CUDA(cudaEventElapsedTime(&total, P.ev[0], P.ev[P.used - 1]));
  const Plan* plan = f->last_plan;
  std::string s = "{\"totalMs\":" + std::to_string(total) + ",\"layers\":[";
  bool first = true;
  // shape: the compile-time shape of a conv3x3_tc launch (0: run-time form)
  auto add = [&](const char* id, int idx, double flop, double bytes, double mma = 0, int shape = 0) {
    if (count[idx] == 0) return;
    char buf[352];
    snprintf(buf, sizeof(buf),
             "%s{\"id\":\"%s\",\"ms\":%.6f,\"launches\":%d,\"flop\":%.0f,\"bytes\":%.0f,\"mmaFlop\":%.0f,"
             "\"shape\":%d}",
             first ? "" : ",", id, ms[idx], count[idx], flop * count[idx], bytes * count[idx],
             mma * count[idx], shape);
    s += buf;
    first = false;
  };
  const int sources = f->in_channels / 3;
  const int bpe = f->precision == OIDNX_PRECISION_FP16 ? 2 : 4;
  const double tile_px = plan ? static_cast<double>(plan->w) * plan->h : 0;
  add("input-pack", 1, 0, tile_px * (16.0 * sources + f->in_channels * bpe));
  double out_px = 0;
  for (const AxisTile& y : f->ty)
    for (const AxisTile& x : f->tx) out_px += static_cast<double>(x.out_size) * y.out_size;
  const int tiles = static_cast<int>(std::max<size_t>(1, f->tx.size() * f->ty.size()));
  const double out_bytes = out_px / tiles * 48.0;  // per tile: net + colour read, image written
  if (plan)
    for (const LayerLaunch& L : plan->launches) {
      if (&L == &plan->launches[0] && plan->head_used) {
        // the input pass and enc_conv0 ran as one kernel: the images read
        // once, the packed input's parity copy and enc_conv0's output
        // written once; its MMAs: per tile of kHeadRows rows, 3 kx x 3 ky
        // row updates of N = 32 per row
        const HeadParams& h = plan->head.p;
        const double mma = static_cast<double>(h.tiles_x) * h.tiles_y * 3.0 * 3 * kHeadRows * 32 * 128 * 16 * 2;
        add("input-pack+enc_conv0", L.layer + 2, L.flop,
            tile_px * (16.0 * sources + 2 * 16 + 2.0 * 32) + static_cast<double>(f->layers[0].weight_bytes), mma);
        continue;
      }
      const bool fused_out =
          &L == &plan->launches.back() && plan->outpass_fused && (L.final || L.tail);
      // with the output pass fused the network output is not stored: the
      // kernel reads the colour and writes the image instead
      add(fused_out ? (L.tail ? "dec_conv1b+dec_conv0+output" : "dec_conv0+output") : L.name,
          L.layer + 2, L.flop,
          fused_out ? L.bytes - tile_px * 16 + out_bytes - out_px / tiles * 16 : L.bytes,
          mma_flop(L), L.pair || L.final || L.tail ? 0 : conv_tc_shape(L.tcl));
    }
  if (plan && plan->stack > 1 && !plan->final_tiles.empty()) {
    const LayerLaunch& L = plan->final_tiles[0];  // per tile, counted per launch
    add(L.tail ? "dec_conv1b+dec_conv0+output" : "dec_conv0+output", L.layer + 2, L.flop,
        L.bytes - tile_px * 16 + out_bytes - out_px / tiles * 16, mma_flop(L));
  }
  add("output", kLayers + 2, 0, out_bytes);
  s += "]}";
  if (s.size() + 1 > cap) return fail(OIDNX_ERR_INVALID_ARGUMENT, "profile buffer too small");
  std::memcpy(json, s.c_str(), s.size() + 1);
  return ok();
}

oidnx_status oidnx_get_resource_info(oidnx_filter* f, char* json, size_t cap) {
  oidnx_status st;
  if (!filter_alive(f, &st)) return st;
  if (!json) return fail(OIDNX_ERR_INVALID_ARGUMENT, "NULL buffer");
  size_t arena = 0;
  for (auto& p : f->plans) arena += p->arena_bytes;
  char buf[512];
  snprintf(buf, sizeof(buf),
           "{\"weightBytes\":%zu,\"arenaBytes\":%zu,\"plans\":%zu,\"retiredPlans\":%zu,"
           "\"graphs\":%d,\"hostImageBytes\":%zu,\"precision\":\"%s\",\"inputChannels\":%d}",
           f->weight_bytes, arena, f->plans.size(), f->retired.size(),
           (f->graphs[0].exec ? 1 : 0) + (f->graphs[1].exec ? 1 : 0),
           f->host_img_bytes * 4 * ((f->host_img[0][0] ? 1 : 0) + (f->host_img[1][0] ? 1 : 0)),
           f->precision == OIDNX_PRECISION_FP16 ? "fp16" : "fp32",
           f->in_channels);
  if (strlen(buf) + 1 > cap) return fail(OIDNX_ERR_INVALID_ARGUMENT, "buffer too small");
  std::memcpy(json, buf, strlen(buf) + 1);
  return ok();
}

oidnx_status oidnx_debug_read_activation(oidnx_filter* f, int layer, void* host_dst, size_t cap,
                                         size_t* bytes_needed) {
  oidnx_status st;
  if (!filter_alive(f, &st)) return st;
  const Plan* P = f->last_plan;
  if (!P) return fail(OIDNX_ERR_INVALID_ARGUMENT, "no network run to read from");
  if (layer < 0 || layer > kLayers) return fail(OIDNX_ERR_INVALID_ARGUMENT, "bad layer %d", layer);
  const int v = layer == 0 ? V_IN : kDefs[layer - 1].dst;
  if (v == V_OUT && !P->out_stored)
    return fail(OIDNX_ERR_INVALID_ARGUMENT,
                "the network output is not stored (the output pass ran in the final conv's "
                "epilogue); set keepActivations");
  if (P->value_bytes[v] == 0)
    return fail(OIDNX_ERR_INVALID_ARGUMENT,
                "the output of layer %d is not stored (fused into the next layer's kernel; "
                "set keepActivations)", layer - 1);
  const Extent e = P->value_ext[v];
  const int C = v == V_OUT ? 3 : P->value_ch[v];
  const size_t need = static_cast<size_t>(e.w) * e.h * C * 4;
  if (bytes_needed) *bytes_needed = need;
  if (!host_dst) return ok();
  if (cap < need) return fail(OIDNX_ERR_INVALID_ARGUMENT, "need %zu bytes", need);
  std::vector<uint8_t> raw(P->value_bytes[v]);
  OIDNX_CUDA(cudaDeviceSynchronize());
  OIDNX_CUDA(cudaMemcpy(raw.data(), P->ptr(v), raw.size(), cudaMemcpyDeviceToHost));
  float* dst = static_cast<float*>(host_dst);
  if (v == V_OUT) {
    const float* src = reinterpret_cast<const float*>(raw.data());
    for (size_t p = 0; p < static_cast<size_t>(e.w) * e.h; ++p)
      for (int c = 0; c < 3; ++c) dst[p * 3 + c] = src[p * 4 + c];
    return ok();
  }
  const int lanes = f->precision == OIDNX_PRECISION_FP16 ? 8 : 4;
  const int chunks = act_chunks(f->precision, C);
  for (int y = 0; y < e.h; ++y)
    for (int x = 0; x < e.w; ++x)
      for (int c = 0; c < C; ++c) {
        const size_t idx = ((static_cast<size_t>(y) * chunks + c / lanes) * e.pitch + x) * lanes + c % lanes;
        float val;
        if (lanes == 8) {
          uint16_t b;
          std::memcpy(&b, raw.data() + idx * 2, 2);
          val = half_bits_to_float(b);
        } else {
          std::memcpy(&val, raw.data() + idx * 4, 4);
        }
        dst[(static_cast<size_t>(y) * e.w + x) * C + c] = val;
      }
  return ok();
}

void oidnx_filter_release(oidnx_filter* f) {
  if (!f || f->released) return;
  f->released = true;
  cudaDeviceSynchronize();
  drop_graphs(f);
  for (auto& p : f->plans) destroy_plan(p.get());
  for (auto& p : f->retired) destroy_plan(p.get());
  f->plans.clear();
  f->retired.clear();
  for (DeviceLayer& L : f->layers) free_layer(L);
  for (int b = 0; b < 2; ++b) {
    for (int i = 0; i < 4; ++i) cudaFree(f->host_img[b][i]);
    if (f->ev_in[b]) cudaEventDestroy(f->ev_in[b]);
    if (f->ev_comp[b]) cudaEventDestroy(f->ev_comp[b]);
    if (f->ev_out[b]) cudaEventDestroy(f->ev_out[b]);
  }
  if (f->host_in) cudaStreamDestroy(f->host_in);
  if (f->host_out) cudaStreamDestroy(f->host_out);
  for (cudaEvent_t e : f->prof.ev) cudaEventDestroy(e);
  if (f->capture_stream) cudaStreamDestroy(f->capture_stream);
  cudaFree(f->status);
  cudaFree(f->log2_tab);
  cudaFree(f->exp2_tab);
  delete f;
}

oidnx_status oidnx_conv_create(const float* weight, const float* bias, int cout, int cin,
                               int precision, oidnx_conv** out) {
  if (!weight || !bias || !out || cout <= 0 || cin <= 0)
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "conv_create: bad arguments");
  if (precision != OIDNX_PRECISION_FP16 && precision != OIDNX_PRECISION_FP32)
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "conv_create: precision must be fp16 or fp32");
  if (cout > 256) return fail(OIDNX_ERR_UNSUPPORTED, "conv_create: more than 256 outputs");
  ConvTensors T;
  T.cout = cout;
  T.cin = cin;
  T.w.assign(weight, weight + static_cast<size_t>(cout) * cin * 9);
  T.b.assign(bias, bias + cout);
  std::unique_ptr<oidnx_conv> c(new oidnx_conv());
  c->precision = precision;
  oidnx_status st = make_device_layer(T, cin, 0, precision, &c->L);
  if (st == OIDNX_OK) {
    cudaError_t e = cudaMalloc(&c->status, 256);
    if (e == cudaSuccess) e = cudaMemset(c->status, 0, 256);
    if (e != cudaSuccess) st = fail(OIDNX_ERR_CUDA, "status word: %s", cudaGetErrorString(e));
  }
  if (st != OIDNX_OK) {
    std::string msg = g_last_error;
    free_layer(c->L);
    cudaFree(c->status);
    g_last_error = msg;
    return st;
  }
  *out = c.release();
  return ok();
}

oidnx_status oidnx_conv_execute(oidnx_conv* c, const void* in, void* out, int w, int h, int relu,
                                void* stream) {
  if (!c || !in || !out || w <= 0 || h <= 0)
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "conv_execute: bad arguments");
  if ((reinterpret_cast<uintptr_t>(in) | reinterpret_cast<uintptr_t>(out)) % 16)
    return fail(OIDNX_ERR_INVALID_ARGUMENT, "conv_execute: pointers must be 16-byte aligned");
  if (!relu) return fail(OIDNX_ERR_UNSUPPORTED, "conv_execute: only relu=1 for hidden layers");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  LayerLaunch LL;
  std::memset(&LL, 0, sizeof(LL));
  LL.layer = 0;
  // caller's buffers: rows of w pixels (128-byte TMA rows when w % 8 == 0)
  OIDNX_TRY(build_tc_launch(c->L, kPlain, in, Extent{w, h, w}, nullptr, Extent{0, 0, 0}, w, h,
                            out, w, c->status, &LL.tcl));
  return run_launch(LL, s);
}

void oidnx_conv_release(oidnx_conv* c) {
  if (!c) return;
  cudaDeviceSynchronize();
  free_layer(c->L);
  cudaFree(c->status);
  delete c;
}

}  // extern "C"

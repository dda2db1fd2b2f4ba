/*
 * oidnx - forward pass of an OIDN-style U-Net image denoiser on one GB300.
 *
 * The calls follow the problem statement of the denoise driver in
 * "oidn-webgpu 0.0.0-stage -> 0.6.0, src/native/denoise.ts"
 * (NativeDenoiseOptions, recordDenoiseExecution): a filter is created from a
 * weight blob; colour / albedo / normal float4 images, width, height, hdr,
 * inputScale and maxTileSize are set; execute runs, per tile of an
 * overlapping grid, the input pass, the 16-layer network and the output pass.
 * The network itself is the executor of "oidn-web 0.3.4 -> 0.4.0,
 * package/src/nativeUNet.ts" (NativeUNetExecutor).
 *
 * Conventions (all calls):
 *   - Every call returns an oidnx_status; on failure oidnx_last_error() holds
 *     a message for the calling thread (the counterpart of the ERRO packet of
 *     "program.ts").  Nothing throws across this boundary.
 *   - The caller owns every image buffer and every stream it passes in; the
 *     library never frees them.  The filter owns its packed weights, its
 *     activation arenas, per-shape plans and CUDA graphs.
 *   - "stream" is a cudaStream_t passed as void*; NULL means the legacy
 *     default stream.  Work is asynchronous on that stream.
 *   - All device pointers must be 16-byte aligned.
 *
 * Activation layout used by oidnx_network_execute, oidnx_conv_execute and
 * oidnx_debug_read_activation (raw form):
 *   fp16: [H][L/8][W][8] halves, L = C rounded up to a multiple of 16;
 *   fp32: [H][L/4][W][4] floats, L = C rounded up to a multiple of 4.
 * That is the pages' channel-blocked NHWC (logical channel c in block c/4,
 * lane c%4) with blocks of 16 bytes and the block index placed above the x
 * index, so that one image row of one block is a contiguous run.  Padded
 * lanes are zero.  Network output: [H][W][4] floats, lane 3 zero.
 */
#ifndef OIDNX_H
#define OIDNX_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct oidnx_filter oidnx_filter;
typedef struct oidnx_conv oidnx_conv;

typedef enum {
  OIDNX_OK = 0,
  OIDNX_ERR_INVALID_ARGUMENT = 1, /* bad pointer, size, name or value      */
  OIDNX_ERR_INVALID_MODEL = 2,    /* weight blob malformed or not a U-Net  */
  OIDNX_ERR_UNSUPPORTED = 3,      /* valid request this build does not do  */
  OIDNX_ERR_OUT_OF_MEMORY = 4,    /* device or host allocation failed      */
  OIDNX_ERR_CUDA = 5,             /* a CUDA runtime/driver call failed     */
  OIDNX_ERR_RELEASED = 6,         /* filter already released               */
  OIDNX_ERR_TIMEOUT = 7,          /* a device-side wait gave up            */
  OIDNX_ERR_NOT_COMMITTED = 8     /* execute before a successful commit    */
} oidnx_status;

enum { OIDNX_IMAGE_COLOR = 0, OIDNX_IMAGE_ALBEDO = 1, OIDNX_IMAGE_NORMAL = 2,
       OIDNX_IMAGE_OUTPUT = 3 };
enum { OIDNX_PRECISION_AUTO = 0, OIDNX_PRECISION_FP32 = 1, OIDNX_PRECISION_FP16 = 2 };
enum { OIDNX_TRANSFER_PU = 0, OIDNX_TRANSFER_LOG = 1 };

/* Create a filter from an "OXW1" weight blob (host memory, copied).
 *   blob: magic "OXW1", u32 version (1), u32 tensor count, then per tensor:
 *         u32 name length, name bytes padded to 4, u32 ndim, u32 dims[ndim],
 *         u32 dtype (0 f32, 1 f16), data padded to 4 bytes.  Little-endian.
 *         Tensors "<layer>.weight" (OIHW, 3x3) and "<layer>.bias" ([O]) for
 *         the 16 layers enc_conv0 .. dec_conv0; the topology is read from
 *         the shapes ("nativeUNet.ts", NativeUNetExecutor constructor:
 *         input channels must be 3, 6 or 9).
 *   precision: OIDNX_PRECISION_*; AUTO means fp16 (the pages' resolution of
 *         'auto' when shader-f16 exists, which holds on this GPU).
 * Weights are packed and uploaded to the current device here.
 * Errors: INVALID_ARGUMENT (NULL), INVALID_MODEL, OUT_OF_MEMORY, CUDA.  */
oidnx_status oidnx_filter_create(const void* blob, size_t bytes, int precision,
                                 oidnx_filter** out);

/* Bind an image: which = OIDNX_IMAGE_*; device_ptr points at float4 RGBA
 * pixels, row-major; row_stride_bytes 0 means width*16.  Inputs are read,
 * the output is written ("denoise.ts": colour, then albedo and normal; the
 * output keeps the input colour's alpha).  The pointer is used by every later
 * execute until rebound.  Errors: INVALID_ARGUMENT.  */
oidnx_status oidnx_filter_set_image(oidnx_filter* f, int which, void* device_ptr,
                                    size_t row_stride_bytes);

/* Integer parameters ("denoise.ts", NativeDenoiseOptions, and the executor's
 * shapeCacheSize):
 *   "width", "height"    image size (> 0)
 *   "hdr"                0 LDR, 1 HDR
 *   "transfer"           OIDNX_TRANSFER_LOG (1); PU (0) is UNSUPPORTED (its
 *                        curve is not defined by the pages)
 *   "maxTileSize"        0 = whole image as one tile, else the tile limit
 *   "overlap"            -1 = alignUp(receptive field / 2, 16) (default)
 *   "shapeCacheSize"     number of per-shape plans kept (LRU, default 2)
 *   "keepActivations"    1 = no activation-slot reuse (for debug reads)
 *   "subpixelDecoder"    1 = decoder convs with even extents compute the
 *                        upsampled part as parity-class 2x2 taps on the
 *                        low-resolution source (fewer MMAs; weights of one
 *                        class are summed, then rounded to fp16, or for fp32
 *                        storage summed in double and rounded to fp32),
 *                        reading parity-split copies of the skip sources
 *                        (default);
 *                        0 builds the upsampled halo in shared memory
 *   "fuseLayers"         1 = with fp16 storage, enc_conv0+enc_conv1 and
 *                        dec_conv1b+dec_conv0 each run as one kernel that
 *                        never stores the first conv's output; default 0:
 *                        on GB300 the separate kernels are faster (the MMAs
 *                        of these layers are bound by shared-memory operand
 *                        reads, which fusion does not reduce)
 *   "fuseInput"          1 = with fp16 storage, frames run one tile at a time
 *                        and the sub-pixel dec_conv1a, the input pass runs
 *                        inside enc_conv0's kernel: the packed input is
 *                        built in shared memory from the source images and
 *                        only its column-parity copy is stored; the results
 *                        equal the separate kernels' bit for bit.  Default
 *                        0 (on GB300 the separate kernels, which overlap
 *                        each other, are as fast).  Off with keepActivations.
 *   "fuseTail"           1 = with fp16 storage, dec_conv1b and dec_conv0 (and
 *                        the output pass when "fuseOutput" is 1) run as one
 *                        kernel, once per tile of a stacked frame:
 *                        dec_conv1b's 32-channel map stays in tensor memory
 *                        and is never stored; the results equal the
 *                        separate kernels' bit for bit (default).  Off with
 *                        keepActivations or fuseLayers 1.
 *   "stackTiles"         frames of several equal tiles stack them: each conv
 *                        runs once over a group of tiles (zero rows between
 *                        them), the input pass and the final conv per tile.
 *                        0 = groups as large as 16 GiB of activations allow
 *                        (default), 1 = tile by tile, n = at most n tiles.
 *                        Off with keepActivations, fuseLayers or fuseOutput 0.
 *                        get_int "stackedTiles": tiles per group of the
 *                        committed plan
 *   "fuseOutput"         1 = the output pass runs in the final conv's
 *                        epilogue (the network output is then not stored
 *                        unless "keepActivations" is 1); default 1
 *   "shapeKernels"       1 = conv layers of the common tile shapes (rows per
 *                        tile, rows stacked per MMA, epilogue) run kernels
 *                        compiled for that shape (default); 0 = every conv
 *                        runs the form that selects its issue sequence at
 *                        run time.  Both issue the same MMAs in the same
 *                        order, so the results are the same bits.
 *   "profile"            1 = record per-kernel events on every execute
 * Errors: INVALID_ARGUMENT for unknown names or out-of-range values.  */
oidnx_status oidnx_filter_set_int(oidnx_filter* f, const char* name, int value);
/* Read-back of the same names plus "inputChannels", "tiles" (grid size of
 * the committed configuration) and "precision" (resolved, 1 or 2).  */
oidnx_status oidnx_filter_get_int(oidnx_filter* f, const char* name, int* value);

/* Float parameters: "inputScale" (HDR only; 0 means 1, as the config word of
 * "program.ts").  Errors: INVALID_ARGUMENT.  */
oidnx_status oidnx_filter_set_float(oidnx_filter* f, const char* name, float value);

/* Validate the parameters and images, plan the tile grid, create (or fetch
 * from the LRU cache) the per-tile-shape network plan: the set-up half of
 * "denoise.ts", recordDenoiseExecution (its dimension checks, the overlap
 * alignUp(receptiveField / 2, 16) and the planTileGrid call), with the plan
 * lookup of "nativeUNet.ts", _execution / _createExecution, made ahead of
 * the first run as NativeUNetExecutor.prewarm does.  Synchronous on the
 * host; allocates device memory.  Errors: INVALID_ARGUMENT, UNSUPPORTED,
 * OUT_OF_MEMORY, CUDA.  */
oidnx_status oidnx_filter_commit(oidnx_filter* f);

/* Run the denoise on `stream`: for every tile, in order, the input pass,
 * the network and the output pass into the tile's output rectangle (the
 * per-tile loop of "denoise.ts", recordDenoiseExecution: inputShader,
 * executePacked, outputShader on one queue).  Asynchronous; the first run of
 * a configuration records a CUDA graph that later runs replay, as
 * "program.ts", recordNetwork records the second execution of a network.
 * Errors: NOT_COMMITTED, RELEASED, CUDA.  */
oidnx_status oidnx_filter_execute(oidnx_filter* f, void* stream);

/* Same denoise with HOST images (float4 RGBA, width*16 bytes per row):
 * copies the inputs to filter-owned device buffers, executes on `stream`,
 * and copies the output back; returns once the output is in `output`.
 * Inputs not used by the model (albedo/normal for 3-channel models) may be
 * NULL.  The device images bound by set_image are not touched.
 * Errors: as execute, plus INVALID_ARGUMENT, OUT_OF_MEMORY.  */
oidnx_status oidnx_filter_execute_host(oidnx_filter* f, const float* color,
                                       const float* albedo, const float* normal,
                                       float* output, void* stream);

/* The same, returning once the work is enqueued, for frame streams.  The
 * inputs are uploaded on an internal stream into one of two filter-owned
 * device staging sets, the denoise runs on `stream`, and the output is
 * downloaded on a second internal stream.  Consecutive calls alternate the
 * sets, so that one call's upload and another's download overlap a
 * denoise.  The caller keeps the input buffers unchanged and does not read
 * `output` until oidnx_filter_wait_host has returned; pinned host memory
 * gives the full link bandwidth.  Errors: as oidnx_filter_execute_host.  */
oidnx_status oidnx_filter_execute_host_async(oidnx_filter* f, const float* color,
                                             const float* albedo, const float* normal,
                                             float* output, void* stream);

/* Block until every download enqueued by the host-buffer calls of `f` has
 * finished.  Errors: RELEASED, CUDA.  */
oidnx_status oidnx_filter_wait_host(oidnx_filter* f);

/* The network alone (conv layers enc_conv0 .. dec_conv0) on one packed input
 * ("nativeUNet.ts", execute / executePacked):
 *   packed_in: device, the activation layout above with C = input channels;
 *   out:       device, [h][w][4] floats (lane 3 zero);
 *   w, h > 0; odd extents are allowed (pools round up).
 * Uses the plan cache of the filter.  Errors: INVALID_ARGUMENT, CUDA.  */
oidnx_status oidnx_network_execute(oidnx_filter* f, const void* packed_in, int w,
                                   int h, void* out, void* stream);

/* The same network forward as oidnx_network_execute, for callers that must
 * not allocate device memory once set-up is over: a renderer whose device
 * memory budget is fixed after start-up (an allocation can synchronise the
 * device and stall the frame), a plug-in whose host application owns all
 * device memory, or any path where an allocation may not fail or wait.
 * The pages have no counterpart of this call; it is an addition of this
 * library.
 *   - Allocates nothing: no cudaMalloc/cudaFree, no plan is created or
 *     cached.  The intermediate activations live in one library-owned
 *     device array of 48 MiB (50331648 bytes), present on every GPU that
 *     loads the library until the process exits.
 *   - Limit: the input must fit that array: fp16 up to 384 x 384 pixels,
 *     fp32 up to 256 x 256 (other shapes: whatever the liveness plan of
 *     the activations fits in 48 MiB).  Larger inputs fail with
 *     INVALID_ARGUMENT and a message stating the bytes needed.
 *   - packed_in / out: as for oidnx_network_execute (the kernels read the
 *     input and write the output in place, without copies).
 *   - Set-up: oidnx_filter_create looks up the array's device address on
 *     the device current at creation; that look-up is when the driver loads
 *     the array (device code loads lazily by default), so its memory is
 *     taken at set-up and calls on that device allocate nothing.  The first
 *     call on any other device makes the look-up itself: make it before any
 *     stream capture and off the frame path.
 *   - All calls on a device share the one array, and it keeps the previous
 *     call's contents (every activation is fully written before it is
 *     read, so nothing is cleared).  Calls that overlap on the GPU (on
 *     different streams, or from several threads) race on the array and
 *     give undefined results: serialise them.
 *   - Device-side timeouts are reported by oidnx_filter_sync_status.
 * Errors: INVALID_ARGUMENT, RELEASED, UNSUPPORTED, CUDA.  */
oidnx_status oidnx_network_execute_noalloc(oidnx_filter* f, const void* packed_in, int w,
                                           int h, void* out, void* stream);

/* The output pass alone on one rectangle ("denoise.ts", outputShader): for
 * every pixel, rgb = sanitize(net.rgb, 0, hdr ? FLT_MAX : 1); with hdr,
 * rgb = (2^rgb - 1) / inputScale (the inverse 'log' transfer), correctly
 * rounded to fp32; alpha = the colour's alpha, copied bit for bit.
 *   net:    device, [h][w] float4 (the network output; lane 3 ignored);
 *   color:  device, float4 RGBA rows of color_stride bytes (0: w*16);
 *   output: device, float4 RGBA rows of output_stride bytes (0: w*16);
 *   hdr 0 or 1; input_scale finite and >= 0 (0 means 1; used with hdr).
 * w > 0, 0 < h <= 65535; pointers and strides 16-byte aligned.  The caller
 * owns every buffer; enqueued on `stream`.  The denoise runs the same
 * per-pixel code for each tile, inside the final conv's epilogue.
 * Errors: INVALID_ARGUMENT, RELEASED, CUDA.  */
oidnx_status oidnx_output_pass(oidnx_filter* f, const void* net, int w, int h, const void* color,
                               size_t color_stride, void* output, size_t output_stride, int hdr,
                               float input_scale, void* stream);

/* Wait for the filter's work, then report and clear the device error word:
 * OK, or TIMEOUT if a kernel's bounded wait gave up (its output is then
 * undefined).  The device-side counterpart of the error packets of
 * "program.ts" (an "ERRO" packet carries the failure of a recorded run);
 * the pages have no device error word, since WebGPU reports failed work
 * through its own error scopes.  Errors: CUDA.  */
oidnx_status oidnx_filter_sync_status(oidnx_filter* f);

/* Failure-detection probe: launch, on `stream`, one thread that waits on a
 * device barrier nothing will complete, bounded by limit_us (1 .. 1e6).  The
 * wait gives up after the limit, records a timeout bit in the filter's device
 * error word and returns, leaving the context usable; the next
 * oidnx_filter_sync_status reports OIDNX_ERR_TIMEOUT.  This exercises the
 * same bounded wait every kernel of the library uses.  Errors:
 * INVALID_ARGUMENT, CUDA.  */
oidnx_status oidnx_debug_wait_probe(oidnx_filter* f, unsigned int limit_us, void* stream);

/* Per-kernel timing of the next execute (or network_execute) only, like
 * "nativeUNet.ts" profileNextExecution (timestamp writes around every pass
 * of the next execution only).  */
oidnx_status oidnx_profile_next(oidnx_filter* f);

/* JSON of the last profiled execution, the record of "nativeUNet.ts",
 * getLastExecutionProfile ({totalMs, layers[{id, durationMs}]} with the ids
 * "input-pack" and the node names), extended with counts:
 * {"totalMs":T,"layers":[{"id":"input-pack","ms":..,"flop":..,"bytes":..,
 *  "launches":..,"mmaFlop":..},...,{"id":"output",...}]} summed over the
 * launches (per tile; with stacked tiles each conv launches once per group);
 * flop and bytes are the algorithmic counts (logical channels; each input
 * activation read once, each output written once); mmaFlop is what the
 * tensor cores execute (padded tiles and channels; 4 of the 9 taps on the
 * upsampled channels of a sub-pixel decoder, three tf32 products per fp32
 * product; 0 where not counted).  Synchronises with the profiled work.
 * Errors: INVALID_ARGUMENT (cap too small or nothing profiled), CUDA.  */
oidnx_status oidnx_get_profile(oidnx_filter* f, char* json, size_t cap);

/* JSON of owned resources: weight bytes, arena bytes, cached plans, graphs,
 * retired plans still waiting for the stream ("nativeUNet.ts",
 * getResourceInfo).  */
oidnx_status oidnx_get_resource_info(oidnx_filter* f, char* json, size_t cap);

/* Copy one stored activation of the last network run on this filter to
 * host memory as float32 [h_l][w_l][C_l] with logical channels: the value
 * buffers of the plan built by "nativeUNet.ts", _createExecution (one per
 * node output, the packed input at index -1), read back the way executeCPU
 * reads the network output.  This is what the per-layer parity checks read.
 * layer: 0 = packed network input, 1..16 = outputs of enc_conv0 ..
 * dec_conv0 in network order (enc_conv1..enc_conv4 store their pooled
 * outputs).  Valid for every layer only with "keepActivations" = 1 (which
 * turns "fuseTail" off) and "fuseLayers" = 0 (the output of a layer fused with the next one is never
 * stored, nor is the network output of a denoise whose output pass ran in
 * the final conv's epilogue without "keepActivations": such reads fail
 * with INVALID_ARGUMENT); the required size is returned in *bytes_needed.
 * Synchronises.
 * Errors: INVALID_ARGUMENT, CUDA.  */
oidnx_status oidnx_debug_read_activation(oidnx_filter* f, int layer, void* host_dst,
                                         size_t cap, size_t* bytes_needed);

/* Message of the last failed call on this thread ("" if none).  */
const char* oidnx_last_error(void);

/* Release a filter and everything it owns, after the work it queued has
 * finished: "nativeUNet.ts", dispose (idempotent, destroys every tracked
 * buffer), with the deferred destruction of _execution's evicted plans,
 * which waits for onSubmittedWorkDone before destroying buffers that
 * commands in flight may still use.  NULL is ignored.  Calls on the handle
 * afterwards are invalid.  */
void oidnx_filter_release(oidnx_filter* f);

/* ---- one conv layer (3x3 same-padded conv + bias (+ReLU)) --------------
 * "nativeUNet.ts", createConvShader / createTiledConvShader.
 * weight: host OIHW float32 [cout][cin][3][3]; bias: host float32 [cout].
 * precision: OIDNX_PRECISION_FP16 (tensor cores, fp32 accumulate) or FP32.
 * in / out: device tensors in the activation layout above (cin / cout
 * channels, w x h pixels, rows of w pixels), 16-byte aligned.  relu must be
 * 1 (the hidden layers' form; the final layer runs inside the network).
 * The caller owns in, out and the stream; the conv owns its packed weights
 * and bias until oidnx_conv_release (NULL is ignored).  execute enqueues on
 * `stream` and returns.
 * Errors: create: INVALID_ARGUMENT (NULL or non-positive sizes, unknown
 * precision), UNSUPPORTED (cout > 256), CUDA (allocation failures too); execute:
 * INVALID_ARGUMENT (NULL, sizes, misaligned pointers), UNSUPPORTED
 * (relu = 0), CUDA.  */
oidnx_status oidnx_conv_create(const float* weight, const float* bias, int cout,
                               int cin, int precision, oidnx_conv** out);
oidnx_status oidnx_conv_execute(oidnx_conv* c, const void* in, void* out, int w,
                                int h, int relu, void* stream);
void oidnx_conv_release(oidnx_conv* c);

/* ---- host-only helpers (no GPU needed) --------------------------------- */

/* Tile grid of a width x height image ("denoise.ts", planTileGrid use):
 * writes up to `cap` tiles as 8 ints each (input x, y, w, h, output x, y,
 * w, h) and the tile count to *count.  overlap < 0 means the default.
 * Errors: INVALID_ARGUMENT (sizes, or maxTileSize too small for overlap).  */
oidnx_status oidnx_plan_tiles(int width, int height, int max_tile_size, int overlap,
                              int* rects, int cap, int* count);

/* Default overlap, alignUp(receptive field / 2, 16), for the 4-level
 * U-Net: the one-sided dependency radius rounded up to 16.  */
int oidnx_default_overlap(void);

/* Version string of the library.  */
const char* oidnx_version(void);

#ifdef __cplusplus
}
#endif

#endif /* OIDNX_H */

// oidnx_network_execute_noalloc: the network forward with its intermediate
// activations in a fixed, library-owned device array instead of memory the
// filter allocates.
//
// Who needs it: callers that must not allocate device memory on their frame
// path, for example a renderer whose device-memory budget is fixed after
// start-up (cudaMalloc/cudaFree can synchronise the whole device and stall
// the frame), a plug-in running under a host application whose own memory
// manager owns all device memory, or any code that runs where a failed or
// slow allocation is not an option.  They create the filter (weights are
// uploaded once, at set-up) and then run the network without any further
// allocation: the caller passes the packed input and the output buffer, and
// every intermediate activation lives in the array below.
//
// The array is a file-scope __device__ variable of kNoAllocScratchBytes
// (48 MiB).  Every GPU that loads this library's device code holds that much
// memory until the process exits.  The driver places it when it loads this
// file's device code on a device; CUDA loads device code lazily (at first
// use) by default, and the first use is the address look-up below, which
// oidnx_filter_create makes on the device it creates the filter on.  So the
// array is taken at set-up, not by the first frame.  It is enough for fp16
// inputs up to 384 x 384 pixels and fp32 inputs up to 256 x 256; larger
// inputs are rejected with OIDNX_ERR_INVALID_ARGUMENT and a message giving
// the bytes needed.
#include <mutex>

#include "../../include/oidnx.h"
#include "internal.h"

namespace oidnx {
oidnx_status report_error(oidnx_status status, const char* message);
oidnx_status network_enqueue_in_arena(oidnx_filter* f, const void* in, int w, int h, void* out,
                                      void* arena, size_t cap, cudaStream_t s);
oidnx_status noalloc_scratch_address(void** out);
}  // namespace oidnx

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(48) << 20;
constexpr int kMaxDevices = 64;

// Device-side scratch shared by every call on a device.  In host code this
// name is only a stand-in for the symbol, not a device address: the address
// comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

// Once per device, with that device current: look up the array's device
// address (the driver loads this file's device code, and so places the
// array, at the first look-up on a device).  oidnx_filter_create calls this
// for its device; later calls on that device only read the cached address.
oidnx_status oidnx::noalloc_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return oidnx::report_error(OIDNX_ERR_CUDA, "network_execute_noalloc: cudaGetDevice failed");
  if (dev < 0 || dev >= kMaxDevices)
    return oidnx::report_error(OIDNX_ERR_UNSUPPORTED,
                               "network_execute_noalloc: device index beyond 63");
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr)
      return oidnx::report_error(OIDNX_ERR_CUDA,
                                 "network_execute_noalloc: cudaGetSymbolAddress of the scratch "
                                 "array failed");
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return OIDNX_OK;
}

extern "C" oidnx_status oidnx_network_execute_noalloc(oidnx_filter* f, const void* packed_in,
                                                      int w, int h, void* out, void* stream) {
  void* scratch = nullptr;
  oidnx_status st = oidnx::noalloc_scratch_address(&scratch);
  if (st != OIDNX_OK) return st;
  // Every intermediate activation is fully written before it is read, so
  // the array's contents from an earlier call need no clearing.
  return oidnx::network_enqueue_in_arena(f, packed_in, w, h, out, scratch, kNoAllocScratchBytes,
                                         static_cast<cudaStream_t>(stream));
}

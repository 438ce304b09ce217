// dpclip_norms_hutch_noalloc: the Hutch norm estimate without any workspace
// from the caller and without any allocation by the library.
//
// Some callers cannot allocate device memory at the point where they need the
// per-sample norms: a host framework that calls into this library from a
// callback in which device allocation is forbidden after initialisation, a
// process whose device memory is entirely handed out by another allocator, or
// a latency-critical loop in which an allocation could stall on the device.
// This entry point serves them with scratch memory that exists for the whole
// life of the process: a file-scope __device__ array of
// DPCLIP_NOALLOC_SCRATCH_BYTES, created when the library is loaded on a GPU
// and held by every GPU that loads the library until the process exits.
//
// In host code the array's name only stands for the array: it is not a device
// address.  The address is obtained once per device and context, with that
// device current, through cudaGetSymbolAddress on the first call made there
// (so make that first call before any stream capture), and is then passed to
// the same kernels as dpclip_norms_hutch uses.  A device reset destroys the
// context and the array with it; the next call sees the new context and
// looks the address up again.
//
// All calls share the one array and it keeps the last call's contents; the
// call clears the parts that must start at zero.  Calls that can overlap on
// the GPU (on different streams, or from several host threads) race on the
// array: serialise them, e.g. by issuing them on one stream.  A bounded wait
// that expires records its error in the array's control word, which
// dpclip_noalloc_status reads.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"

namespace dpclip {
namespace {

__device__ __align__(256) uint8_t g_noalloc_scratch[DPCLIP_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

using CtxGetCurrentFn = PFN_cuCtxGetCurrent_v4000;

CtxGetCurrentFn ctx_get_current_fn() {
  static CtxGetCurrentFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (CtxGetCurrentFn) nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  return fn;
}

// The device address of g_noalloc_scratch on the current device, looked up
// once per device and context.  Returns a status.
int scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return DPCLIP_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return DPCLIP_ERR_UNSUPPORTED;
  CtxGetCurrentFn get_ctx = ctx_get_current_fn();
  if (!get_ctx) return DPCLIP_ERR_CUDA;
  // no context is current yet on a thread where the runtime has not been used
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return DPCLIP_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!ctx || !g_scratch_ptr[dev] || g_scratch_ctx[dev] != ctx) {
    // the lookup makes the device's primary context current if it was not
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
      (void)cudaGetLastError();
      g_scratch_ptr[dev] = nullptr;
      return DPCLIP_ERR_CUDA;
    }
    if (get_ctx(&ctx) != CUDA_SUCCESS || !ctx) return DPCLIP_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
    g_scratch_ctx[dev] = ctx;
  }
  *out = g_scratch_ptr[dev];
  return DPCLIP_OK;
}

}  // namespace
}  // namespace dpclip

extern "C" int dpclip_norms_hutch_noalloc(const void* A, const void* G, int B, int T, int d,
                                          int p, int dtype, int k, uint64_t seed,
                                          uint64_t offset, float* sqnorms,
                                          dpclip_stream_t stream) {
  if (!A || !G || !sqnorms) return DPCLIP_ERR_INVALID_ARG;
  size_t need = 0;
  const int st = dpclip_workspace_size(DPCLIP_OP_NORMS_HUTCH, B, T, d, p, dtype, k, &need);
  if (st != DPCLIP_OK) return st;
  if (need > (size_t)DPCLIP_NOALLOC_SCRATCH_BYTES) return DPCLIP_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st2 = dpclip::scratch_for_current_device(&scratch);
  if (st2 != DPCLIP_OK) return st2;
  return dpclip_norms_hutch(A, G, B, T, d, p, dtype, k, seed, offset, sqnorms, scratch,
                            (size_t)DPCLIP_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" int dpclip_noalloc_status(dpclip_stream_t stream) {
  void* scratch = nullptr;
  const int st = dpclip::scratch_for_current_device(&scratch);
  if (st != DPCLIP_OK) return st;
  return dpclip_workspace_status(scratch, stream);
}

// ssd_fwd_noalloc: the SSD forward for callers that cannot allocate device
// memory.  Some callers own no allocator at all, or must not call one while
// they run: a host runtime whose memory pool already claimed the device's
// memory, a plugin that is handed only its input and output buffers, or a
// latency-critical loop that cannot pay for cudaMalloc, which may synchronise
// the device and take milliseconds.  This entry point needs no workspace from
// them: its scratch lives in one file-scope device array of fixed size that
// the library holds on every GPU that loads it, until the process exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "ssd_internal.h"

namespace {

// The fixed scratch: large enough for the forward workspace of small and
// medium problems (SSD_NOALLOC_SCRATCH_BYTES in ssd.h).
constexpr size_t kScratchBytes = SSD_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Cached {
  CUcontext ctx;
  void* addr;
};
Cached g_cache[kMaxDevices] = {};

// The driver context current on this thread (null if the query is unavailable).
CUcontext current_context() {
  static PFN_cuCtxGetCurrent_v4000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuCtxGetCurrent_v4000>(nullptr);
    return reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  }();
  CUcontext c = nullptr;
  if (fn) fn(&c);
  return c;
}

// Device address of the scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up with
// the device current, once per device and driver context, and cached with
// the context: after cudaDeviceReset, or under another context, it is looked
// up again instead of reusing an address of a context that is gone.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSD_ERR_CUDA;
  const CUcontext ctx = current_context();
  std::lock_guard<std::mutex> lk(g_mu);
  Cached& c = g_cache[dev];
  if (!c.addr || !ctx || c.ctx != ctx) {
    // (the lookup also makes the device's primary context current if this
    // thread had none, so the context is read again after it)
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SSD_ERR_CUDA;
    c.addr = p;
    c.ctx = current_context();
  }
  *out = c.addr;
  return SSD_OK;
}

}  // namespace

extern "C" {

size_t ssd_noalloc_scratch_bytes(void) { return kScratchBytes; }

int ssd_fwd_noalloc(const ssd_shape* shape, const void* x, const void* dt, const float* dt_bias,
                    const float* A, const void* B, const void* C, const float* D,
                    const float* init_states, void* y, float* final_states, void* stream) {
  const size_t need = ssd_fwd_workspace_size(shape);
  if (need == 0) return SSD_ERR_INVALID_ARG;
  if (need > kScratchBytes) return SSD_ERR_WORKSPACE;
  void* scratch = nullptr;
  const int st = scratch_address(&scratch);
  if (st != SSD_OK) return st;
  // Nothing in the scratch has to start at zero: the forward writes every
  // byte of its workspace that it later reads, within the same call.
  return ssd_fwd(shape, x, dt, dt_bias, A, B, C, D, init_states, y, final_states, scratch,
                 kScratchBytes, stream);
}

}  // extern "C"

// ssd_fwd_noalloc: the SSD forward for callers that cannot allocate device
// memory.  Some callers own no allocator at all, or must not call one while
// they run: a host runtime whose memory pool already claimed the device's
// memory, a plugin that is handed only its input and output buffers, or a
// latency-critical loop that cannot pay for cudaMalloc, which may synchronise
// the device and take milliseconds.  This entry point needs no workspace from
// them: its scratch lives in one file-scope device array of fixed size that
// the library holds on every GPU that loads it, until the process exits.
#include <mutex>

#include "ssd_internal.h"

namespace {

// The fixed scratch: large enough for the forward workspace of small and
// medium problems (see SSD_NOALLOC_SCRATCH_BYTES in ssd.h).
constexpr size_t kScratchBytes = (size_t)64 << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device.  In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached.
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SSD_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return SSD_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
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

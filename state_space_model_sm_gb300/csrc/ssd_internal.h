// Internal declarations shared by the translation units of libssd.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/ssd.h"

namespace ssd {

// Problem dimensions after host validation.
struct Dims {
  int B, T, H, P, N, G, L, nc;
  int in_bf16, out_bf16;
  // log2 of the 64-wide parts a head is split into on the tensor-core path
  // (tc_dims): H and P then count parts; dt, dt_bias, A, D and the per-head
  // vectors delta / a are indexed by the head, (b * H + h) >> hs
  int hs = 0;
};

// Device address of the status word of the current device (defined in
// ssd_api.cu).  Kernels whose bounded waits expire store SSD_ERR_TIMEOUT there.
int* device_status_ptr();

// The opt-in NaN / Inf scan of outputs (ssd_set_check_finite): whether it is
// on, and one scan launch over n values (f32, or bf16 when is_bf16).
bool check_finite_enabled();
cudaError_t launch_check_finite(const void* p, int64_t n, bool is_bf16, cudaStream_t s);

// Brackets one kernel launch: counts it and, when profiling is enabled,
// records CUDA events around it on the launch stream (ssd_profile.cu).
class LaunchScope {
 public:
  LaunchScope(const char* name, cudaStream_t s);
  ~LaunchScope();
  LaunchScope(const LaunchScope&) = delete;
  LaunchScope& operator=(const LaunchScope&) = delete;

 private:
  const char* name_;
  cudaStream_t s_;
  cudaEvent_t start_ = nullptr;
};

#define SSD_LAUNCH(name, stream, ...)                  \
  do {                                                 \
    ::ssd::LaunchScope ssd_scope_(name, stream);       \
    __VA_ARGS__;                                       \
  } while (0)

// Programmatic dependent launch.  A kernel launched with launch_pdl may
// start while the previous kernel on its stream is still running (once every
// CTA of that one has called griddep_launch_dependents or exited), so its
// prologue (TMEM, barriers, operand loads that depend on no earlier kernel)
// overlaps that kernel's last wave.  Every such kernel calls griddep_wait
// before it reads anything an earlier kernel of the call wrote, or writes
// anything an earlier kernel may still read; griddep_wait returns once the
// previous grid has completed and its writes are visible.  The first kernel
// of an ssd_fwd / ssd_bwd call is launched normally: its inputs may come from
// the caller's previous kernel.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// ---------------------------------------------------------------- pointers
// delta = softplus(dt + dt_bias): the linear branch above 20, where
// log(1 + e^v) equals v in fp32.
__device__ __forceinline__ float dt_softplus(float v) { return v > 20.f ? v : log1pf(expf(v)); }

struct FwdArgs {
  const void* x;
  const void* dt;
  const float* dt_bias;
  const float* A;
  const void* B;
  const void* C;
  const float* D;
  const float* init;
  void* y;
  float* final_state;
};

struct BwdArgs {
  FwdArgs f;
  const void* dy;
  const float* dfinal;
  float* dx;
  float* ddt;
  float* dA;
  float* dB;
  float* dC;
  float* dD;
  float* ddt_bias;
  float* dinit;
};

// Workspace carving for the generic path.
struct FwdWs {
  float* delta;  // (B, H, nc, L)
  float* acs;    // (B, H, nc, L)
  float* S;      // (B, nc, H, P, N)
  float* Hprev;  // (B, nc, H, P, N)
  float* CB;     // (B, nc, G, L, L)
  void* Himg = nullptr;  // optional (B, nc, H) bf16 hi/lo images of Hprev (tensor-core path)
  float* seg = nullptr;  // optional two-level state passing scratch (see seg_max_segments)
};

// Two-level state passing (image path) for shapes with few (batch, head)
// pairs: the chunks are cut into K segments processed in parallel.  The
// workspace holds 2 * B * seg_max_segments(d) * H * P * N floats for it;
// 0 segments means the single-level walk only.
int seg_max_segments(const Dims& d);

struct BwdWs {
  FwdWs f;
  float* dHs;    // (B, nc, H, P, N)
  float* dS;     // (B, nc, H, P, N)
  float* dlast;  // (B, H, nc, nsplit) partial sums of dlast
  float* dyx;    // (B, nc, H, L, L)
  float* qrow;   // (B, H, nc, L)  delta_s <x_s, state part of u_s>
  float* ddir;   // (B, H, nc, L)  <x_s, u_s>
  float* ycs;    // (B, H, nc, L)  exp(a_l) <dy_l, H_c C_l>
  float* dBh;    // (B, T, H, N)
  float* dCh;    // (B, T, H, N)
  float* part;   // (B, H, nc, 3)  per-chunk partial sums of dA, ddt_bias, dD
  void* dSimg = nullptr;  // optional bf16 hi/lo images of dS (tensor-core path)
};

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Generic SIMT path (ssd_simt.cu).  Return cudaGetLastError() of the launches.
cudaError_t simt_forward(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s);
cudaError_t simt_backward(const Dims& d, const BwdArgs& a, const BwdWs& w, cudaStream_t s);
// The bandwidth-bound steps shared by both paths: chunk_cumsum (delta, a)
// and state_passing (Hprev, final) on the generic kernels.
void simt_cumsum(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s);
void simt_state_passing(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s);

// The first passes of context parallelism: the front of the forward (cumsum,
// chunk states, state passing: final state and Hprev) and the per-chunk
// dstates of the backward (dH^scan_c from dy, C, delta, a).
void simt_front(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s);
void simt_dstates(const Dims& d, const void* dy, const void* C, const float* delta,
                  const float* acs, float* dHs, cudaStream_t s);
cudaError_t tc_front_final(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s);
cudaError_t tc_dstates(const Dims& d, const void* dy, const void* C, const float* delta,
                       const float* acs, float* dHs, cudaStream_t s);
// dinit = G_0 of G_c = dH^scan_c + exp(a_c[L-1]) G_{c+1}, G_nc = dfinal (or 0).
void cp_dinit_chain(const Dims& d, const float* dHs, const float* acs, const float* dfinal,
                    float* dinit, cudaStream_t s);

int simt_state_passing_bwd(const Dims& d, const float* dHs, const float* acs, const float* Hprev,
                           const float* dfinal, float* dS, float* dlast, float* dinit,
                           void* dSimg, const void* Himg, float* seg,
                           cudaStream_t s);  // returns the dlast partials per chunk
void simt_param_grads(const Dims& d, const float* part, float* dA, float* ddt_bias, float* dD,
                      cudaStream_t s);

// Head blocks per group of the chunk kernels' two row tiles (see
// tc_scan_blocks below).
struct HeadBlocks {
  int heavy, light;
  int max() const { return heavy > light ? heavy : light; }
};

// Workspace of the tensor-core backward.
struct TcBwdWs {
  float* delta;   // (B, H, nc, L)
  float* acs;     // (B, H, nc, L)
  float* S;       // (B, nc, H, P, N)
  float* dHs;     // (B, nc, H, P, N)
  void* Himg;     // (B, nc, H) split-bf16 shared-memory images of Hprev
  void* dSimg;    // (B, nc, H) split-bf16 shared-memory images of dS
  float* dlast;   // (B, H, nc, <= 16) partials
  float* rowsum;  // (B, H, nc, L) strict row sums of M (dC kernel)
  float* colsum;  // (B, H, nc, L) strict column sums of M (dB kernel)
  float* ycs;     // (B, H, nc, L)
  float* qrow;    // (B, H, nc, L)
  float* ddir;    // (B, H, nc, L)
  float* ddiag;   // (B, H, nc, L)  <dy_t, x_t>
  float* dBp;     // (B, T, G, nblk, N) head-block partials of dB
  float* dCp;     // (B, T, G, nblk, N)
  float* part;    // (B, H, nc, 3)
  int* done;      // finalize blocks done (zeroed by the chunk_state recompute)
  float* seg;     // two-level state passing scratch, or nullptr
  HeadBlocks nb;  // head blocks of dB / dC (read from the launch table once per call)
};

// tcgen05 path (ssd_tc.cu): bf16 inputs, headdim 64, d_state 64 / 128,
// chunk 128 / 256, an even number of heads per group.
bool tc_forward_supported(const Dims& d);
// The tensor-core path's view of a shape: headdim 128 as two 64-wide parts
// per head (hs = 1); other shapes unchanged.
Dims tc_dims(const Dims& d);
cudaError_t tc_forward(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s);
// Head blocks per group of the chunk kernels' row tiles: `heavy` for the tile
// with more column panels (first in the grid), `light` for the other (chunk
// 256; equal to heavy at chunk 128, one tile).  From the launch table's entry
// for the shape (ssd_scan_set_config), else the built-in rule.  The workspace
// size and the launch read the same table, so they agree as long as the
// entry does not change between the size query and the call.
HeadBlocks tc_bwd_blocks(const Dims& d);
HeadBlocks tc_scan_blocks(const Dims& d);
cudaError_t tc_backward(const Dims& d, const BwdArgs& a, const TcBwdWs& w, cudaStream_t s);

// Tensor map (for TMA) of a (B, T, X, inner) bf16 tensor, 128-byte swizzle,
// boxes of 64 inner elements x box_x x box_t rows x 1; false if the driver
// entry point is missing or rejects the layout (ssd_chunk_tc.cu).
bool make_tma_map(CUtensorMap* m, const void* ptr, int inner, int X, int T, int B, int box_x,
                  int box_t);
// Tensor map of a (rows, inner) fp32 matrix, 128-byte swizzle, boxes of
// box_inner (32: 128 bytes) x box_rows, for TMA stores.
bool make_tma_map_f32(CUtensorMap* m, void* ptr, int inner, int64_t rows, int box_inner,
                      int box_rows);
// Map of an fp32 (B, T, H, 64) tensor (y, dx) for TMA stores: boxes of cols
// (16 or 32) columns x one head x 32 rows, 64- or 128-byte swizzle to match.
bool make_y_map(CUtensorMap* m, void* y, int H, int T, int B, int cols);

// The TMA-fed chunk kernels (ssd_chunk_tc.cu), over (batch, chunk, row tile,
// group, block of nblk heads): chunk_scan (y from the state images in w.Himg),
// and the backward's dC and dB (with the ddA row / column sums and ycs).
// dCout / dBout receive (B, T, G, nblk, N) partials.
cudaError_t tc_chunk_forward(const Dims& d, const FwdArgs& f, const FwdWs& w, HeadBlocks nb,
                             cudaStream_t s);
cudaError_t tc_chunk_backward(const Dims& d, const BwdArgs& a, const TcBwdWs& w, HeadBlocks nb,
                              float* dCout, float* dBout, cudaStream_t s);

// The TMA-fed chunk_state kernels (ssd_state_tc.cu): chunk_cumsum + chunk
// state (writes delta, acs and S; and 0 to *zero when zero is not null), and
// dstates (dHs from dy, C and acs).
cudaError_t tc_chunk_state(const Dims& d, const FwdArgs& f, float* delta, float* acs, float* S,
                           int* zero, cudaStream_t s);
// pdl: launched with launch_pdl (inside a call, after its other kernels).
cudaError_t tc_chunk_dstates(const Dims& d, const void* dy, const void* C, const float* acs,
                             float* dHs, bool pdl, cudaStream_t s);

}  // namespace ssd

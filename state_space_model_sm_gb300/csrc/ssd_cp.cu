// Context (sequence) parallel building blocks.  With the sequence split into
// contiguous segments r = 0 .. R-1, one per rank, the SSD recurrence over a
// segment maps its incoming state affinely:
//     H_out(r) = D_r * H_in(r) + F_r,    D_r[b,h] = exp(A[h] * sum_{t in r} delta_t)
// (F_r: the segment's final state from a zero initial state; the recurrence
// h_t = exp(delta_t A) h_{t-1} + delta_t x_t B_t of "Mamba-2 offers a
// different scaling path", applied over the whole segment).  The incoming
// states are an exclusive scan of these maps over the ranks, and the
// gradients of the outgoing states the same scan in reverse.
#include <cuda_bf16.h>

#include "ssd_internal.h"

namespace ssd {
namespace {

template <typename T>
__device__ __forceinline__ float load_dt(const T* p);
template <>
__device__ __forceinline__ float load_dt<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float load_dt<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

// One warp per (b, h): decay[b, h] = exp(A[h] * sum_t softplus(dt[b,t,h] +
// dt_bias[h])), the sum in fp64.
template <typename Tin>
__global__ void k_segment_decay(const Tin* __restrict__ dt, const float* __restrict__ dt_bias,
                                const float* __restrict__ A, float* __restrict__ decay, int B,
                                int T, int H) {
  const int wid = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (wid >= B * H) return;
  const int b = wid / H, h = wid % H;
  const float bias = dt_bias ? dt_bias[h] : 0.f;
  double s = 0.0;
  for (int t = lane; t < T; t += 32)
    s += (double)dt_softplus(load_dt(dt + ((int64_t)b * T + t) * H + h) + bias);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) decay[wid] = (float)exp((double)A[h] * s);
}

// One thread per element of the (BH, PN) state: acc <- D_k * acc + S_k over
// the ranks k < rank (direction 0, ascending) or k > rank (direction 1,
// descending), starting from zero.
__global__ void k_state_scan(const float* __restrict__ decays, const float* __restrict__ states,
                             float* __restrict__ out, int R, int rank, int direction, int64_t BH,
                             int64_t PN) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= BH * PN) return;
  const int64_t bh = i / PN;
  float acc = 0.f;
  if (direction == 0) {
    for (int k = 0; k < rank; ++k) acc = fmaf(decays[k * BH + bh], acc, states[k * BH * PN + i]);
  } else {
    for (int k = R - 1; k > rank; --k)
      acc = fmaf(decays[k * BH + bh], acc, states[k * BH * PN + i]);
  }
  out[i] = acc;
}

// grid (ceil(PN / 256), H, B): one thread per element of a (b, h) state,
// walking the chunks backwards with the next kPf chunks' dH^scan loads in
// flight: G <- exp(a_c[L-1]) G + dH^scan_c, from G = dfinal (or 0).
__global__ void __launch_bounds__(256)
    k_dinit_chain(const float* __restrict__ dHs, const float* __restrict__ acs,
                  const float* __restrict__ dfinal, float* __restrict__ dinit, int H, int PN,
                  int L, int nc) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x, h = blockIdx.y, b = blockIdx.z;
  if (e >= PN) return;
  const int64_t step = (int64_t)H * PN;
  const float* src = dHs + ((int64_t)b * nc * H + h) * PN + e;
  const float* alast = acs + ((int64_t)b * H + h) * (int64_t)nc * L + (L - 1);
  const int64_t st = ((int64_t)b * H + h) * PN + e;
  float G = dfinal ? dfinal[st] : 0.f;
  constexpr int kPf = 4;
  for (int c1 = nc - 1; c1 >= 0; c1 -= kPf) {
    float v[kPf], dec[kPf];
#pragma unroll
    for (int k = 0; k < kPf; ++k) {
      const int c = c1 - k;
      if (c >= 0) {
        v[k] = src[c * step];
        dec[k] = __expf(alast[(int64_t)c * L]);
      }
    }
#pragma unroll
    for (int k = 0; k < kPf; ++k)
      if (c1 - k >= 0) G = fmaf(dec[k], G, v[k]);
  }
  dinit[st] = G;
}

}  // namespace

void cp_dinit_chain(const Dims& d, const float* dHs, const float* acs, const float* dfinal,
                    float* dinit, cudaStream_t s) {
  const int PN = d.P * d.N;
  const dim3 grid((PN + 255) / 256, d.H, d.B);
  SSD_LAUNCH("k_dinit_chain", s, k_dinit_chain<<<grid, 256, 0, s>>>(dHs, acs, dfinal, dinit, d.H,
                                                                    PN, d.L, d.nc));
}

}  // namespace ssd

extern "C" int ssd_segment_decay(const ssd_shape* shape, const void* dt, const float* dt_bias,
                                 const float* A, float* decay, void* stream) {
  if (!shape || !dt || !A || !decay) return SSD_ERR_INVALID_ARG;
  if (shape->batch < 1 || shape->seqlen < 1 || shape->nheads < 1) return SSD_ERR_INVALID_ARG;
  if (shape->in_dtype != SSD_F32 && shape->in_dtype != SSD_BF16) return SSD_ERR_INVALID_ARG;
  const int64_t warps = shape->batch * shape->nheads;
  if (warps > (int64_t)1 << 30 || shape->seqlen > ((int64_t)1 << 31) - 1) return SSD_ERR_INVALID_ARG;
  const int blocks = (int)((warps + 7) / 8);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int B = (int)shape->batch, T = (int)shape->seqlen, H = (int)shape->nheads;
  if (shape->in_dtype == SSD_BF16)
    SSD_LAUNCH("k_segment_decay", s, ssd::k_segment_decay<__nv_bfloat16><<<blocks, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(dt), dt_bias, A, decay, B, T, H));
  else
    SSD_LAUNCH("k_segment_decay", s, ssd::k_segment_decay<float><<<blocks, 256, 0, s>>>(
        static_cast<const float*>(dt), dt_bias, A, decay, B, T, H));
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

extern "C" int ssd_state_scan(int nranks, int rank, int direction, int64_t bh, int64_t pn,
                              const float* decays, const float* states, float* out,
                              void* stream) {
  if (nranks < 1 || rank < 0 || rank >= nranks || (direction != 0 && direction != 1))
    return SSD_ERR_INVALID_ARG;
  if (bh < 1 || pn < 1 || !decays || !states || !out) return SSD_ERR_INVALID_ARG;
  const int64_t n = bh * pn;
  const int64_t blocks = (n + 255) / 256;
  if (blocks > ((int64_t)1 << 31) - 1) return SSD_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  SSD_LAUNCH("k_state_scan", s, ssd::k_state_scan<<<(unsigned)blocks, 256, 0, s>>>(
      decays, states, out, nranks, rank, direction, bh, pn));
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

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

// decay[b, h] = exp(A[h] * sum_t softplus(dt[b,t,h] + dt_bias[h])), the sum
// in fp64, in two deterministic stages.  Stage 1: grid (ceil(H / 32), B, KT),
// 256 threads; lane = head (a warp's loads at one position are 32
// consecutive heads), warp w sums positions w, w + 8, ... of the block's
// range [kt * span, (kt + 1) * span); the 8 warp sums are added in warp
// order into part[(b * H + h) * KT + kt].
template <typename Tin>
__global__ void __launch_bounds__(256)
    k_segment_decay_part(const Tin* __restrict__ dt, const float* __restrict__ dt_bias,
                         double* __restrict__ part, int T, int H, int KT, int span) {
  __shared__ double red[8][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int h = blockIdx.x * 32 + lane, b = blockIdx.y, kt = blockIdx.z;
  const int t0 = kt * span, t1 = min(T, t0 + span);
  double s = 0.0;
  if (h < H) {
    const float bias = dt_bias ? dt_bias[h] : 0.f;
    const Tin* p = dt + (int64_t)b * T * H + h;
    int t = t0 + warp;
    for (; t + 24 < t1; t += 32) {  // four positions in flight per lane
      const float v0 = load_dt(p + (int64_t)t * H), v1 = load_dt(p + (int64_t)(t + 8) * H);
      const float v2 = load_dt(p + (int64_t)(t + 16) * H), v3 = load_dt(p + (int64_t)(t + 24) * H);
      s += (double)dt_softplus(v0 + bias);
      s += (double)dt_softplus(v1 + bias);
      s += (double)dt_softplus(v2 + bias);
      s += (double)dt_softplus(v3 + bias);
    }
    for (; t < t1; t += 8) s += (double)dt_softplus(load_dt(p + (int64_t)t * H) + bias);
  }
  red[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && h < H) {
    double tot = 0.0;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += red[w][lane];
    part[((int64_t)b * H + h) * KT + kt] = tot;
  }
}

// Stage 2: one thread per (b, h): the KT partials in order, then the decay.
__global__ void __launch_bounds__(256)
    k_segment_decay_finish(const double* __restrict__ part, const float* __restrict__ A,
                           float* __restrict__ decay, int BH, int H, int KT) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= BH) return;
  double s = 0.0;
  for (int k = 0; k < KT; ++k) s += part[(int64_t)i * KT + k];
  decay[i] = (float)exp((double)A[i % H] * s);
}

// positions per stage-1 block: about 4 blocks per SM over the whole grid,
// at least 256 positions a block
int decay_span(const ssd_shape* s, int sms) {
  const int64_t hb = (s->nheads + 31) / 32;
  const int64_t want = 4 * (int64_t)sms;
  int64_t kt = (want + s->batch * hb - 1) / (s->batch * hb);
  const int64_t kt_max = (s->seqlen + 255) / 256;
  if (kt > kt_max) kt = kt_max;
  if (kt < 1) kt = 1;
  return (int)((s->seqlen + kt - 1) / kt);
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

namespace {
bool decay_shape_ok(const ssd_shape* shape) {
  if (!shape || shape->batch < 1 || shape->seqlen < 1 || shape->nheads < 1) return false;
  if (shape->in_dtype != SSD_F32 && shape->in_dtype != SSD_BF16) return false;
  // positions are int in the kernels, with t + span computed: keep seqlen < 2^30
  return shape->batch < 65536 && shape->nheads < ((int64_t)1 << 20) &&
         shape->seqlen < ((int64_t)1 << 30);
}
int current_sms() {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = 148;
  return sms;
}
}  // namespace

extern "C" size_t ssd_segment_decay_workspace_size(const ssd_shape* shape) {
  if (!decay_shape_ok(shape)) return 0;
  const int span = ssd::decay_span(shape, current_sms());
  const int64_t kt = (shape->seqlen + span - 1) / span;
  return (size_t)(shape->batch * shape->nheads * kt) * sizeof(double);
}

extern "C" int ssd_segment_decay(const ssd_shape* shape, const void* dt, const float* dt_bias,
                                 const float* A, float* decay, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  if (!decay_shape_ok(shape) || !dt || !A || !decay) return SSD_ERR_INVALID_ARG;
  const int span = ssd::decay_span(shape, current_sms());
  const int KT = (int)((shape->seqlen + span - 1) / span);
  const int B = (int)shape->batch, T = (int)shape->seqlen, H = (int)shape->nheads;
  if (!workspace || workspace_bytes < (size_t)B * H * KT * sizeof(double) ||
      (reinterpret_cast<uintptr_t>(workspace) & 7))
    return SSD_ERR_WORKSPACE;
  double* part = static_cast<double*>(workspace);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const dim3 grid((H + 31) / 32, B, KT);
  if (shape->in_dtype == SSD_BF16)
    SSD_LAUNCH("k_segment_decay", s, ssd::k_segment_decay_part<__nv_bfloat16><<<grid, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(dt), dt_bias, part, T, H, KT, span));
  else
    SSD_LAUNCH("k_segment_decay", s, ssd::k_segment_decay_part<float><<<grid, 256, 0, s>>>(
        static_cast<const float*>(dt), dt_bias, part, T, H, KT, span));
  const int BH = B * H;
  SSD_LAUNCH("k_segment_decay_finish", s, ssd::k_segment_decay_finish<<<(BH + 255) / 256, 256, 0, s>>>(
      part, A, decay, BH, H, KT));
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

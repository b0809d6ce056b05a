// Generic SIMT kernels of the SSD chunked scan (any headdim / dstate /
// chunk_size within the documented limits, fp32 or bf16 inputs).  fp32 inputs
// always take this path: it keeps full fp32 arithmetic.
//
// Every kernel works on one chunk of one (batch, head) -- or (batch, group) --
// pair and uses the same small building block: a 256-thread block computes a
// 64x64 output tile of sum_k A(m,k) B(k,n), where A(m,k) and B(k,n) are
// element functors (so decay, mask and dt factors are applied on load).
#include <algorithm>

#include "ssd_internal.h"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 64;
constexpr int kTK = 16;
constexpr int kMaxStatePerThread = 64;  // headdim * dstate <= 256 * 64

template <typename T>
__device__ __forceinline__ float ldf(const T* p);
template <>
__device__ __forceinline__ float ldf<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

template <typename T>
__device__ __forceinline__ void stf(T* p, float v);
template <>
__device__ __forceinline__ void stf<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void stf<__nv_bfloat16>(__nv_bfloat16* p, float v) {
  *p = __float2bfloat16_rn(v);
}

__device__ __forceinline__ float softplus_f(float v) { return dt_softplus(v); }
__device__ __forceinline__ float softplus_grad_f(float v) {
  return v > 20.f ? 1.f : 1.f / (1.f + expf(-v));
}

struct TileSmem {
  float As[kTK][kTile + 4];
  float Bs[kTK][kTile + 4];
};

// acc[i][j] += sum_{k in [kb, ke)} fa(m0 + 4*ty + i, k) * fb(k, n0 + 4*tx + j)
// with tx = tid % 16, ty = tid / 16.  A_KC / B_KC say whether the operand is
// contiguous along k in memory; they pick the load order that coalesces.
// Out-of-range m (>= M) or n (>= N) read as zero.  All threads must call it.
template <bool A_KC, bool B_KC, class FA, class FB>
__device__ __forceinline__ void tile_accum(float (&acc)[4][4], int M, int N, int m0, int n0,
                                           int kb, int ke, FA fa, FB fb, TileSmem& sm) {
  const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
  for (int k0 = kb; k0 < ke; k0 += kTK) {
    for (int i = tid; i < kTile * kTK; i += kThreads) {
      int mm, kk;
      if (A_KC) { mm = i >> 4; kk = i & 15; } else { kk = i >> 6; mm = i & 63; }
      const int m = m0 + mm, k = k0 + kk;
      sm.As[kk][mm] = (m < M && k < ke) ? fa(m, k) : 0.f;
    }
    for (int i = tid; i < kTile * kTK; i += kThreads) {
      int nn, kk;
      if (B_KC) { nn = i >> 4; kk = i & 15; } else { kk = i >> 6; nn = i & 63; }
      const int n = n0 + nn, k = k0 + kk;
      sm.Bs[kk][nn] = (n < N && k < ke) ? fb(k, n) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < kTK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = sm.As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = sm.Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
}

__device__ __forceinline__ void zero_acc(float (&acc)[4][4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
}

// Sum over the 16 threads that share a tile row (same ty), result in all 16.
__device__ __forceinline__ float row16_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 8);
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  return v;
}

// Deterministic block sum (fixed tree), result valid in thread 0.
__device__ __forceinline__ float block_sum(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float s = 0.f;
  if (threadIdx.x == 0)
    for (int i = 0; i < kThreads / 32; ++i) s += red[i];
  return s;
}

__device__ __forceinline__ int64_t chunk_vec(int b, int h, int c, int H, int nc, int L) {
  return (((int64_t)b * H + h) * nc + c) * L;
}

// ------------------------------------------------------------ chunk_cumsum
// delta = softplus(dt + dt_bias) (0 past seqlen), a = inclusive in-chunk
// cumsum of delta * A, both laid out (B, H, nc, L).
// Warp-per-chunk variant: grid ceil(B*nc*H / 8) blocks of 8 warps; warp w
// handles (b, c, h) = unravel(w); lane k the E = ceil(L/32) consecutive
// positions starting at k*E.  All dt loads of a lane are issued together.
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
    k_chunk_cumsum_warp(const Tin* __restrict__ dt, const float* __restrict__ dt_bias,
                        const float* __restrict__ A, float* __restrict__ delta,
                        float* __restrict__ acs, int B, int T, int H, int L, int nc) {
  const int64_t wid = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (wid >= (int64_t)B * nc * H) return;
  const int h = (int)(wid % H);
  const int64_t bc = wid / H;
  const int c = (int)(bc % nc), b = (int)(bc / nc);
  const int E = (L + 31) / 32;
  const float bias = dt_bias ? dt_bias[h] : 0.f, Ah = A[h];
  float dv[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int l = lane * E + e, t = c * L + l;
    dv[e] = (e < E && l < L && t < T) ? ldf(dt + ((int64_t)b * T + t) * H + h) : 0.f;
  }
  float run = 0.f, vals[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int l = lane * E + e, t = c * L + l;
    const float d = (e < E && l < L && t < T) ? softplus_f(dv[e] + bias) : 0.f;
    dv[e] = d;
    run += d * Ah;
    vals[e] = run;
  }
  float tot = run;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float o = __shfl_up_sync(0xffffffffu, tot, off);
    if (lane >= off) tot += o;
  }
  const float excl = tot - run;
  const int64_t base = chunk_vec(b, h, c, H, nc, L);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int l = lane * E + e;
    if (e < E && l < L) {
      delta[base + l] = dv[e];
      acs[base + l] = excl + vals[e];
    }
  }
}

// -------------------------------------------------------------- C . B^T
// grid (nc, G, B).  CB[b,c,g,l,s] = sum_n C[l,n] B[s,n] for s <= l.
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
    k_bmm_cb(const Tin* __restrict__ Bm, const Tin* __restrict__ Cm, float* __restrict__ CB,
             int T, int G, int N, int L, int nc) {
  __shared__ TileSmem sm;
  const int c = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int Lv = min(L, T - c * L);
  const Tin* Cc = Cm + (((int64_t)b * T + (int64_t)c * L) * G + g) * N;
  const Tin* Bc = Bm + (((int64_t)b * T + (int64_t)c * L) * G + g) * N;
  const int64_t rs = (int64_t)G * N;
  float* out = CB + (((int64_t)b * nc + c) * G + g) * L * L;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  for (int m0 = 0; m0 < Lv; m0 += kTile)
    for (int n0 = 0; n0 <= m0; n0 += kTile) {
      float acc[4][4];
      zero_acc(acc);
      tile_accum<true, true>(acc, Lv, Lv, m0, n0, 0, N,
                             [&](int l, int n) { return ldf(Cc + l * rs + n); },
                             [&](int n, int s) { return ldf(Bc + s * rs + n); }, sm);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int l = m0 + ty * 4 + i, s = n0 + tx * 4 + j;
          if (l < Lv && s < Lv) out[(int64_t)l * L + s] = acc[i][j];
        }
    }
}

// ------------------------------------------------------------ chunk_state
// grid (nc, H, B).  MODE 0 (chunk_state):  S = sum_l exp(a_last - a_l) delta_l x_l (x) B_l
//                   MODE 1 (dstates):      dHs = sum_l exp(a_l) dy_l (x) C_l
template <typename Tin, int MODE>
__global__ void __launch_bounds__(kThreads)
    k_chunk_state(const Tin* __restrict__ X, const Tin* __restrict__ Y,
                  const float* __restrict__ delta, const float* __restrict__ acs,
                  float* __restrict__ S, int T, int H, int G, int P, int N, int L, int nc) {
  __shared__ TileSmem sm;
  __shared__ float w[256];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z, g = h / (H / G);
  const int Lv = min(L, T - c * L);
  const int64_t cv = chunk_vec(b, h, c, H, nc, L);
  const float alast = acs[cv + L - 1];
  for (int l = threadIdx.x; l < L; l += kThreads)
    w[l] = MODE == 0 ? expf(alast - acs[cv + l]) * delta[cv + l] : expf(acs[cv + l]);
  __syncthreads();
  const Tin* Xc = X + (((int64_t)b * T + (int64_t)c * L) * H + h) * P;
  const Tin* Yc = Y + (((int64_t)b * T + (int64_t)c * L) * G + g) * N;
  const int64_t xs = (int64_t)H * P, ys = (int64_t)G * N;
  float* Sc = S + (((int64_t)b * nc + c) * H + h) * (int64_t)P * N;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  for (int m0 = 0; m0 < P; m0 += kTile)
    for (int n0 = 0; n0 < N; n0 += kTile) {
      float acc[4][4];
      zero_acc(acc);
      tile_accum<false, false>(acc, P, N, m0, n0, 0, Lv,
                               [&](int p, int l) { return w[l] * ldf(Xc + l * xs + p); },
                               [&](int l, int n) { return ldf(Yc + l * ys + n); }, sm);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int p = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
          if (p < P && n < N) Sc[(int64_t)p * N + n] = acc[i][j];
        }
    }
}

// ---------------------------------------------------------- state_passing
// grid (ceil(P*N/256), H, B).  Hprev[c] = H_c;  H_{c+1} = exp(a_c[L-1]) H_c + S_c.
__global__ void __launch_bounds__(kThreads)
    k_state_passing(const float* __restrict__ S, const float* __restrict__ acs,
                    const float* __restrict__ init, float* __restrict__ Hprev,
                    float* __restrict__ final_state, int H, int PN, int L, int nc) {
  const int e = blockIdx.x * kThreads + threadIdx.x, h = blockIdx.y, b = blockIdx.z;
  if (e >= PN) return;
  float cur = init ? init[((int64_t)b * H + h) * PN + e] : 0.f;
  for (int c = 0; c < nc; ++c) {
    const int64_t off = (((int64_t)b * nc + c) * H + h) * PN + e;
    const float s = S[off];
    const float dec = expf(acs[chunk_vec(b, h, c, H, nc, L) + L - 1]);
    Hprev[off] = cur;
    cur = fmaf(dec, cur, s);
  }
  if (final_state) final_state[((int64_t)b * H + h) * PN + e] = cur;
}

// Vectorised state_passing: grid (ceil(P*N/1024), H, B); each thread carries 4
// consecutive state elements (float4) through the chunk recurrence.  The
// loads of S_c do not depend on the recurrence, so they are issued kPrefetch
// chunks ahead to keep enough bytes in flight per SM.
constexpr int kPrefetch = 8;

__global__ void __launch_bounds__(kThreads)
    k_state_passing_v4(const float4* __restrict__ S, const float* __restrict__ acs,
                       const float4* __restrict__ init, float4* __restrict__ Hprev,
                       float4* __restrict__ final_state, int H, int PN4, int L, int nc) {
  const int e = blockIdx.x * kThreads + threadIdx.x, h = blockIdx.y, b = blockIdx.z;
  if (e >= PN4) return;
  const int64_t step = (int64_t)H * PN4;
  const int64_t base = ((int64_t)b * nc * H + h) * PN4 + e;
  const float* ab = acs + ((int64_t)b * H + h) * (int64_t)nc * L + (L - 1);
  float4 cur = init ? init[((int64_t)b * H + h) * PN4 + e] : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < nc; c0 += kPrefetch) {
    float4 sv[kPrefetch];
    float dec[kPrefetch];
#pragma unroll
    for (int k = 0; k < kPrefetch; ++k)
      if (c0 + k < nc) {
        sv[k] = S[base + (c0 + k) * step];
        dec[k] = __expf(ab[(int64_t)(c0 + k) * L]);
      }
#pragma unroll
    for (int k = 0; k < kPrefetch; ++k)
      if (c0 + k < nc) {
        Hprev[base + (c0 + k) * step] = cur;
        cur.x = fmaf(dec[k], cur.x, sv[k].x);
        cur.y = fmaf(dec[k], cur.y, sv[k].y);
        cur.z = fmaf(dec[k], cur.z, sv[k].z);
        cur.w = fmaf(dec[k], cur.w, sv[k].w);
      }
  }
  if (final_state) final_state[((int64_t)b * H + h) * PN4 + e] = cur;
}

// Image-mode state passing (tensor-core path, headdim 64, N % 64 == 0):
// grid (P*N/2048, H, B); a thread carries 8 consecutive elements of one state
// row through the recurrence and writes each H_c as one 16-byte hi chunk and
// one 16-byte lo chunk of the state image.
__device__ __forceinline__ uint32_t image_chunk_off(int e8, int N) {
  const int n = (e8 * 8) % N, p = (e8 * 8) / N;
  return (n >> 6) * 8192u + p * 128u + ((((n & 63) >> 3) ^ (p & 7)) << 4);
}

__device__ __forceinline__ void split8_store(unsigned char* hi, unsigned char* lo,
                                             const float4& a, const float4& b) {
  const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 hb = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    const float2 hf = __bfloat1622float2(hb);
    const __nv_bfloat162 lb = __floats2bfloat162_rn(v[2 * i] - hf.x, v[2 * i + 1] - hf.y);
    h[i] = *reinterpret_cast<const uint32_t*>(&hb);
    l[i] = *reinterpret_cast<const uint32_t*>(&lb);
  }
  *reinterpret_cast<uint4*>(hi) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(lo) = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ void image_load8(const unsigned char* hi, const unsigned char* lo,
                                            float4& a, float4& b) {
  const uint4 h = *reinterpret_cast<const uint4*>(hi);
  const uint4 l = *reinterpret_cast<const uint4*>(lo);
  a.x = __uint_as_float(h.x << 16) + __uint_as_float(l.x << 16);
  a.y = __uint_as_float(h.x & 0xFFFF0000u) + __uint_as_float(l.x & 0xFFFF0000u);
  a.z = __uint_as_float(h.y << 16) + __uint_as_float(l.y << 16);
  a.w = __uint_as_float(h.y & 0xFFFF0000u) + __uint_as_float(l.y & 0xFFFF0000u);
  b.x = __uint_as_float(h.z << 16) + __uint_as_float(l.z << 16);
  b.y = __uint_as_float(h.z & 0xFFFF0000u) + __uint_as_float(l.z & 0xFFFF0000u);
  b.z = __uint_as_float(h.w << 16) + __uint_as_float(l.w << 16);
  b.w = __uint_as_float(h.w & 0xFFFF0000u) + __uint_as_float(l.w & 0xFFFF0000u);
}

__device__ __forceinline__ float4 fma4(float d, const float4& c, const float4& s) {
  return make_float4(fmaf(d, c.x, s.x), fmaf(d, c.y, s.y), fmaf(d, c.z, s.z), fmaf(d, c.w, s.w));
}

// NT = 256: three blocks per SM (registers capped); NT = 128: seven, for
// grids that three blocks of 256 per SM would hold in more than one wave (the
// walk is as long for every block, so a second, partial wave costs a whole
// walk); four chunks in flight per thread.
// grid (P*N/(8 NT), H, B*K): segment k = z % K of batch b = z / K walks chunks
// [k*lseg, min(nc, (k+1)*lseg)) from its entering state (init for K == 1,
// else seg_in (B, K, H, P, N)); only the last segment writes final_state.
// kSeg = false is the single-level walk (K = 1), compiled on its own.
constexpr int kPrefetchImg = 4;
template <bool kSeg, int NT>
__global__ void __launch_bounds__(NT, NT == 256 ? 3 : 7)
    k_state_passing_img(const float4* __restrict__ S, const float* __restrict__ acs,
                        const float4* __restrict__ init, unsigned char* __restrict__ img,
                        float4* __restrict__ final_state, int N, int H, int PN8, int L, int nc,
                        int K, int lseg, const float4* __restrict__ seg_in, int hs) {
  griddep_launch_dependents();
  griddep_wait();  // S and a come from the previous kernel (launched with launch_pdl)
  const int e = blockIdx.x * NT + threadIdx.x, h = blockIdx.y;
  const int b = kSeg ? blockIdx.z / K : blockIdx.z, sk = kSeg ? blockIdx.z % K : 0;
  if (e >= PN8) return;
  const int cb = kSeg ? sk * lseg : 0, ce = kSeg ? min(nc, cb + lseg) : nc;
  const int64_t step = (int64_t)H * PN8 * 2;             // float4 units between chunks
  const int64_t base = ((int64_t)b * nc * H + h) * PN8 * 2;  // (b, c=0, h) state, float4 units
  const uint32_t off = image_chunk_off(e, N), lo_off = (N / 64) * 8192u;
  const float* ab = acs + (((int64_t)b * H + h) >> hs) * (int64_t)nc * L + (L - 1);
  const int64_t sb = ((int64_t)b * H + h) * PN8 * 2 + 2 * e;
  const float4* in = nullptr;  // the state entering the segment (null: zero)
  if constexpr (!kSeg) {
    if (init) in = init + sb;
  } else {
    in = seg_in + (((int64_t)b * K + sk) * H + h) * PN8 * 2 + 2 * e;
  }
  float4 c0 = in ? in[0] : make_float4(0.f, 0.f, 0.f, 0.f);
  float4 c1 = in ? in[1] : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = cb; k0 < ce; k0 += kPrefetchImg) {
    float4 s0[kPrefetchImg], s1[kPrefetchImg];
    float dec[kPrefetchImg];
#pragma unroll
    for (int k = 0; k < kPrefetchImg; ++k)
      if (k0 + k < ce) {
        s0[k] = S[base + (k0 + k) * step + 2 * e];
        s1[k] = S[base + (k0 + k) * step + 2 * e + 1];
        dec[k] = __expf(ab[(int64_t)(k0 + k) * L]);
      }
#pragma unroll
    for (int k = 0; k < kPrefetchImg; ++k)
      if (k0 + k < ce) {
        unsigned char* dst = img + (base + (k0 + k) * step) * 16;
        split8_store(dst + off, dst + off + lo_off, c0, c1);
        c0 = fma4(dec[k], c0, s0[k]);
        c1 = fma4(dec[k], c1, s1[k]);
      }
  }
  if (final_state && (!kSeg || sk == K - 1)) {
    final_state[sb] = c0;
    final_state[sb + 1] = c1;
  }
}

// Two-level pass 1: grid (P*N/2048, H, B*K); segment k's end state from a
// zero start, E[b, k] = sum over its chunks c of (product of the later
// chunks' decays in the segment) S_c.  The last segment's is not needed.
__global__ void __launch_bounds__(kThreads, 3)
    k_state_passing_seg_end(const float4* __restrict__ S, const float* __restrict__ acs,
                            float4* __restrict__ E, int H, int PN8, int L, int nc, int K,
                            int lseg, int hs) {
  const int e = blockIdx.x * kThreads + threadIdx.x, h = blockIdx.y;
  const int b = blockIdx.z / K, sk = blockIdx.z % K;
  if (e >= PN8 || sk == K - 1) return;
  const int cb = sk * lseg, ce = min(nc, cb + lseg);
  const int64_t step = (int64_t)H * PN8 * 2;
  const int64_t base = ((int64_t)b * nc * H + h) * PN8 * 2;
  const float* ab = acs + (((int64_t)b * H + h) >> hs) * (int64_t)nc * L + (L - 1);
  float4 c0 = make_float4(0.f, 0.f, 0.f, 0.f), c1 = c0;
  for (int k0 = cb; k0 < ce; k0 += kPrefetchImg) {
    float4 s0[kPrefetchImg], s1[kPrefetchImg];
    float dec[kPrefetchImg];
#pragma unroll
    for (int k = 0; k < kPrefetchImg; ++k)
      if (k0 + k < ce) {
        s0[k] = S[base + (k0 + k) * step + 2 * e];
        s1[k] = S[base + (k0 + k) * step + 2 * e + 1];
        dec[k] = __expf(ab[(int64_t)(k0 + k) * L]);
      }
#pragma unroll
    for (int k = 0; k < kPrefetchImg; ++k)
      if (k0 + k < ce) {
        c0 = fma4(dec[k], c0, s0[k]);
        c1 = fma4(dec[k], c1, s1[k]);
      }
  }
  const int64_t eo = (((int64_t)b * K + sk) * H + h) * PN8 * 2 + 2 * e;
  E[eo] = c0;
  E[eo + 1] = c1;
}

// Two-level pass 2: grid (P*N/2048, H, B); the state entering each segment,
// In[b, 0] = init (or 0), In[b, k+1] = D_k In[b, k] + E[b, k] with D_k the
// product of segment k's chunk decays.
__global__ void __launch_bounds__(kThreads)
    k_state_passing_seg_in(const float4* __restrict__ E, const float* __restrict__ acs,
                           const float4* __restrict__ init, float4* __restrict__ In, int H,
                           int PN8, int L, int nc, int K, int lseg, int hs) {
  const int e = blockIdx.x * kThreads + threadIdx.x, h = blockIdx.y, b = blockIdx.z;
  if (e >= PN8) return;
  const float* ab = acs + (((int64_t)b * H + h) >> hs) * (int64_t)nc * L + (L - 1);
  const int64_t sb = ((int64_t)b * H + h) * PN8 * 2 + 2 * e;
  float4 c0 = init ? init[sb] : make_float4(0.f, 0.f, 0.f, 0.f);
  float4 c1 = init ? init[sb + 1] : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int sk = 0; sk < K; ++sk) {
    const int64_t o = (((int64_t)b * K + sk) * H + h) * PN8 * 2 + 2 * e;
    In[o] = c0;
    In[o + 1] = c1;
    if (sk == K - 1) break;
    float D = 1.f;
    const int cb = sk * lseg, ce = min(nc, cb + lseg);
    for (int c = cb; c < ce; ++c) D *= __expf(ab[(int64_t)c * L]);
    c0 = fma4(D, c0, E[o]);
    c1 = fma4(D, c1, E[o + 1]);
  }
}

// Image-mode state passing backward: grid (nsplit = P*N/(8 NT), H, B); reads
// the H_c images, writes the dS_c images; dlast partials as in the float4
// kernel (one per warp: P*N/256 per chunk for either NT).  NT as in the
// forward.
template <bool kSeg, int NT>
__global__ void __launch_bounds__(NT, NT == 256 ? 3 : 7)
    k_state_passing_bwd_img(const float4* __restrict__ dHs, const float* __restrict__ acs,
                            const unsigned char* __restrict__ himg,
                            const float4* __restrict__ dfinal, unsigned char* __restrict__ dsimg,
                            float* __restrict__ dlast_part, float4* __restrict__ dinit, int N,
                            int H, int PN8, int L, int nc, int K, int lseg,
                            const float4* __restrict__ seg_out, int hs) {
  griddep_launch_dependents();
  griddep_wait();  // dHs comes from the previous kernel (launched with launch_pdl)
  // grid (nsplit, H, B*K): segment sk = z % K walks chunks [sk*lseg, min(nc,
  // (sk+1)*lseg)) backwards from the gradient leaving it (dfinal for K == 1,
  // else seg_out (B, K, H, P, N)); only segment 0 writes dinit
  const int split = blockIdx.x, nsplit = gridDim.x, h = blockIdx.y;
  const int b = kSeg ? blockIdx.z / K : blockIdx.z, sk = kSeg ? blockIdx.z % K : 0;
  const int cb = kSeg ? sk * lseg : 0, ce = kSeg ? min(nc, cb + lseg) : nc;
  const int e = split * NT + threadIdx.x;
  const bool live = e < PN8;
  const int64_t step = (int64_t)H * PN8 * 2;
  const int64_t base = ((int64_t)b * nc * H + h) * PN8 * 2;
  const uint32_t off = live ? image_chunk_off(e, N) : 0u, lo_off = (N / 64) * 8192u;
  const float* ab = acs + (((int64_t)b * H + h) >> hs) * (int64_t)nc * L + (L - 1);
  const int64_t sb = ((int64_t)b * H + h) * PN8 * 2 + 2 * e;
  const float4* gin = nullptr;  // the gradient leaving the segment (null: zero)
  if constexpr (!kSeg) {
    if (dfinal) gin = dfinal + sb;
  } else {
    gin = seg_out + (((int64_t)b * K + sk) * H + h) * PN8 * 2 + 2 * e;
  }
  float4 g0 = (live && gin) ? gin[0] : make_float4(0.f, 0.f, 0.f, 0.f);
  float4 g1 = (live && gin) ? gin[1] : make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int kPf = 3;
  for (int c1 = ce - 1; c1 >= cb; c1 -= kPf) {
    float4 h0[kPf], h1[kPf], d0[kPf], d1[kPf];
    float dec[kPf];
#pragma unroll
    for (int k = 0; k < kPf; ++k) {
      const int c = c1 - k;
      if (c >= cb) {
        dec[k] = __expf(ab[(int64_t)c * L]);
        if (live) {
          const unsigned char* src = himg + (base + c * step) * 16;
          image_load8(src + off, src + off + lo_off, h0[k], h1[k]);
          d0[k] = dHs[base + c * step + 2 * e];
          d1[k] = dHs[base + c * step + 2 * e + 1];
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kPf; ++k) {
      const int c = c1 - k;
      if (c < cb) break;
      float part = 0.f;
      if (live) {
        unsigned char* dst = dsimg + (base + c * step) * 16;
        split8_store(dst + off, dst + off + lo_off, g0, g1);
        part = h0[k].x * g0.x + h0[k].y * g0.y + h0[k].z * g0.z + h0[k].w * g0.w +
               h1[k].x * g1.x + h1[k].y * g1.y + h1[k].z * g1.z + h1[k].w * g1.w;
        g0 = fma4(dec[k], g0, d0[k]);
        g1 = fma4(dec[k], g1, d1[k]);
      }
      // one partial per warp (fixed-order sums later, no block barrier here)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
      if ((threadIdx.x & 31) == 0)
        dlast_part[((((int64_t)b * H + h) * nc + c) * nsplit + split) * (NT / 32) +
                   (threadIdx.x >> 5)] = dec[k] * part;
    }
  }
  if (live && dinit && (!kSeg || sk == 0)) {
    dinit[sb] = g0;
    dinit[sb + 1] = g1;
  }
}

// Two-level backward pass 1: grid (P*N/2048, H, B*K); segment k's own part of
// the gradient entering its first chunk, from a zero gradient leaving it:
// G <- dHs_c + dec_c G for c = last .. first chunk of the segment.  Segment
// 0's is not needed.
__global__ void __launch_bounds__(kThreads, 3)
    k_state_passing_bwd_seg_end(const float4* __restrict__ dHs, const float* __restrict__ acs,
                                float4* __restrict__ E, int H, int PN8, int L, int nc, int K,
                                int lseg, int hs) {
  const int e = blockIdx.x * kThreads + threadIdx.x, h = blockIdx.y;
  const int b = blockIdx.z / K, sk = blockIdx.z % K;
  if (e >= PN8 || sk == 0) return;
  const int cb = sk * lseg, ce = min(nc, cb + lseg);
  const int64_t step = (int64_t)H * PN8 * 2;
  const int64_t base = ((int64_t)b * nc * H + h) * PN8 * 2;
  const float* ab = acs + (((int64_t)b * H + h) >> hs) * (int64_t)nc * L + (L - 1);
  float4 g0 = make_float4(0.f, 0.f, 0.f, 0.f), g1 = g0;
  for (int c1 = ce - 1; c1 >= cb; c1 -= kPrefetchImg) {
    float4 d0[kPrefetchImg], d1[kPrefetchImg];
    float dec[kPrefetchImg];
#pragma unroll
    for (int k = 0; k < kPrefetchImg; ++k)
      if (c1 - k >= cb) {
        d0[k] = dHs[base + (c1 - k) * step + 2 * e];
        d1[k] = dHs[base + (c1 - k) * step + 2 * e + 1];
        dec[k] = __expf(ab[(int64_t)(c1 - k) * L]);
      }
#pragma unroll
    for (int k = 0; k < kPrefetchImg; ++k)
      if (c1 - k >= cb) {
        g0 = fma4(dec[k], g0, d0[k]);
        g1 = fma4(dec[k], g1, d1[k]);
      }
  }
  const int64_t eo = (((int64_t)b * K + sk) * H + h) * PN8 * 2 + 2 * e;
  E[eo] = g0;
  E[eo + 1] = g1;
}

// Two-level backward pass 2: grid (P*N/2048, H, B); the gradient leaving
// each segment, Out[b, K-1] = dfinal (or 0), Out[b, k-1] = D_k Out[b, k] +
// E[b, k] with D_k the product of segment k's chunk decays.
__global__ void __launch_bounds__(kThreads)
    k_state_passing_bwd_seg_in(const float4* __restrict__ E, const float* __restrict__ acs,
                               const float4* __restrict__ dfinal, float4* __restrict__ Out,
                               int H, int PN8, int L, int nc, int K, int lseg, int hs) {
  const int e = blockIdx.x * kThreads + threadIdx.x, h = blockIdx.y, b = blockIdx.z;
  if (e >= PN8) return;
  const float* ab = acs + (((int64_t)b * H + h) >> hs) * (int64_t)nc * L + (L - 1);
  const int64_t sb = ((int64_t)b * H + h) * PN8 * 2 + 2 * e;
  float4 g0 = dfinal ? dfinal[sb] : make_float4(0.f, 0.f, 0.f, 0.f);
  float4 g1 = dfinal ? dfinal[sb + 1] : make_float4(0.f, 0.f, 0.f, 0.f);
  for (int sk = K - 1; sk >= 0; --sk) {
    const int64_t o = (((int64_t)b * K + sk) * H + h) * PN8 * 2 + 2 * e;
    Out[o] = g0;
    Out[o + 1] = g1;
    if (sk == 0) break;
    float D = 1.f;
    const int cb = sk * lseg, ce = min(nc, cb + lseg);
    for (int c = cb; c < ce; ++c) D *= __expf(ab[(int64_t)c * L]);
    g0 = fma4(D, g0, E[o]);
    g1 = fma4(D, g1, E[o + 1]);
  }
}

// Vectorised state_passing backward: grid (nsplit = ceil(P*N/1024), H, B).
// Each block owns 1024 state elements of one (b, h) and walks the chunks in
// reverse; the partial dot products <H_c, G_{c+1}> of its slice go to
// dlast_part[((b*H + h)*nc + c)*nsplit + split] (summed in a fixed order later).
__global__ void __launch_bounds__(kThreads)
    k_state_passing_bwd_v4(const float4* __restrict__ dHs, const float* __restrict__ acs,
                           const float4* __restrict__ Hprev, const float4* __restrict__ dfinal,
                           float4* __restrict__ dS, float* __restrict__ dlast_part,
                           float4* __restrict__ dinit, int H, int PN4, int L, int nc) {
  __shared__ float red[kThreads / 32];
  const int split = blockIdx.x, nsplit = gridDim.x, h = blockIdx.y, b = blockIdx.z;
  const int e = split * kThreads + threadIdx.x;
  const bool live = e < PN4;
  const int64_t step = (int64_t)H * PN4;
  const int64_t base = ((int64_t)b * nc * H + h) * PN4 + e;
  const float* ab = acs + ((int64_t)b * H + h) * (int64_t)nc * L + (L - 1);
  float4 G = (live && dfinal) ? dfinal[((int64_t)b * H + h) * PN4 + e]
                              : make_float4(0.f, 0.f, 0.f, 0.f);
  constexpr int kPf = 4;
  for (int c1 = nc - 1; c1 >= 0; c1 -= kPf) {
    float4 hv[kPf], gv[kPf];
    float dec[kPf];
#pragma unroll
    for (int k = 0; k < kPf; ++k) {
      const int c = c1 - k;
      if (c >= 0) {
        dec[k] = __expf(ab[(int64_t)c * L]);
        if (live) {
          hv[k] = Hprev[base + c * step];
          gv[k] = dHs[base + c * step];
        }
      }
    }
#pragma unroll
    for (int k = 0; k < kPf; ++k) {
      const int c = c1 - k;
      if (c < 0) break;
      float part = 0.f;
      if (live) {
        dS[base + c * step] = G;
        part = hv[k].x * G.x + hv[k].y * G.y + hv[k].z * G.z + hv[k].w * G.w;
        G.x = fmaf(dec[k], G.x, gv[k].x);
        G.y = fmaf(dec[k], G.y, gv[k].y);
        G.z = fmaf(dec[k], G.z, gv[k].z);
        G.w = fmaf(dec[k], G.w, gv[k].w);
      }
      const float tot = block_sum(part, red);
      if (threadIdx.x == 0)
        dlast_part[(((int64_t)b * H + h) * nc + c) * nsplit + split] = dec[k] * tot;
    }
  }
  if (live && dinit) dinit[((int64_t)b * H + h) * PN4 + e] = G;
}

// ------------------------------------------------------------- chunk_scan
// grid (nc, H, B).  y_l = sum_{s<=l} CB[l,s] exp(a_l - a_s) delta_s x_s
//                        + exp(a_l) H_c C_l + D x_l
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kThreads)
    k_chunk_scan(const Tin* __restrict__ x, const Tin* __restrict__ Cm,
                 const float* __restrict__ CB, const float* __restrict__ delta,
                 const float* __restrict__ acs, const float* __restrict__ Hprev,
                 const float* __restrict__ D, Tout* __restrict__ y, int T, int H, int G, int P,
                 int N, int L, int nc) {
  __shared__ TileSmem sm;
  __shared__ float sa[256], sd[256];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z, g = h / (H / G);
  const int Lv = min(L, T - c * L);
  const int64_t cv = chunk_vec(b, h, c, H, nc, L);
  for (int l = threadIdx.x; l < L; l += kThreads) {
    sa[l] = acs[cv + l];
    sd[l] = delta[cv + l];
  }
  __syncthreads();
  const int64_t xs = (int64_t)H * P, cs = (int64_t)G * N;
  const Tin* xc = x + (((int64_t)b * T + (int64_t)c * L) * H + h) * P;
  const Tin* Cc = Cm + (((int64_t)b * T + (int64_t)c * L) * G + g) * N;
  const float* CBc = CB + (((int64_t)b * nc + c) * G + g) * L * L;
  const float* Hc = Hprev + (((int64_t)b * nc + c) * H + h) * (int64_t)P * N;
  Tout* yc = y + (((int64_t)b * T + (int64_t)c * L) * H + h) * P;
  const float Dh = D ? D[h] : 0.f;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  for (int m0 = 0; m0 < Lv; m0 += kTile)
    for (int n0 = 0; n0 < P; n0 += kTile) {
      float acc[4][4];
      zero_acc(acc);
      // state term: exp(a_l) sum_n C[l,n] H_c[p,n]
      tile_accum<true, true>(acc, Lv, P, m0, n0, 0, N,
                             [&](int l, int n) { return expf(sa[l]) * ldf(Cc + l * cs + n); },
                             [&](int n, int p) { return Hc[(int64_t)p * N + n]; }, sm);
      // intra-chunk term over s <= l
      tile_accum<true, false>(
          acc, Lv, P, m0, n0, 0, min(m0 + kTile, Lv),
          [&](int l, int s) {
            return s <= l ? CBc[(int64_t)l * L + s] * expf(sa[l] - sa[s]) * sd[s] : 0.f;
          },
          [&](int s, int p) { return ldf(xc + s * xs + p); }, sm);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int l = m0 + ty * 4 + i, p = n0 + tx * 4 + j;
          if (l < Lv && p < P) stf(yc + l * xs + p, acc[i][j] + Dh * ldf(xc + l * xs + p));
        }
    }
}

// ======================================================= backward kernels

// grid (B*H).  Reverse recurrence over chunks:
//   dS_c = G_{c+1};  dlast_c = exp(a_c[L-1]) <H_c, G_{c+1}>;
//   G_c = dHs_c + exp(a_c[L-1]) G_{c+1};   G_nc = dfinal, dinit = G_0.
__global__ void __launch_bounds__(kThreads)
    k_state_passing_bwd(const float* __restrict__ dHs, const float* __restrict__ acs,
                        const float* __restrict__ Hprev, const float* __restrict__ dfinal,
                        float* __restrict__ dS, float* __restrict__ dlast,
                        float* __restrict__ dinit, int H, int PN, int L, int nc) {
  __shared__ float red[kThreads / 32];
  const int b = blockIdx.x / H, h = blockIdx.x % H;
  float Gv[kMaxStatePerThread];
  const int64_t bh = ((int64_t)b * H + h) * PN;
#pragma unroll
  for (int e = 0; e < kMaxStatePerThread; ++e) {
    const int idx = threadIdx.x + e * kThreads;
    Gv[e] = (idx < PN && dfinal) ? dfinal[bh + idx] : 0.f;
  }
  for (int c = nc - 1; c >= 0; --c) {
    const int64_t off = (((int64_t)b * nc + c) * H + h) * PN;
    const float dec = expf(acs[chunk_vec(b, h, c, H, nc, L) + L - 1]);
    float part = 0.f;
#pragma unroll
    for (int e = 0; e < kMaxStatePerThread; ++e) {
      const int idx = threadIdx.x + e * kThreads;
      if (idx < PN) {
        dS[off + idx] = Gv[e];
        part = fmaf(Hprev[off + idx], Gv[e], part);
        Gv[e] = fmaf(dec, Gv[e], dHs[off + idx]);
      }
    }
    const float tot = block_sum(part, red);
    if (threadIdx.x == 0) dlast[((int64_t)b * H + h) * nc + c] = dec * tot;
  }
  if (dinit) {
#pragma unroll
    for (int e = 0; e < kMaxStatePerThread; ++e) {
      const int idx = threadIdx.x + e * kThreads;
      if (idx < PN) dinit[bh + idx] = Gv[e];
    }
  }
}

// grid (nc, H, B).  dyx[l,s] = <dy_l, x_s> for s <= l.
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
    k_dyx(const Tin* __restrict__ x, const Tin* __restrict__ dy, float* __restrict__ dyx, int T,
          int H, int P, int L, int nc) {
  __shared__ TileSmem sm;
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int Lv = min(L, T - c * L);
  const int64_t xs = (int64_t)H * P;
  const Tin* xc = x + (((int64_t)b * T + (int64_t)c * L) * H + h) * P;
  const Tin* dyc = dy + (((int64_t)b * T + (int64_t)c * L) * H + h) * P;
  float* out = dyx + (((int64_t)b * nc + c) * H + h) * L * L;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  for (int m0 = 0; m0 < Lv; m0 += kTile)
    for (int n0 = 0; n0 <= m0; n0 += kTile) {
      float acc[4][4];
      zero_acc(acc);
      tile_accum<true, true>(acc, Lv, Lv, m0, n0, 0, P,
                             [&](int l, int p) { return ldf(dyc + l * xs + p); },
                             [&](int p, int s) { return ldf(xc + s * xs + p); }, sm);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int l = m0 + ty * 4 + i, s = n0 + tx * 4 + j;
          if (l < Lv && s < Lv) out[(int64_t)l * L + s] = acc[i][j];
        }
    }
}

// grid (nc, H, B).  u_s = sum_{l>=s} CB[l,s] exp(a_l - a_s) dy_l
//                        + exp(a_last - a_s) dS_c B_s
//   dx_s = delta_s u_s + D dy_s;  ddir_s = <x_s, u_s>;  qrow_s = delta_s <x_s, state part>
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
    k_bwd_dx(const Tin* __restrict__ x, const Tin* __restrict__ Bm, const Tin* __restrict__ dy,
             const float* __restrict__ CB, const float* __restrict__ delta,
             const float* __restrict__ acs, const float* __restrict__ dS,
             const float* __restrict__ D, float* __restrict__ dx, float* __restrict__ ddir,
             float* __restrict__ qrow, int T, int H, int G, int P, int N, int L, int nc) {
  __shared__ TileSmem sm;
  __shared__ float sa[256], sd[256], sq[256], su[256];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z, g = h / (H / G);
  const int Lv = min(L, T - c * L);
  const int64_t cv = chunk_vec(b, h, c, H, nc, L);
  for (int l = threadIdx.x; l < L; l += kThreads) {
    sa[l] = acs[cv + l];
    sd[l] = delta[cv + l];
    sq[l] = 0.f;
    su[l] = 0.f;
  }
  __syncthreads();
  const float alast = sa[L - 1];
  const int64_t xs = (int64_t)H * P, bs = (int64_t)G * N;
  const Tin* xc = x + (((int64_t)b * T + (int64_t)c * L) * H + h) * P;
  const Tin* dyc = dy + (((int64_t)b * T + (int64_t)c * L) * H + h) * P;
  const Tin* Bc = Bm + (((int64_t)b * T + (int64_t)c * L) * G + g) * N;
  const float* CBc = CB + (((int64_t)b * nc + c) * G + g) * L * L;
  const float* dSc = dS + (((int64_t)b * nc + c) * H + h) * (int64_t)P * N;
  float* dxc = dx + (((int64_t)b * T + (int64_t)c * L) * H + h) * P;
  const float Dh = D ? D[h] : 0.f;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  for (int m0 = 0; m0 < Lv; m0 += kTile)
    for (int n0 = 0; n0 < P; n0 += kTile) {
      float acc[4][4];
      zero_acc(acc);
      tile_accum<true, true>(
          acc, Lv, P, m0, n0, 0, N,
          [&](int s, int n) { return expf(alast - sa[s]) * ldf(Bc + s * bs + n); },
          [&](int n, int p) { return dSc[(int64_t)p * N + n]; }, sm);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int s = m0 + ty * 4 + i;
        float r = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int p = n0 + tx * 4 + j;
          if (s < Lv && p < P) r = fmaf(ldf(xc + s * xs + p), acc[i][j], r);
        }
        r = row16_sum(r);
        if (tx == 0 && s < Lv) sq[s] += sd[s] * r;
      }
      tile_accum<false, false>(
          acc, Lv, P, m0, n0, m0, Lv,
          [&](int s, int l) {
            return l >= s ? CBc[(int64_t)l * L + s] * expf(sa[l] - sa[s]) : 0.f;
          },
          [&](int l, int p) { return ldf(dyc + l * xs + p); }, sm);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int s = m0 + ty * 4 + i;
        float r = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int p = n0 + tx * 4 + j;
          if (s < Lv && p < P) {
            r = fmaf(ldf(xc + s * xs + p), acc[i][j], r);
            dxc[s * xs + p] = fmaf(sd[s], acc[i][j], Dh * ldf(dyc + s * xs + p));
          }
        }
        r = row16_sum(r);
        if (tx == 0 && s < Lv) su[s] += r;
      }
      __syncthreads();
    }
  for (int l = threadIdx.x; l < L; l += kThreads) {
    ddir[cv + l] = l < Lv ? su[l] : 0.f;
    qrow[cv + l] = l < Lv ? sq[l] : 0.f;
  }
}

// grid (nc, H, B).  This head's share of dC:
//   dC_l = sum_{s<=l} exp(a_l - a_s) delta_s <dy_l, x_s> B_s + exp(a_l) H_c^T dy_l
//   ycs_l = exp(a_l) <dy_l, H_c C_l> = <C_l, state part of dC_l>
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
    k_bwd_dC(const Tin* __restrict__ Bm, const Tin* __restrict__ Cm, const Tin* __restrict__ dy,
             const float* __restrict__ dyx, const float* __restrict__ delta,
             const float* __restrict__ acs, const float* __restrict__ Hprev,
             float* __restrict__ dCh, float* __restrict__ ycs, int T, int H, int G, int P, int N,
             int L, int nc) {
  __shared__ TileSmem sm;
  __shared__ float sa[256], sd[256], sy[256];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z, g = h / (H / G);
  const int Lv = min(L, T - c * L);
  const int64_t cv = chunk_vec(b, h, c, H, nc, L);
  for (int l = threadIdx.x; l < L; l += kThreads) {
    sa[l] = acs[cv + l];
    sd[l] = delta[cv + l];
    sy[l] = 0.f;
  }
  __syncthreads();
  const int64_t xs = (int64_t)H * P, bs = (int64_t)G * N, hs = (int64_t)H * N;
  const Tin* dyc = dy + (((int64_t)b * T + (int64_t)c * L) * H + h) * P;
  const Tin* Bc = Bm + (((int64_t)b * T + (int64_t)c * L) * G + g) * N;
  const Tin* Cc = Cm + (((int64_t)b * T + (int64_t)c * L) * G + g) * N;
  const float* Hc = Hprev + (((int64_t)b * nc + c) * H + h) * (int64_t)P * N;
  const float* M = dyx + (((int64_t)b * nc + c) * H + h) * L * L;
  float* out = dCh + (((int64_t)b * T + (int64_t)c * L) * H + h) * N;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  for (int m0 = 0; m0 < Lv; m0 += kTile)
    for (int n0 = 0; n0 < N; n0 += kTile) {
      float acc[4][4];
      zero_acc(acc);
      tile_accum<true, false>(
          acc, Lv, N, m0, n0, 0, P,
          [&](int l, int p) { return expf(sa[l]) * ldf(dyc + l * xs + p); },
          [&](int p, int n) { return Hc[(int64_t)p * N + n]; }, sm);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int l = m0 + ty * 4 + i;
        float r = 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int n = n0 + tx * 4 + j;
          if (l < Lv && n < N) r = fmaf(ldf(Cc + l * bs + n), acc[i][j], r);
        }
        r = row16_sum(r);
        if (tx == 0 && l < Lv) sy[l] += r;
      }
      tile_accum<true, false>(
          acc, Lv, N, m0, n0, 0, min(m0 + kTile, Lv),
          [&](int l, int s) {
            return s <= l ? expf(sa[l] - sa[s]) * sd[s] * M[(int64_t)l * L + s] : 0.f;
          },
          [&](int s, int n) { return ldf(Bc + s * bs + n); }, sm);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int l = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
          if (l < Lv && n < N) out[l * hs + n] = acc[i][j];
        }
      __syncthreads();
    }
  for (int l = threadIdx.x; l < L; l += kThreads) ycs[cv + l] = l < Lv ? sy[l] : 0.f;
}

// grid (nc, H, B).  This head's share of dB:
//   dB_s = delta_s [ sum_{l>=s} exp(a_l - a_s) <dy_l, x_s> C_l + exp(a_last - a_s) dS_c^T x_s ]
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
    k_bwd_dB(const Tin* __restrict__ x, const Tin* __restrict__ Cm, const float* __restrict__ dyx,
             const float* __restrict__ delta, const float* __restrict__ acs,
             const float* __restrict__ dS, float* __restrict__ dBh, int T, int H, int G, int P,
             int N, int L, int nc) {
  __shared__ TileSmem sm;
  __shared__ float sa[256], sd[256];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z, g = h / (H / G);
  const int Lv = min(L, T - c * L);
  const int64_t cv = chunk_vec(b, h, c, H, nc, L);
  for (int l = threadIdx.x; l < L; l += kThreads) {
    sa[l] = acs[cv + l];
    sd[l] = delta[cv + l];
  }
  __syncthreads();
  const float alast = sa[L - 1];
  const int64_t xs = (int64_t)H * P, bs = (int64_t)G * N, hs = (int64_t)H * N;
  const Tin* xc = x + (((int64_t)b * T + (int64_t)c * L) * H + h) * P;
  const Tin* Cc = Cm + (((int64_t)b * T + (int64_t)c * L) * G + g) * N;
  const float* dSc = dS + (((int64_t)b * nc + c) * H + h) * (int64_t)P * N;
  const float* M = dyx + (((int64_t)b * nc + c) * H + h) * L * L;
  float* out = dBh + (((int64_t)b * T + (int64_t)c * L) * H + h) * N;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  for (int m0 = 0; m0 < Lv; m0 += kTile)
    for (int n0 = 0; n0 < N; n0 += kTile) {
      float acc[4][4];
      zero_acc(acc);
      tile_accum<true, false>(
          acc, Lv, N, m0, n0, 0, P,
          [&](int s, int p) { return expf(alast - sa[s]) * sd[s] * ldf(xc + s * xs + p); },
          [&](int p, int n) { return dSc[(int64_t)p * N + n]; }, sm);
      tile_accum<false, false>(
          acc, Lv, N, m0, n0, m0, Lv,
          [&](int s, int l) {
            return l >= s ? expf(sa[l] - sa[s]) * sd[s] * M[(int64_t)l * L + s] : 0.f;
          },
          [&](int l, int n) { return ldf(Cc + l * bs + n); }, sm);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int s = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
          if (s < Lv && n < N) out[s * hs + n] = acc[i][j];
        }
    }
}

// grid (nc, H, B).  Gradient w.r.t. dA_r = delta_r A (per position r):
//   ddA_r = sum_{l>=r} sum_{s<r} M[l,s] + sum_{l>=r} ycs_l + sum_{s<r} qrow_s + dlast_c,
//   M[l,s] = CB[l,s] exp(a_l - a_s) delta_s <dy_l, x_s>.
// The double sum is taken as the exclusive prefix over r of
// (strict column sum - strict row sum) of M, which equals it exactly and
// only exponentiates a_l - a_s with s <= l.  Then
//   ddt_r = (ddir_r + A ddA_r) * softplus'(dt_r + dt_bias);
//   partials of dA = sum delta ddA, ddt_bias = sum ddt, dD = sum <dy, x>.
template <typename Tin>
__global__ void __launch_bounds__(kThreads)
    k_bwd_ddA(const Tin* __restrict__ dt, const float* __restrict__ dt_bias,
              const float* __restrict__ A, const float* __restrict__ CB,
              const float* __restrict__ dyx, const float* __restrict__ delta,
              const float* __restrict__ acs, const float* __restrict__ ddir,
              const float* __restrict__ qrow, const float* __restrict__ ycs,
              const float* __restrict__ dlast, int nsplit, float* __restrict__ ddt,
              float* __restrict__ part, int T, int H, int G, int L, int nc) {
  __shared__ float sa[256], sd[256], dr[256], sdd[256], red[kThreads / 32];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z, g = h / (H / G);
  const int Lv = min(L, T - c * L);
  const int64_t cv = chunk_vec(b, h, c, H, nc, L);
  for (int l = threadIdx.x; l < L; l += kThreads) {
    sa[l] = acs[cv + l];
    sd[l] = delta[cv + l];
  }
  __syncthreads();
  const float* CBc = CB + (((int64_t)b * nc + c) * G + g) * L * L;
  const float* Mc = dyx + (((int64_t)b * nc + c) * H + h) * L * L;
  float dpart = 0.f;
  for (int j = threadIdx.x; j < Lv; j += kThreads) {
    float col = 0.f, row = 0.f;
    for (int l = j + 1; l < Lv; ++l)
      col += CBc[(int64_t)l * L + j] * expf(sa[l] - sa[j]) * sd[j] * Mc[(int64_t)l * L + j];
    for (int s = 0; s < j; ++s)
      row += CBc[(int64_t)j * L + s] * expf(sa[j] - sa[s]) * sd[s] * Mc[(int64_t)j * L + s];
    dr[j] = col - row;
    dpart += Mc[(int64_t)j * L + j];
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // sequential prefix / suffix sums (L <= 256) in a fixed order
    float dl = 0.f;
    for (int k = 0; k < nsplit; ++k) dl += dlast[(((int64_t)b * H + h) * nc + c) * nsplit + k];
    float pre = 0.f, qpre = 0.f;
    for (int r = 0; r < Lv; ++r) {
      sdd[r] = pre + qpre + dl;
      pre += dr[r];
      qpre += qrow[cv + r];
    }
    float suf = 0.f;
    for (int r = Lv - 1; r >= 0; --r) {
      suf += ycs[cv + r];
      sdd[r] += suf;
    }
  }
  __syncthreads();
  const float Ah = A[h], bias = dt_bias ? dt_bias[h] : 0.f;
  float pA = 0.f, pbias = 0.f;
  for (int r = threadIdx.x; r < Lv; r += kThreads) {
    const int t = c * L + r;
    const float v = ldf(dt + ((int64_t)b * T + t) * H + h) + bias;
    const float g_delta = fmaf(Ah, sdd[r], ddir[cv + r]);
    const float gv = g_delta * softplus_grad_f(v);
    ddt[((int64_t)b * T + t) * H + h] = gv;
    pA = fmaf(sd[r], sdd[r], pA);
    pbias += gv;
  }
  const float sA = block_sum(pA, red);
  const float sB = block_sum(pbias, red);
  const float sD = block_sum(dpart, red);
  if (threadIdx.x == 0) {
    float* o = part + (((int64_t)b * H + h) * nc + c) * 3;
    o[0] = sA;
    o[1] = sB;
    o[2] = sD;
  }
}

// dB[b,t,g,:] = sum over the heads of group g (in increasing order).
__global__ void k_group_reduce(const float* __restrict__ perhead, float* __restrict__ out,
                               int64_t BT, int H, int G, int N) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= BT * G * N) return;
  const int n = (int)(i % N);
  const int64_t bg = i / N;
  const int g = (int)(bg % G);
  const int64_t bt = bg / G;
  const int hpg = H / G;
  float s = 0.f;
  for (int k = 0; k < hpg; ++k) s += perhead[(bt * H + (int64_t)g * hpg + k) * N + n];
  out[i] = s;
}

// grid (H), 32 threads.  Per-head parameter gradients from the per-chunk
// partials: lane k sums the chunks k, k+32, ... in order, then a fixed
// xor-tree combines the lanes (bit-reproducible).
__global__ void k_param_grads(const float* __restrict__ part, float* __restrict__ dA,
                              float* __restrict__ ddt_bias, float* __restrict__ dD, int B, int H,
                              int nc) {
  griddep_wait();  // the partials come from the previous kernel (launched with launch_pdl)
  const int h = blockIdx.x, lane = threadIdx.x;
  float a = 0.f, bb = 0.f, dd = 0.f;
  for (int i = lane; i < B * nc; i += 32) {
    const int b = i / nc, c = i % nc;
    const float* o = part + (((int64_t)b * H + h) * nc + c) * 3;
    a += o[0];
    bb += o[1];
    dd += o[2];
  }
  for (int off = 16; off > 0; off >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, off);
    bb += __shfl_xor_sync(0xffffffffu, bb, off);
    dd += __shfl_xor_sync(0xffffffffu, dd, off);
  }
  if (lane == 0) {
    dA[h] = a;
    if (ddt_bias) ddt_bias[h] = bb;
    if (dD) dD[h] = dd;
  }
}

template <typename Tin>
void launch_cumsum(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s) {
  const int64_t warps = (int64_t)d.B * d.nc * d.H;
  const int blocks = (int)((warps + kThreads / 32 - 1) / (kThreads / 32));
  SSD_LAUNCH("k_chunk_cumsum", s, k_chunk_cumsum_warp<Tin><<<blocks, kThreads, 0, s>>>(
      static_cast<const Tin*>(a.dt), a.dt_bias, a.A, w.delta, w.acs, d.B, d.T, d.H, d.L, d.nc));
}

bool vec4_ok(const void* p) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int sm_count() {
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return sms;
}

// Blocks of 128 threads (seven per SM) for the image-mode walks when a
// single-level grid of 256-thread blocks (gx per (batch, head)) would not fit
// in one wave at three per SM.
bool narrow_walk(const Dims& d, int gx, int K) {
  return K == 1 && (int64_t)gx * d.H * d.B > 3 * (int64_t)sm_count();
}

// Segments of the two-level state passing: two levels only when the
// (batch, head) grid alone (gx blocks per pair) would leave at least half the
// SMs idle (the backward: any SM idle, its per-chunk walk being longer); then
// K segments of lseg chunks, about three blocks per SM in all.
void seg_plan(const Dims& d, int gx, bool have_scratch, bool bwd, int* K, int* lseg) {
  *K = 1;
  *lseg = d.nc;
  const int kmax = have_scratch ? seg_max_segments(d) : 0;
  if (kmax < 2) return;
  const int sms = sm_count();
  const int64_t base = (int64_t)gx * d.H * d.B;
  if (bwd ? base >= sms : 2 * base > sms) return;
  // at most three blocks per SM in all, so the segments run in one wave
  int k = (int)std::min<int64_t>(kmax, std::max<int64_t>(2, (3 * sms) / base));
  *lseg = (d.nc + k - 1) / k;
  *K = (d.nc + *lseg - 1) / *lseg;
}

void launch_state_passing(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s) {
  const int PN = d.P * d.N;
  if (w.Himg) {  // tensor-core path: states as split-bf16 images only
    const int PN8 = PN / 8, gx = (PN8 + kThreads - 1) / kThreads;
    int K, lseg;
    seg_plan(d, gx, w.seg != nullptr, false, &K, &lseg);
    const float4* in = nullptr;
    if (K > 1) {
      float4* E = reinterpret_cast<float4*>(w.seg);
      float4* In = E + (size_t)d.B * K * d.H * PN8 * 2;
      SSD_LAUNCH("k_state_passing_seg", s, k_state_passing_seg_end<<<dim3(gx, d.H, d.B * K), kThreads, 0, s>>>(
          reinterpret_cast<const float4*>(w.S), w.acs, E, d.H, PN8, d.L, d.nc, K, lseg, d.hs));
      SSD_LAUNCH("k_state_passing_seg", s, k_state_passing_seg_in<<<dim3(gx, d.H, d.B), kThreads, 0, s>>>(
          E, w.acs, reinterpret_cast<const float4*>(a.init), In, d.H, PN8, d.L, d.nc, K, lseg, d.hs));
      in = In;
    }
    const bool nw = narrow_walk(d, gx, K);
    auto kern = K > 1 ? k_state_passing_img<true, 256>
                      : (nw ? k_state_passing_img<false, 128> : k_state_passing_img<false, 256>);
    const int nt = nw ? 128 : 256;
    SSD_LAUNCH("k_state_passing", s, launch_pdl(kern, dim3((PN8 + nt - 1) / nt, d.H, d.B * K),
        dim3(nt), 0, s,
        reinterpret_cast<const float4*>(w.S), w.acs, reinterpret_cast<const float4*>(a.init),
        static_cast<unsigned char*>(w.Himg), reinterpret_cast<float4*>(a.final_state), d.N, d.H,
        PN8, d.L, d.nc, K, lseg, in, d.hs));
    return;
  }
  if (PN % 4 == 0 && vec4_ok(a.init) && vec4_ok(a.final_state)) {
    const int PN4 = PN / 4;
    SSD_LAUNCH("k_state_passing", s, k_state_passing_v4<<<dim3((PN4 + kThreads - 1) / kThreads, d.H, d.B), kThreads, 0, s>>>(
        reinterpret_cast<const float4*>(w.S), w.acs, reinterpret_cast<const float4*>(a.init),
        reinterpret_cast<float4*>(w.Hprev), reinterpret_cast<float4*>(a.final_state), d.H, PN4,
        d.L, d.nc));
    return;
  }
  SSD_LAUNCH("k_state_passing", s, k_state_passing<<<dim3((PN + kThreads - 1) / kThreads, d.H, d.B), kThreads, 0, s>>>(
      w.S, w.acs, a.init, w.Hprev, a.final_state, d.H, PN, d.L, d.nc));
}

template <typename Tin>
void launch_forward_front(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s) {
  launch_cumsum<Tin>(d, a, w, s);
  SSD_LAUNCH("k_bmm_cb", s, k_bmm_cb<Tin><<<dim3(d.nc, d.G, d.B), kThreads, 0, s>>>(
      static_cast<const Tin*>(a.B), static_cast<const Tin*>(a.C), w.CB, d.T, d.G, d.N, d.L, d.nc));
  SSD_LAUNCH("k_chunk_state", s, k_chunk_state<Tin, 0><<<dim3(d.nc, d.H, d.B), kThreads, 0, s>>>(
      static_cast<const Tin*>(a.x), static_cast<const Tin*>(a.B), w.delta, w.acs, w.S, d.T, d.H,
      d.G, d.P, d.N, d.L, d.nc));
  launch_state_passing(d, a, w, s);
}

template <typename Tin, typename Tout>
void launch_forward(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s) {
  launch_forward_front<Tin>(d, a, w, s);
  SSD_LAUNCH("k_chunk_scan", s, k_chunk_scan<Tin, Tout><<<dim3(d.nc, d.H, d.B), kThreads, 0, s>>>(
      static_cast<const Tin*>(a.x), static_cast<const Tin*>(a.C), w.CB, w.delta, w.acs, w.Hprev,
      a.D, static_cast<Tout*>(a.y), d.T, d.H, d.G, d.P, d.N, d.L, d.nc));
}

// Returns the number of dlast partials per (b, h, c) it wrote.
int launch_state_passing_bwd(const Dims& d, const BwdArgs& a, const BwdWs& w, cudaStream_t s) {
  const int PN = d.P * d.N;
  if (w.f.Himg && w.dSimg) {  // tensor-core path
    const int PN8 = PN / 8, nsplit = (PN8 + kThreads - 1) / kThreads;
    int K, lseg;
    seg_plan(d, nsplit, w.f.seg != nullptr, true, &K, &lseg);
    const float4* out = nullptr;
    if (K > 1) {
      float4* E = reinterpret_cast<float4*>(w.f.seg);
      float4* Out = E + (size_t)d.B * K * d.H * PN8 * 2;
      SSD_LAUNCH("k_state_passing_bwd_seg", s, k_state_passing_bwd_seg_end<<<dim3(nsplit, d.H, d.B * K), kThreads, 0, s>>>(
          reinterpret_cast<const float4*>(w.dHs), w.f.acs, E, d.H, PN8, d.L, d.nc, K, lseg, d.hs));
      SSD_LAUNCH("k_state_passing_bwd_seg", s, k_state_passing_bwd_seg_in<<<dim3(nsplit, d.H, d.B), kThreads, 0, s>>>(
          E, w.f.acs, reinterpret_cast<const float4*>(a.dfinal), Out, d.H, PN8, d.L, d.nc, K,
          lseg, d.hs));
      out = Out;
    }
    const bool nw = narrow_walk(d, nsplit, K);
    auto kern = K > 1 ? k_state_passing_bwd_img<true, 256>
                      : (nw ? k_state_passing_bwd_img<false, 128>
                            : k_state_passing_bwd_img<false, 256>);
    const int nt = nw ? 128 : 256;
    SSD_LAUNCH("k_state_passing_bwd", s, launch_pdl(kern, dim3((PN8 + nt - 1) / nt, d.H, d.B * K),
        dim3(nt), 0, s,
        reinterpret_cast<const float4*>(w.dHs), w.f.acs,
        static_cast<const unsigned char*>(w.f.Himg), reinterpret_cast<const float4*>(a.dfinal),
        static_cast<unsigned char*>(w.dSimg), w.dlast, reinterpret_cast<float4*>(a.dinit), d.N,
        d.H, PN8, d.L, d.nc, K, lseg, out, d.hs));
    return (PN8 + nt - 1) / nt * (nt / 32);  // one partial per warp
  }
  if (PN % 4 == 0 && vec4_ok(a.dfinal) && vec4_ok(a.dinit)) {
    const int PN4 = PN / 4, nsplit = (PN4 + kThreads - 1) / kThreads;
    SSD_LAUNCH("k_state_passing_bwd", s, k_state_passing_bwd_v4<<<dim3(nsplit, d.H, d.B), kThreads, 0, s>>>(
        reinterpret_cast<const float4*>(w.dHs), w.f.acs, reinterpret_cast<const float4*>(w.f.Hprev),
        reinterpret_cast<const float4*>(a.dfinal), reinterpret_cast<float4*>(w.dS), w.dlast,
        reinterpret_cast<float4*>(a.dinit), d.H, PN4, d.L, d.nc));
    return nsplit;
  }
  SSD_LAUNCH("k_state_passing_bwd", s, k_state_passing_bwd<<<d.B * d.H, kThreads, 0, s>>>(
      w.dHs, w.f.acs, w.f.Hprev, a.dfinal, w.dS, w.dlast, a.dinit, d.H, PN, d.L, d.nc));
  return 1;
}

template <typename Tin>
void launch_backward(const Dims& d, const BwdArgs& a, const BwdWs& w, cudaStream_t s) {
  FwdArgs f = a.f;
  f.final_state = nullptr;
  launch_forward_front<Tin>(d, f, w.f, s);
  const Tin* x = static_cast<const Tin*>(a.f.x);
  const Tin* Bm = static_cast<const Tin*>(a.f.B);
  const Tin* Cm = static_cast<const Tin*>(a.f.C);
  const Tin* dy = static_cast<const Tin*>(a.dy);
  const dim3 grid(d.nc, d.H, d.B);
  SSD_LAUNCH("k_chunk_state", s, k_chunk_state<Tin, 1><<<grid, kThreads, 0, s>>>(dy, Cm, w.f.delta, w.f.acs, w.dHs, d.T, d.H,
                                                  d.G, d.P, d.N, d.L, d.nc));
  const int PN = d.P * d.N;
  const int nsplit = launch_state_passing_bwd(d, a, w, s);
  SSD_LAUNCH("k_dyx", s, k_dyx<Tin><<<grid, kThreads, 0, s>>>(x, dy, w.dyx, d.T, d.H, d.P, d.L, d.nc));
  SSD_LAUNCH("k_bwd_dx", s, k_bwd_dx<Tin><<<grid, kThreads, 0, s>>>(x, Bm, dy, w.f.CB, w.f.delta, w.f.acs, w.dS, a.f.D,
                                          a.dx, w.ddir, w.qrow, d.T, d.H, d.G, d.P, d.N, d.L,
                                          d.nc));
  SSD_LAUNCH("k_bwd_dC", s, k_bwd_dC<Tin><<<grid, kThreads, 0, s>>>(Bm, Cm, dy, w.dyx, w.f.delta, w.f.acs, w.f.Hprev,
                                          w.dCh, w.ycs, d.T, d.H, d.G, d.P, d.N, d.L, d.nc));
  SSD_LAUNCH("k_bwd_dB", s, k_bwd_dB<Tin><<<grid, kThreads, 0, s>>>(x, Cm, w.dyx, w.f.delta, w.f.acs, w.dS, w.dBh, d.T,
                                          d.H, d.G, d.P, d.N, d.L, d.nc));
  SSD_LAUNCH("k_bwd_ddA", s, k_bwd_ddA<Tin><<<grid, kThreads, 0, s>>>(static_cast<const Tin*>(a.f.dt), a.f.dt_bias, a.f.A,
                                           w.f.CB, w.dyx, w.f.delta, w.f.acs, w.ddir, w.qrow,
                                           w.ycs, w.dlast, nsplit, a.ddt, w.part, d.T, d.H, d.G, d.L,
                                           d.nc));
  const int64_t BT = (int64_t)d.B * d.T;
  const int64_t nred = BT * d.G * d.N;
  const int rb = (int)((nred + kThreads - 1) / kThreads);
  SSD_LAUNCH("k_group_reduce", s, k_group_reduce<<<rb, kThreads, 0, s>>>(w.dBh, a.dB, BT, d.H, d.G, d.N));
  SSD_LAUNCH("k_group_reduce", s, k_group_reduce<<<rb, kThreads, 0, s>>>(w.dCh, a.dC, BT, d.H, d.G, d.N));
  SSD_LAUNCH("k_param_grads", s, k_param_grads<<<d.H, 32, 0, s>>>(w.part, a.dA, a.ddt_bias, a.dD, d.B, d.H, d.nc));
}

}  // namespace

cudaError_t simt_forward(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s) {
  if (d.in_bf16) {
    if (d.out_bf16) launch_forward<__nv_bfloat16, __nv_bfloat16>(d, a, w, s);
    else launch_forward<__nv_bfloat16, float>(d, a, w, s);
  } else {
    if (d.out_bf16) launch_forward<float, __nv_bfloat16>(d, a, w, s);
    else launch_forward<float, float>(d, a, w, s);
  }
  return cudaGetLastError();
}

int seg_max_segments(const Dims& d) {
  // a property of the shape, so workspace sizes do not depend on the device:
  // scratch only where the (batch, head) grid is small and there are chunks
  // to split (at most 16 segments of at least 4 chunks)
  const int64_t ctas =
      (int64_t)(((d.P << d.hs) * d.N / 8 + kThreads - 1) / kThreads) * (d.H >> d.hs) * d.B;
  if (d.nc < 8 || ctas >= 256) return 0;
  return std::min(16, d.nc / 4);
}

void simt_cumsum(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s) {
  if (d.in_bf16) launch_cumsum<__nv_bfloat16>(d, a, w, s);
  else launch_cumsum<float>(d, a, w, s);
}

void simt_state_passing(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s) {
  launch_state_passing(d, a, w, s);
}

void simt_front(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s) {
  // chunk_cumsum, chunk_state, state_passing (no C B^T: the states do not need C)
  const dim3 grid(d.nc, d.H, d.B);
  if (d.in_bf16) {
    using T = __nv_bfloat16;
    launch_cumsum<T>(d, a, w, s);
    SSD_LAUNCH("k_chunk_state", s, k_chunk_state<T, 0><<<grid, kThreads, 0, s>>>(
        static_cast<const T*>(a.x), static_cast<const T*>(a.B), w.delta, w.acs, w.S, d.T, d.H,
        d.G, d.P, d.N, d.L, d.nc));
  } else {
    launch_cumsum<float>(d, a, w, s);
    SSD_LAUNCH("k_chunk_state", s, k_chunk_state<float, 0><<<grid, kThreads, 0, s>>>(
        static_cast<const float*>(a.x), static_cast<const float*>(a.B), w.delta, w.acs, w.S, d.T,
        d.H, d.G, d.P, d.N, d.L, d.nc));
  }
  launch_state_passing(d, a, w, s);
}

void simt_dstates(const Dims& d, const void* dy, const void* C, const float* delta,
                  const float* acs, float* dHs, cudaStream_t s) {
  const dim3 grid(d.nc, d.H, d.B);
  if (d.in_bf16) {
    using T = __nv_bfloat16;
    SSD_LAUNCH("k_chunk_state", s, k_chunk_state<T, 1><<<grid, kThreads, 0, s>>>(
        static_cast<const T*>(dy), static_cast<const T*>(C), delta, acs, dHs, d.T, d.H, d.G, d.P,
        d.N, d.L, d.nc));
  } else {
    SSD_LAUNCH("k_chunk_state", s, k_chunk_state<float, 1><<<grid, kThreads, 0, s>>>(
        static_cast<const float*>(dy), static_cast<const float*>(C), delta, acs, dHs, d.T, d.H,
        d.G, d.P, d.N, d.L, d.nc));
  }
}

int simt_state_passing_bwd(const Dims& d, const float* dHs, const float* acs, const float* Hprev,
                           const float* dfinal, float* dS, float* dlast, float* dinit,
                           void* dSimg, const void* Himg, float* seg, cudaStream_t s) {
  BwdArgs a{};
  a.dfinal = dfinal;
  a.dinit = dinit;
  BwdWs w{};
  w.dSimg = dSimg;
  w.f.Himg = const_cast<void*>(Himg);
  w.dHs = const_cast<float*>(dHs);
  w.f.acs = const_cast<float*>(acs);
  w.f.Hprev = const_cast<float*>(Hprev);
  w.dS = dS;
  w.dlast = dlast;
  w.f.seg = seg;
  return launch_state_passing_bwd(d, a, w, s);
}

void simt_param_grads(const Dims& d, const float* part, float* dA, float* ddt_bias, float* dD,
                      cudaStream_t s) {
  SSD_LAUNCH("k_param_grads", s, launch_pdl(k_param_grads, dim3(d.H), dim3(32), 0, s, part, dA,
                                            ddt_bias, dD, d.B, d.H, d.nc));
}

cudaError_t simt_backward(const Dims& d, const BwdArgs& a, const BwdWs& w, cudaStream_t s) {
  if (d.in_bf16) launch_backward<__nv_bfloat16>(d, a, w, s);
  else launch_backward<float>(d, a, w, s);
  return cudaGetLastError();
}

}  // namespace ssd

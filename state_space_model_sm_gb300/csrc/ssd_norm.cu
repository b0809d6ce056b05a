// Gated RMSNorm, the step after the SSD output in a Mamba-2 layer (its
// backward is the pages' _layer_norm_bwd, step bwd_2 of "Latency and speedup
// by kernel"): with u = y * silu(z), per row and group g of group_size
// features
//     rstd_g = 1 / sqrt(mean_g(u^2) + eps),   out = u * rstd_g * w
// and the backward
//     xhat = u rstd, gx = dout w, c = mean_g(gx xhat)
//     du = rstd (gx - xhat c);  dy = du silu(z);  dz = du y silu'(z)
//     dw = sum over rows of dout xhat.
//
// Both passes are HBM-bound streams: the lesson the pages draw for this
// kernel ("The highway got wider, but we didn't add any cars") is that it
// needs enough independent requests in flight per SM.  Here the rows reach
// shared memory by bulk asynchronous copies: each persistent CTA owns a ring
// of NS stages, a stage holds one block of RPC consecutive rows of every input
// tensor (one contiguous copy per tensor, completing on the stage's
// mbarrier), and NS - 1 stages are in flight while the CTA computes the
// current one, so the bytes in flight per SM are set by the ring, not by
// registers or the row count.  Every thread owns 8 consecutive features of a
// row; group sums are warp butterflies (plus shared memory when a group spans
// several warps).  dw is reduced per CTA and then summed over CTAs in a fixed
// order (deterministic).  Waits are bounded (1 s): on expiry the kernel
// records SSD_ERR_TIMEOUT in the status word, drains its copies in flight
// (again bounded) and returns.
#include <cuda_bf16.h>

#include <mutex>

#include "ssd_internal.h"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

using namespace tc;

constexpr int kV = 8;                 // features per thread
constexpr int kMaxNT = 512;           // threads per CTA at most
constexpr int kMaxStages = 8;         // ring depth at most
constexpr int kRingBytes = 96 * 1024;  // ring size aimed at (two CTAs per SM)
constexpr int kNormMaxCtasPerSm = 8;  // persistent grid: at most this many CTAs per SM

// 8 consecutive elements as 4 pairs (packed fp32x2 arithmetic below)
__device__ __forceinline__ void lds8(const __nv_bfloat16* p, float2 (&v)[4]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __bfloat1622float2(h[i]);
}

__device__ __forceinline__ void lds8(const float* p, float2 (&v)[4]) {
  const float4 a = reinterpret_cast<const float4*>(p)[0];
  const float4 b = reinterpret_cast<const float4*>(p)[1];
  v[0] = make_float2(a.x, a.y), v[1] = make_float2(a.z, a.w);
  v[2] = make_float2(b.x, b.y), v[3] = make_float2(b.z, b.w);
}

__device__ __forceinline__ void store8(__nv_bfloat16* p, const float2 (&v)[4]) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __float22bfloat162_rn(v[i]);
  __stcs(reinterpret_cast<uint4*>(p), u);
}

__device__ __forceinline__ void store8(float* p, const float2 (&v)[4]) {
  __stcs(reinterpret_cast<float4*>(p), make_float4(v[0].x, v[0].y, v[1].x, v[1].y));
  __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(v[2].x, v[2].y, v[3].x, v[3].y));
}

__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }

// sigmoid of a pair: 1 / (1 + e^-z) with the fast exponential and divide
// (e^-z overflowing to inf for z < -88 gives exactly 0)
__device__ __forceinline__ float2 sigmoid2(float2 z) {
  const float2 d = __fadd2_rn(make_float2(__expf(-z.x), __expf(-z.y)), f2(1.f));
  return make_float2(__fdividef(1.f, d.x), __fdividef(1.f, d.y));
}

struct NormDims {
  int M, D, gs;
  int VPT;     // 8-feature vectors per thread (1, or 2 in the forward where it fits)
  int TPR;     // threads per row = D / (8 VPT)
  int TPG;     // threads per group = gs / (8 VPT)
  int RPC;     // rows per item (one ring stage); NT = RPC * TPR threads
  int n_iter;  // items: ceil(M / RPC)
  int NS;      // ring stages
  float eps;
  int ring_cap;  // ring bytes aimed at
  int cta_cap;   // CTAs per SM at most
};

// This thread's place: its row slot and 8 features within an item, its
// group, and the shape of its group sum (all loop-invariant).
struct ThreadMap {
  int slot;   // row slot within an item
  int f0;     // first feature
  int off;    // element offset within one tensor's block: slot * D + f0
  int grp;    // group index within the row (rstd column)
  bool lead;  // first thread of its group (writes rstd)
  int wl;     // butterfly width: min(TPG, 32)
  int g0;     // first warp of the group (groups spanning warps)
  int wpg;    // warps per group (groups spanning warps)
};

__device__ __forceinline__ ThreadMap thread_map(const NormDims& d) {
  ThreadMap m;
  const int tid = threadIdx.x;
  m.slot = tid / d.TPR;
  const int v = tid - m.slot * d.TPR;
  m.f0 = v * kV * d.VPT;
  m.off = m.slot * d.D + m.f0;
  m.grp = v / d.TPG;
  m.lead = v == m.grp * d.TPG;
  m.wl = d.TPG < 32 ? d.TPG : 32;
  m.wpg = d.TPG >> 5;
  m.g0 = m.wpg > 0 ? ((tid >> 5) / m.wpg) * m.wpg : 0;
  return m;
}

// Sum of v over the threads of the caller's group; every thread of the
// group gets the same value.  Groups of <= 32 threads are aligned segments
// of a warp (xor butterfly); larger ones are whole warps, combined through
// shared memory in warp order.  Called by every thread of the CTA; the
// partials alternate between two buffers (call parity `ph`), so one barrier
// per call suffices: a buffer is rewritten two calls later, after the
// barrier of the call in between.
template <bool kBig>
__device__ __forceinline__ float group_sum(float v, const ThreadMap& m, float (*red)[32], int ph) {
  if constexpr (kBig) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  } else {
    for (int o = m.wl >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  }
  if constexpr (kBig) {
    if ((threadIdx.x & 31) == 0) red[ph][threadIdx.x >> 5] = v;
    __syncthreads();
    float s = 0.f;
    for (int k = 0; k < m.wpg; ++k) s += red[ph][m.g0 + k];
    v = s;
  }
  return v;
}

// The ring of one CTA: NTENS tensors' row blocks per stage, stage s at
// base + s * NTENS * tile; item j of this CTA (the j-th it takes) uses stage
// j % NS in phase (j / NS) & 1.  Issue / drain are called by thread 0.
template <int NTENS, typename Tin>
struct RowRing {
  unsigned char* base;
  uint64_t* full;
  size_t tile;  // bytes of one tensor's block: RPC * D * sizeof(Tin)
  const Tin* src[NTENS];

  __device__ void issue(const NormDims& d, int item, int s) const {
    const int r0 = item * d.RPC;
    const int nr = min(d.RPC, d.M - r0);
    const uint32_t bytes = (uint32_t)nr * d.D * sizeof(Tin);
    // write-after-read on the stage: every thread's reads of it precede the CTA
    // barrier that thread 0 passed before calling this (no proxy fence, which
    // would also wait for this thread's global stores)
    mbar_arrive_expect_tx(&full[s], NTENS * bytes);
#pragma unroll
    for (int t = 0; t < NTENS; ++t)
      bulk_g2s(base + ((size_t)s * NTENS + t) * tile, src[t] + (int64_t)r0 * d.D, bytes, &full[s]);
  }
  __device__ const Tin* at(int s, int t) const {
    return reinterpret_cast<const Tin*>(base + ((size_t)s * NTENS + t) * tile);
  }
  // waits (bounded, without the abort flag) for items [from, to) of this CTA
  __device__ void drain(const NormDims& d, int from, int to) const {
    for (int j = from; j < to; ++j) {
      const uint32_t a = smem_u32(&full[j % d.NS]), par = (j / d.NS) & 1;
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(a, par) && globaltimer_ns() - t0 < kWaitLimitNs) {
      }
    }
  }
};

// Start of a CTA: barriers, abort flag and w (D floats, after the ring) in
// shared memory, and the first NS items in flight.  Returns the number of
// items this CTA takes.
template <int NTENS, typename Tin>
__device__ __forceinline__ int ring_start(const NormDims& d, const RowRing<NTENS, Tin>& ring,
                                          const float* w, float* sw, int* abort_flag,
                                          int& issued) {
  const int mine = d.n_iter > (int)blockIdx.x
                       ? (d.n_iter - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < d.NS; ++s) mbar_init(&ring.full[s], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  for (int f = threadIdx.x; f < d.D; f += blockDim.x) sw[f] = w[f];
  __syncthreads();
  issued = 0;
  if (threadIdx.x == 0)
    for (; issued < d.NS && issued < mine; ++issued)
      ring.issue(d, blockIdx.x + issued * gridDim.x, issued);
  return mine;
}

// Item k's stage (s, phase) is full: warp 0 waits on its barrier (bounded,
// suspending between tries) while the other warps wait at the CTA barrier,
// neither of which costs issue slots;
// the barrier also tells thread 0 that every thread is past item k - 1, so it
// refills item k - 1's stage (sprev).  False (for every thread) after a
// timeout.
template <int NTENS, typename Tin>
__device__ __forceinline__ bool ring_acquire(const NormDims& d, const RowRing<NTENS, Tin>& ring,
                                             int k, int s, uint32_t phase, int sprev, int mine,
                                             int& issued, int* status, int* abort_flag) {
  bool got = true;
  if (threadIdx.x < 32) got = mbar_wait_suspend(&ring.full[s], phase, status, abort_flag);
  if (!__syncthreads_and(got)) return false;
  if (threadIdx.x == 0 && k > 0 && issued < mine) {
    ring.issue(d, blockIdx.x + issued * gridDim.x, sprev);
    ++issued;
  }
  return true;
}

template <typename Tin, typename Tout, bool kBig, int VPT>
__global__ void __launch_bounds__(kMaxNT, 2)
    k_gated_norm_fwd(const Tin* __restrict__ y, const Tin* __restrict__ z,
                     const float* __restrict__ w, Tout* __restrict__ out,
                     float* __restrict__ rstd, NormDims d, int* status) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t full[kMaxStages];
  __shared__ float red[2][32];
  __shared__ int abort_flag;
  const size_t tile = (size_t)d.RPC * d.D * sizeof(Tin);
  RowRing<2, Tin> ring{smem, full, tile, {y, z}};
  float* sw = reinterpret_cast<float*>(smem + (size_t)d.NS * 2 * tile);
  int issued;
  const int mine = ring_start(d, ring, w, sw, &abort_flag, issued);
  const ThreadMap m = thread_map(d);
  const int ngr = d.D / d.gs;
  const int tile_e = d.RPC * d.D;  // elements of one tensor's block
  const Tin* sy = reinterpret_cast<const Tin*>(smem) + m.off;
  float2 wv[4 * VPT];
#pragma unroll
  for (int q = 0; q < VPT; ++q) lds8(sw + m.f0 + 8 * q, *reinterpret_cast<float2(*)[4]>(wv + 4 * q));
  int row = blockIdx.x * d.RPC + m.slot;
  const int row_step = gridDim.x * d.RPC;
  int s = 0, sprev = 0;
  uint32_t phase = 0;
  int k = 0;
  for (; k < mine; ++k) {
    if (!ring_acquire(d, ring, k, s, phase, sprev, mine, issued, status, &abort_flag)) break;
    const bool live = row < d.M;
    float2 u[4 * VPT];
    float2 ss2 = f2(0.f);
    const Tin* st = sy + s * 2 * tile_e;
#pragma unroll
    for (int q = 0; q < VPT; ++q) {
      float2 yv[4], zv[4];
      lds8(st + 8 * q, yv);
      lds8(st + tile_e + 8 * q, zv);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        u[4 * q + i] = __fmul2_rn(yv[i], __fmul2_rn(zv[i], sigmoid2(zv[i])));
        ss2 = __ffma2_rn(u[4 * q + i], u[4 * q + i], ss2);
      }
    }
    const float ss = group_sum<kBig>(live ? ss2.x + ss2.y : 0.f, m, red, 0);
    const float r = rsqrtf(ss / (float)d.gs + d.eps);
    if (live) {
#pragma unroll
      for (int q = 0; q < VPT; ++q) {
        float2 o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = __fmul2_rn(__fmul2_rn(u[4 * q + i], f2(r)), wv[4 * q + i]);
        store8(out + (int64_t)row * d.D + m.f0 + 8 * q, o);
      }
      if (rstd && m.lead) rstd[(int64_t)row * ngr + m.grp] = r;
    }
    row += row_step;
    sprev = s;
    if (++s == d.NS) s = 0, phase ^= 1u;
  }
  if (threadIdx.x == 0 && k < issued) ring.drain(d, k, issued);  // only after a timeout
}

template <typename Tin, typename Tout, bool kBig>
__global__ void __launch_bounds__(kMaxNT, 2)
    k_gated_norm_bwd(const Tin* __restrict__ y, const Tin* __restrict__ z,
                     const float* __restrict__ w, const float* __restrict__ rstd,
                     const Tin* __restrict__ dout, Tout* __restrict__ dy, Tout* __restrict__ dz,
                     float* __restrict__ dw_part, NormDims d, int* status) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ uint64_t full[kMaxStages];
  __shared__ float red[2][32];
  __shared__ int abort_flag;
  const size_t tile = (size_t)d.RPC * d.D * sizeof(Tin);
  RowRing<3, Tin> ring{smem, full, tile, {y, z, dout}};
  float* sw = reinterpret_cast<float*>(smem + (size_t)d.NS * 3 * tile);  // D floats
  float* dsm = reinterpret_cast<float*>(smem);  // NT * 8 floats, on the ring once it is idle
  int issued;
  const int mine = ring_start(d, ring, w, sw, &abort_flag, issued);
  const ThreadMap m = thread_map(d);
  const int ngr = d.D / d.gs;
  const int tile_e = d.RPC * d.D;
  const Tin* sy = reinterpret_cast<const Tin*>(smem) + m.off;
  float2 dw2[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) dw2[i] = f2(0.f);
  int row = blockIdx.x * d.RPC + m.slot;
  const int row_step = gridDim.x * d.RPC;
  // the saved rstd of this thread's next row, loaded one item ahead
  float r_next = (rstd && row < d.M) ? rstd[(int64_t)row * ngr + m.grp] : 0.f;
  int s = 0, sprev = 0;
  uint32_t phase = 0;
  int k = 0;
  for (; k < mine; ++k) {
    if (!ring_acquire(d, ring, k, s, phase, sprev, mine, issued, status, &abort_flag)) break;
    const bool live = row < d.M;
    float r = r_next;
    if (rstd && row + row_step < d.M) r_next = rstd[(int64_t)(row + row_step) * ngr + m.grp];
    const Tin* st = sy + s * 3 * tile_e;
    // live across the group sums: silu(z), y silu'(z), xhat, dout w, dw
    float2 sl[4], yd[4], xh[4], gv[4];
    {
      float2 yv[4];
      lds8(st, yv);
      lds8(st + tile_e, sl);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 zz = sl[i], sg = sigmoid2(zz);
        sl[i] = __fmul2_rn(zz, sg);                                           // silu(z)
        xh[i] = __fmul2_rn(yv[i], sl[i]);                                     // u for now
        const float2 dsg = __fmul2_rn(sg, __ffma2_rn(zz, __ffma2_rn(sg, f2(-1.f), f2(1.f)),
                                                     f2(1.f)));               // silu'(z)
        yd[i] = __fmul2_rn(yv[i], dsg);
      }
    }
    lds8(st + 2 * tile_e, gv);
    int ph = 0;
    if (!rstd) {
      float2 ss2 = f2(0.f);
#pragma unroll
      for (int i = 0; i < 4; ++i) ss2 = __ffma2_rn(xh[i], xh[i], ss2);
      const float ss = group_sum<kBig>(live ? ss2.x + ss2.y : 0.f, m, red, ph);
      ph = 1;
      r = rsqrtf(ss / (float)d.gs + d.eps);
    }
    float2 dot2 = f2(0.f);
    {
      float2 wv[4];
      lds8(sw + m.f0, wv);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xh[i] = __fmul2_rn(xh[i], f2(r));
        if (live) dw2[i] = __ffma2_rn(gv[i], xh[i], dw2[i]);
        gv[i] = __fmul2_rn(gv[i], wv[i]);  // dout w
        dot2 = __ffma2_rn(gv[i], xh[i], dot2);
      }
    }
    const float c = group_sum<kBig>(live ? dot2.x + dot2.y : 0.f, m, red, ph) / (float)d.gs;
    if (live) {
      float2 a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // du = r (dout w - xhat c); dy = du silu(z); dz = du y silu'(z)
        const float2 du = __fmul2_rn(f2(r), __ffma2_rn(xh[i], f2(-c), gv[i]));
        a[i] = __fmul2_rn(du, sl[i]);
        b[i] = __fmul2_rn(du, yd[i]);
      }
      const int64_t go = (int64_t)row * d.D + m.f0;
      store8(dy + go, a);
      store8(dz + go, b);
    }
    row += row_step;
    sprev = s;
    if (++s == d.NS) s = 0, phase ^= 1u;
  }
  if (threadIdx.x == 0 && k < issued) ring.drain(d, k, issued);  // only after a timeout
  __syncthreads();  // the ring is idle: no copy in flight, every read of it done
  // the CTA's dw: row slots summed in order, one partial row per CTA
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    dsm[m.off + 2 * i] = dw2[i].x;
    dsm[m.off + 2 * i + 1] = dw2[i].y;
  }
  __syncthreads();
  for (int f = threadIdx.x; f < d.D; f += blockDim.x) {
    float sum = 0.f;
    for (int sl = 0; sl < d.RPC; ++sl) sum += dsm[sl * d.D + f];
    dw_part[(int64_t)blockIdx.x * d.D + f] = sum;
  }
}

// dw[f] = the sum over parts p of part[p][f] in a fixed order.  Grid
// ceil(D / 32) blocks of 512 threads: thread (slice, c) sums parts slice,
// slice + 16, ... of column c into four interleaved accumulators (loads in
// flight), then the 16 slice sums are added in slice order.
__global__ void __launch_bounds__(512)
    k_norm_dw_reduce(const float* __restrict__ part, float* __restrict__ dw, int nparts, int D) {
  __shared__ float ssum[16][32];
  const int c = threadIdx.x & 31, sl = threadIdx.x >> 5;
  const int f = blockIdx.x * 32 + c;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  if (f < D) {
    int p = sl;
    for (; p + 48 < nparts; p += 64) {
      a0 += part[(int64_t)p * D + f];
      a1 += part[(int64_t)(p + 16) * D + f];
      a2 += part[(int64_t)(p + 32) * D + f];
      a3 += part[(int64_t)(p + 48) * D + f];
    }
    for (; p < nparts; p += 16) a0 += part[(int64_t)p * D + f];
  }
  ssum[sl][c] = (a0 + a1) + (a2 + a3);
  __syncthreads();
  if (sl == 0 && f < D) {
    float t = 0.f;
#pragma unroll
    for (int q = 0; q < 16; ++q) t += ssum[q][c];
    dw[f] = t;
  }
}

// ------------------------------------------------------ launch-config table
// Per-shape launch parameters set through ssd_gated_norm_set_config (an
// offline sweep's table, loaded at start-up); a zero field keeps the
// built-in choice.  Keyed by (features, group_size, in_dtype, out_dtype):
// the row count does not change the best launch once there are many rows.
struct NormEntry {
  int64_t features, group_size;
  int32_t in_dtype, out_dtype;
  ssd_norm_config cfg;
};
constexpr int kMaxNormEntries = 64;
NormEntry g_norm_table[kMaxNormEntries];
int g_norm_entries = 0;
std::mutex g_norm_mu;

bool same_key(const NormEntry& e, const ssd_norm_shape* s) {
  return e.features == s->features && e.group_size == s->group_size &&
         e.in_dtype == s->in_dtype && e.out_dtype == s->out_dtype;
}

bool table_lookup(const ssd_norm_shape* s, ssd_norm_config* out) {
  std::lock_guard<std::mutex> lk(g_norm_mu);
  for (int i = 0; i < g_norm_entries; ++i)
    if (same_key(g_norm_table[i], s)) {
      *out = g_norm_table[i].cfg;
      return true;
    }
  return false;
}

// rows per item valid for a row of TPR threads: the CTA (RPC * TPR threads)
// stays within kMaxNT and tiles whole warps
bool rpc_ok(int rpc, int TPR) {
  const int nt = rpc * TPR;
  return rpc >= 1 && nt <= kMaxNT && nt % 32 == 0;
}

bool norm_dims(const ssd_norm_shape* s, NormDims* d) {
  if (!s || s->rows < 0 || s->features < 8 || s->group_size < 8) return false;
  if (s->features % 8 || s->group_size % 8 || s->features % s->group_size) return false;
  if (!(s->eps >= 0.f)) return false;
  if ((s->in_dtype != SSD_F32 && s->in_dtype != SSD_BF16) ||
      (s->out_dtype != SSD_F32 && s->out_dtype != SSD_BF16))
    return false;
  // rows advance by a grid stride in int arithmetic: keep them below 2^30
  if (s->features > 65536 || s->rows >= ((int64_t)1 << 30)) return false;
  d->M = (int)s->rows;
  d->D = (int)s->features;
  d->gs = (int)s->group_size;
  d->VPT = 1;
  d->TPR = d->D / kV;
  d->TPG = d->gs / kV;
  d->eps = s->eps;
  d->RPC = d->TPR < kMaxNT ? kMaxNT / d->TPR : 1;
  d->ring_cap = kRingBytes;
  d->cta_cap = kNormMaxCtasPerSm;
  ssd_norm_config cfg;
  if (table_lookup(s, &cfg)) {
    if (cfg.rows_per_item > 0 && rpc_ok(cfg.rows_per_item, d->TPR)) d->RPC = cfg.rows_per_item;
    if (cfg.ring_kb > 0) d->ring_cap = cfg.ring_kb * 1024;
    if (cfg.ctas_per_sm > 0) d->cta_cap = cfg.ctas_per_sm;
  }
  d->n_iter = (int)((s->rows + d->RPC - 1) / d->RPC);
  d->NS = 0;
  return true;
}

// what the kernels implement: a row of at most 512 threads (features <=
// 4096) that tiles warps (a multiple of 32 threads, or a power of two below
// 32), and groups that are aligned power-of-two warp segments or whole warps
int norm_supported(const NormDims& d) {
  if (d.TPR > kMaxNT) return SSD_ERR_UNSUPPORTED;
  const bool tpr_ok = d.TPR % 32 == 0 || (32 % d.TPR == 0);
  const bool tpg_ok = d.TPG % 32 == 0 || (d.TPG < 32 && (d.TPG & (d.TPG - 1)) == 0);
  return tpr_ok && tpg_ok ? SSD_OK : SSD_ERR_UNSUPPORTED;
}

// ring depth for ntens tensors of elt bytes: as many stages as fit in the
// shared memory left to each CTA when registers allow `ctas` CTAs per SM
// (at most kRingBytes), between 2 and kMaxStages
int ring_stages(const NormDims& d, int ntens, int elt, int ctas, size_t other) {
  const size_t stage = (size_t)ntens * d.RPC * d.D * elt;
  const size_t per_cta = (size_t)(220 * 1024) / (size_t)(ctas < 2 ? 2 : ctas);
  size_t budget = per_cta > other ? per_cta - other : 0;
  if (budget > (size_t)d.ring_cap) budget = d.ring_cap;
  const size_t ns = budget / stage;
  return ns < 2 ? 2 : (ns > (size_t)kMaxStages ? kMaxStages : (int)ns);
}

// CTAs per SM that the kernel's registers and threads allow (at most 4)
int reg_ctas(const void* kern, int nt) {
  int per = 1;
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kern, nt, 0);
  return per < 1 ? 1 : (per > 4 ? 4 : per);
}

int norm_grid(const NormDims& d, const void* kern, int nt, size_t smem) {
  int dev = 0, sms = 148, per = 1;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, kern, nt, smem);
  per = per < 1 ? 1 : (per > d.cta_cap ? d.cta_cap : per);
  const int64_t g = (int64_t)per * sms;
  return (int)(d.n_iter < g ? d.n_iter : g);
}

// The forward's thread map with two vectors per thread, when the row and
// group widths allow it (the same rules as for one vector); false if not.
bool fwd_two_vectors(NormDims* d) {
  if (d->D % 16 || d->gs % 16) return false;
  NormDims e = *d;
  e.VPT = 2;
  e.TPR = d->D / 16;
  e.TPG = d->gs / 16;
  if (norm_supported(e) != SSD_OK) return false;
  e.RPC = e.TPR < kMaxNT ? kMaxNT / e.TPR : 1;
  if ((e.RPC * e.TPR) % 32) return false;
  e.n_iter = (e.M + e.RPC - 1) / e.RPC;
  *d = e;
  return true;
}

template <typename Tin, typename Tout, int VPT>
int launch_norm_fwd_v(NormDims d, const void* y, const void* z, const float* w, void* out,
                      float* rstd, cudaStream_t s, int* status) {
  const int nt = d.RPC * d.TPR;
  const bool big = d.TPG > 32;
  auto kb = k_gated_norm_fwd<Tin, Tout, true, VPT>;
  auto ks = k_gated_norm_fwd<Tin, Tout, false, VPT>;
  const void* kern = big ? (const void*)kb : (const void*)ks;
  d.NS = ring_stages(d, 2, sizeof(Tin), reg_ctas(kern, nt), (size_t)d.D * sizeof(float));
  const size_t smem = (size_t)d.NS * 2 * d.RPC * d.D * sizeof(Tin) + (size_t)d.D * sizeof(float);
  const int grid = norm_grid(d, kern, nt, smem);
  const Tin* yy = static_cast<const Tin*>(y);
  const Tin* zz = static_cast<const Tin*>(z);
  Tout* oo = static_cast<Tout*>(out);
  if (big)
    SSD_LAUNCH("k_gated_norm_fwd", s,
               kb<<<grid, nt, smem, s>>>(yy, zz, w, oo, rstd, d, status));
  else
    SSD_LAUNCH("k_gated_norm_fwd", s,
               ks<<<grid, nt, smem, s>>>(yy, zz, w, oo, rstd, d, status));
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

template <typename Tin, typename Tout>
int launch_norm_fwd(NormDims d, const void* y, const void* z, const float* w, void* out,
                    float* rstd, cudaStream_t s) {
  int* status = device_status_ptr();
  if (!status) return SSD_ERR_CUDA;
  // two 8-feature vectors per thread halve the per-row fixed work (the
  // backward keeps one: its live set would not fit the register budget)
  if (fwd_two_vectors(&d)) return launch_norm_fwd_v<Tin, Tout, 2>(d, y, z, w, out, rstd, s, status);
  return launch_norm_fwd_v<Tin, Tout, 1>(d, y, z, w, out, rstd, s, status);
}

template <typename Tin, typename Tout>
int launch_norm_bwd(NormDims d, const void* y, const void* z, const float* w,
                    const float* rstd, const void* dout, void* dy, void* dz, float* dw,
                    float* part, cudaStream_t s) {
  int* status = device_status_ptr();
  if (!status) return SSD_ERR_CUDA;
  const int nt = d.RPC * d.TPR;
  const bool big = d.TPG > 32;
  auto kb = k_gated_norm_bwd<Tin, Tout, true>;
  auto ks = k_gated_norm_bwd<Tin, Tout, false>;
  const void* kern = big ? (const void*)kb : (const void*)ks;
  d.NS = ring_stages(d, 3, sizeof(Tin), reg_ctas(kern, nt), (size_t)d.D * sizeof(float));
  const size_t ring_b = (size_t)d.NS * 3 * d.RPC * d.D * sizeof(Tin);
  const size_t part_b = (size_t)nt * kV * sizeof(float);  // dw partials alias the ring
  const size_t smem = (ring_b > part_b ? ring_b : part_b) + (size_t)d.D * sizeof(float);
  const int grid = norm_grid(d, kern, nt, smem);
  const Tin* yy = static_cast<const Tin*>(y);
  const Tin* zz = static_cast<const Tin*>(z);
  const Tin* gg = static_cast<const Tin*>(dout);
  Tout* a = static_cast<Tout*>(dy);
  Tout* b = static_cast<Tout*>(dz);
  if (big)
    SSD_LAUNCH("k_gated_norm_bwd", s,
               kb<<<grid, nt, smem, s>>>(yy, zz, w, rstd, gg, a, b, part, d, status));
  else
    SSD_LAUNCH("k_gated_norm_bwd", s,
               ks<<<grid, nt, smem, s>>>(yy, zz, w, rstd, gg, a, b, part, d, status));
  SSD_LAUNCH("k_norm_dw_reduce", s,
             k_norm_dw_reduce<<<(d.D + 31) / 32, 512, 0, s>>>(part, dw, grid, d.D));
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace
}  // namespace ssd

using namespace ssd;

extern "C" {

size_t ssd_gated_norm_workspace_size(const ssd_norm_shape* shape) {
  NormDims d;
  if (!norm_dims(shape, &d) || norm_supported(d) != SSD_OK) return 0;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) sms = 256;
  return (size_t)kNormMaxCtasPerSm * sms * d.D * sizeof(float);
}

int ssd_gated_norm_set_config(const ssd_norm_shape* shape, const ssd_norm_config* config) {
  NormDims d;
  if (!norm_dims(shape, &d) || norm_supported(d) != SSD_OK) return SSD_ERR_INVALID_ARG;
  if (config) {
    if (config->rows_per_item < 0 || config->ring_kb < 0 || config->ctas_per_sm < 0)
      return SSD_ERR_INVALID_ARG;
    if (config->rows_per_item > 0 && !rpc_ok(config->rows_per_item, d.TPR))
      return SSD_ERR_INVALID_ARG;
    if (config->ring_kb > 0 && (config->ring_kb < 8 || config->ring_kb > 200))
      return SSD_ERR_INVALID_ARG;
    if (config->ctas_per_sm > kNormMaxCtasPerSm) return SSD_ERR_INVALID_ARG;
  }
  std::lock_guard<std::mutex> lk(g_norm_mu);
  int i = 0;
  while (i < g_norm_entries && !same_key(g_norm_table[i], shape)) ++i;
  if (!config) {  // remove
    if (i < g_norm_entries) g_norm_table[i] = g_norm_table[--g_norm_entries];
    return SSD_OK;
  }
  if (i == g_norm_entries) {
    if (g_norm_entries == kMaxNormEntries) return SSD_ERR_UNSUPPORTED;
    ++g_norm_entries;
  }
  g_norm_table[i] = NormEntry{shape->features, shape->group_size, shape->in_dtype,
                              shape->out_dtype, *config};
  return SSD_OK;
}

int ssd_gated_norm_get_config(const ssd_norm_shape* shape, ssd_norm_config* out) {
  NormDims d;
  if (!out || !norm_dims(shape, &d) || norm_supported(d) != SSD_OK) return -SSD_ERR_INVALID_ARG;
  ssd_norm_config cfg;
  const bool set = table_lookup(shape, &cfg);
  out->rows_per_item = d.RPC;
  out->ring_kb = d.ring_cap / 1024;
  out->ctas_per_sm = d.cta_cap;
  return set ? 1 : 0;
}

int ssd_gated_norm_fwd(const ssd_norm_shape* shape, const void* y, const void* z,
                       const float* w, void* out, float* rstd, void* stream) {
  NormDims d;
  if (!norm_dims(shape, &d)) return SSD_ERR_INVALID_ARG;
  const int st = norm_supported(d);
  if (st != SSD_OK) return st;
  if (d.M == 0) return SSD_OK;
  if (!y || !z || !w || !out) return SSD_ERR_INVALID_ARG;
  if (!al16(y) || !al16(z) || !al16(out) || (reinterpret_cast<uintptr_t>(w) & 3) ||
      (reinterpret_cast<uintptr_t>(rstd) & 3))
    return SSD_ERR_INVALID_ARG;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool ib = shape->in_dtype == SSD_BF16, ob = shape->out_dtype == SSD_BF16;
  using bf = __nv_bfloat16;
  if (ib) return ob ? launch_norm_fwd<bf, bf>(d, y, z, w, out, rstd, s)
                    : launch_norm_fwd<bf, float>(d, y, z, w, out, rstd, s);
  return ob ? launch_norm_fwd<float, bf>(d, y, z, w, out, rstd, s)
            : launch_norm_fwd<float, float>(d, y, z, w, out, rstd, s);
}

int ssd_gated_norm_bwd(const ssd_norm_shape* shape, const void* y, const void* z,
                       const float* w, const float* rstd, const void* dout, void* dy, void* dz,
                       float* dw, void* workspace, size_t workspace_bytes, void* stream) {
  NormDims d;
  if (!norm_dims(shape, &d)) return SSD_ERR_INVALID_ARG;
  const int st = norm_supported(d);
  if (st != SSD_OK) return st;
  if (!w || !dw) return SSD_ERR_INVALID_ARG;
  if (d.M > 0 && (!y || !z || !dout || !dy || !dz)) return SSD_ERR_INVALID_ARG;
  if (!al16(y) || !al16(z) || !al16(dout) || !al16(dy) || !al16(dz) ||
      (reinterpret_cast<uintptr_t>(w) & 3) || (reinterpret_cast<uintptr_t>(rstd) & 3) ||
      (reinterpret_cast<uintptr_t>(dw) & 3))
    return SSD_ERR_INVALID_ARG;
  const size_t need = ssd_gated_norm_workspace_size(shape);
  if (!workspace || workspace_bytes < need || !al16(workspace)) return SSD_ERR_WORKSPACE;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (d.M == 0) {  // no rows: dw = 0
    return cudaMemsetAsync(dw, 0, (size_t)d.D * sizeof(float), s) == cudaSuccess ? SSD_OK
                                                                               : SSD_ERR_CUDA;
  }
  float* part = static_cast<float*>(workspace);
  const bool ib = shape->in_dtype == SSD_BF16, ob = shape->out_dtype == SSD_BF16;
  using bf = __nv_bfloat16;
  if (ib) return ob ? launch_norm_bwd<bf, bf>(d, y, z, w, rstd, dout, dy, dz, dw, part, s)
                    : launch_norm_bwd<bf, float>(d, y, z, w, rstd, dout, dy, dz, dw, part, s);
  return ob ? launch_norm_bwd<float, bf>(d, y, z, w, rstd, dout, dy, dz, dw, part, s)
            : launch_norm_bwd<float, float>(d, y, z, w, rstd, dout, dy, dz, dw, part, s);
}

}  // extern "C"

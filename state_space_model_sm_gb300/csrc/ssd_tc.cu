// tcgen05 tensor-core kernels of the SSD forward (bf16 inputs, headdim 64,
// d_state 64 or 128, chunk 128 or 256): chunk_state and chunk_scan.
//
// Precision: operands that the method forms in fp32 before a contraction
// (the decay-weighted x of chunk_state, the masked decay-weighted C.B^T of
// chunk_scan, the fp32 inter-chunk state) are split into two bf16 terms,
// v = hi + lo with hi = rn_bf16(v), and both terms are multiplied; raw bf16
// inputs enter as they are.  Every product is accumulated in fp32 in TMEM,
// so the results carry ~16 significant bits per operand instead of bf16's 8.
#include <algorithm>

#include "ssd_internal.h"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

using namespace tc;
using bf16 = __nv_bfloat16;

constexpr int kP = 64;  // headdim of the tensor-core path

__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                          ~uintptr_t(1023));
}

// Write 8 fp32 values as one 16-byte bf16 chunk (hi part) and, when lo is
// non-null, the rounding remainder as a second chunk.
__device__ __forceinline__ void store_split8(unsigned char* hi, unsigned char* lo,
                                             const float (&v)[8]) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float h0, l0, h1, l1;
    split_bf16(v[2 * i], h0, l0);
    split_bf16(v[2 * i + 1], h1, l1);
    h[i] = pack_bf16(h0, h1);
    l[i] = pack_bf16(l0, l1);
  }
  *reinterpret_cast<uint4*>(hi) = make_uint4(h[0], h[1], h[2], h[3]);
  if (lo) *reinterpret_cast<uint4*>(lo) = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// =============================================================== chunk_state
// grid (nc, B, ceil(H / (2 * pairs))), 256 threads.  For a head pair (h, h+1)
// of one group and chunk c:
//   D[m = 64 hh + p, n] = sum_l w_hh[l] x[l, h+hh, p] B[l, n],
//   w_hh[l] = exp(a_last - a_l) delta_l     ->  S[b, c, h+hh, p, n]
// A = (w x)^T as an MN-major operand (rows l, 128 columns = two heads x 64),
// B = the chunk's B rows as an MN-major operand (rows l, N columns).
template <int N, int L>
struct StateSmem {
  static constexpr int kPanelB = L * 128;        // bytes of one 64-column panel of L rows
  static constexpr int kB = (N / 64) * kPanelB;  // B tile
  static constexpr int kX = 2 * kPanelB;         // w x for a head pair (hi or lo)
  static constexpr int kBytes = kB + 2 * kX + 2 * L * 4 + 1024;
};

template <int N, int L>
__global__ void __launch_bounds__(256, 1)
    k_state_tc(const bf16* __restrict__ x, const bf16* __restrict__ Bm,
               const float* __restrict__ delta, const float* __restrict__ acs,
               float* __restrict__ S, int T, int H, int G, int nc, int pairs_per_cta,
               int* status) {
  using SM = StateSmem<N, L>;
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  unsigned char* base = align1024(smem_raw);
  unsigned char* sB = base;
  unsigned char* sXh = sB + SM::kB;
  unsigned char* sXl = sXh + SM::kX;
  float* sw = reinterpret_cast<float*>(sXl + SM::kX);  // [2][L]

  const int c = blockIdx.x, b = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hpg = H / G;
  const int pair0 = blockIdx.z * pairs_per_cta;
  const int npairs = min(pairs_per_cta, H / 2 - pair0);
  const int g = (2 * pair0) / hpg;
  const int64_t t0 = (int64_t)c * L;
  const int Lv = min(L, T - (int)t0);

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 128);

  // B rows of the chunk: N/8 chunks of 16 bytes per row, zero past seqlen.
  constexpr int kBC = N / 8;
  for (int i = tid; i < L * kBC; i += 256) {
    const int l = i / kBC, j = i % kBC;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (l < Lv)
      v = *reinterpret_cast<const uint4*>(Bm + ((((int64_t)b * T + t0 + l) * G + g) * N) + j * 8);
    *reinterpret_cast<uint4*>(sB + (j / 8) * SM::kPanelB + sw128(l, j % 8)) = v;
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tm = tmem_base;
  constexpr uint32_t idesc = idesc_bf16(128, N, 1, 1);

  for (int ip = 0; ip < npairs; ++ip) {
    const int h = 2 * (pair0 + ip);
    for (int i = tid; i < 2 * L; i += 256) {
      const int hh = i / L, l = i % L;
      const int64_t cv = (((int64_t)b * H + h + hh) * nc + c) * L;
      sw[i] = __expf(acs[cv + L - 1] - acs[cv + l]) * delta[cv + l];
    }
    __syncthreads();
    // w x for both heads: a row l holds x[l, h:h+2, 0:64] (256 contiguous bytes)
    for (int i = tid; i < L * 16; i += 256) {
      const int l = i >> 4, j = i & 15, hh = j >> 3;
      float v[8];
      if (l < Lv) {
        const uint4 u =
            *reinterpret_cast<const uint4*>(x + (((int64_t)b * T + t0 + l) * H + h) * kP + j * 8);
        unpack8(u, v);
        const float wl = sw[hh * L + l];
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] *= wl;
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) v[q] = 0.f;
      }
      const uint32_t off = hh * SM::kPanelB + sw128(l, j & 7);
      store_split8(sXh + off, sXl + off, v);
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      fence_after_sync();
      for (int ks = 0; ks < L / 16; ++ks) {
        const uint64_t bd = sdesc(smem_u32(sB) + ks * 2048, SM::kPanelB, 1024);
        mma_bf16(tm, sdesc(smem_u32(sXh) + ks * 2048, SM::kPanelB, 1024), bd, idesc,
                 ks > 0 ? 1u : 0u);
        mma_bf16(tm, sdesc(smem_u32(sXl) + ks * 2048, SM::kPanelB, 1024), bd, idesc, 1u);
      }
      mma_commit(&bar);
    }
    const bool ok = mbar_wait(&bar, ip & 1, status, &abort_flag);
    fence_after_sync();
    if (ok) {
      // lanes 32 q .. 32 q + 31 = rows m; warps q and q + 4 split the N columns
      const int q = warp & 3, half = warp >> 2;
      const int m = 32 * q + lane, hh = m >> 6, p = m & 63;
      float* out = S + ((((int64_t)b * nc + c) * H + h + hh) * kP + p) * N;
      const uint32_t ta = tm + ((uint32_t)(32 * q) << 16);
#pragma unroll
      for (int c0 = half * (N / 2); c0 < (half + 1) * (N / 2); c0 += 16) {
        float v[16];
        tmem_ld16(ta + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 16; k += 4)
          *reinterpret_cast<float4*>(out + c0 + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
      }
    }
    fence_before_sync();
    __syncthreads();
  }
  if (warp == 0) tmem_dealloc(tm, 128);
}

// ================================================================ chunk_scan
// grid (nc * L/128, B, ceil(H / heads_per_cta)), 256 threads.  CTA = rows
// l0 .. l0+127 of chunk c for a block of heads of one group:
//   CB[l, s] = C_l . B_s                         (TMEM cols 0 .. s_end-1, once)
//   per head:  Y  = sum_s P[l, s] x[s, :],  P = CB e^{a_l - a_s} delta_s [s <= l]
//              ST = C_l . H_c[p, :]
//              y  = Y + e^{a_l} ST + D x_l
template <int N, int L>
struct ScanSmem {
  static constexpr int kLT = 128;
  static constexpr int kC = (N / 64) * kLT * 128;           // C rows of the tile
  static constexpr int kBrows = (N / 64) * L * 128;         // B rows of the chunk
  static constexpr int kPbuf = 2 * kLT * 128;               // one P panel, hi + lo
  static constexpr int kBP = kBrows > 2 * kPbuf ? kBrows : 2 * kPbuf;
  static constexpr int kX = L * 128;                        // x rows, one MN panel
  static constexpr int kHhalf = (N / 64) * 64 * 128;        // H (hi or lo), K-major
  static constexpr int kBytes = kC + kBP + kX + 2 * kHhalf + 2 * L * 4 + 1024;
};

template <int N, int L, typename Tout>
__global__ void __launch_bounds__(256, 1)
    k_scan_tc(const bf16* __restrict__ x, const bf16* __restrict__ Bm,
              const bf16* __restrict__ Cm, const float* __restrict__ delta,
              const float* __restrict__ acs, const float* __restrict__ Hprev,
              const float* __restrict__ D, Tout* __restrict__ y, int T, int H, int G, int nc,
              int heads_per_cta, int* status) {
  using SM = ScanSmem<N, L>;
  constexpr int LT = SM::kLT, NLT = L / LT, NKP = N / 64;
  constexpr uint32_t kColY = 256, kColST = 320;
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t bar_cb, bar_done, bar_p[2];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  unsigned char* base = align1024(smem_raw);
  unsigned char* sC = base;
  unsigned char* sBP = sC + SM::kC;
  unsigned char* sX = sBP + SM::kBP;
  unsigned char* sHh = sX + SM::kX;
  unsigned char* sHl = sHh + SM::kHhalf;
  float* sa = reinterpret_cast<float*>(sHl + SM::kHhalf);
  float* sd = sa + L;

  const int c = blockIdx.x / NLT, lt = blockIdx.x % NLT, b = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hpg = H / G;
  const int h_begin = blockIdx.z * heads_per_cta;
  const int h_end = min(H, h_begin + heads_per_cta);
  const int g = h_begin / hpg;
  const int l0 = lt * LT, s_end = l0 + LT, nsp = s_end / 64;
  const int64_t t0 = (int64_t)c * L;
  const int Lv = min(L, T - (int)t0);

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bar_cb, 1);
    mbar_init(&bar_done, 1);
    mbar_init(&bar_p[0], 1);
    mbar_init(&bar_p[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 512);

  // C rows l0 .. l0+127 and B rows 0 .. s_end-1 (K-major, N/64 panels each)
  constexpr int kRC = N / 8;
  for (int i = tid; i < LT * kRC; i += 256) {
    const int r = i / kRC, j = i % kRC, l = l0 + r;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (l < Lv)
      v = *reinterpret_cast<const uint4*>(Cm + ((((int64_t)b * T + t0 + l) * G + g) * N) + j * 8);
    *reinterpret_cast<uint4*>(sC + (j / 8) * (LT * 128) + sw128(r, j % 8)) = v;
  }
  for (int i = tid; i < s_end * kRC; i += 256) {
    const int s = i / kRC, j = i % kRC;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (s < Lv)
      v = *reinterpret_cast<const uint4*>(Bm + ((((int64_t)b * T + t0 + s) * G + g) * N) + j * 8);
    *reinterpret_cast<uint4*>(sBP + (j / 8) * (L * 128) + sw128(s, j % 8)) = v;
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tm = tmem_base;
  if (tid == 0) {
    const uint32_t id = idesc_bf16(128, s_end, 0, 0);
    for (int ks = 0; ks < N / 16; ++ks) {
      const uint32_t kp = ks / 4, ko = (ks % 4) * 32;
      mma_bf16(tm, sdesc(smem_u32(sC) + kp * (LT * 128) + ko, 16, 1024),
               sdesc(smem_u32(sBP) + kp * (L * 128) + ko, 16, 1024), id, ks > 0 ? 1u : 0u);
    }
    mma_commit(&bar_cb);
  }
  mbar_wait(&bar_cb, 0, status, &abort_flag);
  fence_after_sync();

  const int q = warp & 3, half = warp >> 2;
  const int r = 32 * q + lane, l = l0 + r;  // this thread's row (TMEM lane)
  const uint32_t tlane = tm + ((uint32_t)(32 * q) << 16);
  unsigned char* Phi[2] = {sBP, sBP + SM::kPbuf};
  uint32_t ncommit[2] = {0, 0};
  constexpr uint32_t id_py = idesc_bf16(128, kP, 0, 1);
  constexpr uint32_t id_st = idesc_bf16(128, kP, 0, 0);

  for (int h = h_begin, it = 0; h < h_end; ++h, ++it) {
    const int64_t cv = (((int64_t)b * H + h) * nc + c) * L;
    for (int i = tid; i < L; i += 256) {
      sa[i] = acs[cv + i];
      sd[i] = delta[cv + i];
    }
    // x rows 0 .. s_end-1 of head h: one MN-major panel (rows s, 64 columns p)
    for (int i = tid; i < s_end * 8; i += 256) {
      const int s = i >> 3, j = i & 7;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (s < Lv)
        v = *reinterpret_cast<const uint4*>(x + (((int64_t)b * T + t0 + s) * H + h) * kP + j * 8);
      *reinterpret_cast<uint4*>(sX + sw128(s, j)) = v;
    }
    // H_c (fp32, 64 x N) as hi / lo bf16, K-major (rows p, N/64 panels)
    const float* Hc = Hprev + (((int64_t)b * nc + c) * H + h) * kP * N;
    for (int i = tid; i < kP * (N / 8); i += 256) {
      const int p = i / (N / 8), j = i % (N / 8);
      const float4 u0 = *reinterpret_cast<const float4*>(Hc + p * N + j * 8);
      const float4 u1 = *reinterpret_cast<const float4*>(Hc + p * N + j * 8 + 4);
      const float v[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
      const uint32_t off = (j / 8) * (64 * 128) + sw128(p, j % 8);
      store_split8(sHh + off, sHl + off, v);
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      fence_after_sync();
      for (int ks = 0; ks < N / 16; ++ks) {
        const uint32_t kp = ks / 4, ko = (ks % 4) * 32;
        const uint64_t ad = sdesc(smem_u32(sC) + kp * (LT * 128) + ko, 16, 1024);
        mma_bf16(tm + kColST, ad, sdesc(smem_u32(sHh) + kp * (64 * 128) + ko, 16, 1024), id_st,
                 ks > 0 ? 1u : 0u);
        mma_bf16(tm + kColST, ad, sdesc(smem_u32(sHl) + kp * (64 * 128) + ko, 16, 1024), id_st,
                 1u);
      }
    }
    const float al = sa[min(l, L - 1)];
    for (int j = 0; j < nsp; ++j) {
      const int buf = j & 1;
      if (ncommit[buf] > 0) mbar_wait(&bar_p[buf], (ncommit[buf] - 1) & 1, status, &abort_flag);
      unsigned char* ph = Phi[buf];
      unsigned char* pl = ph + LT * 128;
      float cb[32];
      tmem_ld16(tlane + 64 * j + 32 * half, *reinterpret_cast<float(*)[16]>(cb));
      tmem_ld16(tlane + 64 * j + 32 * half + 16, *reinterpret_cast<float(*)[16]>(cb + 16));
      tmem_wait_ld();
#pragma unroll
      for (int k8 = 0; k8 < 4; ++k8) {
        float v[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int s = 64 * j + 32 * half + 8 * k8 + e;
          v[e] = s <= l ? cb[8 * k8 + e] * __expf(al - sa[s]) * sd[s] : 0.f;
        }
        const uint32_t off = sw128(r, 4 * half + k8);
        store_split8(ph + off, pl + off, v);
      }
      fence_async_smem();
      fence_before_sync();
      __syncthreads();
      if (tid == 0) {
        fence_after_sync();
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t bd = sdesc(smem_u32(sX) + (64 * j + 16 * ks) * 128, L * 128, 1024);
          mma_bf16(tm + kColY, sdesc(smem_u32(ph) + ks * 32, 16, 1024), bd, id_py,
                   (j > 0 || ks > 0) ? 1u : 0u);
          mma_bf16(tm + kColY, sdesc(smem_u32(pl) + ks * 32, 16, 1024), bd, id_py, 1u);
        }
        mma_commit(&bar_p[buf]);
      }
      ncommit[buf]++;
    }
    if (tid == 0) mma_commit(&bar_done);
    const bool ok = mbar_wait(&bar_done, it & 1, status, &abort_flag);
    fence_after_sync();
    if (ok) {
      float yv[32], st[32];
      tmem_ld16(tlane + kColY + 32 * half, *reinterpret_cast<float(*)[16]>(yv));
      tmem_ld16(tlane + kColY + 32 * half + 16, *reinterpret_cast<float(*)[16]>(yv + 16));
      tmem_ld16(tlane + kColST + 32 * half, *reinterpret_cast<float(*)[16]>(st));
      tmem_ld16(tlane + kColST + 32 * half + 16, *reinterpret_cast<float(*)[16]>(st + 16));
      tmem_wait_ld();
      if (l < Lv) {
        const float ea = __expf(al), Dh = D ? D[h] : 0.f;
        Tout* out = y + (((int64_t)b * T + t0 + l) * H + h) * kP + 32 * half;
#pragma unroll
        for (int k8 = 0; k8 < 4; ++k8) {
          float xv[8];
          unpack8(*reinterpret_cast<const uint4*>(sX + sw128(l, 4 * half + k8)), xv);
          float o[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            o[e] = yv[8 * k8 + e] + ea * st[8 * k8 + e] + Dh * xv[e];
          if constexpr (sizeof(Tout) == 4) {
            float* of = reinterpret_cast<float*>(out) + 8 * k8;
            *reinterpret_cast<float4*>(of) = make_float4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<float4*>(of + 4) = make_float4(o[4], o[5], o[6], o[7]);
          } else {
            *reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(out) + 8 * k8) =
                make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]), pack_bf16(o[4], o[5]),
                           pack_bf16(o[6], o[7]));
          }
        }
      }
    }
    fence_before_sync();
    __syncthreads();
  }
  if (warp == 0) tmem_dealloc(tm, 512);
}

// ------------------------------------------------------------------ launch
int pick_heads_per_cta(int hpg, int units, int sms, int target_waves) {
  // largest divisor of hpg that still gives >= target_waves * sms CTAs
  int best = 1;
  for (int d = 1; d <= hpg; ++d)
    if (hpg % d == 0 && (int64_t)units * (hpg / d) * 1 >= (int64_t)target_waves * sms) best = d;
  return best;
}

template <int N, int L, typename Tout>
cudaError_t launch_tc_forward_t(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s,
                                int* status, int sms) {
  simt_cumsum(d, a, w, s);
  {
    using SM = StateSmem<N, L>;
    auto kern = k_state_tc<N, L>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
    const int pairs_total = d.H / 2;
    const int ppc = pick_heads_per_cta((d.H / d.G) / 2, d.B * d.nc * d.G, sms, 4);
    const dim3 grid(d.nc, d.B, (pairs_total + ppc - 1) / ppc);
    SSD_LAUNCH("k_state_tc", s,
               kern<<<grid, 256, SM::kBytes, s>>>(
                   static_cast<const bf16*>(a.x), static_cast<const bf16*>(a.B), w.delta, w.acs,
                   w.S, d.T, d.H, d.G, d.nc, ppc, status));
  }
  simt_state_passing(d, a, w, s);
  {
    using SM = ScanSmem<N, L>;
    auto kern = k_scan_tc<N, L, Tout>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
    const int hpc = pick_heads_per_cta(d.H / d.G, d.B * d.nc * (L / 128) * d.G, sms, 4);
    const dim3 grid(d.nc * (L / 128), d.B, (d.H + hpc - 1) / hpc);
    SSD_LAUNCH("k_scan_tc", s,
               kern<<<grid, 256, SM::kBytes, s>>>(
                   static_cast<const bf16*>(a.x), static_cast<const bf16*>(a.B),
                   static_cast<const bf16*>(a.C), w.delta, w.acs, w.Hprev, a.D,
                   static_cast<Tout*>(a.y), d.T, d.H, d.G, d.nc, hpc, status));
  }
  return cudaGetLastError();
}

template <int N, int L>
cudaError_t launch_tc_forward_nl(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s,
                                 int* status, int sms) {
  return d.out_bf16 ? launch_tc_forward_t<N, L, bf16>(d, a, w, s, status, sms)
                    : launch_tc_forward_t<N, L, float>(d, a, w, s, status, sms);
}

}  // namespace

bool tc_forward_supported(const Dims& d) {
  return d.in_bf16 && d.P == kP && (d.N == 64 || d.N == 128) && (d.L == 128 || d.L == 256) &&
         (d.H / d.G) % 2 == 0;
}

cudaError_t tc_forward(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s) {
  int* status = device_status_ptr();
  if (!status) return cudaErrorUnknown;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (d.N == 128 && d.L == 256) return launch_tc_forward_nl<128, 256>(d, a, w, s, status, sms);
  if (d.N == 128 && d.L == 128) return launch_tc_forward_nl<128, 128>(d, a, w, s, status, sms);
  if (d.N == 64 && d.L == 256) return launch_tc_forward_nl<64, 256>(d, a, w, s, status, sms);
  return launch_tc_forward_nl<64, 128>(d, a, w, s, status, sms);
}

}  // namespace ssd

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
//   D[m = 64 hh + p, n] = sum_l w_hh[l] X[l, h+hh, p] Y[l, n]  ->  out[b, c, h+hh, p, n]
//   MODE 0 (chunk_state): X = x,  Y = B, w = exp(a_last - a_l) delta_l  (S_c)
//   MODE 1 (dstates):     X = dy, Y = C, w = exp(a_l)                   (dHs_c)
// A = (w X)^T as an MN-major operand (rows l, 128 columns = two heads x 64),
// B = the chunk's Y rows as an MN-major operand (rows l, N columns).
template <int N, int L>
struct StateSmem {
  static constexpr int kPanelB = L * 128;        // bytes of one 64-column panel of L rows
  static constexpr int kB = (N / 64) * kPanelB;  // B tile
  static constexpr int kX = 2 * kPanelB;         // w x for a head pair (hi or lo)
  static constexpr int kBytes = kB + 2 * kX + 2 * L * 4 + 1024;
};

template <int N, int L, int MODE>
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
      sw[i] = MODE == 0 ? __expf(acs[cv + L - 1] - acs[cv + l]) * delta[cv + l]
                        : __expf(acs[cv + l]);
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
// One kernel, two directions.
//   forward (REV = false), rows r = l of chunk c, columns s in [0, l0 + 128):
//     CB[l, s] = C_l . B_s                       (TMEM cols 0.., once per CTA)
//     per head: Y  = sum_s P[l, s] x_s,  P = CB e^{a_l - a_s} delta_s [s <= l]
//               ST = C_l . H_c[p, :]
//               y_l = Y + e^{a_l} ST + D x_l
//   backward dx (REV = true), rows r = s, columns l in [s0, L):
//     CBT[s, l] = B_s . C_l
//     per head: Y  = sum_l P[s, l] dy_l,  P = CBT e^{a_l - a_s} [l >= s]
//               ST = B_s . dS_c[p, :]
//               u_s = Y + e^{a_last - a_s} ST;  dx_s = delta_s u_s + D dy_s
//               ddir_s = <x_s, u_s>,  qrow_s = delta_s <x_s, e^{a_last - a_s} ST>
// grid (nc * L/128, B, ceil(H / heads_per_cta)), 256 threads; the heads of a
// CTA belong to one group.
template <int N, int L>
struct ScanSmem {
  static constexpr int kLT = 128;
  static constexpr int kC = (N / 64) * kLT * 128;           // row-operand rows of the tile
  static constexpr int kBrows = (N / 64) * L * 128;         // column-operand rows
  static constexpr int kPbuf = 2 * kLT * 128;               // one P panel, hi + lo
  static constexpr int kBP = kBrows > 2 * kPbuf ? kBrows : 2 * kPbuf;
  static constexpr int kX = L * 128;                        // x or dy rows, one MN panel
  static constexpr int kHhalf = (N / 64) * 64 * 128;        // H or dS (hi or lo), K-major
  static constexpr int kBytes = kC + kBP + kX + 2 * kHhalf + (2 * L + 3 * 128) * 4 + 1024;
};

template <int N, int L, typename Tout, bool REV>
__global__ void __launch_bounds__(256, 1)
    k_scan_tc(const bf16* __restrict__ x, const bf16* __restrict__ Bm,
              const bf16* __restrict__ Cm, const bf16* __restrict__ dy,
              const float* __restrict__ delta, const float* __restrict__ acs,
              const float* __restrict__ state, const float* __restrict__ D,
              Tout* __restrict__ out, float* __restrict__ ddir, float* __restrict__ qrow,
              float* __restrict__ ddiag, int T, int H, int G, int nc, int heads_per_cta,
              int* status) {
  using SM = ScanSmem<N, L>;
  constexpr int LT = SM::kLT, NLT = L / LT;
  constexpr uint32_t kColY = 256, kColST = 320;
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t bar_cb, bar_done, bar_p[2];
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  unsigned char* base = align1024(smem_raw);
  unsigned char* sR = base;               // row operand: C (fwd) or B (rev) rows of the tile
  unsigned char* sBP = sR + SM::kC;       // column operand rows, later the P panels
  unsigned char* sX = sBP + SM::kBP;      // x (fwd) or dy (rev) rows of the columns
  unsigned char* sHh = sX + SM::kX;
  unsigned char* sHl = sHh + SM::kHhalf;
  float* sa = reinterpret_cast<float*>(sHl + SM::kHhalf);
  float* sd = sa + L;
  float* sred = sd + L;                   // [3][128] half-row partial sums (rev)

  const int c = blockIdx.x / NLT, tile = blockIdx.x % NLT, b = blockIdx.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hpg = H / G;
  const int h_begin = blockIdx.z * heads_per_cta;
  const int h_end = min(H, h_begin + heads_per_cta);
  const int g = h_begin / hpg;
  const int r0 = tile * LT;                       // first row (chunk-local)
  const int col0 = REV ? r0 : 0;                  // first column
  const int ncol = REV ? L - r0 : r0 + LT;        // number of columns
  const int nsp = ncol / 64;
  const int64_t t0 = (int64_t)c * L;
  const int Lv = min(L, T - (int)t0);
  const bf16* rowsrc = REV ? Bm : Cm;             // row operand of the score tile
  const bf16* colsrc = REV ? Cm : Bm;             // column operand
  const bf16* opsrc = REV ? dy : x;               // second MMA operand (per head)

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bar_cb, 1);
    mbar_init(&bar_done, 1);
    mbar_init(&bar_p[0], 1);
    mbar_init(&bar_p[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 512);

  constexpr int kRC = N / 8;
  for (int i = tid; i < LT * kRC; i += 256) {
    const int rr = i / kRC, j = i % kRC, row = r0 + rr;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < Lv)
      v = *reinterpret_cast<const uint4*>(rowsrc + ((((int64_t)b * T + t0 + row) * G + g) * N) +
                                          j * 8);
    *reinterpret_cast<uint4*>(sR + (j / 8) * (LT * 128) + sw128(rr, j % 8)) = v;
  }
  for (int i = tid; i < ncol * kRC; i += 256) {
    const int cc = i / kRC, j = i % kRC, col = col0 + cc;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (col < Lv)
      v = *reinterpret_cast<const uint4*>(colsrc + ((((int64_t)b * T + t0 + col) * G + g) * N) +
                                          j * 8);
    *reinterpret_cast<uint4*>(sBP + (j / 8) * (L * 128) + sw128(cc, j % 8)) = v;
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tm = tmem_base;
  if (tid == 0) {
    const uint32_t id = idesc_bf16(128, ncol, 0, 0);
    for (int ks = 0; ks < N / 16; ++ks) {
      const uint32_t kp = ks / 4, ko = (ks % 4) * 32;
      mma_bf16(tm, sdesc(smem_u32(sR) + kp * (LT * 128) + ko, 16, 1024),
               sdesc(smem_u32(sBP) + kp * (L * 128) + ko, 16, 1024), id, ks > 0 ? 1u : 0u);
    }
    mma_commit(&bar_cb);
  }
  mbar_wait(&bar_cb, 0, status, &abort_flag);
  fence_after_sync();

  const int q = warp & 3, half = warp >> 2;
  const int rr = 32 * q + lane, r = r0 + rr;  // this thread's row (TMEM lane)
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
    // second operand rows (columns of the score tile): one MN-major panel
    for (int i = tid; i < ncol * 8; i += 256) {
      const int cc = i >> 3, j = i & 7, col = col0 + cc;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (col < Lv)
        v = *reinterpret_cast<const uint4*>(opsrc + (((int64_t)b * T + t0 + col) * H + h) * kP +
                                            j * 8);
      *reinterpret_cast<uint4*>(sX + sw128(cc, j)) = v;
    }
    // inter-chunk state (H_c forward, dS_c backward), fp32 64 x N -> hi / lo
    const float* Sc = state + (((int64_t)b * nc + c) * H + h) * kP * N;
    for (int i = tid; i < kP * (N / 8); i += 256) {
      const int p = i / (N / 8), j = i % (N / 8);
      const float4 u0 = *reinterpret_cast<const float4*>(Sc + p * N + j * 8);
      const float4 u1 = *reinterpret_cast<const float4*>(Sc + p * N + j * 8 + 4);
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
        const uint64_t ad = sdesc(smem_u32(sR) + kp * (LT * 128) + ko, 16, 1024);
        mma_bf16(tm + kColST, ad, sdesc(smem_u32(sHh) + kp * (64 * 128) + ko, 16, 1024), id_st,
                 ks > 0 ? 1u : 0u);
        mma_bf16(tm + kColST, ad, sdesc(smem_u32(sHl) + kp * (64 * 128) + ko, 16, 1024), id_st,
                 1u);
      }
    }
    const float ar = sa[r];
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
          const int cl = col0 + 64 * j + 32 * half + 8 * k8 + e;  // chunk-local column
          if constexpr (REV)
            v[e] = cl >= r ? cb[8 * k8 + e] * __expf(sa[cl] - ar) : 0.f;
          else
            v[e] = cl <= r ? cb[8 * k8 + e] * __expf(ar - sa[cl]) * sd[cl] : 0.f;
        }
        const uint32_t off = sw128(rr, 4 * half + k8);
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
    float pd = 0.f, pq = 0.f, pdd = 0.f;  // rev: partial <x, u>, <x, state part>, <x, dy>
    if (ok) {
      float yv[32], st[32];
      tmem_ld16(tlane + kColY + 32 * half, *reinterpret_cast<float(*)[16]>(yv));
      tmem_ld16(tlane + kColY + 32 * half + 16, *reinterpret_cast<float(*)[16]>(yv + 16));
      tmem_ld16(tlane + kColST + 32 * half, *reinterpret_cast<float(*)[16]>(st));
      tmem_ld16(tlane + kColST + 32 * half + 16, *reinterpret_cast<float(*)[16]>(st + 16));
      tmem_wait_ld();
      if (r < Lv) {
        const float Dh = D ? D[h] : 0.f;
        const int64_t rowoff = (((int64_t)b * T + t0 + r) * H + h) * kP + 32 * half;
        if constexpr (!REV) {
          const float ea = __expf(ar);
#pragma unroll
          for (int k8 = 0; k8 < 4; ++k8) {
            float xv[8], o[8];
            unpack8(*reinterpret_cast<const uint4*>(sX + sw128(rr + r0 - col0, 4 * half + k8)),
                    xv);
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = yv[8 * k8 + e] + ea * st[8 * k8 + e] + Dh * xv[e];
            if constexpr (sizeof(Tout) == 4) {
              float* of = reinterpret_cast<float*>(out + rowoff) + 8 * k8;
              *reinterpret_cast<float4*>(of) = make_float4(o[0], o[1], o[2], o[3]);
              *reinterpret_cast<float4*>(of + 4) = make_float4(o[4], o[5], o[6], o[7]);
            } else {
              *reinterpret_cast<uint4*>(reinterpret_cast<bf16*>(out + rowoff) + 8 * k8) =
                  make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]),
                             pack_bf16(o[4], o[5]), pack_bf16(o[6], o[7]));
            }
          }
        } else {
          const float es = __expf(sa[L - 1] - ar), dr = sd[r];
#pragma unroll
          for (int k8 = 0; k8 < 4; ++k8) {
            float dyv[8], xv[8], o[8];
            unpack8(*reinterpret_cast<const uint4*>(sX + sw128(rr + r0 - col0, 4 * half + k8)),
                    dyv);
            unpack8(*reinterpret_cast<const uint4*>(x + rowoff + 8 * k8), xv);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
              const float us = es * st[8 * k8 + e];
              const float u = yv[8 * k8 + e] + us;
              o[e] = fmaf(dr, u, Dh * dyv[e]);
              pd = fmaf(xv[e], u, pd);
              pq = fmaf(xv[e], us, pq);
              pdd = fmaf(xv[e], dyv[e], pdd);
            }
            float* of = reinterpret_cast<float*>(out + rowoff) + 8 * k8;
            *reinterpret_cast<float4*>(of) = make_float4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<float4*>(of + 4) = make_float4(o[4], o[5], o[6], o[7]);
          }
        }
      }
    }
    if constexpr (REV) {
      if (half == 1) {
        sred[rr] = pd;
        sred[128 + rr] = pq;
        sred[256 + rr] = pdd;
      }
      __syncthreads();
      if (half == 0 && r < Lv) {
        ddir[cv + r] = pd + sred[rr];
        qrow[cv + r] = sd[r] * (pq + sred[128 + rr]);
        ddiag[cv + r] = pdd + sred[256 + rr];
      }
    }
    fence_before_sync();
    __syncthreads();
  }
  if (warp == 0) tmem_dealloc(tm, 512);
}

// ================================================================ dB and dC
// grid (nc * L/128, B, G * nblk), 256 threads.  CTA = a 128-row tile of chunk
// c and one block of hb consecutive heads of group g (blockIdx.z = g*nblk + k);
// its accumulator sums the block's heads, so out holds one partial per block.
// REV = false -> dC (rows l, columns s in [0, l0 + 128)):
//   per head and 128-column panel: S0 = C_l . B_s (K = N), S1 = dy_l . x_s (K = P)
//     P2[l,s] = e^{a_l - a_s} delta_s S1 [s <= l];  ACC += P2 . B  (K = s)
//     msum_l += sum_{s < l} S0 P2
//   then ACC += (e^{a_l} dy_l) . H_c (K = p);  ST = C_l . H_c^T (K = n)
//     ycs_l = e^{a_l} <dy_l, ST_l>
// REV = true -> dB (rows s, columns l in [s0, L)):
//   S0 = B_s . C_l, S1 = x_s . dy_l
//     P2[s,l] = e^{a_l - a_s} delta_s S1 [l >= s];  ACC += P2 . C  (K = l)
//     msum_s += sum_{l > s} S0 P2
//   then ACC += (delta_s e^{a_last - a_s} x_s) . dS_c (K = p)
// msum holds the strict row (dC) or column (dB) sums of
// M[l,s] = C_l.B_s e^{a_l - a_s} delta_s <dy_l, x_s> for the ddA gradient.
template <int N, int L>
struct BcSmem {
  static constexpr int kLT = 128;
  static constexpr int kGR = (N / 64) * kLT * 128;
  static constexpr int kGC = (N / 64) * L * 128;
  static constexpr int kHR = kLT * 128;
  static constexpr int kHC = L * 128;
  static constexpr int kPP = 4 * kLT * 128;  // P2 panel (2 x 64 columns, hi + lo); state operands later
  static constexpr int kBytes = kGR + kGC + kHR + kHC + kPP + (2 * L + 4 * 128) * 4 + 1024;
};

template <int N, int L, bool REV>
__global__ void __launch_bounds__(256, 1)
    k_bwd_bc_tc(const bf16* __restrict__ x, const bf16* __restrict__ Bm,
                const bf16* __restrict__ Cm, const bf16* __restrict__ dy,
                const float* __restrict__ delta, const float* __restrict__ acs,
                const float* __restrict__ state, float* __restrict__ out,
                float* __restrict__ msum, float* __restrict__ ycs, int T, int H, int G, int nc,
                int hb, int* status) {
  using SM = BcSmem<N, L>;
  constexpr int LT = SM::kLT, NLT = L / LT, NKP = N / 64;
  constexpr uint32_t kColS0 = 0, kColS1 = 128, kColAcc = 256, kColST = 384;
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t bar_s, bar_acc, bar_st;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  unsigned char* base = align1024(smem_raw);
  unsigned char* sGR = base;
  unsigned char* sGC = sGR + SM::kGR;
  unsigned char* sHR = sGC + SM::kGC;
  unsigned char* sHC = sHR + SM::kHR;
  unsigned char* sP = sHC + SM::kHC;
  float* sa = reinterpret_cast<float*>(sP + SM::kPP);
  float* sd = sa + L;
  float* sred = sd + L;  // [4][128]

  const int c = blockIdx.x / NLT, tile = blockIdx.x % NLT, b = blockIdx.y;
  const int nblk = gridDim.z / G, g = blockIdx.z / nblk, kb = blockIdx.z % nblk;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h_begin = g * (H / G) + kb * hb, h_end = h_begin + hb;
  const int r0 = tile * LT, col0 = REV ? r0 : 0, ncol = REV ? L - r0 : r0 + LT;
  const int npan = ncol / 128;
  const int64_t t0 = (int64_t)c * L;
  const int Lv = min(L, T - (int)t0);
  const bf16* grow = REV ? Bm : Cm;
  const bf16* gcol = REV ? Cm : Bm;
  const bf16* hrow = REV ? x : dy;
  const bf16* hcol = REV ? dy : x;

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bar_s, 1);
    mbar_init(&bar_acc, 1);
    mbar_init(&bar_st, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 512);
  constexpr int kRC = N / 8;
  for (int i = tid; i < LT * kRC; i += 256) {
    const int rr = i / kRC, j = i % kRC, row = r0 + rr;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (row < Lv)
      v = *reinterpret_cast<const uint4*>(grow + ((((int64_t)b * T + t0 + row) * G + g) * N) +
                                          j * 8);
    *reinterpret_cast<uint4*>(sGR + (j / 8) * (LT * 128) + sw128(rr, j % 8)) = v;
  }
  for (int i = tid; i < ncol * kRC; i += 256) {
    const int cc = i / kRC, j = i % kRC, col = col0 + cc;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (col < Lv)
      v = *reinterpret_cast<const uint4*>(gcol + ((((int64_t)b * T + t0 + col) * G + g) * N) +
                                          j * 8);
    *reinterpret_cast<uint4*>(sGC + (j / 8) * (L * 128) + sw128(cc, j % 8)) = v;
  }
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tm = tmem_base;
  const int q = warp & 3, half = warp >> 2;
  const int rr = 32 * q + lane, r = r0 + rr;
  const uint32_t tlane = tm + ((uint32_t)(32 * q) << 16);
  uint32_t n_s = 0, n_acc = 0, n_st = 0;
  bool acc_started = false;  // meaningful in thread 0 only
  constexpr uint32_t id_sc0 = idesc_bf16(128, 128, 0, 0);
  constexpr uint32_t id_acc = idesc_bf16(128, N, 0, 1);
  constexpr uint32_t id_st = idesc_bf16(128, kP, 0, 0);
  unsigned char* sAh = sP;                      // state A operand hi / lo (128 x 64)
  unsigned char* sAl = sP + LT * 128;
  unsigned char* sBh = sP + 2 * LT * 128;       // state B operand hi / lo (64 x N)
  unsigned char* sBl = sBh + NKP * 64 * 128;

  for (int h = h_begin; h < h_end; ++h) {
    const int64_t cv = (((int64_t)b * H + h) * nc + c) * L;
    for (int i = tid; i < L; i += 256) {
      sa[i] = acs[cv + i];
      sd[i] = delta[cv + i];
    }
    for (int i = tid; i < LT * 8; i += 256) {
      const int r2 = i >> 3, j = i & 7, row = r0 + r2;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (row < Lv)
        v = *reinterpret_cast<const uint4*>(hrow + (((int64_t)b * T + t0 + row) * H + h) * kP +
                                            j * 8);
      *reinterpret_cast<uint4*>(sHR + sw128(r2, j)) = v;
    }
    for (int i = tid; i < ncol * 8; i += 256) {
      const int cc = i >> 3, j = i & 7, col = col0 + cc;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (col < Lv)
        v = *reinterpret_cast<const uint4*>(hcol + (((int64_t)b * T + t0 + col) * H + h) * kP +
                                            j * 8);
      *reinterpret_cast<uint4*>(sHC + sw128(cc, j)) = v;
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    const float ar = sa[r], dr = sd[r];
    float mpart = 0.f;
    for (int k = 0; k < npan; ++k) {
      if (tid == 0) {
        fence_after_sync();
        for (int ks = 0; ks < N / 16; ++ks) {
          const uint32_t kp = ks / 4, ko = (ks % 4) * 32;
          mma_bf16(tm + kColS0, sdesc(smem_u32(sGR) + kp * (LT * 128) + ko, 16, 1024),
                   sdesc(smem_u32(sGC) + kp * (L * 128) + k * 128 * 128 + ko, 16, 1024), id_sc0,
                   ks > 0 ? 1u : 0u);
        }
        for (int ks = 0; ks < 4; ++ks)
          mma_bf16(tm + kColS1, sdesc(smem_u32(sHR) + ks * 32, 16, 1024),
                   sdesc(smem_u32(sHC) + k * 128 * 128 + ks * 32, 16, 1024), id_sc0,
                   ks > 0 ? 1u : 0u);
        mma_commit(&bar_s);
      }
      ++n_s;
      mbar_wait(&bar_s, (n_s - 1) & 1, status, &abort_flag);
      if (n_acc > 0) mbar_wait(&bar_acc, (n_acc - 1) & 1, status, &abort_flag);
      fence_after_sync();
#pragma unroll
      for (int g32 = 0; g32 < 2; ++g32) {
        float s0[32], s1[32];
        const uint32_t cb = 64 * half + 32 * g32;
        tmem_ld16(tlane + kColS0 + cb, *reinterpret_cast<float(*)[16]>(s0));
        tmem_ld16(tlane + kColS0 + cb + 16, *reinterpret_cast<float(*)[16]>(s0 + 16));
        tmem_ld16(tlane + kColS1 + cb, *reinterpret_cast<float(*)[16]>(s1));
        tmem_ld16(tlane + kColS1 + cb + 16, *reinterpret_cast<float(*)[16]>(s1 + 16));
        tmem_wait_ld();
#pragma unroll
        for (int k8 = 0; k8 < 4; ++k8) {
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int cl = col0 + 128 * k + cb + 8 * k8 + e;  // chunk-local column
            float p2;
            bool strict;
            if constexpr (REV) {
              p2 = cl >= r ? __expf(sa[cl] - ar) * dr * s1[8 * k8 + e] : 0.f;
              strict = cl > r;
            } else {
              p2 = cl <= r ? __expf(ar - sa[cl]) * sd[cl] * s1[8 * k8 + e] : 0.f;
              strict = cl < r;
            }
            if (strict) mpart = fmaf(s0[8 * k8 + e], p2, mpart);
            v[e] = p2;
          }
          const uint32_t off = half * (LT * 128) + sw128(rr, 4 * g32 + k8);
          store_split8(sP + off, sP + 2 * LT * 128 + off, v);
        }
      }
      fence_async_smem();
      fence_before_sync();
      __syncthreads();
      if (tid == 0) {
        fence_after_sync();
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t sub = ks / 4, ko = (ks % 4) * 32;
          const uint64_t bd = sdesc(smem_u32(sGC) + (k * 128 + ks * 16) * 128, L * 128, 1024);
          mma_bf16(tm + kColAcc, sdesc(smem_u32(sP) + sub * (LT * 128) + ko, 16, 1024), bd, id_acc,
                   acc_started ? 1u : 0u);
          acc_started = true;
          mma_bf16(tm + kColAcc,
                   sdesc(smem_u32(sP) + 2 * LT * 128 + sub * (LT * 128) + ko, 16, 1024), bd,
                   id_acc, 1u);
        }
        mma_commit(&bar_acc);
      }
      ++n_acc;
    }
    // state term of this head
    mbar_wait(&bar_acc, (n_acc - 1) & 1, status, &abort_flag);
    for (int i = tid; i < LT * 8; i += 256) {
      const int r2 = i >> 3, j = i & 7, row = r0 + r2;
      float v[8];
      unpack8(*reinterpret_cast<const uint4*>(sHR + sw128(r2, j)), v);
      const float sc = REV ? sd[row] * __expf(sa[L - 1] - sa[row]) : __expf(sa[row]);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[e] *= sc;
      store_split8(sAh + sw128(r2, j), sAl + sw128(r2, j), v);
    }
    const float* Sc = state + (((int64_t)b * nc + c) * H + h) * kP * N;
    for (int i = tid; i < kP * (N / 8); i += 256) {
      const int p = i / (N / 8), j = i % (N / 8);
      const float4 u0 = *reinterpret_cast<const float4*>(Sc + p * N + j * 8);
      const float4 u1 = *reinterpret_cast<const float4*>(Sc + p * N + j * 8 + 4);
      const float v[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
      const uint32_t off = (j / 8) * (64 * 128) + sw128(p, j % 8);
      store_split8(sBh + off, sBl + off, v);
    }
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    if (tid == 0) {
      fence_after_sync();
      for (int ks = 0; ks < 4; ++ks) {
        const uint64_t ah = sdesc(smem_u32(sAh) + ks * 32, 16, 1024);
        const uint64_t al = sdesc(smem_u32(sAl) + ks * 32, 16, 1024);
        const uint64_t bh = sdesc(smem_u32(sBh) + ks * 2048, 64 * 128, 1024);
        const uint64_t bl = sdesc(smem_u32(sBl) + ks * 2048, 64 * 128, 1024);
        mma_bf16(tm + kColAcc, ah, bh, id_acc, 1u);
        mma_bf16(tm + kColAcc, ah, bl, id_acc, 1u);
        mma_bf16(tm + kColAcc, al, bh, id_acc, 1u);
      }
      if constexpr (!REV) {
        for (int ks = 0; ks < N / 16; ++ks) {
          const uint32_t kp = ks / 4, ko = (ks % 4) * 32;
          const uint64_t ad = sdesc(smem_u32(sGR) + kp * (LT * 128) + ko, 16, 1024);
          mma_bf16(tm + kColST, ad, sdesc(smem_u32(sBh) + kp * (64 * 128) + ko, 16, 1024), id_st,
                   ks > 0 ? 1u : 0u);
          mma_bf16(tm + kColST, ad, sdesc(smem_u32(sBl) + kp * (64 * 128) + ko, 16, 1024), id_st,
                   1u);
        }
      }
      mma_commit(&bar_st);
    }
    ++n_st;
    const bool ok = mbar_wait(&bar_st, (n_st - 1) & 1, status, &abort_flag);
    fence_after_sync();
    float ypart = 0.f;
    if constexpr (!REV) {
      if (ok) {
        float st[32];
        tmem_ld16(tlane + kColST + 32 * half, *reinterpret_cast<float(*)[16]>(st));
        tmem_ld16(tlane + kColST + 32 * half + 16, *reinterpret_cast<float(*)[16]>(st + 16));
        tmem_wait_ld();
#pragma unroll
        for (int k8 = 0; k8 < 4; ++k8) {
          float dv[8];
          unpack8(*reinterpret_cast<const uint4*>(sHR + sw128(rr, 4 * half + k8)), dv);
#pragma unroll
          for (int e = 0; e < 8; ++e) ypart = fmaf(dv[e], st[8 * k8 + e], ypart);
        }
        ypart *= __expf(ar);
      }
    }
    if (half == 1) {
      sred[rr] = mpart;
      sred[128 + rr] = ypart;
    }
    __syncthreads();
    if (half == 0 && r < Lv) {
      msum[cv + r] = mpart + sred[rr];
      if constexpr (!REV) ycs[cv + r] = ypart + sred[128 + rr];
    }
    fence_before_sync();
    __syncthreads();
  }
  // the block's accumulated dB / dC rows
  if (!abort_flag) {  // CTA-uniform: the TMEM loads below are warp-collective
    float* o = out + (((((int64_t)b * T + t0 + r) * G + g) * nblk + kb) * N) + half * (N / 2);
#pragma unroll
    for (int c0 = 0; c0 < N / 2; c0 += 16) {
      float v[16];
      tmem_ld16(tlane + kColAcc + half * (N / 2) + c0, v);
      tmem_wait_ld();
      if (r < Lv) {
#pragma unroll
        for (int k4 = 0; k4 < 16; k4 += 4)
          *reinterpret_cast<float4*>(o + c0 + k4) =
              make_float4(v[k4], v[k4 + 1], v[k4 + 2], v[k4 + 3]);
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, 512);
}

// grid (nc, H, B).  Gradient w.r.t. dA_r = delta_r A from the strict row sums
// (dC kernel) and column sums (dB kernel) of M:
//   ddA_r = sum_{j<r} (colsum_j - rowsum_j) + sum_{l>=r} ycs_l + sum_{s<r} qrow_s + dlast_c
//   ddt_r = (ddir_r + A ddA_r) softplus'(dt_r + dt_bias);  partials of dA, ddt_bias, dD.
__global__ void __launch_bounds__(256)
    k_bwd_finalize_tc(const bf16* __restrict__ dt, const float* __restrict__ dt_bias,
                      const float* __restrict__ A, const float* __restrict__ delta,
                      const float* __restrict__ rowsum, const float* __restrict__ colsum,
                      const float* __restrict__ ycs, const float* __restrict__ qrow,
                      const float* __restrict__ ddir, const float* __restrict__ ddiag,
                      const float* __restrict__ dlast, int nsplit, float* __restrict__ ddt,
                      float* __restrict__ part, int T, int H, int L, int nc) {
  __shared__ float sdd[256], red[8];
  const int c = blockIdx.x, h = blockIdx.y, b = blockIdx.z, tid = threadIdx.x;
  const int Lv = min(L, T - c * L);
  const int64_t cv = (((int64_t)b * H + h) * nc + c) * L;
  if (tid == 0) {
    float dl = 0.f;
    for (int k = 0; k < nsplit; ++k) dl += dlast[(((int64_t)b * H + h) * nc + c) * nsplit + k];
    float pre = 0.f;
    for (int r = 0; r < Lv; ++r) {
      sdd[r] = pre + dl;
      pre += colsum[cv + r] - rowsum[cv + r] + qrow[cv + r];
    }
    float suf = 0.f;
    for (int r = Lv - 1; r >= 0; --r) {
      suf += ycs[cv + r];
      sdd[r] += suf;
    }
  }
  __syncthreads();
  const float Ah = A[h], bias = dt_bias ? dt_bias[h] : 0.f;
  float pA = 0.f, pB = 0.f, pD = 0.f;
  for (int r = tid; r < Lv; r += 256) {
    const int64_t ti = ((int64_t)b * T + (int64_t)c * L + r) * H + h;
    const float v = __bfloat162float(dt[ti]) + bias;
    const float sg = v > 20.f ? 1.f : 1.f / (1.f + __expf(-v));
    const float gv = fmaf(Ah, sdd[r], ddir[cv + r]) * sg;
    ddt[ti] = gv;
    pA = fmaf(delta[cv + r], sdd[r], pA);
    pB += gv;
    pD += ddiag[cv + r];
  }
  float vals[3] = {pA, pB, pD};
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    float v = vals[k];
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    __syncthreads();
    if ((tid & 31) == 0) red[tid >> 5] = v;
    __syncthreads();
    if (tid == 0) {
      float t = 0.f;
      for (int i = 0; i < 8; ++i) t += red[i];
      part[(((int64_t)b * H + h) * nc + c) * 3 + k] = t;
    }
  }
}

// out[i, :] = sum_k in[i, k, :] over the nblk head-block partials, in order.
__global__ void k_block_reduce(const float* __restrict__ in, float* __restrict__ out,
                               int64_t rows, int nblk, int N) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows * N) return;
  const int64_t row = i / N;
  const int n = (int)(i % N);
  float s = 0.f;
  for (int k = 0; k < nblk; ++k) s += in[(row * nblk + k) * N + n];
  out[i] = s;
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
    auto kern = k_state_tc<N, L, 0>;
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
    auto kern = k_scan_tc<N, L, Tout, false>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
    const int hpc = pick_heads_per_cta(d.H / d.G, d.B * d.nc * (L / 128) * d.G, sms, 4);
    const dim3 grid(d.nc * (L / 128), d.B, (d.H + hpc - 1) / hpc);
    SSD_LAUNCH("k_scan_tc", s,
               kern<<<grid, 256, SM::kBytes, s>>>(
                   static_cast<const bf16*>(a.x), static_cast<const bf16*>(a.B),
                   static_cast<const bf16*>(a.C), nullptr, w.delta, w.acs, w.Hprev, a.D,
                   static_cast<Tout*>(a.y), nullptr, nullptr, nullptr, d.T, d.H, d.G, d.nc, hpc,
                   status));
  }
  return cudaGetLastError();
}

template <int N, int L>
cudaError_t launch_tc_forward_nl(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s,
                                 int* status, int sms) {
  return d.out_bf16 ? launch_tc_forward_t<N, L, bf16>(d, a, w, s, status, sms)
                    : launch_tc_forward_t<N, L, float>(d, a, w, s, status, sms);
}

template <int N, int L>
cudaError_t launch_tc_backward_nl(const Dims& d, const BwdArgs& a, const TcBwdWs& w,
                                  cudaStream_t s, int* status, int sms) {
  const bf16* x = static_cast<const bf16*>(a.f.x);
  const bf16* Bm = static_cast<const bf16*>(a.f.B);
  const bf16* Cm = static_cast<const bf16*>(a.f.C);
  const bf16* dy = static_cast<const bf16*>(a.dy);
  FwdArgs f = a.f;
  f.final_state = nullptr;
  FwdWs fw{w.delta, w.acs, w.S, w.Hprev, nullptr};
  simt_cumsum(d, f, fw, s);
  using SS = StateSmem<N, L>;
  const int ppc = pick_heads_per_cta((d.H / d.G) / 2, d.B * d.nc * d.G, sms, 4);
  const dim3 sgrid(d.nc, d.B, (d.H / 2 + ppc - 1) / ppc);
  {
    auto kern = k_state_tc<N, L, 0>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SS::kBytes);
    SSD_LAUNCH("k_state_tc", s, kern<<<sgrid, 256, SS::kBytes, s>>>(
        x, Bm, w.delta, w.acs, w.S, d.T, d.H, d.G, d.nc, ppc, status));
  }
  simt_state_passing(d, f, fw, s);
  {
    auto kern = k_state_tc<N, L, 1>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SS::kBytes);
    SSD_LAUNCH("k_dstates_tc", s, kern<<<sgrid, 256, SS::kBytes, s>>>(
        dy, Cm, w.delta, w.acs, w.dHs, d.T, d.H, d.G, d.nc, ppc, status));
  }
  const int nsplit = simt_state_passing_bwd(d, w.dHs, w.acs, w.Hprev, a.dfinal, w.dS, w.dlast,
                                            a.dinit, s);
  {
    using SM = ScanSmem<N, L>;
    auto kern = k_scan_tc<N, L, float, true>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
    const int hpc = pick_heads_per_cta(d.H / d.G, d.B * d.nc * (L / 128) * d.G, sms, 4);
    const dim3 grid(d.nc * (L / 128), d.B, (d.H + hpc - 1) / hpc);
    SSD_LAUNCH("k_scan_tc_dx", s, kern<<<grid, 256, SM::kBytes, s>>>(
        x, Bm, Cm, dy, w.delta, w.acs, w.dS, a.f.D, a.dx, w.ddir, w.qrow, w.ddiag, d.T, d.H,
        d.G, d.nc, hpc, status));
  }
  const int nblk = tc_bwd_nblk(d), hb = (d.H / d.G) / nblk;
  const dim3 bgrid(d.nc * (L / 128), d.B, d.G * nblk);
  float* dCout = nblk == 1 ? a.dC : w.dCp;
  float* dBout = nblk == 1 ? a.dB : w.dBp;
  {
    using SM = BcSmem<N, L>;
    auto kern = k_bwd_bc_tc<N, L, false>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
    SSD_LAUNCH("k_bwd_dc_tc", s, kern<<<bgrid, 256, SM::kBytes, s>>>(
        x, Bm, Cm, dy, w.delta, w.acs, w.Hprev, dCout, w.rowsum, w.ycs, d.T, d.H, d.G, d.nc, hb,
        status));
  }
  {
    using SM = BcSmem<N, L>;
    auto kern = k_bwd_bc_tc<N, L, true>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
    SSD_LAUNCH("k_bwd_db_tc", s, kern<<<bgrid, 256, SM::kBytes, s>>>(
        x, Bm, Cm, dy, w.delta, w.acs, w.dS, dBout, w.colsum, nullptr, d.T, d.H, d.G, d.nc, hb,
        status));
  }
  SSD_LAUNCH("k_bwd_finalize_tc", s, k_bwd_finalize_tc<<<dim3(d.nc, d.H, d.B), 256, 0, s>>>(
      static_cast<const bf16*>(a.f.dt), a.f.dt_bias, a.f.A, w.delta, w.rowsum, w.colsum, w.ycs,
      w.qrow, w.ddir, w.ddiag, w.dlast, nsplit, a.ddt, w.part, d.T, d.H, d.L, d.nc));
  if (nblk > 1) {
    const int64_t rows = (int64_t)d.B * d.T * d.G;
    const int blocks = (int)((rows * d.N + 255) / 256);
    SSD_LAUNCH("k_block_reduce", s, k_block_reduce<<<blocks, 256, 0, s>>>(w.dCp, a.dC, rows, nblk, d.N));
    SSD_LAUNCH("k_block_reduce", s, k_block_reduce<<<blocks, 256, 0, s>>>(w.dBp, a.dB, rows, nblk, d.N));
  }
  simt_param_grads(d, w.part, a.dA, a.ddt_bias, a.dD, s);
  return cudaGetLastError();
}

}  // namespace

bool tc_forward_supported(const Dims& d) {
  return d.in_bf16 && d.P == kP && (d.N == 64 || d.N == 128) && (d.L == 128 || d.L == 256) &&
         (d.H / d.G) % 2 == 0;
}

int tc_bwd_nblk(const Dims& d) {
  // fewest head blocks per group that still give >= 2 x 152 CTAs
  const int hpg = d.H / d.G;
  const int64_t units = (int64_t)d.B * d.nc * (d.L / 128) * d.G;
  for (int nb = 1; nb <= hpg; ++nb)
    if (hpg % nb == 0 && units * nb >= 2 * 152) return nb;
  return hpg;
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

cudaError_t tc_backward(const Dims& d, const BwdArgs& a, const TcBwdWs& w, cudaStream_t s) {
  int* status = device_status_ptr();
  if (!status) return cudaErrorUnknown;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (d.N == 128 && d.L == 256) return launch_tc_backward_nl<128, 256>(d, a, w, s, status, sms);
  if (d.N == 128 && d.L == 128) return launch_tc_backward_nl<128, 128>(d, a, w, s, status, sms);
  if (d.N == 64 && d.L == 256) return launch_tc_backward_nl<64, 256>(d, a, w, s, status, sms);
  return launch_tc_backward_nl<64, 128>(d, a, w, s, status, sms);
}

}  // namespace ssd

// chunk_state and dstates on the tensor cores, fed by TMA (sm_103a), with
// chunk_cumsum inside chunk_state ("Optimizing Mamba-2 kernels for the B200",
// Stage 1 kernel table: _chunk_state_fwd fwd_2 / bwd_5 and
// _chunk_scan_bwd_dstates bwd_8):
//
//   MODE 0  S_c[h, p, n]   = sum_l e^{a_last - a_l} delta_l x[l, h, p] B[l, n]
//           with delta = softplus(dt + dt_bias) and a = the in-chunk inclusive
//           cumsum of delta A, both also written for the later kernels
//   MODE 1  dHs_c[h, p, n] = sum_l e^{a_l} dy[l, h, p] C[l, n]
//
// An item is (batch, chunk, two heads h, h + 1 of one group).  Its product is
//   D[m = 64 hh + p, n] = sum_l A[m, l] Y[l, n],  A = (w X)^T,  Y = B or C,
// one M = 128 accumulator per item (the pair's two heads), N = d_state, K =
// the chunk's rows in blocks of 64.
//
// Warp roles (704 threads, one persistent CTA per SM over items k =
// blockIdx.x, blockIdx.x + gridDim.x, ...; head pair fastest, so the CTAs
// running side by side share a chunk's Y rows in L2):
//   warps 0-15  convert: per block the TMA-landed x (dy) rows times the
//               item's weights w, split into bf16 hi + lo, stored as the A
//               operand in tensor memory (lane m = 64 hh + p, two bf16 of
//               consecutive l per column), so A costs shared memory neither
//               a write nor the tensor core's read;
//   warps 16-19 epilogue: TMEM accumulator -> shared-memory slabs -> TMA
//               stores of the item's two 64 x N states; between items they
//               also form the weights two items ahead (chunk_cumsum in MODE
//               0), off the converters' path;
//   warp 20     issues every tcgen05.mma (hi and lo A against the same Y);
//   warp 21     issues every TMA copy (x / dy pair boxes, Y panels).
// Rings: four raw-x stages, three Y stages, two TMEM A stages and two TMEM
// accumulators, each handed over by full / empty mbarriers; every wait is
// bounded and records SSD_ERR_TIMEOUT on expiry.
//
// Precision: w X is formed in fp32 and both bf16 parts are multiplied (about
// 16 significant bits instead of bf16's 8); Y enters as stored; the products
// accumulate in fp32 in TMEM.
#include <cuda.h>

#include "ssd_internal.h"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

using namespace tc;
using bf16 = __nv_bfloat16;

constexpr int kSP = 64;         // headdim
constexpr int kKB = 64;         // rows of l per block
constexpr int kNX = 4;          // raw x stages
constexpr int kNY = 3;          // Y stages
constexpr int kNA = 2;          // A operand stages
constexpr int kConvW = 16;      // converter warps
constexpr int kEpiW = 4;        // epilogue warps (one per TMEM lane quarter)
constexpr int kEpi0 = kConvW;   // first epilogue warp
constexpr int kMmaW = kConvW + kEpiW;
constexpr int kProdW = kMmaW + 1;
constexpr int kStateThreads = 32 * (kProdW + 1);
constexpr int kConvT = 32 * kConvW;
constexpr int kEpiT = 32 * kEpiW;

template <int N, int L>
struct StateLayout {
  static constexpr int kX = kKB * 2 * 128;           // a block's x rows of the pair
  static constexpr int kYPanel = kKB * 128;          // 64 of Y's columns
  static constexpr int kY = (N / 64) * kYPanel;      // a block's Y rows
  static constexpr int oX = 0;
  static constexpr int oY = oX + kNX * kX;
  static constexpr int oW = oY + kNY * kY;            // [2 items][2 heads][L] weights
  static constexpr int kStg = (N / 32) * 32 * 128;     // per epilogue warp: an item's 32 x N rows
  static constexpr int oStg = (oW + 2 * 2 * L * 4 + 1023) / 1024 * 1024;
  static constexpr int kBytes = oStg + kEpiW * kStg + 1024;
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
  static_assert(kX % 1024 == 0 && kY % 1024 == 0, "1024-byte stages");
  // TMEM: two N-column accumulators, then two 64-column A stages (a block's
  // 64 values of l as hi / lo bf16 per 16-wide K group)
  static constexpr uint32_t kColA = 2 * N;
  static constexpr uint32_t kTmemCols = 2 * N + 2 * 64 > 256 ? 512 : 256;
};

__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                          ~uintptr_t(1023));
}

__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiT) : "memory");
}

// 16 fp32 values of this thread's TMEM lane -> one 16-wide K group of an A
// operand in tensor memory: hi = rn_bf16(v) packed two per column in
// [col, col + 8), lo = rn_bf16(v - hi) in [col + 8, col + 16).
// Warp-collective.
__device__ __forceinline__ void tmem_store_split16(uint32_t col, const float (&v)[16]) {
  uint32_t h[8], l[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) split2_bf16(v[2 * e], v[2 * e + 1], h[e], l[e]);
  tmem_st8u(col, h);
  tmem_st8u(col + 8, l);
}

__device__ __forceinline__ void warp_arrive(uint64_t* bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

struct StateArgs {
  const bf16* dt;        // MODE 0: (B, T, H)
  const float* dt_bias;  // MODE 0: (H) or null
  const float* A;        // MODE 0: (H)
  float* delta;          // MODE 0 writes (B, H, nc, L)
  float* acs;            // MODE 0 writes, MODE 1 reads (B, H, nc, L)
  float* out;            // (B, nc, H, P, N)
  int T, H, G, nc, n_items;
  int hs;  // log2 of the 64-wide parts per head: dt, dt_bias, A, delta, a index (b, h) >> hs
  int* status;
  int* zero;  // MODE 0: a word set to 0 before anything after this kernel reads it, or null
};

template <int N, int L, int MODE>
__global__ void __launch_bounds__(kStateThreads, 1)
    k_state_tc(const __grid_constant__ CUtensorMap mX, const __grid_constant__ CUtensorMap mY,
               const __grid_constant__ CUtensorMap mOut, const StateArgs a) {
  using LY = StateLayout<N, L>;
  constexpr int NKB = L / kKB, NP = N / 64;
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t bar_xf[kNX], bar_xe[kNX], bar_yf[kNY], bar_ye[kNY], bar_af[kNA],
      bar_ae[kNA], bar_accf[2], bar_acce[2], bar_wf[2], bar_final;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  __shared__ float s_scan[kEpiW], s_alast[2];
  unsigned char* base = align1024(smem_raw);
  float* sw = reinterpret_cast<float*>(base + LY::oW);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int H = a.H, T = a.T, nc = a.nc, hpg = H / a.G, npairs = H / 2;
  int* status = a.status;
  const int nk = (int)blockIdx.x < a.n_items
                     ? (a.n_items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x
                     : 0;
  // item k of this CTA -> batch, chunk, first head of the pair
  auto decode = [&](int k, int& b, int& c, int& h) {
    const int item = (int)blockIdx.x + k * (int)gridDim.x;
    const int pp = item % npairs, bc = item / npairs;
    c = bc % nc;
    b = bc / nc;
    h = 2 * pp;
  };

  if (tid == 0) {
    abort_flag = 0;
    for (int i = 0; i < kNX; ++i) {
      mbar_init(&bar_xf[i], 1);
      mbar_init(&bar_xe[i], kConvW);
    }
    for (int i = 0; i < kNY; ++i) {
      mbar_init(&bar_yf[i], 1);
      mbar_init(&bar_ye[i], 1);
    }
    for (int i = 0; i < kNA; ++i) {
      mbar_init(&bar_af[i], kConvW);
      mbar_init(&bar_ae[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_accf[i], 1);
      mbar_init(&bar_acce[i], kEpiW);
      mbar_init(&bar_wf[i], kEpiW);
    }
    mbar_init(&bar_final, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, LY::kTmemCols);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  // the next kernel may start once every CTA of this one holds its TMEM: a
  // dependent CTA that allocates TMEM on the same SM then only waits for CTAs
  // that need nothing from it
  griddep_launch_dependents();
  if (MODE == 0 && a.zero && blockIdx.x == 0 && tid == 0) *a.zero = 0;
  const uint32_t tm = tmem_base;

  if (warp == kProdW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&mX);
      tma_prefetch_map(&mY);
      bool ok = true;
      uint32_t n_x[kNX] = {}, n_y[kNY] = {};  // phases armed per stage
      for (int k = 0; ok && k < nk; ++k) {
        int b, c, h;
        decode(k, b, c, h);
        const int g = h / hpg, t0 = c * L;
        for (int kb = 0; kb < NKB; ++kb) {
          const int u = k * NKB + kb;
          const int sx = u % kNX, sy = u % kNY;
          if (u >= kNX && !mbar_wait(&bar_xe[sx], ((u / kNX) - 1) & 1, status, &abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bar_xf[sx], LY::kX);
          ++n_x[sx];
          tma_load_4d(base + LY::oX + sx * LY::kX, &mX, 0, h, t0 + kb * kKB, b, &bar_xf[sx]);
          if (u >= kNY && !mbar_wait(&bar_ye[sy], ((u / kNY) - 1) & 1, status, &abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bar_yf[sy], LY::kY);
          ++n_y[sy];
          for (int kp = 0; kp < NP; ++kp)
            tma_load_4d(base + LY::oY + sy * LY::kY + kp * LY::kYPanel, &mY, 64 * kp, g,
                        t0 + kb * kKB, b, &bar_yf[sy]);
        }
      }
      // copies still in flight (after an expired wait) land before the CTA
      // exits: wait for the last phase each stage was armed for
      for (int s = 0; s < kNX; ++s)
        if (n_x[s] > 0) mbar_drain(&bar_xf[s], (n_x[s] - 1) & 1);
      for (int s = 0; s < kNY; ++s)
        if (n_y[s] > 0) mbar_drain(&bar_yf[s], (n_y[s] - 1) & 1);
    }
  } else if (warp == kMmaW) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16(128, N, 0, 1);  // A in TMEM, B MN-major
      const uint64_t dY0 = sdesc(smem_u32(base + LY::oY), LY::kYPanel, 1024);
      bool ok = true;
      for (int k = 0; ok && k < nk; ++k) {
        const int buf = k & 1;
        if (k >= 2 && !mbar_wait(&bar_acce[buf], ((k >> 1) - 1) & 1, status, &abort_flag)) break;
        fence_after_sync();
        for (int kb = 0; kb < NKB; ++kb) {
          const int u = k * NKB + kb;
          const int sa = u % kNA, sy = u % kNY;
          if (!mbar_wait(&bar_af[sa], (u / kNA) & 1, status, &abort_flag) ||
              !mbar_wait(&bar_yf[sy], (u / kNY) & 1, status, &abort_flag)) {
            ok = false;
            break;
          }
          fence_after_sync();
          const uint32_t at = tm + LY::kColA + 64 * sa;
          const uint64_t yd = desc_add(dY0, sy * LY::kY);
#pragma unroll
          for (int ks = 0; ks < kKB / 16; ++ks) {
            mma_bf16_ta(tm + buf * N, at + 16 * ks, desc_add(yd, ks * 2048), idesc,
                        (kb > 0 || ks > 0) ? 1u : 0u);
            mma_bf16_ta(tm + buf * N, at + 16 * ks + 8, desc_add(yd, ks * 2048), idesc, 1u);
          }
          mma_commit(&bar_ae[sa]);
          mma_commit(&bar_ye[sy]);
        }
        if (ok) mma_commit(&bar_accf[buf]);
      }
      // every product issued has completed before TMEM is released
      mma_commit(&bar_final);
      mbar_drain(&bar_final, 0);
    }
  } else if (warp >= kEpi0) {
    // ------------------------------------------------------------ epilogue
    // Each warp owns 32 accumulator rows (its TMEM lane quarter) and writes
    // them 32 columns at a time: registers -> a 128-byte-swizzled slab in
    // shared memory -> one TMA store; a warp's slabs hold a whole item, so it
    // waits for its stores to have read them only once per item.
    // the epilogue warps read a (dstates) and write every global output, so
    // they alone wait for the previous kernel (x / dy, B / C are inputs)
    griddep_wait();
    const int q = warp & 3;               // TMEM lane quarter of this warp
    const int et = tid - 32 * kEpi0;      // 0 .. 127
    unsigned char* stg = base + LY::oStg + q * LY::kStg;
    if (lane == 0) tma_prefetch_map(&mOut);

    // The weights of item k into sw[k & 1]: 64 threads per head, EV
    // consecutive positions each.  MODE 0 also runs chunk_cumsum for the
    // pair (delta = softplus(dt + dt_bias), a = in-chunk inclusive cumsum of
    // delta A, both written out) and w = e^{a_last - a} delta; MODE 1 w = e^a.
    // Every epilogue thread calls it for every item (it holds named barriers).
    constexpr int EV = L / 64;
    const int eh = et >> 6, ev = et & 63;
    // The inputs of item k's weights are loaded into registers before the
    // epilogue of item k - 2 and used after it, so the epilogue hides their
    // latency (every address is valid: positions past seqlen re-read the
    // last one and are masked at use).
    unsigned short vdt[EV];
    float vin[EV], vbias = 0.f, vA = 0.f;
    auto load_w = [&](int k) {
      int b, c, h;
      decode(k, b, c, h);
      const int hd = h + eh, t0 = c * L, Lv = min(L, T - t0);
      if constexpr (MODE == 0) {
        vbias = (a.dt_bias ? a.dt_bias : a.A)[hd >> a.hs];
        vA = a.A[hd >> a.hs];
#pragma unroll
        for (int e = 0; e < EV; ++e)
          vdt[e] = reinterpret_cast<const unsigned short*>(
              a.dt)[(((int64_t)b * T + t0 + min(ev * EV + e, Lv - 1)) * H + hd) >> a.hs];
      } else {
        const int64_t cv = ((((int64_t)b * H + hd) >> a.hs) * nc + c) * L;
#pragma unroll
        for (int e = 0; e < EV; ++e) vin[e] = a.acs[cv + ev * EV + e];
      }
    };
    auto compute_w = [&](int k) {
      int b, c, h;
      decode(k, b, c, h);
      const int hd = h + eh, t0 = c * L, Lv = min(L, T - t0);
      float* w = sw + (k & 1) * 2 * L + eh * L;
      const int64_t cv = ((((int64_t)b * H + hd) >> a.hs) * nc + c) * L;
      // a head split in parts: its first part writes delta and a
      const bool wr = (hd & ((1 << a.hs) - 1)) == 0;
      if constexpr (MODE == 0) {
        const float bias = a.dt_bias ? vbias : 0.f, Ah = vA;
        float dl[EV], al[EV], run = 0.f;
#pragma unroll
        for (int e = 0; e < EV; ++e) {
          const int l = ev * EV + e;
          dl[e] = l < Lv ? dt_softplus(__uint_as_float((uint32_t)vdt[e] << 16) + bias) : 0.f;
          run += dl[e] * Ah;
          al[e] = run;
        }
        float incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const float o = __shfl_up_sync(0xffffffffu, incl, off);
          if (lane >= off) incl += o;
        }
        if (lane == 31) s_scan[q] = incl;
        epi_sync();
        const float pre = incl - run + ((q & 1) ? s_scan[q - 1] : 0.f);  // exclusive prefix
#pragma unroll
        for (int e = 0; e < EV; ++e) {
          const int l = ev * EV + e;
          al[e] += pre;
          if (wr) {
            a.delta[cv + l] = dl[e];
            a.acs[cv + l] = al[e];
          }
        }
        if (ev == 63) s_alast[eh] = al[EV - 1];  // a[L-1] as written
        epi_sync();
        const float alast = s_alast[eh];
#pragma unroll
        for (int e = 0; e < EV; ++e) w[ev * EV + e] = __expf(alast - al[e]) * dl[e];
      } else {
#pragma unroll
        for (int e = 0; e < EV; ++e) w[ev * EV + e] = __expf(vin[e]);
      }
    };

    bool ok = true;
    for (int k = 0; k < 2 && k < nk; ++k) {
      load_w(k);
      compute_w(k);
      warp_arrive(&bar_wf[k], lane);
    }
    int js = 0;                           // slabs this warp has stored
    // after an expired wait the loop still runs to the end (its waits return
    // at once), so all four warps meet the same named barriers
    for (int k = 0; k < nk; ++k) {
      const int buf = k & 1;
      if (k + 2 < nk) load_w(k + 2);
      ok = ok && __all_sync(0xffffffffu,
                            mbar_wait(&bar_accf[buf], (k >> 1) & 1, status, &abort_flag));
      fence_after_sync();
      if (ok) {
        int b, c, h;
        decode(k, b, c, h);
        const int row0 = (((b * nc + c) * H + h) * kSP) + 32 * q;  // rows (b, c, h, p) of out
        const uint32_t ta = tm + buf * N + ((uint32_t)(32 * q) << 16);
        if (js > 0) {  // the previous item's stores have read the slabs
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
        }
#pragma unroll
        for (int s = 0; s < N / 32; ++s, ++js) {
          float v[32];
          tmem_ld16(ta + 32 * s, *reinterpret_cast<float(*)[16]>(v));
          tmem_ld16(ta + 32 * s + 16, *reinterpret_cast<float(*)[16]>(v + 16));
          tmem_wait_ld();
          unsigned char* slab = stg + s * (32 * 128);
#pragma unroll
          for (int j = 0; j < 8; ++j)
            *reinterpret_cast<float4*>(slab + sw128(lane, j)) =
                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
          fence_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&mOut, 32 * s, row0, slab);
            bulk_commit_group();
          }
        }
        fence_before_sync();
        warp_arrive(&bar_acce[buf], lane);
      }
      // item k's products are complete, so the converters no longer read
      // sw[k & 1]: the weights of item k + 2 go there
      if (k + 2 < nk) {
        compute_w(k + 2);
        if (ok) warp_arrive(&bar_wf[buf], lane);
      }
    }
    if (lane == 0) bulk_wait_all();  // the stores have read shared memory and landed
  } else {
    // ------------------------------------------------------------ converters
    bool ok = true;
    for (int k = 0; ok && k < nk; ++k) {
      const float* w = sw + (k & 1) * 2 * L;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_wf[k & 1], (k >> 1) & 1, status, &abort_flag));
      for (int kb = 0; kb < NKB; ++kb) {
        const int u = k * NKB + kb;
        const int sx = u % kNX, sa = u % kNA;
        ok = ok && __all_sync(0xffffffffu,
                              mbar_wait(&bar_xf[sx], (u / kNX) & 1, status, &abort_flag));
        if (ok && u >= kNA)
          ok = __all_sync(0xffffffffu,
                          mbar_wait(&bar_ae[sa], ((u / kNA) - 1) & 1, status, &abort_flag));
        if (!ok) continue;
        // this warp: TMEM lane quarter q (A rows m = 64 hh + p), K group lg
        // (16 of the block's 64 values of l); a lane reads its (hh, p) column
        // of 16 box rows R = 2 l + hh (2 bytes each; a warp's 32 lanes read
        // 64 contiguous bytes of one row)
        const unsigned char* xs = base + LY::oX + sx * LY::kX;
        const int q = warp & 3, lg = warp >> 2;
        const int m = 32 * q + lane, hx = m >> 6, p = m & 63;
        const float* wb = w + hx * L + kb * kKB + 16 * lg;
        const uint32_t pb = ((uint32_t)(p & 7)) * 2;
        float v[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int R = 2 * (16 * lg + e) + hx;
          const unsigned short raw = *reinterpret_cast<const unsigned short*>(
              xs + sw128(R, (uint32_t)(p >> 3)) + pb);
          v[e] = __uint_as_float((uint32_t)raw << 16) * wb[e];
        }
        warp_arrive(&bar_xe[sx], lane);  // the x rows are read
        const uint32_t at = tm + ((uint32_t)(32 * q) << 16) + LY::kColA + 64 * sa;
        tmem_store_split16(at + 16 * lg, v);
        tmem_wait_st();
        fence_before_sync();  // the A operand is read by the tensor core
        warp_arrive(&bar_af[sa], lane);
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, LY::kTmemCols);
}

template <int N, int L, int MODE>
cudaError_t launch_state(const Dims& d, const void* X, const void* Y, const StateArgs& a0,
                         const char* name, bool pdl, cudaStream_t s) {
  using LY = StateLayout<N, L>;
  CUtensorMap mX, mY, mOut;
  if (!make_tma_map(&mX, X, kSP, d.H, d.T, d.B, 2, kKB) ||
      !make_tma_map(&mY, Y, d.N, d.G, d.T, d.B, 1, kKB) ||
      !make_tma_map_f32(&mOut, a0.out, d.N, (int64_t)d.B * d.nc * d.H * kSP, 32, 32))
    return cudaErrorInvalidValue;
  StateArgs a = a0;
  a.T = d.T;
  a.H = d.H;
  a.G = d.G;
  a.nc = d.nc;
  a.hs = d.hs;
  a.n_items = d.B * d.nc * (d.H / 2);
  a.status = device_status_ptr();
  if (!a.status) return cudaErrorUnknown;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  auto kern = k_state_tc<N, L, MODE>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kBytes);
  const int grid = a.n_items < sms ? a.n_items : sms;
  if (grid <= 0) return cudaSuccess;
  if (pdl)
    SSD_LAUNCH(name, s, launch_pdl(kern, dim3(grid), dim3(kStateThreads), LY::kBytes, s, mX, mY,
                                   mOut, a));
  else
    SSD_LAUNCH(name, s, kern<<<grid, kStateThreads, LY::kBytes, s>>>(mX, mY, mOut, a));
  return cudaGetLastError();
}

template <int MODE>
cudaError_t state_dispatch(const Dims& d, const void* X, const void* Y, const StateArgs& a,
                           const char* name, bool pdl, cudaStream_t s) {
  if (d.N == 128 && d.L == 256) return launch_state<128, 256, MODE>(d, X, Y, a, name, pdl, s);
  if (d.N == 128 && d.L == 128) return launch_state<128, 128, MODE>(d, X, Y, a, name, pdl, s);
  if (d.N == 64 && d.L == 256) return launch_state<64, 256, MODE>(d, X, Y, a, name, pdl, s);
  return launch_state<64, 128, MODE>(d, X, Y, a, name, pdl, s);
}

}  // namespace

cudaError_t tc_chunk_state(const Dims& d, const FwdArgs& f, float* delta, float* acs, float* S,
                           int* zero, cudaStream_t s) {
  StateArgs a{};
  a.dt = static_cast<const bf16*>(f.dt);
  a.dt_bias = f.dt_bias;
  a.A = f.A;
  a.delta = delta;
  a.acs = acs;
  a.out = S;
  a.zero = zero;
  // a call's first kernel: launched in stream order (a programmatic launch
  // here measured 15 us slower per layer step)
  return state_dispatch<0>(d, f.x, f.B, a, "k_state_tc", false, s);
}

cudaError_t tc_chunk_dstates(const Dims& d, const void* dy, const void* C, const float* acs,
                             float* dHs, bool pdl, cudaStream_t s) {
  StateArgs a{};
  a.acs = const_cast<float*>(acs);
  a.out = dHs;
  return state_dispatch<1>(d, dy, C, a, "k_dstates_tc", pdl, s);
}

}  // namespace ssd

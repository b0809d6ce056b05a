// tcgen05 tensor-core path of the SSD forward and backward (bf16 inputs,
// headdim 64, d_state 64 or 128, chunk 128 or 256): the launch sequences of
// both directions, the backward's dx kernel and its tail.  chunk_state /
// dstates run in ssd_state_tc.cu, chunk_scan, dC and dB in ssd_chunk_tc.cu.
//
// Precision: operands that the method forms in fp32 before a contraction
// (the masked decay-weighted C.B^T of dx, the fp32 inter-chunk state) are
// split into two bf16 terms,
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
  for (int i = 0; i < 4; ++i) split2_bf16(v[2 * i], v[2 * i + 1], h[i], l[i]);
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

// Copies rows [0, rows) of 8*nchunk bf16 each into 128-byte-swizzle panels
// (chunk j of row r -> dst + (j/8)*panel + sw128(r, j%8)) with cp.async;
// rows >= valid are zero-filled (their source is not read).  The caller
// commits and waits.
template <class RowPtr>
__device__ __forceinline__ void stage_rows_async(unsigned char* dst, int rows, int nchunk,
                                                 uint32_t panel, int valid, const bf16* safe,
                                                 RowPtr rowptr) {
  for (int i = threadIdx.x; i < rows * nchunk; i += blockDim.x) {
    const int r = i / nchunk, j = i % nchunk;
    const bool v = r < valid;
    cp_async16(dst + (j / 8) * panel + sw128(r, j % 8), v ? rowptr(r) + j * 8 : safe, v);
  }
}

// ================================================================ dx
// The backward's dx ("Optimizing Mamba-2 kernels for the B200", Stage 1
// kernel table: _chunk_scan_chunk_state_bwd_dx, bwd_10), rows r = s of chunk
// c, columns l in [s0, L):
//     CBT[s, l] = B_s . C_l                      (TMEM cols 0.., once per unit)
//     per head: Y  = sum_l P[s, l] dy_l,  P = CBT e^{a_l - a_s} [l >= s]
//               ST = B_s . dS_c[p, :]
//               u_s = Y + e^{a_last - a_s} ST;  dx_s = delta_s u_s + D dy_s
//               ddir_s = <x_s, u_s>,  qrow_s = delta_s <x_s, e^{a_last - a_s} ST>,
//               ddiag_s = <x_s, dy_s>
// Persistent, one CTA (512 threads) per SM over a balanced range of (batch,
// chunk, 128-row tile, group) x head items.  Per unit the score tile is
// formed once; then the two 8-warp pipelines run chains on alternate heads
// (own TMEM accumulators, P buffer, operand rows and mbarriers), the second
// starting each unit once the first has issued its state products, so one
// forms P while the other waits for the tensor core.
template <int N, int L>
struct ScanSmem {
  static constexpr int kLT = 128;
  static constexpr int kC = (N / 64) * kLT * 128;           // row-operand rows of the tile
  static constexpr int kBrows = (N / 64) * L * 128;         // column-operand rows
  static constexpr int kPw = 2 * kLT * 128;                 // per group: P panel hi + lo
  static constexpr int kBP = kBrows > 2 * kPw ? kBrows : 2 * kPw;
  static constexpr int kX = L * 128;                        // per group: dy rows
  // Where the dy rows alone cannot stage every warp's 32 x 32 fp32 block of
  // dx (4 KB each, 128-byte swizzle) for its TMA store, the tile's x rows
  // come by TMA into a buffer right after them, and the two together are
  // the staging
  static constexpr bool kXT = kX < 8 * 4096;
  static constexpr int kXr = kXT ? kLT * 128 : 0;
  static constexpr int kXg = kX + kXr;                      // per group: dy (+ x) rows
  static_assert(kXg >= 8 * 4096, "dx staging: eight warps' 4 KB blocks");
  static constexpr int kHlo = (N / 64) * 64 * 128;          // offset of the state's lo part
  static constexpr int kImg = 2 * kHlo;                     // bytes of one state image
  static constexpr int kBytes = kC + kBP + 2 * kXg + (8 * L + 6 * 128) * 4 + 1024;
};

__device__ __forceinline__ void group_sync(int id) {
  asm volatile("bar.sync %0, 256;" ::"r"(id) : "memory");
}

// The persistent grid's split of the (batch, chunk, row tile, group) x head
// items into contiguous ranges of equal cost: a head of row tile t costs its
// 64-column panels, (L - 128 t) / 64, plus about two panels of fixed work
// (state products, epilogue), so a CTA is not left with heavy-tile heads
// only.  Returns the first item of range k of `parts`; range `parts` starts
// at n_items.  Items run unit by unit, tile 0's groups before tile 1's, so
// the cost is periodic in NLT * H items.
template <int L>
__device__ __forceinline__ int64_t dx_range_start(int k, int parts, int64_t n_items, int H) {
  constexpr int NLT = L / 128, kOver = 2;
  int64_t pc = 0;  // cost of one period (one chunk's tiles, all heads)
#pragma unroll
  for (int t = 0; t < NLT; ++t) pc += (int64_t)H * ((L - 128 * t) / 64 + kOver);
  const int64_t periods = n_items / ((int64_t)NLT * H);
  const int64_t target = (periods * pc * k) / parts;  // cost before range k
  const int64_t q = target / pc;
  int64_t rem = target - q * pc, i = q * NLT * H;
#pragma unroll
  for (int t = 0; t < NLT; ++t) {
    const int64_t w = (L - 128 * t) / 64 + kOver;
    if (rem <= (int64_t)H * w) return i + (rem + w - 1) / w;  // first item whose prefix reaches it
    rem -= (int64_t)H * w;
    i += H;
  }
  return i;
}

template <int N, int L>
__global__ void __launch_bounds__(512, 1)
    k_scan_tc(const __grid_constant__ CUtensorMap mOut, const __grid_constant__ CUtensorMap mOp,
              const __grid_constant__ CUtensorMap mX, const bf16* __restrict__ x,
              const bf16* __restrict__ Bm,
              const bf16* __restrict__ Cm,
              const float* __restrict__ delta, const float* __restrict__ acs,
              const unsigned char* __restrict__ simg, const float* __restrict__ D,
              float* __restrict__ ddir, float* __restrict__ qrow,
              float* __restrict__ ddiag, int B_, int T, int H, int G, int nc, int hs,
              int* status) {
  using SM = ScanSmem<N, L>;
  constexpr int LT = SM::kLT, NLT = L / LT;
  griddep_wait();  // the state images and vectors come from the previous kernels
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t bar_cb, bar_p[2], bar_st[2], bar_done[2], bar_ld[2], bar_xr[2], bar_xx[2],
      bar_stg;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  unsigned char* base = align1024(smem_raw);
  unsigned char* sR = base;               // row operand: B rows of the tile
  unsigned char* sBP = sR + SM::kC;       // column operand rows, later the groups' P buffers
  unsigned char* sXall = sBP + SM::kBP;   // per group: dy rows (and the tile's x rows)
  float* sAall = reinterpret_cast<float*>(sXall + 2 * SM::kXg);  // per group: a [L], delta [L]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int hpg = H / G;
  const int64_t n_items = (int64_t)B_ * nc * NLT * H;  // (batch, chunk, tile, group) x head
  const int64_t it_begin = dx_range_start<L>(blockIdx.x, gridDim.x, n_items, H);
  const int64_t it_end = dx_range_start<L>(blockIdx.x + 1, gridDim.x, n_items, H);
  const bf16* rowsrc = Bm;
  const bf16* colsrc = Cm;

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bar_cb, 1);
    mbar_init(&bar_stg, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_p[i], 1);
      mbar_init(&bar_st[i], 1);
      mbar_init(&bar_done[i], 1);
      mbar_init(&bar_ld[i], 1);
      mbar_init(&bar_xr[i], 1);
      mbar_init(&bar_xx[i], 1);
    }
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 512);
  // TMEM and the per-group state live across the CTA's whole item range
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  // the next kernel may start once every CTA of this one holds its TMEM: a
  // dependent CTA that allocates TMEM on the same SM then only waits for CTAs
  // that need nothing from it
  griddep_launch_dependents();
  const uint32_t tm = tmem_base;
  // two pipelines of 8 warps; a TMEM row is shared by the warps q and q + 4
  // of a pipeline, each taking 32 of a panel's 64 columns
  const int wg = tid >> 8, wtid = tid & 255, wq = wtid >> 5, q = wq & 3, half = wq >> 2;
  const int rr = 32 * q + lane;
  const uint32_t tlane = tm + ((uint32_t)(32 * q) << 16);
  const uint32_t colY = 256 + 128 * wg, colST = colY + 64;
  const int gbar = 1 + wg;
  float* sred = sAall + 8 * L + wg * 3 * 128;  // [3][128] per pipeline: half-row partial sums
  uint32_t n_p = 0, n_st = 0, n_done = 0, n_units = 0;
  // per pipeline: heads started (all threads), and (thread wtid 0) the copies
  // issued of the image + vectors and of the operand rows
  uint32_t n_heads = 0, n_ld = 0, n_xr = 0, n_xx = 0;
  uint32_t n_stg = 0;  // units in which pipeline 0 has released pipeline 1

  for (int64_t item = it_begin; item < it_end;) {
    // one unit = (batch, chunk, row tile, group); this CTA's heads of it
    const int64_t unit = item / hpg;
    const int j0 = (int)(item % hpg);
    const int j1 = (int)min((int64_t)hpg, j0 + (it_end - item));
    item += j1 - j0;
    const int g = (int)(unit % G);
    const int64_t bct = unit / G;
    const int tile = (int)(bct % NLT);
    const int64_t bc = bct / NLT;
    const int c = (int)(bc % nc), b = (int)(bc / nc);
    const int h_begin = g * hpg + j0, h_end = g * hpg + j1;
    const int r0 = tile * LT;                       // first row (chunk-local)
    const int col0 = r0;                            // first column
    const int ncol = L - r0;                        // number of columns
    const int nsp = ncol / 64;
    const int64_t t0 = (int64_t)c * L;
    const int Lv = min(L, T - (int)t0);
    const int r = r0 + rr;                          // this thread's row (TMEM lane)
    // pipeline 1 starts a unit once pipeline 0 has issued its first head's
    // state products, so the two alternate between forming P and waiting
    // for the tensor core instead of doing both at the same time
    const uint32_t stg_par = n_stg & 1;
    if (h_begin < h_end) ++n_stg;

  stage_rows_async(sR, LT, N / 8, LT * 128, Lv - r0, rowsrc, [&](int rr2) {
      return rowsrc + (((int64_t)b * T + t0 + r0 + rr2) * G + g) * N;
    });
    stage_rows_async(sBP, ncol, N / 8, L * 128, Lv - col0, colsrc, [&](int cc) {
      return colsrc + (((int64_t)b * T + t0 + col0 + cc) * G + g) * N;
    });
    cp_async_commit();
    cp_async_wait<0>();
    fence_async_smem();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    if (tid == 0) {
      const uint32_t id = idesc_bf16(128, ncol, 0, 0);
      for (int ks = 0; ks < N / 16; ++ks) {
        const uint32_t kp = ks / 4, ko = (ks % 4) * 32;
        mma_bf16(tm, sdesc(smem_u32(sR) + kp * (LT * 128) + ko, 16, 1024),
                 sdesc(smem_u32(sBP) + kp * (L * 128) + ko, 16, 1024), id, ks > 0 ? 1u : 0u);
      }
      mma_commit(&bar_cb);
    }
    mbar_wait(&bar_cb, n_units & 1, status, &abort_flag);
    ++n_units;
    fence_after_sync();
    // sBP (the column operand) is free from here on: it becomes the P buffers.
    __syncthreads();

  unsigned char* Pw = sBP + wg * SM::kPw;
  unsigned char* sX = sXall + wg * SM::kXg;
  unsigned char* sXr = sX + SM::kX;
  float* sa2 = sAall + wg * 4 * L;  // a * log2(e)
  float* sx = sa2 + L;              // delta
  float* sraw = sx + L;             // prefetched a [L], delta [L] of the next head
  constexpr uint32_t id_py = idesc_bf16(128, kP, 0, 1);
  constexpr uint32_t id_st = idesc_bf16(128, kP, 0, 0);
  // shared-memory descriptors formed once; each product adds its offset (the
  // issuing thread shares its scheduler with the group's other warps)
  const uint64_t dR = sdesc(smem_u32(sR), 16, 1024);        // row operand, K-major
  const uint64_t dP = sdesc(smem_u32(Pw), 16, 1024);        // P panel / state image, K-major
  const uint64_t dX = sdesc(smem_u32(sX), L * 128, 1024);   // dy rows, MN-major

  // Each head's epilogue reads its own dy row from sX (and x row from sXr);
  // its block of dx is then staged there for a TMA store.  Only after that do
  // the next head's rows come in.
  constexpr bool kXT = SM::kXT;
  // What a head needs, copied by thread wtid 0 of its pipeline: its
  // inter-chunk state image (into the P buffer) and raw a / delta with bulk
  // copies on bar_ld, issued once the previous head's products are done; its
  // second-operand rows (sX, 128-byte swizzle; rows past seqlen read as
  // zeros) with TMA on bar_xr, issued at the head's start, which the first P
  // product waits for.
  auto prefetch_x = [&](int hh) {
    mbar_arrive_expect_tx(&bar_xr[wg], (uint32_t)(ncol * 128));
    ++n_xr;
    for (int k2 = 0; k2 < ncol / 128; ++k2)
      tma_load_4d(sX + k2 * 128 * 128, &mOp, 0, hh, (int)t0 + col0 + 128 * k2, b, &bar_xr[wg]);
  };
  // (kXT) the tile's rows of x, which only the epilogue reads: on bar_xx,
  // issued once the previous head's epilogue is over (rows past seqlen read
  // as zeros)
  auto prefetch_xr = [&](int hh) {
    mbar_arrive_expect_tx(&bar_xx[wg], (uint32_t)(LT * 128));
    ++n_xx;
    tma_load_4d(sXr, &mX, 0, hh, (int)t0 + r0, b, &bar_xx[wg]);
  };
  auto prefetch = [&](int hh) {
    const unsigned char* img = simg + ((((int64_t)b * nc + c) * H + hh) * (int64_t)SM::kImg);
    const int64_t cvh = ((((int64_t)b * H + hh) >> hs) * nc + c) * L;
    mbar_arrive_expect_tx(&bar_ld[wg], (uint32_t)(SM::kImg + 2 * L * 4));
    ++n_ld;
    bulk_g2s(Pw, img, SM::kImg, &bar_ld[wg]);
    bulk_g2s(sraw, acs + cvh, L * 4, &bar_ld[wg]);
    bulk_g2s(sraw + L, delta + cvh, L * 4, &bar_ld[wg]);
  };
  if (wtid == 0 && h_begin + wg < h_end) {
    prefetch(h_begin + wg);
    prefetch_x(h_begin + wg);
    if constexpr (kXT) prefetch_xr(h_begin + wg);
  }

  for (int h = h_begin + wg; h < h_end; h += 2) {
    const int64_t cv = (((int64_t)b * H + h) * nc + c) * L;
    const float Dh = D ? D[h >> hs] : 0.f;
    // the image and vectors (the operand rows may still be in flight)
    const uint32_t hpar = n_heads & 1;
    ++n_heads;
    mbar_wait(&bar_ld[wg], hpar, status, &abort_flag);
    if (wg == 1 && h == h_begin + 1) mbar_wait(&bar_stg, stg_par, status, &abort_flag);
    for (int i = wtid; i < L; i += 256) {
      const float a2 = sraw[i] * kLog2e, dl = sraw[L + i];
      sa2[i] = a2;
      sx[i] = dl;
    }
    // (TMA epilogue) the previous head's dx stores have read their staging
    // in sX before this head's operand rows are copied over it
    if (lane == 0) bulk_wait_read<0>();
    fence_async_smem();
    fence_before_sync();
    group_sync(gbar);
    if (wtid == 0 && h != h_begin + wg) {
      prefetch_x(h);
      if constexpr (kXT) prefetch_xr(h);
    }
    if (wtid == 0) {
      fence_after_sync();
#pragma unroll
      for (int ks = 0; ks < N / 16; ++ks) {
        const uint32_t kp = ks / 4, ko = (ks % 4) * 32;
        const uint64_t ad = desc_add(dR, kp * (LT * 128) + ko);
        mma_bf16(tm + colST, ad, desc_add(dP, kp * (64 * 128) + ko), id_st, ks > 0 ? 1u : 0u);
        mma_bf16(tm + colST, ad, desc_add(dP, SM::kHlo + kp * (64 * 128) + ko), id_st, 1u);
      }
      mma_commit(&bar_st[wg]);
      if (wg == 0 && h == h_begin) mbar_arrive(&bar_stg);
    }
    ++n_st;
    mbar_wait(&bar_st[wg], (n_st - 1) & 1, status, &abort_flag);  // P buffer free again
    fence_after_sync();
    const float ar2 = sa2[r];
    for (int j = 0; j < nsp; ++j) {
      if (j > 0) mbar_wait(&bar_p[wg], (n_p - 1) & 1, status, &abort_flag);
      const float* colv = sa2 + col0 + 64 * j;  // per-column a log2(e)
      // the thread's 32 columns as two 16-column groups; the second group's
      // TMEM load is in flight while the first is formed
      float cbA[16], cbB[16];
      tmem_ld16(tlane + 64 * j + 32 * half, cbA);
      tmem_wait_ld();
#pragma unroll
      for (int qg = 0; qg < 2; ++qg) {
        float(&cur)[16] = qg ? cbB : cbA;
        if (qg == 0) tmem_ld16(tlane + 64 * j + 32 * half + 16, cbB);
        // P[s, l] = CBT e^{a_l - a_s} for l >= s (one exponential per element)
#pragma unroll
        for (int k8 = 0; k8 < 2; ++k8) {
          const int c8 = 32 * half + 16 * qg + 8 * k8;  // panel-local column of the chunk
          const float4 w0 = *reinterpret_cast<const float4*>(colv + c8);
          const float4 w1 = *reinterpret_cast<const float4*>(colv + c8 + 4);
          const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
          float v[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int cl = col0 + 64 * j + c8 + e;  // chunk-local column
            v[e] = cl >= r ? cur[8 * k8 + e] * ex2_approx(wv[e] - ar2) : 0.f;
          }
          const uint32_t off = sw128(rr, c8 / 8);
          store_split8(Pw + off, Pw + LT * 128 + off, v);
        }
        if (qg == 0) tmem_wait_ld();
      }
      fence_async_smem();
      fence_before_sync();
      group_sync(gbar);
      if (wtid == 0) {
        if (j == 0) mbar_wait(&bar_xr[wg], hpar, status, &abort_flag);  // the operand rows
        fence_after_sync();
        const uint64_t dXj = desc_add(dX, 64 * j * 128);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t bd = desc_add(dXj, 16 * ks * 128);
          mma_bf16(tm + colY, desc_add(dP, ks * 32), bd, id_py, (j > 0 || ks > 0) ? 1u : 0u);
          mma_bf16(tm + colY, desc_add(dP, LT * 128 + ks * 32), bd, id_py, 1u);
        }
        mma_commit(&bar_p[wg]);
        if (j == nsp - 1) mma_commit(&bar_done[wg]);  // one phase per head
      }
      ++n_p;
    }
    // (without kXT) this thread's 32 columns of its row of x: loaded now, so
    // the latency overlaps the last MMAs
    const int64_t rowoff = (((int64_t)b * T + t0 + r) * H + h) * kP;
    const bool live = r < Lv;
    uint4 orow[4], xrow[4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      if constexpr (!kXT)
        xrow[kk] = live ? *reinterpret_cast<const uint4*>(x + rowoff + 32 * half + 8 * kk)
                        : make_uint4(0, 0, 0, 0);
    }
    ++n_done;
    const bool ok = __all_sync(
        0xffffffffu, mbar_wait(&bar_done[wg], (n_done - 1) & 1, status, &abort_flag) &&
                         (!kXT || mbar_wait(&bar_xx[wg], hpar, status, &abort_flag)));
    fence_after_sync();
    if constexpr (kXT) {
      // the row of x, from the tile's x rows
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        xrow[kk] = *reinterpret_cast<const uint4*>(sXr + sw128(rr, 4 * half + kk));
    }
    // this head's MMAs are done: the P buffer takes the next head's image
    if (wtid == 0 && h + 2 < h_end) prefetch(h + 2);
    unsigned char* stg = sX + wq * 4096;  // this warp's staging (TMA epilogue; spans sXr)
    {
      // the row of the operand this thread's outputs need, from sX (rows
      // past seqlen were zero-filled), before any warp stages over it (and
      // over the x rows, read above)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        orow[kk] = *reinterpret_cast<const uint4*>(sX + sw128(r - col0, 4 * half + kk));
      group_sync(gbar);
    }
    float pd = 0.f, pq = 0.f, pdd = 0.f;  // partial <x, u>, <x, state part>, <x, dy>
    if (ok) {
      const float es = ex2_approx(sa2[L - 1] - ar2);
      const float dr = sx[r];
#pragma unroll
      for (int c16 = 0; c16 < 2; ++c16) {
        float yv[16], st[16];
        tmem_ld16(tlane + colY + 32 * half + 16 * c16, yv);
        tmem_ld16(tlane + colST + 32 * half + 16 * c16, st);
        tmem_wait_ld();
        // (rows past seqlen: x reads as zeros, and the store clips them)
#pragma unroll
        for (int k8 = 0; k8 < 2; ++k8) {
          float ov[8], o[8];
          unpack8(orow[2 * c16 + k8], ov);
          float xv[8];
          unpack8(xrow[2 * c16 + k8], xv);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float us = es * st[8 * k8 + e];
            const float u = yv[8 * k8 + e] + us;
            o[e] = fmaf(dr, u, Dh * ov[e]);
            pd = fmaf(xv[e], u, pd);
            pq = fmaf(xv[e], us, pq);
            pdd = fmaf(xv[e], ov[e], pdd);
          }
          const int j = 4 * c16 + 2 * k8;  // 16-byte chunks j, j + 1 of the 128-byte row
          *reinterpret_cast<float4*>(stg + sw128(lane, j)) = make_float4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<float4*>(stg + sw128(lane, j + 1)) =
              make_float4(o[4], o[5], o[6], o[7]);
        }
      }
      // one store of the warp's 32 rows x 32 columns (rows past seqlen are
      // clipped by it); the next head (or unit) waits for its reads of the
      // staging before sX is refilled
      fence_async_smem();
      __syncwarp();
      if (lane == 0 && t0 + r0 + 32 * q < T) {
        tma_store_4d(&mOut, 32 * half, h, (int)t0 + r0 + 32 * q, b, stg);
        bulk_commit_group();
      }
    }
    // combine the two half-rows (pipeline-local barrier)
    if (half == 1) {
      sred[rr] = pd;
      sred[128 + rr] = pq;
      sred[256 + rr] = pdd;
    }
    group_sync(gbar);
    if (half == 0 && r < Lv) {
      ddir[cv + r] = pd + sred[rr];
      qrow[cv + r] = sx[r] * (pq + sred[128 + rr]);
      ddiag[cv + r] = pdd + sred[256 + rr];
    }
    fence_before_sync();
    group_sync(gbar);  // sX, sa, sd and the accumulators are reused by the next head
  }
    // both groups are done with this unit's C.B^T tile and buffers (and the
    // dx stores with their staging, before the next unit's rows come in)
    if (lane == 0) bulk_wait_read<0>();
    fence_before_sync();
    __syncthreads();
  }
  if (lane == 0) bulk_wait_all();  // the dx stores have landed
  if (wtid == 0) {  // copies still in flight (after an expired wait) land before the CTA exits
    if (n_ld > 0) mbar_drain(&bar_ld[wg], (n_ld - 1) & 1);
    if (n_xr > 0) mbar_drain(&bar_xr[wg], (n_xr - 1) & 1);
    if (n_xx > 0) mbar_drain(&bar_xx[wg], (n_xx - 1) & 1);
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, 512);
}

// grid (nc, H, B).  Gradient w.r.t. dA_r = delta_r A from the strict row sums
// (dC kernel) and column sums (dB kernel) of M:
//   ddA_r = sum_{j<r} (colsum_j - rowsum_j) + sum_{l>=r} ycs_l + sum_{s<r} qrow_s + dlast_c
//   ddt_r = (ddir_r + A ddA_r) softplus'(dt_r + dt_bias);  partials of dA, ddt_bias, dD.
struct FinalizeArgs {
  const bf16* dt;
  const float *dt_bias, *A, *delta, *rowsum, *colsum, *ycs, *qrow, *ddir, *ddiag, *dlast;
  int nsplit;
  float *ddt, *part;
  int T, H, L, nc;
  int hs;  // H counts 64-wide head parts, 1 << hs per head of dt / delta / ddt / part
  int B;
  float *dA, *ddt_bias, *dD;  // per head (ddt_bias / dD may be null)
  int* done;                  // finalize blocks finished, 0 at launch
};

// One (chunk c, head h, batch b) of the finalize step, by W = L / 128 warps:
// lane k of the item's warp w takes the four consecutive rows from
// 128 w + 4 k, so its loads are float4 and the scans are a lane-local pass,
// one warp scan and, for W > 1, the warps' totals through shared memory (a
// barrier of the item's warps only).  A head of 1 << hs parts sums its
// parts' row vectors first: every term of ddA and of the direct dt gradient
// is a sum over the head's channels.
template <int L>
__device__ __forceinline__ void finalize_item(const FinalizeArgs& f, int c, int h, int b,
                                              int w, int bar_id, float4* xch) {
  constexpr int R = 4, W = L / 128;
  const int lane = threadIdx.x & 31;
  const int nsplit = f.nsplit, T = f.T, H = f.H >> f.hs, nc = f.nc, V = 1 << f.hs;
  const int Lv = min(L, T - c * L);
  const int r0 = 128 * w + lane * R;
  const int64_t cv = (((int64_t)b * H + h) * nc + c) * L + r0;
  const int64_t ti0 = ((int64_t)b * T + (int64_t)c * L + r0) * H + h;
  float vdt[R], jump[R], y[R], dirr[R];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    vdt[i] = r0 + i < Lv ? __bfloat162float(f.dt[ti0 + (int64_t)i * H]) : 0.f;
    jump[i] = y[i] = dirr[i] = 0.f;
  }
  const float4 d4 = *reinterpret_cast<const float4*>(f.delta + cv);
  float dlt[R] = {d4.x, d4.y, d4.z, d4.w}, dg[R] = {0.f, 0.f, 0.f, 0.f};
  for (int j = 0; j < V; ++j) {
    const int64_t bhc = ((int64_t)b * H + h) * V + j;  // the part's (b, part) row
    const int64_t cp = (bhc * nc + c) * L + r0;
    const float4 cs = *reinterpret_cast<const float4*>(f.colsum + cp);
    const float4 rs = *reinterpret_cast<const float4*>(f.rowsum + cp);
    const float4 qr = *reinterpret_cast<const float4*>(f.qrow + cp);
    const float4 yc = *reinterpret_cast<const float4*>(f.ycs + cp);
    const float4 di = *reinterpret_cast<const float4*>(f.ddir + cp);
    const float4 dd = *reinterpret_cast<const float4*>(f.ddiag + cp);
    const float csv[R] = {cs.x, cs.y, cs.z, cs.w}, rsv[R] = {rs.x, rs.y, rs.z, rs.w};
    const float qrv[R] = {qr.x, qr.y, qr.z, qr.w}, ycv[R] = {yc.x, yc.y, yc.z, yc.w};
    const float div[R] = {di.x, di.y, di.z, di.w}, ddv[R] = {dd.x, dd.y, dd.z, dd.w};
#pragma unroll
    for (int e = 0; e < R; ++e) {
      jump[e] += csv[e] - rsv[e] + qrv[e];
      y[e] += ycv[e];
      dirr[e] += div[e];
      dg[e] += ddv[e];
    }
  }
  // rows past seqlen take no part (their entries are not defined)
#pragma unroll
  for (int i = 0; i < R; ++i)
    if (r0 + i >= Lv) dlt[i] = jump[i] = y[i] = dirr[i] = dg[i] = 0.f;
  // dlast: the state-passing partials of every part (lane k takes the
  // partials k, k + 32, ..., then a fixed xor tree)
  float dl = 0.f;
  for (int j = 0; j < V; ++j) {
    const int64_t bhc = ((int64_t)b * H + h) * V + j;
    for (int k = lane; k < nsplit; k += 32) dl += f.dlast[(bhc * nc + c) * nsplit + k];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) dl += __shfl_xor_sync(0xffffffffu, dl, o);
  // ddA_r = prefix_{j<r}(jump_j) + dlast + suffix_{l>=r}(ycs_l): the lane's
  // totals, their scan over the lanes, then over the item's warps
  const float tj = (jump[0] + jump[1]) + (jump[2] + jump[3]);
  const float ty = (y[0] + y[1]) + (y[2] + y[3]);
  float ij = tj, iy = ty;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float oj = __shfl_up_sync(0xffffffffu, ij, off);
    const float oy = __shfl_up_sync(0xffffffffu, iy, off);
    if (lane >= off) {
      ij += oj;
      iy += oy;
    }
  }
  float pj = ij - tj, py = iy - ty;  // before the lane's first row, within the warp
  float toty = __shfl_sync(0xffffffffu, iy, 31);
  if constexpr (W > 1) {
    if (lane == 31) xch[w] = make_float4(ij, iy, 0.f, 0.f);
    asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(32 * W) : "memory");
    float bj = 0.f, by = 0.f, ay = 0.f;
#pragma unroll
    for (int k = 0; k < W; ++k) {
      const float4 t = xch[k];
      if (k < w) {
        bj += t.x;
        by += t.y;
      }
      ay += t.y;
    }
    pj += bj;
    py += by;
    toty = ay;
  }
  const float Ah = f.A[h], bias = f.dt_bias ? f.dt_bias[h] : 0.f;
  float pA = 0.f, pB = 0.f, pD = 0.f;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const float dd = pj + dl + (toty - py);
    pj += jump[i];
    py += y[i];
    if (r0 + i < Lv) {
      const float v = vdt[i] + bias;
      const float sg = v > 20.f ? 1.f : 1.f / (1.f + __expf(-v));
      const float gv = fmaf(Ah, dd, dirr[i]) * sg;
      f.ddt[ti0 + (int64_t)i * H] = gv;
      pA += dlt[i] * dd;
      pB += gv;
      pD += dg[i];
    }
  }
  // the item's partials of dA, ddt_bias and dD: a fixed xor tree per warp,
  // then the warps in order
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    pA += __shfl_xor_sync(0xffffffffu, pA, o);
    pB += __shfl_xor_sync(0xffffffffu, pB, o);
    pD += __shfl_xor_sync(0xffffffffu, pD, o);
  }
  if constexpr (W > 1) {
    if (lane == 0) xch[W + w] = make_float4(pA, pB, pD, 0.f);
    asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(32 * W) : "memory");
    if (w == 0) {
      pA = pB = pD = 0.f;
#pragma unroll
      for (int k = 0; k < W; ++k) {
        const float4 t = xch[W + k];
        pA += t.x;
        pB += t.y;
        pD += t.z;
      }
    }
  }
  if (w == 0 && lane == 0) {
    float* o = f.part + (((int64_t)b * H + h) * nc + c) * 3;
    o[0] = pA;
    o[1] = pB;
    o[2] = pD;
    __threadfence();  // before the block counts itself finished
  }
}

// Head-block partials of dC / dB: row (b, t, g) holds `stride` slots, of
// which the first nb[tile of t] were written (the chunk's 128-row tile; each
// tile has its own block count).
struct PartialRows {
  int stride, G, T, L;
  int nb[2];
};

// out[i, :] = sum_k in[i, k, :] over the row's head-block partials, in order
// (float4 per element; N % 4 == 0), for the elements i0 and i0 + stride: the
// first four partials of both are loaded before any is added, so eight
// loads are in flight at once.
__device__ __forceinline__ void reduce_elem2(const float4* __restrict__ in,
                                             float4* __restrict__ out, int64_t i0, int stride,
                                             int64_t n, const PartialRows& pr, int N4) {
  const float4* p[2];
  int nb[2];
  float4 v[2][4];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const int64_t i = i0 + (int64_t)u * stride;
    const int64_t row = (i < n ? i : 0) / N4;
    const int t = (int)((row / pr.G) % pr.T);
    nb[u] = i < n ? ((t % pr.L) < 128 ? pr.nb[0] : pr.nb[1]) : 0;
    p[u] = in + (row * pr.stride) * N4 + (i < n ? i : 0) % N4;
#pragma unroll
    for (int k = 0; k < 4; ++k)
      if (k < nb[u]) v[u][k] = p[u][(int64_t)k * N4];
  }
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    if (nb[u] == 0) continue;
    float4 s = v[u][0];
#pragma unroll
    for (int k = 1; k < 4; ++k)
      if (k < nb[u]) {
        s.x += v[u][k].x;
        s.y += v[u][k].y;
        s.z += v[u][k].z;
        s.w += v[u][k].w;
      }
    for (int k = 4; k < nb[u]; ++k) {
      const float4 w = p[u][(int64_t)k * N4];
      s.x += w.x;
      s.y += w.y;
      s.z += w.z;
      s.w += w.w;
    }
    out[i0 + (int64_t)u * stride] = s;
  }
}

// The backward's tail in one launch of NT-thread blocks (NT = L): the first
// ceil(nfin / 4) blocks run the finalize step, four items i = (h, c, b) =
// (i % H, (i / H) % nc, i / (nc H)) per block, 128 rows per warp; the rest
// sum the dC, then the dB head-block partials (nred blocks each).  The two parts are independent, so
// the latency-bound finalize blocks and the bandwidth-bound sums share the SMs.
// dA, ddt_bias, dD of every head from the per-chunk partials, by the block
// that finishes the finalize step last: per head, lane k of a warp sums the
// chunks k, k + 32, ... of every batch row in order, then a fixed xor tree
// combines the lanes (bit-reproducible).  part was written by other blocks:
// it is read around L1.
template <int NT>
__device__ __forceinline__ void param_grads_block(const FinalizeArgs& f) {
  const int H = f.H >> f.hs, n = f.B * f.nc, lane = threadIdx.x & 31;
  for (int h = threadIdx.x >> 5; h < H; h += NT / 32) {
    float a = 0.f, bb = 0.f, dd = 0.f;
    for (int i = lane; i < n; i += 32) {
      const int b = i / f.nc, c = i % f.nc;
      const float* o = f.part + (((int64_t)b * H + h) * f.nc + c) * 3;
      a += __ldcg(o);
      bb += __ldcg(o + 1);
      dd += __ldcg(o + 2);
    }
    for (int off = 16; off > 0; off >>= 1) {
      a += __shfl_xor_sync(0xffffffffu, a, off);
      bb += __shfl_xor_sync(0xffffffffu, bb, off);
      dd += __shfl_xor_sync(0xffffffffu, dd, off);
    }
    if (lane == 0) {
      f.dA[h] = a;
      if (f.ddt_bias) f.ddt_bias[h] = bb;
      if (f.dD) f.dD[h] = dd;
    }
  }
}

// (1024 threads per SM: four 256-thread or eight 128-thread blocks, 64
// registers each, for the four rows of six vectors a finalize lane holds)
template <int NT>
__global__ void __launch_bounds__(NT, 1024 / NT)
    k_bwd_tail_tc(FinalizeArgs f, int nfin, const float4* __restrict__ dCp,
                  float4* __restrict__ dC, const float4* __restrict__ dBp, float4* __restrict__ dB,
                  int nred, int64_t rows, PartialRows prC, PartialRows prB, int N4) {
  griddep_launch_dependents();
  griddep_wait();  // every input comes from the previous kernels
  const int blk = blockIdx.x;
  constexpr int W = NT / 128, IPB = NT / 32 / W;  // warps per item, items per block
  const int nfb = (nfin + IPB - 1) / IPB;        // finalize blocks
  if (blk < nfb) {
    __shared__ float4 xch[NT / 32][2];  // per item: its warps' totals, then partials
    const int H = f.H >> f.hs, warp = (int)(threadIdx.x >> 5), k = warp / W;
    const int item = blk * IPB + k;
    // heads fastest: a block's items share their (batch, chunk) rows of dt
    // and ddt, which are head-interleaved
    if (item < nfin)
      finalize_item<NT>(f, (item / H) % f.nc, item % H, item / (f.nc * H), warp % W, 1 + k,
                        &xch[k * W][0]);
    // the last finalize block to finish also forms the parameter gradients
    // (each item's first lane wrote and fenced its partials)
    __shared__ int last;
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      last = atomicAdd(f.done, 1) == nfb - 1;
    }
    __syncthreads();
    if (last) {
      __threadfence();
      param_grads_block<NT>(f);
    }
    return;
  }
  const int rb = blk - nfb, which = rb / nred;
  const int64_t i0 = (int64_t)(rb % nred) * (2 * NT) + threadIdx.x;  // two elements a thread
  reduce_elem2(which ? dBp : dCp, which ? dB : dC, i0, NT, rows * N4, which ? prB : prC, N4);
}

// ------------------------------------------------------------------ launch
// The persistent dx kernel: one CTA per SM (at most one per item), each
// taking a contiguous range of the (batch, chunk, row tile, group) x head
// items of equal cost (dx_range_start).
int scan_grid(const Dims& d, int sms) {
  const int64_t items = (int64_t)d.B * d.nc * (d.L / 128) * d.H;
  return (int)(items < sms ? items : sms);
}

template <int N, int L, typename Tout>
cudaError_t launch_tc_forward_t(const Dims& d, const FwdArgs& a, const FwdWs& w, cudaStream_t s,
                                int* status, int sms) {
  {
    const cudaError_t e = tc_chunk_state(d, a, w.delta, w.acs, w.S, nullptr, s);  // + cumsum
    if (e != cudaSuccess) return e;
  }
  simt_state_passing(d, a, w, s);
  const cudaError_t e = tc_chunk_forward(d, a, w, tc_scan_blocks(d), s);
  if (e != cudaSuccess) return e;
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
  const bf16* Cm = static_cast<const bf16*>(a.f.C);
  const bf16* dy = static_cast<const bf16*>(a.dy);
  FwdArgs f = a.f;
  f.final_state = nullptr;
  FwdWs fw{w.delta, w.acs, w.S, nullptr, nullptr, w.Himg, w.seg};
  {
    // with chunk_cumsum; zeroes the tail's count of finished finalize blocks
    cudaError_t e = tc_chunk_state(d, f, w.delta, w.acs, w.S, w.done, s);
    if (e != cudaSuccess) return e;
    simt_state_passing(d, f, fw, s);
    e = tc_chunk_dstates(d, dy, Cm, w.acs, w.dHs, true, s);
    if (e != cudaSuccess) return e;
  }
  const int nsplit = simt_state_passing_bwd(d, w.dHs, w.acs, nullptr, a.dfinal, nullptr, w.dlast,
                                            a.dinit, w.dSimg, w.Himg, w.seg, s);
  {
    using SM = ScanSmem<N, L>;
    auto kern = k_scan_tc<N, L>;
    cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, SM::kBytes);
    const int grid = scan_grid(d, sms);
    CUtensorMap mDX, mDY, mXr;
    if (!make_y_map(&mDX, a.dx, d.H, d.T, d.B, 32) ||
        !make_tma_map(&mDY, dy, 64, d.H, d.T, d.B, 1, 128) ||
        !make_tma_map(&mXr, a.f.x, 64, d.H, d.T, d.B, 1, 128))
      return cudaErrorInvalidValue;
    SSD_LAUNCH("k_scan_tc_dx", s, launch_pdl(kern, dim3(grid), dim3(512), SM::kBytes, s,
        mDX, mDY, mXr, static_cast<const bf16*>(a.f.x), static_cast<const bf16*>(a.f.B), Cm, w.delta, w.acs,
        static_cast<const unsigned char*>(w.dSimg), a.f.D, w.ddir, w.qrow, w.ddiag, d.B, d.T,
        d.H, d.G, d.nc, d.hs, status));
  }
  const int nblk = w.nb.max();  // partial slots per row
  float* dCout = nblk == 1 ? a.dC : w.dCp;
  float* dBout = nblk == 1 ? a.dB : w.dBp;
  {
    const cudaError_t e = tc_chunk_backward(d, a, w, w.nb, dCout, dBout, s);
    if (e != cudaSuccess) return e;
  }
  {
    const FinalizeArgs fa{static_cast<const bf16*>(a.f.dt), a.f.dt_bias, a.f.A, w.delta,
                          w.rowsum, w.colsum, w.ycs, w.qrow, w.ddir, w.ddiag, w.dlast, nsplit,
                          a.ddt, w.part, d.T, d.H, d.L, d.nc, d.hs, d.B, a.dA, a.ddt_bias,
                          a.dD, w.done};
    const int nfin = d.nc * (d.H >> d.hs) * d.B;
    const int64_t rows = (int64_t)d.B * d.T * d.G;
    const int N4 = d.N / 4;
    const int nred = nblk > 1 ? (int)((rows * N4 + 2 * L - 1) / (2 * L)) : 0;
    // dC's heavy tile is the chunk's last (its rows see more columns), dB's
    // the first; with one tile both counts are the heavy one
    const int c0 = L > 128 ? w.nb.light : w.nb.heavy;
    const PartialRows prC{nblk, d.G, d.T, d.L, {c0, w.nb.heavy}};
    const PartialRows prB{nblk, d.G, d.T, d.L, {w.nb.heavy, w.nb.light}};
    const int nfb = (nfin + 3) / 4;  // finalize blocks: four items each (128 rows per warp)
    SSD_LAUNCH("k_bwd_tail_tc", s, launch_pdl(k_bwd_tail_tc<L>, dim3(nfb + 2 * nred), dim3(L), 0, s,
        fa, nfin, reinterpret_cast<const float4*>(w.dCp), reinterpret_cast<float4*>(a.dC),
        reinterpret_cast<const float4*>(w.dBp), reinterpret_cast<float4*>(a.dB),
        nred > 0 ? nred : 1, rows, prC, prB, N4));
  }
  return cudaGetLastError();
}

}  // namespace

bool tc_forward_supported(const Dims& d) {
  const Dims v = tc_dims(d);
  return d.in_bf16 && v.P == kP && (d.N == 64 || d.N == 128) && (d.L == 128 || d.L == 256) &&
         (v.H / d.G) % 2 == 0;
}

// A head of 128 channels runs as two 64-wide parts (the kernels' M = 128
// operand rows hold two parts, i.e. the whole head): the parts share the
// head's dt, A, D and decay vectors, and their x, y, states and images are
// the head's own bytes (channel p of head h is channel p % 64 of part
// 2h + p / 64).  Each part writes its own row vectors of the backward, which
// the finalize step sums per head.
Dims tc_dims(const Dims& d) {
  Dims v = d;
  if (d.hs == 0 && d.P == 2 * kP) {
    v.H = 2 * d.H;
    v.P = kP;
    v.hs = 1;
  }
  return v;
}


cudaError_t tc_forward(const Dims& d0, const FwdArgs& a, const FwdWs& w, cudaStream_t s) {
  const Dims d = tc_dims(d0);
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

cudaError_t tc_front_final(const Dims& d0, const FwdArgs& a, const FwdWs& w, cudaStream_t s) {
  const Dims d = tc_dims(d0);
  const cudaError_t e = tc_chunk_state(d, a, w.delta, w.acs, w.S, nullptr, s);
  if (e != cudaSuccess) return e;
  simt_state_passing(d, a, w, s);
  return cudaGetLastError();
}

cudaError_t tc_dstates(const Dims& d, const void* dy, const void* C, const float* delta,
                       const float* acs, float* dHs, cudaStream_t s) {
  (void)delta;
  return tc_chunk_dstates(tc_dims(d), dy, C, acs, dHs, false, s);  // the call's first kernel
}

cudaError_t tc_backward(const Dims& d0, const BwdArgs& a, const TcBwdWs& w, cudaStream_t s) {
  const Dims d = tc_dims(d0);
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

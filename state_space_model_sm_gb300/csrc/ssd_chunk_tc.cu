// tcgen05 chunk kernels of the SSD, fed by TMA (sm_103a).  One template,
// three roles, each over a 128-row tile of one chunk and a block of heads of
// one group ("Optimizing Mamba-2 kernels for the B200", Stage 1 kernel table:
// _chunk_scan_fwd fwd_5, _chunk_scan_bwd_dC bwd_12, _chunk_state_bwd_db
// bwd_11; the backward's dx, bwd_10, runs in ssd_tc.cu):
//
//   FWD  rows l, columns s <= l:  P  = CB[l,s] e^{a_l-a_s} delta_s
//        y_l  = sum_s P[l,s] x_s + e^{a_l} C_l.H_c^T + D x_l
//   DC   rows l, columns s <= l:  P2 = e^{a_l-a_s} delta_s <dy_l, x_s>
//        dC_l += sum_s P2[l,s] B_s + e^{a_l} dy_l.H_c   (summed over the block's heads)
//        rowsum_l = sum_{s<l} CB[l,s] P2[l,s];  ycs_l = e^{a_l} <dy_l, C_l.H_c^T>
//   DB   rows s, columns l >= s:  P2 = e^{a_l-a_s} delta_s <x_s, dy_l>
//        dB_s += sum_l P2[s,l] C_l + delta_s e^{a_last-a_s} x_s.dS_c
//        colsum_s = sum_{l>s} CB[l,s] P2[s,l]
// with CB = C.B^T of the chunk (the column-row orientation in DB).
//
// CB of the tile is formed once per CTA into TMEM and read by every head: it is
// P's base in FWD and gives the ddA sums of DC / DB directly, element by
// element, so no per-head accumulator is needed for them.
//
// Warp roles (576 threads): warps 0-15 convert (TMEM -> decay, mask, hi/lo
// bf16 split -> a TMEM operand slot, and the epilogues), warp 16 issues every
// tcgen05.mma, warp 17 issues every copy (TMA tiles of x, dy, B, C through
// tensor maps; bulk copies of the state images and the per-head a / delta
// vectors).  Full / empty mbarriers hand each buffer over; every wait is
// bounded and records SSD_ERR_TIMEOUT on expiry.
//
// Precision: P and P2 are formed in fp32 and split into bf16 hi + lo; both
// parts are multiplied (a single bf16 rounding of either exceeds the 2e-2
// max-abs bar at the layer and hybrid workloads, measured on the CPU); state
// images are split likewise; raw bf16 inputs enter unchanged; every product
// accumulates in fp32 in TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "ssd_internal.h"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

using namespace tc;
using bf16 = __nv_bfloat16;

enum : int { kFwd = 0, kDc = 2, kDb = 3 };

constexpr int kConvWarps = 16;  // 4 TMEM lane quarters x 4 column groups
constexpr int kConv = 32 * kConvWarps;
// A thread owns 64 / kCG of a row's columns in every panel and epilogue.
constexpr int kCG = kConvWarps / 4;
constexpr int kPC = 64 / kCG;
constexpr int kNG = kPC / 16;        // 16-column groups per thread
constexpr int kCPT = kPC / 8;        // 16-byte bf16 chunks per thread
constexpr int kMmaWarp = kConvWarps;
constexpr int kProdWarp = kConvWarps + 1;
constexpr int kChunkThreads = 32 * (kConvWarps + 2);

// Shared memory carving (byte offsets from a 1024-aligned base).  Only B
// operands and the row operand live here: every A operand of the big
// products (P, P2, the state terms' scaled rows) is written by the
// conversion warps into tensor memory.
template <int N, int L, int MODE>
struct ChunkLayout {
  static constexpr bool kRev = MODE == kDb;
  static constexpr bool kS1 = MODE == kDc || MODE == kDb;
  static constexpr int kLT = 128;                 // rows of a tile
  static constexpr int kNP = N / 64;              // 64-wide panels of a B / C row
  static constexpr int kRow = kNP * kLT * 128;    // the tile's row operand (C or B rows)
  static constexpr int kCol = kNP * L * 128;      // column operand rows (B or C), up to L
  static constexpr int kHlo = kNP * 64 * 128;     // offset of a state image's lo panels
  static constexpr int kImg = 2 * kHlo;           // one state image
  static constexpr int kOps = L * 128;            // one head's x or dy rows (64 wide)
  static constexpr int kHR = kLT * 128;           // DC / DB: the tile's dy (x) rows
  static constexpr int oRow = 0;
  static constexpr int oCol = oRow + kRow;
  static constexpr int oOps = oCol + kCol;                          // FWD: two stages
  static constexpr int oHR = oOps + (kS1 ? kOps : 2 * kOps);
  static constexpr int oImg = oHR + (kS1 ? kHR : 0);
  static constexpr int oVec = oImg + kImg;                         // raw [2 stages][a, delta][L]
  // derived per-head arrays: FWD keeps three heads (a head's epilogue runs
  // during the next one), DC / DB two
  static constexpr int kNDer = kS1 ? 2 : 3;
  static constexpr int oDer = oVec + 4 * L * 4;                    // [kNDer][a2, sx, cf][L]
  static constexpr int oRed = oDer + kNDer * 3 * L * 4;            // [3][kCG][128] row partials
  static constexpr int kEnd = (oRed + 3 * kCG * 128 * 4 + 1023) / 1024 * 1024;
  // FWD: each conversion warp stages its 32 x 16 block of a head's y (2 KB)
  // for one TMA store; the column operand's rows are dead once C.B^T
  // is formed, so the staging reuses them when they are large enough
  static constexpr int kStg = MODE == kFwd ? kConvWarps * 2048 : 0;
  static constexpr bool kStgInCol = kCol >= kStg;
  static constexpr int oStg = kStgInCol ? oCol : kEnd;
  static constexpr int kBytes = kEnd + (kStgInCol ? 0 : kStg) + 1024;
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
};

struct ChunkArgs {
  const float* delta;        // (B, H >> hs, nc, L)
  const float* acs;          // (B, H >> hs, nc, L)
  const unsigned char* img;  // state images (B, nc, H): H_c (FWD, DC) or dS_c (DB)
  const float* D;            // (H >> hs) or null
  void* out;                 // FWD y, DC / DB partials (B, T, G, nblk, N)
  float* msum;               // DC rowsum, DB colsum  (B, H, nc, L)
  float* ycs;                // DC
  int T, H, G, nc;
  int hs;      // H counts 64-wide head parts, 1 << hs per head of delta / a / D
  int nbt[2];  // head blocks per group of row tile 0 / 1 (the grid holds the heavier first)
  int nblk;    // DC / DB: head-block slots per row of the partials (the larger of nbt)
  int* status;
};

__device__ __forceinline__ unsigned char* align1024(unsigned char* p) {
  return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                          ~uintptr_t(1023));
}

__device__ __forceinline__ void conv_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConv) : "memory");
}

__device__ __forceinline__ void unpack8(const uint4& u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// 16 fp32 values of this thread's row -> a 16-wide K group of a TMEM A operand:
// hi = rn_bf16(v) packed in columns [col, col + 8), lo = rn_bf16(v - hi) in
// [col + 8, col + 16).  Warp-collective.
__device__ __forceinline__ void tmem_store_split16(uint32_t col, const float (&v)[16]) {
  uint32_t h[8], l[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) split2_bf16(v[2 * e], v[2 * e + 1], h[e], l[e]);
  tmem_st8u(col, h);
  tmem_st8u(col + 8, l);
}

// Arrive once per warp (lane 0) after the warp's own work.
__device__ __forceinline__ void warp_arrive(uint64_t* bar, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

template <int N, int L, int MODE, typename Tout>
__global__ void __launch_bounds__(kChunkThreads, 1)
    k_chunk_tc(const __grid_constant__ CUtensorMap mRow, const __grid_constant__ CUtensorMap mCol,
               const __grid_constant__ CUtensorMap mOps, const __grid_constant__ CUtensorMap mHR,
               const ChunkArgs a) {
  // mHR: DC / DB the tile's dy (x) rows; FWD (fp32 y) the map y is stored
  // through (fp32 (B, T, H, 64), boxes of 16 x 1 x 32, 64-byte swizzle)
  using LY = ChunkLayout<N, L, MODE>;
  constexpr bool REV = LY::kRev, S1M = LY::kS1;
  constexpr int LT = LY::kLT, NLT = L / LT, NP = LY::kNP;
  // TMEM columns: C.B^T of the tile [0, 256); two 64-column operand slots
  // (a 64-wide K panel as hi / lo bf16 per 16-wide group; in DC / DB first the
  // fp32 S1 panel, converted in place); accumulators from 384: FWD Y per head
  // parity, DC / DB the block's dC / dB rows
  constexpr uint32_t kColSlot = 256, kColAcc = 384;
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t bar_unit, bar_cb, bar_ops_full[2], bar_ops_empty[2], bar_vec_full[2],
      bar_vec_empty[2], bar_img_full, bar_img_empty, bar_slot_ready[2], bar_slot_full[2],
      bar_slot_free[2], bar_acc_full[2], bar_acc_empty[2], bar_tot, bar_final;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  unsigned char* base = align1024(smem_raw);
  unsigned char* sRow = base + LY::oRow;
  unsigned char* sCol = base + LY::oCol;
  unsigned char* sOps = base + LY::oOps;
  unsigned char* sHR = base + LY::oHR;
  unsigned char* sImg = base + LY::oImg;
  float* sVec = reinterpret_cast<float*>(base + LY::oVec);
  float* sDer = reinterpret_cast<float*>(base + LY::oDer);
  float* sRed = reinterpret_cast<float*>(base + LY::oRed);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // heavier row tiles (more columns) first: FWD / DC the last tile, DB the
  // first; each tile cuts a group's heads into its own number of blocks
  const int th = REV ? 0 : NLT - 1;  // the heavier tile
  const int zh = NLT > 1 ? a.G * a.nbt[th] : 0;
  const int tile = (int)blockIdx.z < zh || NLT == 1 ? th : NLT - 1 - th;
  // (a select, not an index: a runtime index into the parameter struct would
  // copy it to local memory)
  const int nbk = tile == 0 ? a.nbt[0] : a.nbt[1];
  const int zr = (int)blockIdx.z - (tile == th ? 0 : zh);
  const int c = blockIdx.x, b = blockIdx.y;
  const int g = zr / nbk, kb = zr % nbk;
  const int H = a.H, T = a.T, nc = a.nc, hb = H / a.G / nbk;
  const int h_begin = g * (H / a.G) + kb * hb;
  const int r0 = tile * LT, col0 = REV ? r0 : 0, ncol = REV ? L - r0 : r0 + LT;
  const int npan = ncol / 64;
  // chunk_scan: the state term C.H_c^T is one product of the tile's C rows
  // (shared memory) with the state image into its own accumulator ST,
  // scaled by e^{a_l} in the epilogue.  A tile of 128 columns leaves TMEM room
  // for Y and ST per head parity (Y at 384 + 64 st, ST at 128 + 64 st); a
  // tile of 256 holds one of each (Y at 384, ST at 448), so a head's first
  // product waits for the previous head's epilogue.
  const bool acc2 = ncol <= 128;
  const int t0 = c * L;
  const int Lv = min(L, T - t0);
  int* status = a.status;

  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bar_unit, 1);
    mbar_init(&bar_cb, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_ops_full[i], 1);
      mbar_init(&bar_ops_empty[i], 1 + kConvWarps);
      mbar_init(&bar_vec_full[i], 1);
      mbar_init(&bar_vec_empty[i], kConvWarps);
      mbar_init(&bar_slot_ready[i], 1);
      mbar_init(&bar_slot_full[i], kConvWarps);
      mbar_init(&bar_slot_free[i], 1);
      mbar_init(&bar_acc_full[i], 1);
      mbar_init(&bar_acc_empty[i], kConvWarps);
    }
    mbar_init(&bar_img_full, 1);
    mbar_init(&bar_img_empty, 1);
    mbar_init(&bar_tot, 1);
    mbar_init(&bar_final, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 512);
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  // the next kernel may start once every CTA of this one holds its TMEM: a
  // dependent CTA that allocates TMEM on the same SM then only waits for CTAs
  // that need nothing from it
  griddep_launch_dependents();
  const uint32_t tm = tmem_base;
  // slot uses per head: FWD the P panels; DC the S1 panels, the state term's
  // A operand and the state dot C.H_c^T; DB the S1 panels and the state term's
  // A operand

  if (warp == kProdWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_map(&mRow);
      tma_prefetch_map(&mCol);
      tma_prefetch_map(&mOps);
      if constexpr (S1M) tma_prefetch_map(&mHR);
      mbar_arrive_expect_tx(&bar_unit, (uint32_t)(NP * LT * 128 + NP * ncol * 128));
      for (int kp = 0; kp < NP; ++kp) {
        tma_load_4d(sRow + kp * LT * 128, &mRow, 64 * kp, g, t0 + r0, b, &bar_unit);
        for (int k2 = 0; k2 < ncol / 128; ++k2)
          tma_load_4d(sCol + kp * L * 128 + k2 * 128 * 128, &mCol, 64 * kp, g,
                      t0 + col0 + 128 * k2, b, &bar_unit);
      }
      // the tile's rows above are inputs; a / delta and the state images
      // come from the previous kernels (launched with launch_pdl)
      griddep_wait();
      uint32_t n_vec[2] = {0, 0}, n_ops[2] = {0, 0}, n_img = 0;  // phases armed
      auto load_vec = [&](int i) -> bool {
        const int v = i & 1;
        if (i >= 2 && !mbar_wait(&bar_vec_empty[v], ((i >> 1) - 1) & 1, status, &abort_flag))
          return false;
        const int64_t cv = ((((int64_t)b * H + h_begin + i) >> a.hs) * nc + c) * L;
        mbar_arrive_expect_tx(&bar_vec_full[v], 2 * L * 4);
        ++n_vec[v];
        bulk_g2s(sVec + v * 2 * L, a.acs + cv, L * 4, &bar_vec_full[v]);
        bulk_g2s(sVec + v * 2 * L + L, a.delta + cv, L * 4, &bar_vec_full[v]);
        return true;
      };
      auto load_ops = [&](int i) -> bool {
        const int h = h_begin + i;
        if constexpr (!S1M) {
          const int st = i & 1;
          if (i >= 2 && !mbar_wait(&bar_ops_empty[st], ((i >> 1) - 1) & 1, status, &abort_flag))
            return false;
          mbar_arrive_expect_tx(&bar_ops_full[st], (uint32_t)(ncol * 128));
          ++n_ops[st];
          for (int k2 = 0; k2 < ncol / 128; ++k2)
            tma_load_4d(sOps + st * LY::kOps + k2 * 128 * 128, &mOps, 0, h, t0 + col0 + 128 * k2,
                        b, &bar_ops_full[st]);
        } else {
          if (i >= 1 && !mbar_wait(&bar_ops_empty[0], (i - 1) & 1, status, &abort_flag))
            return false;
          mbar_arrive_expect_tx(&bar_ops_full[0], (uint32_t)(LT * 128 + ncol * 128));
          ++n_ops[0];
          tma_load_4d(sHR, &mHR, 0, h, t0 + r0, b, &bar_ops_full[0]);
          for (int k2 = 0; k2 < ncol / 128; ++k2)
            tma_load_4d(sOps + k2 * 128 * 128, &mOps, 0, h, t0 + col0 + 128 * k2, b,
                        &bar_ops_full[0]);
        }
        return true;
      };
      auto load_img = [&](int i) -> bool {
        if (i >= 1 && !mbar_wait(&bar_img_empty, (i - 1) & 1, status, &abort_flag)) return false;
        const unsigned char* src = a.img + (((int64_t)b * nc + c) * H + h_begin + i) * LY::kImg;
        mbar_arrive_expect_tx(&bar_img_full, LY::kImg);
        ++n_img;
        bulk_g2s(sImg, src, LY::kImg, &bar_img_full);
        return true;
      };
      bool ok = hb > 0 && load_vec(0) && load_ops(0) && load_img(0);
      for (int i = 0; ok && i + 1 < hb; ++i)
        ok = load_vec(i + 1) && load_ops(i + 1) && load_img(i + 1);
      // copies still in flight (after an expired wait) land before the CTA exits
      mbar_drain(&bar_unit, 0);
      for (int v = 0; v < 2; ++v)
        if (n_vec[v] > 0) mbar_drain(&bar_vec_full[v], (n_vec[v] - 1) & 1);
      for (int v = 0; v < 2; ++v)
        if (n_ops[v] > 0) mbar_drain(&bar_ops_full[v], (n_ops[v] - 1) & 1);
      if (n_img > 0) mbar_drain(&bar_img_full, (n_img - 1) & 1);
    }
  } else if (warp == kMmaWarp) {
    // ---------------------------------------------------------------- MMA
    if (lane == 0) {
      // Shared-memory descriptors are formed once; each product adds a
      // compile-time offset (the issuing thread would otherwise spend more
      // cycles building descriptors than the tensor pipe spends per product).
      const uint64_t dRowK = sdesc(smem_u32(sRow), 16, 1024);
      const uint64_t dColK = sdesc(smem_u32(sCol), 16, 1024);
      const uint64_t dColMN = sdesc(smem_u32(sCol), L * 128, 1024);
      const uint64_t dOpsK = sdesc(smem_u32(sOps), 16, 1024);
      const uint64_t dOpsMN = sdesc(smem_u32(sOps), L * 128, 1024);
      const uint64_t dHRK = sdesc(smem_u32(sHR), 16, 1024);
      const uint64_t dImgK = sdesc(smem_u32(sImg), 16, 1024);
      const uint64_t dImgMN = sdesc(smem_u32(sImg), 64 * 128, 1024);
      bool ok = mbar_wait(&bar_unit, 0, status, &abort_flag);
      fence_after_sync();
      if (ok) {
        const uint32_t id_cb = idesc_bf16(128, ncol, 0, 0);
#pragma unroll
        for (int ks = 0; ks < N / 16; ++ks) {
          constexpr int kR = LT * 128, kC = L * 128;
          const uint32_t oa = (ks / 4) * kR + (ks % 4) * 32, ob = (ks / 4) * kC + (ks % 4) * 32;
          mma_bf16(tm, desc_add(dRowK, oa), desc_add(dColK, ob), id_cb, ks > 0 ? 1u : 0u);
        }
        mma_commit(&bar_cb);
      }
      constexpr uint32_t id_n64k = idesc_bf16(128, 64, 0, 0);   // B K-major, N = 64
      constexpr uint32_t id_n64m = idesc_bf16(128, 64, 0, 1);   // B MN-major, N = 64
      constexpr uint32_t id_nNm = idesc_bf16(128, N, 0, 1);     // B MN-major, N = d_state
      if constexpr (!S1M) {
        uint32_t u = 0;  // slot uses
        for (int i = 0; ok && i < hb; ++i) {
          const int st = i & 1;
          const int ab = acc2 ? st : 0;             // the accumulator pair of this head
          const int na = acc2 ? (i >> 1) : i;       // earlier uses of that pair
          const uint32_t colY = kColAcc + (acc2 ? 64 * st : 0);
          const uint32_t colS = acc2 ? 128 + 64 * st : kColAcc + 64;
          ok = mbar_wait(&bar_ops_full[st], (i >> 1) & 1, status, &abort_flag);
          if (ok && na >= 1)
            ok = mbar_wait(&bar_acc_empty[ab], (na - 1) & 1, status, &abort_flag);
          if (!ok) break;
          const uint64_t dops = desc_add(dOpsMN, st * LY::kOps);
          for (int k = 0; k < npan; ++k, ++u) {
            const int s = u & 1;
            if (!mbar_wait(&bar_slot_full[s], (u >> 1) & 1, status, &abort_flag)) {
              ok = false;
              break;
            }
            fence_after_sync();
            const uint32_t sc = tm + kColSlot + 64 * s;
            const uint64_t bp = desc_add(dops, k * 64 * 128);
            const uint32_t acc0 = k > 0 ? 1u : 0u;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t bd = desc_add(bp, ks * 16 * 128);
              mma_bf16_ta(tm + colY, sc + 16 * ks, bd, id_n64m, ks > 0 ? 1u : acc0);
              mma_bf16_ta(tm + colY, sc + 16 * ks + 8, bd, id_n64m, 1u);
            }
            if (k == npan - 1) mma_commit(&bar_ops_empty[st]);  // x rows read
            mma_commit(&bar_slot_ready[s]);  // the slot may be written again
          }
          // the state term: ST = C . H_c^T (hi and lo parts of the image)
          if (ok) {
            ok = mbar_wait(&bar_img_full, i & 1, status, &abort_flag);
            fence_after_sync();
            if (ok) {
#pragma unroll
              for (int ks = 0; ks < N / 16; ++ks) {
                const uint32_t oa = (ks / 4) * (LT * 128) + (ks % 4) * 32;
                const uint32_t ob = (ks / 4) * (64 * 128) + (ks % 4) * 32;
                const uint64_t ad = desc_add(dRowK, oa);
                mma_bf16(tm + colS, ad, desc_add(dImgK, ob), id_n64k, ks > 0 ? 1u : 0u);
                mma_bf16(tm + colS, ad, desc_add(dImgK, LY::kHlo + ob), id_n64k, 1u);
              }
            }
          }
          if (!ok) break;
          mma_commit(&bar_img_empty);
          mma_commit(&bar_acc_full[ab]);
        }
      } else {
        uint32_t pu = 0, cu = 0;  // slot uses produced (MMA side) and consumed
        uint32_t acc_first = 0;   // 0 until TOT holds its first product
        auto slot_take = [&]() -> int {  // the next slot, once its previous use is over
          const int s = pu & 1;
          if (pu >= 2 && !mbar_wait(&bar_slot_free[s], ((pu >> 1) - 1) & 1, status, &abort_flag))
            return -1;
          ++pu;
          fence_after_sync();
          return s;
        };
        auto slot_wait_full = [&]() -> int {
          const int s = cu & 1;
          if (!mbar_wait(&bar_slot_full[s], (cu >> 1) & 1, status, &abort_flag)) return -1;
          ++cu;
          fence_after_sync();
          return s;
        };
        auto produce_s1 = [&](int j) -> bool {
          const int s = slot_take();
          if (s < 0) return false;
          const uint64_t bp = desc_add(dOpsK, j * 64 * 128);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks)
            mma_bf16(tm + kColSlot + 64 * s, desc_add(dHRK, ks * 32), desc_add(bp, ks * 32),
                     id_n64k, ks > 0 ? 1u : 0u);
          mma_commit(&bar_slot_ready[s]);
          return true;
        };
        auto consume_p2 = [&](int j) -> bool {
          const int s = slot_wait_full();
          if (s < 0) return false;
          const uint32_t sc = tm + kColSlot + 64 * s;
          const uint64_t bp = desc_add(dColMN, j * 64 * 128);
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const uint64_t bd = desc_add(bp, ks * 16 * 128);
            mma_bf16_ta(tm + kColAcc, sc + 16 * ks, bd, id_nNm, ks > 0 ? 1u : acc_first);
            mma_bf16_ta(tm + kColAcc, sc + 16 * ks + 8, bd, id_nNm, 1u);
          }
          acc_first = 1u;
          mma_commit(&bar_slot_free[s]);
          return true;
        };
        for (int i = 0; ok && i < hb; ++i) {
          ok = mbar_wait(&bar_ops_full[0], i & 1, status, &abort_flag);
          if (!ok) break;
          fence_after_sync();
          ok = produce_s1(0) && (npan < 2 || produce_s1(1));
          if (ok && npan <= 2) mma_commit(&bar_ops_empty[0]);  // x / dy rows read
          int sa = -1;
          for (int j = 0; ok && j < npan; ++j) {
            ok = consume_p2(j);
            if (ok && j + 2 < npan) {
              ok = produce_s1(j + 2);
              if (ok && j + 3 == npan) mma_commit(&bar_ops_empty[0]);
            }
            if (ok && j == npan - 2) {
              // the state term's A operand: the slot the next-to-last P2 frees
              // goes to the conversion warps now, so they form it right after
              // the last P2 panel instead of after its products
              sa = slot_take();
              if (sa < 0) ok = false;
              else mbar_arrive(&bar_slot_ready[sa]);
            }
          }
          if (!ok) break;
          if (!mbar_wait(&bar_img_full, i & 1, status, &abort_flag)) break;
          fence_after_sync();
          int sst = -1;
          if constexpr (MODE == kDc) {
            // the state dot C.H_c^T (for ycs) into the other slot
            sst = slot_take();
            if (sst < 0) break;
#pragma unroll
            for (int ks = 0; ks < N / 16; ++ks) {
              constexpr int kR = LT * 128;
              const uint32_t oa = (ks / 4) * kR + (ks % 4) * 32;
              const uint32_t ob = (ks / 4) * (64 * 128) + (ks % 4) * 32;
              const uint64_t ad = desc_add(dRowK, oa);
              mma_bf16(tm + kColSlot + 64 * sst, ad, desc_add(dImgK, ob), id_n64k,
                       ks > 0 ? 1u : 0u);
              mma_bf16(tm + kColSlot + 64 * sst, ad, desc_add(dImgK, LY::kHlo + ob), id_n64k, 1u);
            }
            mma_commit(&bar_slot_ready[sst]);
          }
          // TOT += A_st . img with A_st = e^{a_l} dy_l (DC) or delta_s e^{a_last-a_s} x_s
          // (DB), the image MN-major (K = p rows, N = d_state)
          sa = slot_wait_full();
          if (sa < 0) break;
          {
            const uint32_t sc = tm + kColSlot + 64 * sa;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint64_t bh = desc_add(dImgMN, ks * 2048);
              const uint64_t bl = desc_add(dImgMN, LY::kHlo + ks * 2048);
              mma_bf16_ta(tm + kColAcc, sc + 16 * ks, bh, id_nNm, 1u);
              mma_bf16_ta(tm + kColAcc, sc + 16 * ks, bl, id_nNm, 1u);
              mma_bf16_ta(tm + kColAcc, sc + 16 * ks + 8, bh, id_nNm, 1u);
            }
            mma_commit(&bar_slot_free[sa]);
          }
          mma_commit(&bar_img_empty);
          if constexpr (MODE == kDc) {
            // the conversion warps have read the state dot: its slot is free
            sst = slot_wait_full();
            if (sst < 0) break;
            mbar_arrive(&bar_slot_free[sst]);
          }
        }
        if (ok) mma_commit(&bar_tot);
      }
      // every product issued has completed before TMEM is released
      mma_commit(&bar_final);
      mbar_drain(&bar_final, 0);
    }
  } else {
    // --------------------------------------------------- conversion warps
    const int q = warp & 3, cq = warp >> 2;     // lane quarter, column group
    const int rr = 32 * q + lane, r = r0 + rr;  // this thread's row (TMEM lane), chunk-local
    const int rw = r0 + 32 * q;                 // the warp's first row
    const uint32_t tl = tm + ((uint32_t)(32 * q) << 16);
    const bool live = r < Lv;
    bool ok = __all_sync(0xffffffffu, mbar_wait(&bar_cb, 0, status, &abort_flag));
    fence_after_sync();

    // per-head vectors -> derived arrays: a2 = a log2 e; sx: FWD / DC / DB
    // a2 - log2 delta (+inf where delta = 0); cf: column factors of the
    // factorized decay inside the causal triangle.  The barriers here keep the
    // conversion warps within one head of each other.
    auto der = [&](int i) { return sDer + (i % LY::kNDer) * 3 * L; };
    auto derive = [&](int i) {
      const int v = i & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_vec_full[v], (i >> 1) & 1, status, &abort_flag)) &&
           ok;
      const float* ra = sVec + v * 2 * L;
      float* da2 = der(i);
      float* dsx = da2 + L;
      float* dcf = dsx + L;
      // the column factor's edge value is recomputed from the raw vector, so
      // one pass and one barrier suffice; it must equal the edge's own entry
      // bit for bit (the group factor R uses that entry and the two cancel),
      // hence rounded products that cannot fuse into the subtraction
      for (int t = tid; t < L; t += kConv) {
        const float a2 = __fmul_rn(ra[t], kLog2e), dl = ra[L + t];
        const float sx = dl > 0.f ? a2 - lg2_approx(dl) : __int_as_float(0x7f800000);
        da2[t] = a2;
        dsx[t] = sx;
        if constexpr (REV) dcf[t] = ex2_approx(a2 - __fmul_rn(ra[t & ~15], kLog2e));
        else dcf[t] = ex2_approx(__fmul_rn(ra[t | 15], kLog2e) - sx);
      }
      warp_arrive(&bar_vec_empty[v], lane);
      conv_sync();
    };

    // slot protocol (conversion side): wait until the MMA warp hands the slot
    // over (FWD: the products that read its previous contents are done;
    // DC / DB: S1, the state dot or an empty slot is there), then work on it
    uint32_t u = 0;  // slot uses
    auto slot_acquire = [&]() -> uint32_t {
      const int s = u & 1;
      if (S1M || u >= 2) {
        const uint32_t par = S1M ? (u >> 1) & 1 : ((u >> 1) - 1) & 1;
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_slot_ready[s], par, status, &abort_flag)) &&
             ok;
      }
      fence_after_sync();
      return tl + kColSlot + 64 * s;
    };
    auto slot_release = [&](bool wrote) {
      if (wrote) tmem_wait_st();
      fence_before_sync();
      warp_arrive(&bar_slot_full[u & 1], lane);
      ++u;
    };

    // one 64-column panel j of head i: P (FWD) or P2 (DC / DB) in fp32,
    // then hi / lo bf16 into the slot; DC / DB also add the row's M terms
    float msum = 0.f;
    auto panel = [&](int i, int j) {
      const float* da2 = der(i);
      const float* dsx = da2 + L;
      const float* dcf = dsx + L;
      const float a2r = da2[r], sxr = dsx[r];
      const int cbase = col0 + 64 * j + kPC * cq;  // chunk-local first column of this thread
      float base[kNG][16], cbv[kNG][16];
      bool outside[kNG], inside[kNG];
#pragma unroll
      for (int qg = 0; qg < kNG; ++qg) {
        const int cg = cbase + 16 * qg;
        outside[qg] = REV ? cg + 15 < rw : cg > rw + 31;
        inside[qg] = REV ? cg > rw + 31 : cg + 15 < rw;
      }
      const uint32_t sc = slot_acquire();
      if (ok) {
#pragma unroll
        for (int qg = 0; qg < kNG; ++qg) {
          if (outside[qg]) continue;
          const uint32_t cb_col = 64 * j + kPC * cq + 16 * qg;  // CB's column (from col0)
          if constexpr (S1M) {
            tmem_ld16(sc + kPC * cq + 16 * qg, base[qg]);
            tmem_ld16(tl + cb_col, cbv[qg]);
          } else {
            tmem_ld16(tl + cb_col, base[qg]);
          }
        }
        tmem_wait_ld();
      }
#pragma unroll
      for (int qg = 0; qg < kNG; ++qg) {
        const int cg = cbase + 16 * qg;
        float* vv = base[qg];  // formed in place
        if (outside[qg] || !ok) {
#pragma unroll
          for (int e = 0; e < 16; ++e) vv[e] = 0.f;
        } else if (inside[qg]) {
          // e^{a_l - a_s} (times delta) = R_row * cf_col, with the group's edge column m
          float R;
          if constexpr (MODE == kFwd || MODE == kDc) R = ex2_approx(a2r - da2[cg + 15]);
          else R = ex2_approx(da2[cg] - sxr);
          const float2 R2 = make_float2(R, R);
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4) {
            const float4 cf = *reinterpret_cast<const float4*>(dcf + cg + 4 * e4);
            const float2 f0 = __fmul2_rn(R2, make_float2(cf.x, cf.y));
            const float2 f1 = __fmul2_rn(R2, make_float2(cf.z, cf.w));
            const float2 p0 = __fmul2_rn(f0, make_float2(vv[4 * e4], vv[4 * e4 + 1]));
            const float2 p1 = __fmul2_rn(f1, make_float2(vv[4 * e4 + 2], vv[4 * e4 + 3]));
            vv[4 * e4] = p0.x;
            vv[4 * e4 + 1] = p0.y;
            vv[4 * e4 + 2] = p1.x;
            vv[4 * e4 + 3] = p1.y;
          }
          if constexpr (S1M) {
            float2 acc = make_float2(0.f, 0.f);
#pragma unroll
            for (int e = 0; e < 16; e += 2)
              acc = __ffma2_rn(make_float2(vv[e], vv[e + 1]),
                               make_float2(cbv[qg][e], cbv[qg][e + 1]), acc);
            msum += acc.x + acc.y;
          }
        } else {
          // across the diagonal: per-element exponent and mask
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int cl = cg + e;
            float f;
            if constexpr (MODE == kFwd || MODE == kDc) f = ex2_approx(a2r - dsx[cl]);
            else f = ex2_approx(da2[cl] - sxr);
            const bool valid = REV ? cl >= r : cl <= r;
            vv[e] = valid ? f * vv[e] : 0.f;
            if constexpr (S1M)
              if (cl != r) msum = fmaf(vv[e], cbv[qg][e], msum);
          }
        }
        tmem_store_split16(sc + kPC * cq + 16 * qg, base[qg]);
      }
      slot_release(true);
    };

    if constexpr (!S1M) {
      // chunk_scan: a head's epilogue runs once the next head's first panel
      // (both of its first two, where Y and ST are double-buffered) is handed
      // over, so the MMA warp has work meanwhile
      int n_ostores = 0;  // TMA stores this warp has issued
      auto epilogue = [&](int i) {
        const int st = i & 1, h = h_begin + i;
        const int ab = acc2 ? st : 0, na = acc2 ? (i >> 1) : i;
        const float* da2 = der(i);
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_acc_full[ab], na & 1, status, &abort_flag)) &&
             ok;
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_ops_full[st], (i >> 1) & 1, status,
                                               &abort_flag)) && ok;
        fence_after_sync();
        float yv[kNG][16], sv[kNG][16];
        const uint32_t colY = kColAcc + (acc2 ? 64 * st : 0);
        const uint32_t colS = acc2 ? 128 + 64 * st : kColAcc + 64;
        if (ok) {
#pragma unroll
          for (int g2 = 0; g2 < kNG; ++g2) {
            tmem_ld16(tl + colY + kPC * cq + 16 * g2, yv[g2]);
            tmem_ld16(tl + colS + kPC * cq + 16 * g2, sv[g2]);
          }
          tmem_wait_ld();
        }
        fence_before_sync();
        warp_arrive(&bar_acc_empty[ab], lane);
        // this thread's row of the stage's x rows
        const unsigned char* orow = sOps + st * LY::kOps;
        const int orr = r - col0;
        const float Dh = a.D ? a.D[h >> a.hs] : 0.f;
        const float ea = ex2_approx(da2[r]);  // e^{a_l}
        // fp32 y leaves through TMA: this warp's 32 x 16 block goes to its
        // staging slot, then one store (rows past seqlen are clipped by it);
        // bf16 y is written directly
        constexpr bool kTmaO = sizeof(Tout) == 4;
        unsigned char* stg = base + LY::oStg + warp * 2048;
        if (kTmaO && ok && n_ostores > 0) {  // the previous head's store has read the slot
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
        }
        if (ok && (kTmaO || live)) {
          const int64_t ooff = (((int64_t)b * T + t0 + r) * H + h) * 64 + kPC * cq;
#pragma unroll
          for (int k8 = 0; k8 < kCPT; ++k8) {
            float ov[8], o[8];
            unpack8(*reinterpret_cast<const uint4*>(orow + sw128(orr, kCPT * cq + k8)), ov);
            const float* yk = yv[k8 >> 1] + 8 * (k8 & 1);
            const float* sk = sv[k8 >> 1] + 8 * (k8 & 1);
#pragma unroll
            for (int e = 0; e < 8; ++e) o[e] = fmaf(Dh, ov[e], fmaf(ea, sk[e], yk[e]));
            if constexpr (kTmaO) {
#pragma unroll
              for (int j2 = 0; j2 < 2; ++j2) {
                const int j = 2 * k8 + j2;  // 16-byte chunk of the 64-byte row (64-byte swizzle)
                *reinterpret_cast<float4*>(stg + lane * 64 + ((j ^ ((lane >> 1) & 3)) << 4)) =
                    make_float4(o[4 * j2], o[4 * j2 + 1], o[4 * j2 + 2], o[4 * j2 + 3]);
              }
            } else {
              Tout* op = static_cast<Tout*>(a.out) + ooff + 8 * k8;
              *reinterpret_cast<uint4*>(op) =
                  make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]), pack_bf16(o[4], o[5]),
                             pack_bf16(o[6], o[7]));
            }
          }
        }
        if (kTmaO && ok) {
          fence_async_smem();
          __syncwarp();
          if (lane == 0 && rw + t0 < T) {
            tma_store_4d(&mHR, kPC * cq, h, t0 + rw, b, stg);
            bulk_commit_group();
          }
          ++n_ostores;
        }
        warp_arrive(&bar_ops_empty[st], lane);
      };
      for (int i = 0; i < hb; ++i) {
        derive(i);
        // the previous head's epilogue runs once two of this head's panels are
        // handed over, so the MMA warp has both to work on meanwhile
        const int jepi = acc2 && npan > 1 ? 1 : 0;
        for (int j = 0; j < npan; ++j) {
          panel(i, j);
          if (j == jepi && i > 0) epilogue(i - 1);
        }
      }
      if (hb > 0) epilogue(hb - 1);
      if (lane == 0) bulk_wait_all();  // the y stores have read the staging and landed
    } else {
      uint4 hrow[kCPT];  // this thread's values of its row of dy (DC) or x (DB)
      for (int i = 0; i < hb; ++i) {
        const int h = h_begin + i;
        ok = __all_sync(0xffffffffu, mbar_wait(&bar_ops_full[0], i & 1, status, &abort_flag)) &&
             ok;
#pragma unroll
        for (int k = 0; k < kCPT; ++k)
          hrow[k] = *reinterpret_cast<const uint4*>(sHR + sw128(rr, kCPT * cq + k));
        warp_arrive(&bar_ops_empty[0], lane);
        derive(i);
        msum = 0.f;
        for (int j = 0; j < npan; ++j) panel(i, j);
        const float* da2 = der(i);
        const float* dsx = da2 + L;
        {
          // the state term's A operand: e^{a_l} dy_l (DC), delta_s e^{a_last-a_s} x_s (DB)
          const float sc_r = MODE == kDc ? ex2_approx(da2[r]) : ex2_approx(da2[L - 1] - dsx[r]);
          const uint32_t sc = slot_acquire();
#pragma unroll
          for (int qg = 0; qg < kNG; ++qg) {
            float vv[16];
#pragma unroll
            for (int k8 = 0; k8 < 2; ++k8) {
              float v8[8];
              unpack8(hrow[2 * qg + k8], v8);
#pragma unroll
              for (int e = 0; e < 8; ++e) vv[8 * k8 + e] = v8[e] * sc_r;
            }
            tmem_store_split16(sc + kPC * cq + 16 * qg, vv);
          }
          slot_release(true);
        }
        float ypart = 0.f;
        if constexpr (MODE == kDc) {
          // ycs_l = e^{a_l} <dy_l, C_l . H_c^T> from the state dot in the other slot
          const uint32_t sc = slot_acquire();
          float sv[kNG][16];
          if (ok) {
#pragma unroll
            for (int g2 = 0; g2 < kNG; ++g2) tmem_ld16(sc + kPC * cq + 16 * g2, sv[g2]);
            tmem_wait_ld();
          }
          slot_release(false);
#pragma unroll
          for (int k = 0; k < kCPT; ++k) {
            float v[8];
            unpack8(hrow[k], v);
#pragma unroll
            for (int e = 0; e < 8; ++e) ypart = fmaf(v[e], sv[k >> 1][8 * (k & 1) + e], ypart);
          }
          ypart *= ex2_approx(da2[r]);
        }
        // the row's column groups meet in shared memory (the next writes come
        // after the next head's derive barriers)
        if (cq > 0) {
          sRed[cq * 128 + rr] = msum;
          if constexpr (MODE == kDc) sRed[(kCG + cq) * 128 + rr] = ypart;
        }
        conv_sync();
        if (cq == 0 && live && ok) {
#pragma unroll
          for (int k = 1; k < kCG; ++k) {
            msum += sRed[k * 128 + rr];
            if constexpr (MODE == kDc) ypart += sRed[(kCG + k) * 128 + rr];
          }
          const int64_t cv = (((int64_t)b * H + h) * nc + c) * L;
          a.msum[cv + r] = msum;
          if constexpr (MODE == kDc) a.ycs[cv + r] = ypart;
        }
      }
      // the block's accumulated dC / dB rows
      constexpr int NT = N / kCG;  // accumulator columns per thread
      ok = __all_sync(0xffffffffu, mbar_wait(&bar_tot, 0, status, &abort_flag)) && ok;
      fence_after_sync();
      if (ok && hb > 0) {
        float* o = static_cast<float*>(a.out) +
                   ((((int64_t)b * T + t0 + r) * a.G + g) * a.nblk + kb) * N + cq * NT;
#pragma unroll
        for (int c0 = 0; c0 < NT; c0 += 16) {
          float v[16];
          tmem_ld16(tl + kColAcc + cq * NT + c0, v);
          tmem_wait_ld();
          if (live) {
#pragma unroll
            for (int k4 = 0; k4 < 16; k4 += 4)
              *reinterpret_cast<float4*>(o + c0 + k4) =
                  make_float4(v[k4], v[k4 + 1], v[k4 + 2], v[k4 + 3]);
          }
        }
      }
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, 512);
}

// ------------------------------------------------------------------ host
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

bool make_map(CUtensorMap* m, const void* ptr, int inner, int X, int T, int B) {
  return make_tma_map(m, ptr, inner, X, T, B, 1, 128);
}

template <int N, int L, int MODE, typename Tout>
cudaError_t launch_chunk(const Dims& d, const CUtensorMap& mRow, const CUtensorMap& mCol,
                         const CUtensorMap& mOps, const CUtensorMap& mHR, const ChunkArgs& a,
                         const char* name, cudaStream_t s) {
  using LY = ChunkLayout<N, L, MODE>;
  auto kern = k_chunk_tc<N, L, MODE, Tout>;
  cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kBytes);
  const dim3 grid(d.nc, d.B, d.G * (L > 128 ? a.nbt[0] + a.nbt[1] : a.nbt[0]));
  SSD_LAUNCH(name, s, launch_pdl(kern, grid, dim3(kChunkThreads), LY::kBytes, s, mRow, mCol, mOps,
                                 mHR, a));
  return cudaGetLastError();
}

template <int N, int L>
cudaError_t chunk_fwd_nl(const Dims& d, const FwdArgs& f, const FwdWs& w, HeadBlocks nb,
                         cudaStream_t s) {
  CUtensorMap mB, mC, mX;
  if (!make_map(&mB, f.B, d.N, d.G, d.T, d.B) || !make_map(&mC, f.C, d.N, d.G, d.T, d.B) ||
      !make_map(&mX, f.x, 64, d.H, d.T, d.B))
    return cudaErrorInvalidValue;
  ChunkArgs a{};
  a.delta = w.delta;
  a.acs = w.acs;
  a.img = static_cast<const unsigned char*>(w.Himg);
  a.D = f.D;
  a.out = f.y;
  a.T = d.T;
  a.H = d.H;
  a.G = d.G;
  a.nc = d.nc;
  a.hs = d.hs;
  // the heavy tile is the chunk's last (its rows see more columns)
  a.nbt[0] = L > 128 ? nb.light : nb.heavy;
  a.nbt[1] = nb.heavy;
  a.nblk = nb.max();
  a.status = device_status_ptr();
  if (!a.status) return cudaErrorUnknown;
  if (d.out_bf16) return launch_chunk<N, L, kFwd, bf16>(d, mC, mB, mX, mX, a, "k_scan_tc", s);
  CUtensorMap mY;
  if (!make_y_map(&mY, f.y, d.H, d.T, d.B, 16)) return cudaErrorInvalidValue;
  return launch_chunk<N, L, kFwd, float>(d, mC, mB, mX, mY, a, "k_scan_tc", s);
}

template <int N, int L>
cudaError_t chunk_bwd_nl(const Dims& d, const BwdArgs& ba, const TcBwdWs& w, HeadBlocks nb,
                         float* dCout, float* dBout, cudaStream_t s) {
  CUtensorMap mB, mC, mX, mDY;
  if (!make_map(&mB, ba.f.B, d.N, d.G, d.T, d.B) || !make_map(&mC, ba.f.C, d.N, d.G, d.T, d.B) ||
      !make_map(&mX, ba.f.x, 64, d.H, d.T, d.B) || !make_map(&mDY, ba.dy, 64, d.H, d.T, d.B))
    return cudaErrorInvalidValue;
  ChunkArgs a{};
  a.delta = w.delta;
  a.acs = w.acs;
  a.D = ba.f.D;
  a.T = d.T;
  a.H = d.H;
  a.G = d.G;
  a.nc = d.nc;
  a.hs = d.hs;
  a.nblk = nb.max();  // partial slots per row
  a.status = device_status_ptr();
  if (!a.status) return cudaErrorUnknown;
  cudaError_t e;
  // dC: rows l, S1 = dy.x^T, H_c images
  ChunkArgs ac = a;  // dC: the heavy tile is the chunk's last
  ac.nbt[0] = L > 128 ? nb.light : nb.heavy;
  ac.nbt[1] = nb.heavy;
  ac.img = static_cast<const unsigned char*>(w.Himg);
  ac.out = dCout;
  ac.msum = w.rowsum;
  ac.ycs = w.ycs;
  e = launch_chunk<N, L, kDc, float>(d, mC, mB, mX, mDY, ac, "k_bwd_dc_tc", s);
  if (e != cudaSuccess) return e;
  // dB: rows s, S1 = x.dy^T, dS images
  ChunkArgs ab = a;  // dB: the heavy tile is the chunk's first
  ab.nbt[0] = nb.heavy;
  ab.nbt[1] = nb.light;
  ab.img = static_cast<const unsigned char*>(w.dSimg);
  ab.out = dBout;
  ab.msum = w.colsum;
  return launch_chunk<N, L, kDb, float>(d, mB, mC, mDY, mX, ab, "k_bwd_db_tc", s);
}

}  // namespace

// Tensor map of a (B, T, X, inner) bf16 tensor read in boxes of 64 inner
// elements (128 bytes, the 128-byte swizzle span) x box_x of X x box_t rows
// of T x one batch index; rows past T read as zeros.
bool make_tma_map(CUtensorMap* m, const void* ptr, int inner, int X, int T, int B, int box_x,
                  int box_t) {
  const auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)X, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)inner * 2, (cuuint64_t)X * inner * 2,
                                 (cuuint64_t)T * X * inner * 2};
  const cuuint32_t box[4] = {64, (cuuint32_t)box_x, (cuuint32_t)box_t, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Map of an fp32 (B, T, H, 64) tensor (y, dx) for TMA stores: boxes of cols
// (16 or 32) columns x one head x 32 rows (one warp's block), 64- or 128-byte
// swizzle to match.
bool make_y_map(CUtensorMap* m, void* y, int H, int T, int B, int cols) {
  const auto fn = encode_fn();
  if (!fn || (cols != 16 && cols != 32)) return false;
  const cuuint64_t dims[4] = {64, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {64 * 4, (cuuint64_t)H * 64 * 4, (cuuint64_t)T * H * 64 * 4};
  const cuuint32_t box[4] = {(cuuint32_t)cols, 1, 32, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, y, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            cols == 16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_tma_map_f32(CUtensorMap* m, void* ptr, int inner, int64_t rows, int box_inner,
                      int box_rows) {
  const auto fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)inner * 4};
  const cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t tc_chunk_forward(const Dims& d, const FwdArgs& f, const FwdWs& w, HeadBlocks nb,
                             cudaStream_t s) {
  if (d.N == 128 && d.L == 256) return chunk_fwd_nl<128, 256>(d, f, w, nb, s);
  if (d.N == 128 && d.L == 128) return chunk_fwd_nl<128, 128>(d, f, w, nb, s);
  if (d.N == 64 && d.L == 256) return chunk_fwd_nl<64, 256>(d, f, w, nb, s);
  return chunk_fwd_nl<64, 128>(d, f, w, nb, s);
}

cudaError_t tc_chunk_backward(const Dims& d, const BwdArgs& a, const TcBwdWs& w, HeadBlocks nb,
                              float* dCout, float* dBout, cudaStream_t s) {
  if (d.N == 128 && d.L == 256) return chunk_bwd_nl<128, 256>(d, a, w, nb, dCout, dBout, s);
  if (d.N == 128 && d.L == 128) return chunk_bwd_nl<128, 128>(d, a, w, nb, dCout, dBout, s);
  if (d.N == 64 && d.L == 256) return chunk_bwd_nl<64, 256>(d, a, w, nb, dCout, dBout, s);
  return chunk_bwd_nl<64, 128>(d, a, w, nb, dCout, dBout, s);
}

}  // namespace ssd

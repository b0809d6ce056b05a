// ssd_selftest_mma: one tcgen05 tile product, D[128][nn] = A[128][k] * B[nn][k]^T,
// with each operand staged K-major or MN-major in the 128-byte-swizzle
// layout the SSD kernels use, or (a_mn == 2) A held in tensor memory as
// packed bf16 pairs.  A diagnostic entry point: it checks the descriptor and
// tensor-memory conventions of tc_ptx.cuh on the device it runs on.
#include "ssd_internal.h"
#include "tc_ptx.cuh"

namespace ssd {
namespace {

using namespace tc;

constexpr int kSmemBytes = 200 * 1024;

__global__ void __launch_bounds__(128)
    k_selftest_mma(const __nv_bfloat16* __restrict__ A, const __nv_bfloat16* __restrict__ B,
                   float* __restrict__ D, int nn, int K, int a_mn, int b_mn, int swap_mn,
                   int* status) {
  extern __shared__ unsigned char smem_raw[];
  __shared__ uint64_t bar;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  unsigned char* sA = base;          // <= 128 x 128 bf16
  unsigned char* sB = base + 32768;  // <= 256 x 128 bf16
  const int tid = threadIdx.x, warp = tid >> 5;
  const int kc = K / 8;  // 16-byte chunks per K row
  const bool a_tm = a_mn == 2;
  if (a_tm) {
    // staged below, in tensor memory
  } else if (!a_mn) {
    for (int i = tid; i < 128 * kc; i += 128) {
      const int m = i / kc, c = i % kc;
      const uint4 v = *reinterpret_cast<const uint4*>(A + (size_t)m * K + c * 8);
      *reinterpret_cast<uint4*>(sA + (c / 8) * (128 * 128) + sw128(m, c % 8)) = v;
    }
  } else {
    for (int i = tid; i < K * 16; i += 128) {
      const int k = i / 16, c = i % 16;
      __align__(16) __nv_bfloat16 t[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) t[q] = A[(size_t)(c * 8 + q) * K + k];
      *reinterpret_cast<uint4*>(sA + (c / 8) * (K * 128) + sw128(k, c % 8)) =
          *reinterpret_cast<const uint4*>(t);
    }
  }
  if (!b_mn) {
    for (int i = tid; i < nn * kc; i += 128) {
      const int n = i / kc, c = i % kc;
      const uint4 v = *reinterpret_cast<const uint4*>(B + (size_t)n * K + c * 8);
      *reinterpret_cast<uint4*>(sB + (c / 8) * (nn * 128) + sw128(n, c % 8)) = v;
    }
  } else {
    const int nchunks = nn / 8;
    for (int i = tid; i < K * nchunks; i += 128) {
      const int k = i / nchunks, c = i % nchunks;
      __align__(16) __nv_bfloat16 t[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) t[q] = B[(size_t)(c * 8 + q) * K + k];
      *reinterpret_cast<uint4*>(sB + (c / 8) * (K * 128) + sw128(k, c % 8)) =
          *reinterpret_cast<const uint4*>(t);
    }
  }
  uint32_t ncols = 32;
  while ((int)ncols < nn + (a_tm ? K / 2 : 0)) ncols <<= 1;
  if (tid == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, ncols);
  fence_async_smem();
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tm = tmem_base;
  const uint32_t acol = (uint32_t)nn;  // A's columns follow D's
  if (a_tm) {
    // row tid of A: column c holds elements 2c (low half) and 2c + 1 (high half)
    const uint32_t lane_addr = tm + ((uint32_t)(warp * 32) << 16) + acol;
    for (int c0 = 0; c0 < K / 2; c0 += 8) {
      uint32_t w[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const __nv_bfloat16 lo = A[(size_t)tid * K + 2 * (c0 + q)];
        const __nv_bfloat16 hi = A[(size_t)tid * K + 2 * (c0 + q) + 1];
        w[q] = (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
      }
      tmem_st8u(lane_addr + c0, w);
    }
    tmem_wait_st();
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
  }
  if (tid == 0) {
    const uint32_t idesc = idesc_bf16(128, nn, a_tm ? 0 : a_mn, b_mn);
    for (int ks = 0; ks < K / 16; ++ks) {
      uint64_t ad = 0, bd;
      if (a_tm) {
      } else if (!a_mn) {
        ad = sdesc(smem_u32(sA) + (ks / 4) * (128 * 128) + (ks % 4) * 32, 16, 1024);
      } else {
        const uint32_t panel = K * 128;
        ad = sdesc(smem_u32(sA) + ks * 2048, swap_mn ? 1024 : panel, swap_mn ? panel : 1024);
      }
      if (!b_mn) {
        bd = sdesc(smem_u32(sB) + (ks / 4) * (nn * 128) + (ks % 4) * 32, 16, 1024);
      } else {
        const uint32_t panel = K * 128;
        bd = sdesc(smem_u32(sB) + ks * 2048, swap_mn ? 1024 : panel, swap_mn ? panel : 1024);
      }
      if (a_tm) mma_bf16_ta(tm, tm + acol + ks * 8, bd, idesc, ks > 0 ? 1u : 0u);
      else mma_bf16(tm, ad, bd, idesc, ks > 0 ? 1u : 0u);
    }
    mma_commit(&bar);
  }
  const bool ok = mbar_wait(&bar, 0, status, &abort_flag);
  fence_after_sync();
  if (ok) {
    const uint32_t lane_addr = tm + ((uint32_t)(warp * 32) << 16);
    for (int c0 = 0; c0 < nn; c0 += 16) {
      float v[16];
      tmem_ld16(lane_addr + c0, v);
      tmem_wait_ld();
#pragma unroll
      for (int q = 0; q < 16; ++q) D[(size_t)tid * nn + c0 + q] = v[q];
    }
  }
  fence_before_sync();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tm, ncols);
}

}  // namespace
}  // namespace ssd

extern "C" int ssd_selftest_mma(int a_mn, int b_mn, int swap_mn_offsets, int nn, int k,
                                const void* A, const void* B, float* D, void* stream) {
  if (nn < 16 || nn > 256 || nn % 16 || k < 16 || k > 128 || k % 16) return SSD_ERR_INVALID_ARG;
  if (!A || !B || !D) return SSD_ERR_INVALID_ARG;
  if (((uintptr_t)A | (uintptr_t)B) % 16) return SSD_ERR_INVALID_ARG;
  if (b_mn && nn % 64) return SSD_ERR_INVALID_ARG;
  if (a_mn < 0 || a_mn > 2 || (a_mn == 2 && nn + k / 2 > 512)) return SSD_ERR_INVALID_ARG;
  int* status = ssd::device_status_ptr();
  if (!status) return SSD_ERR_CUDA;
  if (cudaFuncSetAttribute(ssd::k_selftest_mma, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           ssd::kSmemBytes) != cudaSuccess)
    return SSD_ERR_CUDA;
  SSD_LAUNCH("k_selftest_mma", static_cast<cudaStream_t>(stream),
             ssd::k_selftest_mma<<<1, 128, ssd::kSmemBytes, static_cast<cudaStream_t>(stream)>>>(
                 static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(B), D,
                 nn, k, a_mn, b_mn, swap_mn_offsets, status));
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

namespace ssd {
namespace {

// One warp waits on an mbarrier that no one arrives on.  The wait is the
// library's bounded wait: after its time limit it records SSD_ERR_TIMEOUT in
// the status word and the kernel returns normally.
__global__ void k_selftest_timeout(int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(&bar, 0, status, &abort_flag);
}

// The same with the suspending wait of the row-streaming kernels.
__global__ void k_selftest_timeout_suspend(int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait_suspend(&bar, 0, status, &abort_flag);
}

}  // namespace
}  // namespace ssd

extern "C" int ssd_selftest_timeout(void* stream) {
  int* status = ssd::device_status_ptr();
  if (!status) return SSD_ERR_CUDA;
  SSD_LAUNCH("k_selftest_timeout", static_cast<cudaStream_t>(stream),
             ssd::k_selftest_timeout<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(status));
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

extern "C" int ssd_selftest_timeout_suspend(void* stream) {
  int* status = ssd::device_status_ptr();
  if (!status) return SSD_ERR_CUDA;
  SSD_LAUNCH("k_selftest_timeout_suspend", static_cast<cudaStream_t>(stream),
             ssd::k_selftest_timeout_suspend<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
                 status));
  return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

// Inline-PTX building blocks for the sm_103a tensor-core kernels: shared
// memory descriptors, the tcgen05 instruction descriptor, TMEM allocation and
// loads, tcgen05.mma / commit, and mbarriers with bounded waits.
//
// Operand tiles live in shared memory in the 128-byte-swizzle layout: a
// "panel" is R rows of 128 bytes (64 bf16), R a multiple of 8, 1024-byte
// aligned; the 16-byte chunk j of row r sits at r*128 + ((j ^ (r % 8)) * 16).
//   K-major operand (rows = M or N index, 64 K values per row): one panel per
//     64 K values; an MMA K-step of 16 starts 32 bytes further in the row;
//     stride between 8-row groups (SBO) = 1024 bytes.
//   MN-major operand (rows = K index, 64 M/N values per row): one panel per
//     64 M/N values, LBO = bytes between panels, SBO = 1024 bytes between
//     8-row groups; an MMA K-step of 16 starts 16 rows (2048 bytes) further.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace ssd {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t sw128(uint32_t row, uint32_t chunk) {
  return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

// Shared memory matrix descriptor (tcgen05 format): start address, leading
// and stride byte offsets (16-byte units), fixed version field 1 at bit 46,
// swizzle mode 2 (128-byte) at bits 61..63.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Descriptor of the operand that starts off bytes after the one d describes:
// the start-address field holds address >> 4 in 14 bits, and shared memory
// addresses stay below 256 KB, so the sum never carries out of the field.
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t off) {
  return d + (uint64_t)(off >> 4);
}

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 accumulator:
// D format bit 4, A format bits 7..9, B format bits 10..12, A/B major bits
// 15/16 (1 = MN-major), N/8 at bits 17..22, M/16 at bits 24..28.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// ------------------------------------------------------------------ fences
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ uint32_t mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s
constexpr int kStatusTimeout = 5;                 // SSD_ERR_TIMEOUT

// Waits for the phase with the given parity to complete, for at most
// kWaitLimitNs.  On expiry it records SSD_ERR_TIMEOUT in *status, raises the
// CTA's abort flag and returns false; once the flag is up, later waits return
// false at once so the CTA reaches its clean-up without spinning again.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int* status,
                                          volatile int* abort_flag) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (*abort_flag) return false;
    if (mbar_try_wait(a, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      if (status) atomicExch(status, kStatusTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}

// As mbar_wait, but each try suspends the thread until the phase completes
// or about kSuspendHintNs pass (the hint of mbarrier.try_wait), so a thread
// that waits long issues a few instructions instead of spinning.
constexpr uint32_t kSuspendHintNs = 20000;
__device__ __forceinline__ uint32_t mbar_try_wait_suspend(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(kSuspendHintNs)
      : "memory");
  return ok;
}
__device__ __forceinline__ bool mbar_wait_suspend(uint64_t* bar, uint32_t parity, int* status,
                                                  volatile int* abort_flag) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait_suspend(a, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (*abort_flag) return false;
    if (mbar_try_wait_suspend(a, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      if (status) atomicExch(status, kStatusTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}

// Arrive (release, CTA scope) on the mbarrier: one of its expected arrivals.
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Arrive on the mbarrier and raise its expected transaction count by bytes.
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// Bulk asynchronous copy of bytes (a multiple of 16; both addresses 16-byte
// aligned) from global to this CTA's shared memory, completing that many
// transaction bytes on bar.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Tiled tensor copy (TMA) of one box from global memory, described by a
// tensor map in kernel-parameter space, into this CTA's shared memory at dst,
// completing the box's bytes on bar.  Coordinates are element indices from
// the innermost dimension out; the innermost one times the element size must
// be a multiple of 16 bytes.  Rows outside the tensor are filled with zeros.
__device__ __forceinline__ void tma_load_4d(void* dst, const void* tmap, int c0, int c1, int c2,
                                            int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_prefetch_map(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(tmap) : "memory");
}

// Tiled tensor store (TMA) of one box from this CTA's shared memory at src to
// global memory, in the issuing thread's current bulk group.  The writes to
// src must be made visible to the async proxy first (fence_async_smem).
// Coordinates: innermost first; the innermost one times the element size is a
// multiple of 16 bytes, and neither is negative.
__device__ __forceinline__ void tma_store_2d(const void* tmap, int c0, int c1, const void* src) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::
                   "l"(tmap), "r"(c0), "r"(c1), "r"(smem_u32(src))
               : "memory");
}
__device__ __forceinline__ void tma_store_4d(const void* tmap, int c0, int c1, int c2, int c3,
                                             const void* src) {
  asm volatile(
      "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
          tmap),
      "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(src))
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until at most N of this thread's bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Waits until every bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Waits for a phase like mbar_wait but ignores the abort flag: used at the
// end of a kernel to let copies or products already in flight land before
// the CTA releases its shared memory and TMEM.  Bounded by kWaitLimitNs.
__device__ __forceinline__ void mbar_drain(uint64_t* bar, uint32_t parity) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(a, parity))
    if (globaltimer_ns() - t0 > kWaitLimitNs) return;
}

// One lane of a converged warp: 1 in the elected lane, 0 in the others.
__device__ __forceinline__ uint32_t elect_one() {
  uint32_t pred;
  asm volatile(
      "{\n\t.reg .b32 rx;\n\t.reg .pred px;\n\telect.sync rx|px, 0xffffffff;\n\t"
      "selp.b32 %0, 1, 0, px;\n\t}"
      : "=r"(pred));
  return pred;
}

// -------------------------------------------------------------------- TMEM
// Whole warp: allocate ncols (power of two >= 32) columns; the TMEM address
// is written to shared memory at dst.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// This thread's lane, 16 consecutive 32-bit columns starting at taddr's column.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// This thread's lane, 16 consecutive 32-bit columns starting at taddr's column.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
// This thread's lane, 16 consecutive 32-bit columns of raw words (packed bf16 pairs).
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t (&w)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]),
      "r"(w[8]), "r"(w[9]), "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]),
      "r"(w[15])
      : "memory");
}
// The same for 8 columns.
__device__ __forceinline__ void tmem_st8u(uint32_t taddr, const uint32_t (&w)[8]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
      "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// --------------------------------------------------------------------- MMA
// D[tmem] (+)= A[smem] * B[smem], one elected thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem], one elected thread: A (M = 128 rows, one per
// TMEM lane) sits in tensor memory at a_tmem, a K-step of 16 bf16 values in 8
// consecutive 32-bit columns, element 2c in the low and 2c + 1 in the high
// half of column c (the packing of tmem_st16 with pack_bf16 pairs).
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on the mbarrier once every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// The same issued only by the lane with leader != 0 of a converged warp.
__device__ __forceinline__ void mma_bf16_if(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                            uint32_t accumulate, uint32_t leader) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "setp.ne.b32 q, %5, 0;\n\t"
      "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate), "r"(leader)
      : "memory");
}
__device__ __forceinline__ void mma_commit_if(uint64_t* bar, uint32_t leader) {
  asm volatile(
      "{\n\t.reg .pred q;\n\t"
      "setp.ne.b32 q, %1, 0;\n\t"
      "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
      ::"r"(smem_u32(bar)), "r"(leader)
      : "memory");
}

// ---------------------------------------------------------------- cp.async
// 16-byte global -> shared copy; valid == false writes 16 zero bytes (the
// source is not read).  Completion: cp_async_commit + cp_async_wait<n>.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// --------------------------------------------------------------- bf16 pack
__device__ __forceinline__ uint32_t pack_bf16(float lo_elem, float hi_elem) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo_elem, hi_elem);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Hardware base-2 exponential / logarithm (MUFU, flush-to-zero); the SSD
// kernels keep cumulative decays in log2 units so each decay factor is one
// subtraction and one ex2.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2_approx(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2e = 1.4426950408889634f;

// Two fp32 values -> packed bf16 pairs hi = rn(v), lo = rn(v - hi).  The
// residual v - hi is exact in fp32; one packed fma (-hi * 1 + v) forms both.
__device__ __forceinline__ void split2_bf16(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(a, b);
  const float2 hf = make_float2(__uint_as_float(hi << 16), __uint_as_float(hi & 0xFFFF0000u));
  const float2 res = __ffma2_rn(hf, make_float2(-1.f, -1.f), make_float2(a, b));
  lo = pack_bf16(res.x, res.y);
}

// Split v into two bf16 whose sum carries ~16 significant bits: hi = rn(v),
// lo = rn(v - hi).
__device__ __forceinline__ void split_bf16(float v, float& hi, float& lo) {
  hi = __bfloat162float(__float2bfloat16_rn(v));
  lo = v - hi;
}

}  // namespace tc
}  // namespace ssd

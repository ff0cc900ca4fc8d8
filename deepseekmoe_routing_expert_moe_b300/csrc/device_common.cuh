// Device-side helpers shared by the kernels of libmoe (sm_103a only).
//
// PTX wrappers are written from the PTX ISA description of mbarrier,
// cp.async.bulk.tensor (TMA) and the tcgen05 family (TMEM alloc, MMA,
// commit, load).  No CUTLASS/CuTe code is used or linked.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/moe.h"

namespace moe {

// ----------------------------------------------------------------- bf16
__device__ __forceinline__ float bf16_lo(uint32_t v) {
  return __uint_as_float(v << 16);
}
__device__ __forceinline__ float bf16_hi(uint32_t v) {
  return __uint_as_float(v & 0xFFFF0000u);
}
// round-to-nearest-even fp32 -> bf16 pair, packed (lo in bits 0..15)
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&p);
}

// ----------------------------------------------------------- error word
// The first 256 bytes of every workspace are the device status block:
//   [0] int32 first error code recorded (moe_status_t), 0 = none
//   [1] int32 site of that error (kernel-specific tag)
struct DevStatus {
  int32_t code;
  int32_t site;
};

__device__ __forceinline__ void record_error(DevStatus* st, int code,
                                             int site) {
  if (st != nullptr && atomicCAS(&st->code, 0, code) == 0) {
    st->site = site;
  }
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar),
               "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar,
                                                      uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
          bar),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with parity `parity` of barrier `bar`.
// Returns false -- without waiting further -- when the CTA's abort flag is
// raised or when `limit_ns` passes; in the latter case it raises the abort
// flag and records MOE_ERR_TIMEOUT with `site`.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar,
                                                  uint32_t parity,
                                                  volatile int* abort_flag,
                                                  uint64_t limit_ns,
                                                  DevStatus* st, int site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (abort_flag != nullptr && *abort_flag) return false;
    if (global_ns() - t0 > limit_ns) {
      if (abort_flag != nullptr) *abort_flag = 1;
      record_error(st, MOE_ERR_TIMEOUT, site);
      return false;
    }
  }
}

// ------------------------------------------------------------------ TMA
// 2-D tiled bulk tensor load global -> shared, completion counted in bytes
// on `bar`.  c0 is the innermost (contiguous) coordinate in elements.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap,
                                            int32_t c0, int32_t c1,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::"
      "complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst,
                                                 const void* tmap, int32_t c0,
                                                 int32_t c1, uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::"
      "complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(bar),
      "l"(policy)
      : "memory");
}

// Four rows of a 2-D tensor gathered into shared memory: rows r0..r3 (any
// order, each a box of one row) at columns c0.., landing as four
// consecutive rows at `dst`; completion counted in bytes on `bar`.
__device__ __forceinline__ void tma_gather4(uint32_t dst, const void* tmap,
                                            int32_t c0, int4 rows,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cta.global.tile::gather4.mbarrier::"
      "complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(rows.x),
      "r"(rows.y), "r"(rows.z), "r"(rows.w), "r"(bar)
      : "memory");
}

// 3-D tiled bulk tensor store shared -> global (bulk-group completion),
// with an L2 cache policy for the written lines
__device__ __forceinline__ void tma_store_3d(const void* tmap, uint32_t src,
                                             int32_t c0, int32_t c1,
                                             int32_t c2, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group"
      ".L2::cache_hint [%0, {%2, %3, %4}], [%1], %5;" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}
// the same, added element-wise to the global tensor (fp32 add in L2)
__device__ __forceinline__ void tma_reduce_add_3d(const void* tmap,
                                                  uint32_t src, int32_t c0,
                                                  int32_t c1, int32_t c2,
                                                  uint64_t policy) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      ".L2::cache_hint [%0, {%2, %3, %4}], [%1], %5;" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// wait until at most one bulk group still reads its shared-memory source
__device__ __forceinline__ void bulk_wait_read_le1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// wait until at most three bulk groups still read their sources
__device__ __forceinline__ void bulk_wait_read_le3() {
  asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory");
}
// wait until every bulk group of this thread has completed
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
// make this thread's generic-proxy shared-memory writes visible to the
// async proxy (TMA) before a bulk copy reads them
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap))
               : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;"
               : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;"
               : "=l"(p));
  return p;
}

// ------------------------------------------------- power-of-two scales
// Exponent e of the least power of two with 448 * 2^e >= amax (amax >= 0,
// finite), at least -127 (the smallest UE8M0 exponent); 0 for amax = 0.
// For a normal amax = 1.m * 2^E: amax / 448 = (1.m / 1.75) * 2^(E - 8), and
// 1.m / 1.75 lies in [4/7, 8/7), so e = E - 8 when 1.m <= 1.75 (mantissa
// field <= 0x600000) and E - 7 otherwise.  A subnormal amax needs an e
// below -134, clamped to -127.
__device__ __forceinline__ int ue8m0_exponent(float amax) {
  const uint32_t b = __float_as_uint(amax);
  if (b == 0u) return 0;
  const int E = (int)(b >> 23) - 127;
  if ((b >> 23) == 0u) return -127;
  const int e = (b & 0x7FFFFFu) <= 0x600000u ? E - 8 : E - 7;
  return e < -127 ? -127 : e;
}
// 2^-e as an fp32 (exact: e in [-127, 127] keeps it a normal number)
__device__ __forceinline__ float pow2_neg(int e) {
  return __uint_as_float((uint32_t)(127 - e) << 23);
}

// -------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile(
      "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::
          "r"(dst_smem),
      "r"(ncols)
      : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile(
      "tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr),
      "r"(ncols)
      : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 in, f32 acc)
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc,
                                           uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(
          d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when all previously issued tcgen05 ops of this
// thread have completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 "
      "[%0];" ::"r"(bar)
      : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: lane i of the warp receives row
// (taddr.lane + i), columns taddr.col .. taddr.col+15.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
      "%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]),
        "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]),
        "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand tile written by TMA
// with 128-byte swizzle: rows of 64 bf16 (128 B), 8-row swizzle atoms of
// 1024 B stacked at a stride of 1024 B.  Fields: start address >> 4
// (bits 0-13), leading byte offset >> 4 (16-29, unused for this layout),
// stride byte offset >> 4 (32-45), fixed 0b001 (46-48), base offset 0
// (49-51), layout SWIZZLE_128B = 2 (61-63).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;          // LBO (ignored): 16 B
  d |= static_cast<uint64_t>(1024u >> 4) << 32;  // SBO: 1024 B
  d |= static_cast<uint64_t>(1u) << 46;          // descriptor version
  d |= static_cast<uint64_t>(2u) << 61;          // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f16: D f32, A and B bf16, both K-major,
// dense, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4)                                   // D format: f32
         | (1u << 7)                                 // A format: bf16
         | (1u << 10)                                // B format: bf16
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

}  // namespace moe

// PTX wrappers shared by the tcgen05 kernels: shared-memory addresses and matrix
// descriptors, bounded mbarrier waits, TMA loads, TMEM loads and stores, a release-acquire
// atomic.  Device code only; every function is inlined into its caller.
#pragma once

#include <cstdint>

namespace dq4d {
namespace {

// A wait gives up after kWaitNs of %globaltimer time (or kWaitLimit polls, should the
// timer not advance); each poll may suspend the thread for up to kSuspendNs, and the
// hardware resumes it as soon as the phase completes, so waiting warps do not spin on
// issue slots the dequantizing warps need.
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr uint32_t kSuspendNs = 1000;  // (0 or 100 ns for the MMA thread measured alike)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
// groups 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  uint64_t d = static_cast<uint64_t>((addr >> 4) & 0x3FFF);
  d |= static_cast<uint64_t>(1) << 16;            // leading byte offset (unused when swizzled)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;    // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;            // descriptor version
  d |= static_cast<uint64_t>(2) << 61;            // 128-byte swizzle
  return d;
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity,
                                         uint32_t suspend_ns = kSuspendNs) {
  uint32_t done;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done) : "r"(bar), "r"(parity), "r"(suspend_ns) : "memory");
  return done != 0;
}

// Poll two barriers at once (their round trips overlap); true when both phases completed.
__device__ __forceinline__ bool mbar_try2(uint32_t bar_a, uint32_t par_a, uint32_t bar_b,
                                          uint32_t par_b) {
  uint32_t done;
  asm volatile(
      "{\n.reg .pred pa, pb;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 pa, [%1], %2, %5;\n"
      "mbarrier.try_wait.parity.shared::cta.b64 pb, [%3], %4, %5;\n"
      "and.pred pa, pa, pb;\n"
      "selp.u32 %0, 1, 0, pa;\n}"
      : "=r"(done) : "r"(bar_a), "r"(par_a), "r"(bar_b), "r"(par_b), "r"(kSuspendNs)
      : "memory");
  return done != 0;
}

// Add v to *p and return the old value, with release and acquire semantics at GPU scope:
// the writes ordered before it are visible to whoever acquires a later value of *p, and
// the writes released with earlier values are visible after it.
__device__ __forceinline__ int atomic_add_acq_rel(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;"
               : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint32_t suspend_ns = kSuspendNs) {
  if (mbar_try(bar, parity, suspend_ns)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0; it < kWaitLimit; ++it) {
    if (mbar_try(bar, parity, suspend_ns)) return true;
    if (global_ns() - t0 > kWaitNs) break;
  }
  return false;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

// Add `bytes` to the transaction count `bar` waits for, and arrive on it.
__device__ __forceinline__ void mbar_expect(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(bar), "r"(bytes) : "memory");
}

// A 2-D tiled TMA copy into shared memory at `dst`, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, uint64_t tmap, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      :: "r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(bar) : "memory");
}

// 8 consecutive accumulator columns of this warp's 32 TMEM lanes.  The load carries no
// memory clobber (it may be issued ahead of earlier stores); the wait names the loaded
// registers, so no use of them precedes it.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7])
               :: "memory");
}

// 32 consecutive accumulator columns: four loads, one wait.  The wait names half the
// registers (an asm statement takes at most 30 operands); the empty statement after it
// (volatile, so it stays after the wait) names the rest, so no use of any of them
// moves above the wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r[8 * q]), "=r"(r[8 * q + 1]), "=r"(r[8 * q + 2]), "=r"(r[8 * q + 3]),
          "=r"(r[8 * q + 4]), "=r"(r[8 * q + 5]), "=r"(r[8 * q + 6]), "=r"(r[8 * q + 7])
        : "r"(taddr + 8 * q));
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                 "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                 "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :: "memory");
  asm volatile(""
               : "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                 "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]),
                 "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]));
}

template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[N]) {
  static_assert(N == 8 || N == 32, "8 or 32 columns");
  if constexpr (N == 8) tmem_ld8(taddr, r); else tmem_ld32(taddr, r);
}

// 16 and 8 bytes at shared-memory byte address `addr` (aligned to their size): shared
// loads named as such, so they need no generic-address resolution.
__device__ __forceinline__ uint4 lds_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds_v2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}

// The 8-byte word at shared-memory byte address `addr` (8-byte aligned).
__device__ __forceinline__ uint64_t lds_b64(uint32_t addr) {
  uint64_t v;
  asm volatile("ld.shared.b64 %0, [%1];" : "=l"(v) : "r"(addr));
  return v;
}

// Store N (8, 16 or 32) consecutive 32-bit columns of this warp's 32 TMEM lanes.  It
// reads registers only, so it carries no memory clobber and the compiler may move
// shared-memory loads across it; tcgen05.wait::st (volatile, in order) completes it.
template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const uint32_t (&v)[N]) {
  if constexpr (N == 32) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
        :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
           "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]),
           "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]),
           "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),
           "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31]));
  } else if constexpr (N == 16) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};"
        :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
           "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]),
           "r"(v[13]), "r"(v[14]), "r"(v[15]));
  } else {
    static_assert(N == 8, "8, 16 or 32 columns");
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
        :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]),
           "r"(v[6]), "r"(v[7]));
  }
}

// Instruction descriptor, kind::f16: FP32 accumulator, A and B both BF16 or both FP16, both
// K-major, M x N.
template <int M, int N>
__device__ __forceinline__ uint32_t instr_desc_f16(bool bf16) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

}  // namespace
}  // namespace dq4d

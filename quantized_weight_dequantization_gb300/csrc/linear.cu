// Nested 4-bit dequantization fused into a tcgen05 GEMM: dq4_nested_linear,
// Y[M, N] = X[M, K] * W[N, K]^T with W given as nested 4-bit codes (the
// rows x cols = N x K weight that dq4_nested would expand) and never written
// out.  This is the dequantize-plus-linear shape of "Fuse nested scale
// reconstruction into SM103 4-bit dequantization" (bitsandbytes issue #21,
// sections "Problem" and "B300 evidence plan": the fallback that rebuilds the
// scales, materialises the whole weight and calls F.linear), done without the
// weight.
//
// The weight sits on the MMA's M side: a CTA owns 128 weight rows (TMEM lanes)
// and BX activation rows (TMEM columns, the MMA's N = 16 .. 256), so a decode
// batch of a few tokens costs an N = 16 MMA instead of a 128-row activation
// tile, and a large batch decodes each weight tile once per 256 activations.
// Eleven warps:
//  * warp 9 (lane 0): streams the packed weight rows of the tile with TMA into
//    a ring of raw 128 x 64-value stages (4 KB each), as far ahead as the
//    ring allows;
//  * warp 10 (lane 0): streams the activation tiles (BX rows x 64 K, 128-byte
//    swizzle, rows past M zero-filled) with TMA into their own ring;
//  * warps 0..7 (256 threads, two per weight row, 32 values each): per stage,
//    the nested scale of the row's block (separately rounded FP32 multiply
//    and add; the scale codes and absmax values are loaded 8 stages ahead
//    into registers), the 32 values (FP32 product, RN to BF16 / FP16) written
//    into the K-major 128-byte-swizzled A tile the MMA reads; afterwards the
//    epilogue: tcgen05.ld of the accumulator, conversion, stores of Y;
//  * warp 8: allocates the TMEM accumulator; lane 0 issues tcgen05.mma
//    (M = 128, N = BX, K = 16) for each stage and commits the stage's weight
//    and activation slots back to their producers.
// Every W value is computed exactly as dq4_nested does, so the GEMM consumes
// the same operand bits as "dequantize, then F.linear".  Waits on mbarriers
// are bounded; a wait that runs out counts into *bad, raises a CTA-wide abort
// flag, and the CTA drains its copies and MMAs, frees its TMEM and returns.
#include "common.cuh"

#include <cuda.h>  // CUtensorMap and its enums (the encoder is reached through the runtime)

#include <mutex>

namespace dq4d {
namespace {

constexpr int kLinThreads = 352;  // 8 dequant/epilogue warps, MMA, weight-TMA, activation-TMA
constexpr int kProducerWarps = 8;
constexpr int kBW = 128;           // weight rows per CTA = MMA M = TMEM lanes
constexpr int kBK = 64;            // 64 16-bit values = one 128-byte swizzle row
constexpr int kRawBytes = kBW * kBK / 2;  // one raw stage: 128 rows x 32 packed bytes
constexpr int kRaw = 16;           // raw weight stages in flight
constexpr int kCodeAhead = 8;      // stages of scale codes / absmax held in registers
// A wait gives up after kWaitNs of %globaltimer time (or kWaitLimit polls, should the
// timer not advance); each poll may suspend the thread for up to kSuspendNs, and the
// hardware resumes it as soon as the phase completes, so waiting warps do not spin on
// issue slots the dequantizing warps need.
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr uint32_t kSuspendNs = 1000;

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

// Instruction descriptor, kind::f16: FP32 accumulator, A and B both BF16 or
// both FP16, both K-major, M = 128, N = BX.
template <int BX>
__device__ __forceinline__ uint32_t instr_desc(bool bf16) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         (static_cast<uint32_t>(BX >> 3) << 17) | (static_cast<uint32_t>(kBW >> 4) << 24);
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      "selp.u32 %0, 1, 0, p;\n}"
      : "=r"(done) : "r"(bar), "r"(parity), "r"(kSuspendNs) : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0; it < kWaitLimit; ++it) {
    if (mbar_try(bar, parity)) return true;
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

// Arm `bar` for `bytes` of TMA data and start a 2-D tiled copy into `dst`.
__device__ __forceinline__ void tma_2d(uint32_t dst, uint64_t tmap, int x, int y, uint32_t bar,
                                       uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(bar), "r"(bytes) : "memory");
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];"
      :: "r"(dst), "l"(tmap), "r"(x), "r"(y), "r"(bar) : "memory");
}

// 8 consecutive accumulator columns of this warp's 32 TMEM lanes.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// (a * s, b * s), each product rounded to nearest FP32 on its own (one packed
// f32x2 multiply; no contraction, so the bits equal two __fmul_rn).
__device__ __forceinline__ void mul2_rn(float a, float b, uint64_t s2, float& x, float& y) {
  uint64_t ab, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ab) : "f"(a), "f"(b));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(ab), "l"(s2));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(r));
}

// Byte offset of 16-byte chunk `ch` of row `r` in a K-major 128-byte-swizzled tile.
__device__ __forceinline__ int swz128(int r, int ch) {
  return (r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4);
}

struct LinArgs {
  Args w;          // the nested 4-bit weight (n = N * K values, row-major N x K)
  void* Y;
  int64_t M, N, K;
  int* bad;        // optional device counter of timed-out waits
  int out_dtype;
  int tiles_x;     // activation-row tiles of Y
};

// Three rings: dequantized weight tiles (A operand, written by the producers),
// activation tiles (B operand, TMA) and raw packed weight stages (TMA).  The
// activation ring is deeper where its tiles are small, so its TMA latency
// stays hidden behind several stages of MMAs.
#ifndef DQ4_LIN_AS_SMALL
#define DQ4_LIN_AS_SMALL 8  // weight operand stages for BX <= 64
#endif
#ifndef DQ4_LIN_AS_LARGE
#define DQ4_LIN_AS_LARGE 4  // weight operand stages for BX >= 128
#endif
template <int BX>
struct LinSmem {
  static constexpr int kAS = BX <= 64 ? DQ4_LIN_AS_SMALL : DQ4_LIN_AS_LARGE;
  static constexpr int kXS = BX <= 32 ? 8 : BX == 64 ? 6 : BX == 128 ? 4 : 3;
  // raw weight stages: what the operand rings leave of a 220 KB budget, at most kRaw
  static constexpr int kRawFit = (220 * 1024 - kAS * kBW * kBK * 2 - kXS * BX * kBK * 2) /
                                 kRawBytes;
  static constexpr int kRawS = kRawFit < kRaw ? kRawFit : kRaw;
  static_assert(kRawS >= 4, "raw ring too shallow");
  static constexpr int kA = kBW * kBK * 2;                         // dequantized weight tile
  static constexpr int kB = BX * kBK * 2;                          // activation tile
  static constexpr int kXOff = kAS * kA;
  static constexpr int kRawOff = kXOff + kXS * kB;
  static constexpr int kBarOff = kRawOff + kRawS * kRawBytes;
  // full_w, empty_a per weight stage; full_x, empty_x per activation stage;
  // raw_full, raw_empty per raw stage; acc_full
  static constexpr int kBars = 2 * kAS + 2 * kXS + 2 * kRawS + 1;
  static constexpr int kBytes = kBarOff + 8 * kBars + 16 + 1024;  // + slot, flag, alignment
  static_assert(kBytes <= 227 * 1024, "shared memory budget");
  static_assert(kB % 1024 == 0 && kA % 1024 == 0, "swizzle atoms stay 1024-byte aligned");
};

template <int BX, bool kBF16>
__global__ void __launch_bounds__(kLinThreads, 1)
    dq4_linear_kernel(const __grid_constant__ CUtensorMap tmap_x,
                      const __grid_constant__ CUtensorMap tmap_w, const LinArgs p) {
  using S = LinSmem<BX>;
  constexpr int kAS = S::kAS, kXS = S::kXS, kRawS = S::kRawS;
  constexpr int kOut = kBF16 ? DQ4_OUT_BF16 : DQ4_OUT_F16;
  constexpr uint32_t kTmemCols = BX < 32 ? 32 : BX;  // a power of two >= 32
  constexpr unsigned kFull = 0xFFFFFFFFu;
  extern __shared__ uint8_t smem_raw[];
  __shared__ float s_vcb[16];
  __shared__ float s_scb[256];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(base);
  const uint32_t bar0 = sbase + S::kBarOff;
  auto full_w = [&](int s) { return bar0 + 8 * s; };              // 8 producer warps
  auto empty_a = [&](int s) { return bar0 + 8 * (kAS + s); };     // MMAs reading it done
  auto full_x = [&](int s) { return bar0 + 8 * (2 * kAS + s); };  // activation TMA
  auto empty_x = [&](int s) { return bar0 + 8 * (2 * kAS + kXS + s); };
  auto raw_full = [&](int s) { return bar0 + 8 * (2 * kAS + 2 * kXS + s); };
  auto raw_empty = [&](int s) { return bar0 + 8 * (2 * kAS + 2 * kXS + kRawS + s); };
  const uint32_t acc_full = bar0 + 8 * (2 * kAS + 2 * kXS + 2 * kRawS);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + S::kBarOff + 8 * S::kBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile_w = blockIdx.x / p.tiles_x, tile_x = blockIdx.x % p.tiles_x;
  const int64_t n0 = int64_t(tile_w) * kBW, m0 = int64_t(tile_x) * BX;
  const int kt_count = int(p.K / kBK);
  auto fail = [&]() {
    *abort_flag = 1;
    if (p.bad) atomicAdd(p.bad, 1);
  };

#if DQ4_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
#endif
  if (tid < 16) s_vcb[tid] = __ldg(p.w.vcb + tid);
  for (int k = tid; k < 256; k += kLinThreads) s_scb[k] = __ldg(p.w.scb + k);
  if (warp == 8) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(tmem_slot)), "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    if (lane == 0) {
      for (int s = 0; s < kAS; ++s) {
        mbar_init(full_w(s), kProducerWarps);
        mbar_init(empty_a(s), 1);
      }
      for (int s = 0; s < kXS; ++s) {
        mbar_init(full_x(s), 1);
        mbar_init(empty_x(s), 1);
      }
      for (int s = 0; s < kRawS; ++s) {
        mbar_init(raw_full(s), 1);
        mbar_init(raw_empty(s), kProducerWarps);
      }
      mbar_init(acc_full, 1);
      *abort_flag = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmap_x)));
      asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmap_w)));
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (warp == 9 || warp == 10) {
    if (lane == 0) {
      // ---- TMA streams: warp 9 the packed weight rows n0 .. n0 + 127 (32 bytes = 64
      // values per stage and row), warp 10 the activation rows m0 .. m0 + BX - 1 (64 K
      // per stage).  Tile j goes to slot j % depth once the consumers of tile j - depth
      // released it.
      const bool raw = warp == 9;
      const int depth = raw ? kRawS : kXS;
      const uint64_t tmap = reinterpret_cast<uint64_t>(raw ? &tmap_w : &tmap_x);
      int issued = 0;
      for (; issued < kt_count; ++issued) {
        const int slot = issued % depth;
        if (issued >= depth) {
          if (*abort_flag) break;
          const uint32_t par = ((issued / depth) - 1) & 1;
          if (!mbar_wait(raw ? raw_empty(slot) : empty_x(slot), par)) {
            fail();
            break;
          }
        }
        if (raw)
          tma_2d(sbase + S::kRawOff + slot * kRawBytes, tmap, issued * (kBK / 2), int(n0),
                 raw_full(slot), kRawBytes);
        else
          tma_2d(sbase + S::kXOff + slot * S::kB, tmap, issued * kBK, int(m0), full_x(slot),
                 S::kB);
      }
      if (*abort_flag)  // copies still in flight land before the CTA leaves
        for (int j = issued - 1; j >= 0 && j >= issued - depth; --j)
          mbar_wait(raw ? raw_full(j % depth) : full_x(j % depth), (j / depth) & 1);
    }
  } else if (warp == 8) {
    if (lane == 0) {
      // ---- the MMA issue: stage kt reads weight slot kt % kAS and activation slot
      // kt % kXS, and releases both when its MMAs complete
      const uint32_t idesc = instr_desc<BX>(kBF16);
      for (int kt = 0; kt < kt_count; ++kt) {
        const int sa = kt % kAS, sx = kt % kXS;
        if (*abort_flag) break;
        if (!mbar_wait(full_x(sx), (kt / kXS) & 1) || !mbar_wait(full_w(sa), (kt / kAS) & 1)) {
          fail();
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t a_addr = sbase + sa * S::kA;             // weights: M side
        const uint32_t b_addr = sbase + S::kXOff + sx * S::kB;  // activations: N side
#pragma unroll
        for (int ks = 0; ks < kBK / 16; ++ks) {
          const uint64_t da = smem_desc(a_addr + ks * 32);
          const uint64_t db = smem_desc(b_addr + ks * 32);
          const uint32_t acc = (kt > 0 || ks > 0) ? 1u : 0u;
          asm volatile(
              "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
              :: "r"(tmem), "l"(da), "l"(db), "r"(idesc), "r"(acc));
        }
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
            :: "r"(empty_a(sa)) : "memory");
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
            :: "r"(empty_x(sx)) : "memory");
      }
      // tracks every MMA issued above, aborted or not
      asm volatile(
          "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
          :: "r"(acc_full) : "memory");
      mbar_wait(acc_full, 0);  // no MMA still writes TMEM when it is freed below
    }
  } else {
    // ---- dequantize: thread tid owns weight row r = tid / 2, values 32 h .. 32 h + 31
    // of every 64-value stage (one block, since blocksize >= 32)
    const int r = tid >> 1, h = tid & 1;
    const int64_t n = n0 + r;
    const bool row_ok = n < p.N;
    const float offset = p.w.offset;
    bool failed = false;
    uint32_t cq[kCodeAhead];  // scale code and absmax of stage kt live in slot kt % kCodeAhead
    float aq[kCodeAhead];
    auto fetch = [&](int kt, uint32_t& c, float& a) {
      c = 0;
      a = 0.f;
      if (row_ok) {
        const int64_t b = (n * p.K + int64_t(kt) * kBK + 32 * h) >> p.w.log2_bs;
        c = __ldg(p.w.codes + b);
        a = __ldg(p.w.absmax + (b >> p.w.log2_nbs));
      }
    };
#pragma unroll
    for (int d = 0; d < kCodeAhead; ++d)
      if (d < kt_count) fetch(d, cq[d], aq[d]);
    for (int kb = 0; kb < kt_count && !failed; kb += kCodeAhead) {
#pragma unroll
      for (int d = 0; d < kCodeAhead; ++d) {
        const int kt = kb + d;
        if (kt >= kt_count) break;
        const float sc = __fadd_rn(__fmul_rn(s_scb[cq[d]], aq[d]), offset);  // two roundings
        if (kt + kCodeAhead < kt_count) fetch(kt + kCodeAhead, cq[d], aq[d]);
        const int s = kt % kAS, slot = kt % kRawS;
        bool ok = !*abort_flag && mbar_wait(raw_full(slot), (kt / kRawS) & 1);
        if (ok && kt >= kAS) ok = mbar_wait(empty_a(s), ((kt / kAS) - 1) & 1);
        if (!__all_sync(kFull, ok)) {  // warp-uniform, so the warp stays converged
          failed = true;
          break;
        }
        const uint4 w4 =
            *reinterpret_cast<const uint4*>(base + S::kRawOff + slot * kRawBytes + tid * 16);
        const uint32_t wd[4] = {w4.x, w4.y, w4.z, w4.w};
        uint8_t* sA = base + s * S::kA;
        uint64_t sc2;
        asm("mov.b64 %0, {%1, %1};" : "=l"(sc2) : "f"(sc));
#pragma unroll
        for (int e = 0; e < 4; ++e) {  // 8 values: one 16-byte chunk of the swizzled row
          uint32_t o[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {  // byte j: the high nibble is the earlier value
            const uint32_t byte = (wd[e] >> (8 * j)) & 0xFFu;
            float v0, v1;
            mul2_rn(s_vcb[byte >> 4], s_vcb[byte & 0xFu], sc2, v0, v1);
            o[j] = pack2<kOut>(v0, v1);
          }
          *reinterpret_cast<uint4*>(sA + swz128(r, 4 * h + e)) =
              row_ok ? make_uint4(o[0], o[1], o[2], o[3]) : make_uint4(0, 0, 0, 0);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // visible to the MMA
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(full_w(s));
          mbar_arrive(raw_empty(slot));
        }
      }
    }
    if (failed && lane == 0) fail();
    // ---- epilogue: warps w and w + 4 read TMEM lanes 32 (w % 4) .. (weight rows), each
    // half of the BX accumulator columns (activation rows)
    bool ok = !failed && !*abort_flag && mbar_wait(acc_full, 0);
    if (__all_sync(kFull, ok && !*abort_flag)) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int quad = warp & 3;
      const int64_t ny = n0 + quad * 32 + lane;  // this lane's column of Y
      constexpr int kHalf = BX / 2;
      const int c_begin = (warp >> 2) * kHalf;
#pragma unroll 1
      for (int c = c_begin; c < c_begin + kHalf; c += 8) {
        if (m0 + c >= p.M) break;  // warp-uniform
        uint32_t v[8];
        tmem_ld8(tmem + (static_cast<uint32_t>(quad * 32) << 16) + c, v);
        if (ny >= p.N) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int64_t m = m0 + c + j;
          if (m >= p.M) break;
          const float f = __uint_as_float(v[j]);
          const int64_t o = m * p.N + ny;  // a warp writes 32 consecutive columns of row m
          if (p.out_dtype == DQ4_OUT_F32) {
            static_cast<float*>(p.Y)[o] = f;
          } else if (p.out_dtype == DQ4_OUT_BF16) {
            static_cast<__nv_bfloat16*>(p.Y)[o] = __float2bfloat16_rn(f);
          } else {
            static_cast<__half*>(p.Y)[o] = __float2half_rn(f);
          }
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 8) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(tmem), "r"(kTmemCols));
  }
}

// ------------------------------------------------------------- host side
using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled tensor_map_encoder() {
  static std::once_flag once;
  static EncodeTiled fn = nullptr;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(ptr);
  });
  return fn;
}

template <int BX, bool kBF16>
int launch_linear(const CUtensorMap& tx, const CUtensorMap& tw, const LinArgs& p, int64_t grid,
                  cudaStream_t stream, int dev) {
  using S = LinSmem<BX>;
  auto kernel = dq4_linear_kernel<BX, kBF16>;
  static std::atomic<int> configured[kMaxDevices];
  if (dev >= 0 && dev < kMaxDevices && !configured[dev].load()) {
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes);
    if (e != cudaSuccess) return fail_cuda(DQ4_ERR_LAUNCH, e);
    configured[dev].store(1);
  }
#if DQ4_PDL
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kLinThreads);
  cfg.dynamicSmemBytes = S::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t le = cudaLaunchKernelEx(&cfg, kernel, tx, tw, p);
  if (le != cudaSuccess) {
    cudaGetLastError();
    return fail_cuda(DQ4_ERR_LAUNCH, le);
  }
  return DQ4_OK;
#else
  kernel<<<static_cast<unsigned>(grid), kLinThreads, S::kBytes, stream>>>(tx, tw, p);
  return check_launch();
#endif
}

// Activation rows per CTA.  A CTA spends max(MMA time ~ BX, decode time of its 128 x K
// weight tile ~ 160 in the same units) per round of the grid, so pick the BX with the
// fewest rounds x that, among the powers of two from 16 up to the first one >= M.
int pick_bx(int64_t M, int64_t N, int sms) {
  const int64_t tiles_w = (N + kBW - 1) / kBW;
  int best = 16;
  int64_t best_cost = INT64_MAX;
  for (int bx = 16; bx <= 256; bx *= 2) {
    const int64_t tiles = tiles_w * ((M + bx - 1) / bx);
    const int64_t rounds = (tiles + sms - 1) / sms;
    const int64_t cost = rounds * (bx > 160 ? bx : 160);
    if (cost < best_cost) {
      best_cost = cost;
      best = bx;
    }
    if (bx >= M) break;
  }
  return best;
}

template <bool kBF16>
int launch_bx(int bx, const CUtensorMap& tx, const CUtensorMap& tw, const LinArgs& p,
              int64_t grid, cudaStream_t st, int dev) {
  switch (bx) {
    case 16: return launch_linear<16, kBF16>(tx, tw, p, grid, st, dev);
    case 32: return launch_linear<32, kBF16>(tx, tw, p, grid, st, dev);
    case 64: return launch_linear<64, kBF16>(tx, tw, p, grid, st, dev);
    case 128: return launch_linear<128, kBF16>(tx, tw, p, grid, st, dev);
    default: return launch_linear<256, kBF16>(tx, tw, p, grid, st, dev);
  }
}

}  // namespace
}  // namespace dq4d

using namespace dq4d;

extern "C" {

int dq4_nested_linear(const void* X, int32_t in_dtype, const uint8_t* packed,
                      const uint8_t* scale_codes, const float* nested_absmax,
                      const float* scale_codebook, const float* value_codebook, float offset,
                      int64_t M, int64_t N, int64_t K, int32_t blocksize,
                      int32_t nested_blocksize, int32_t out_dtype, void* Y, int* bad,
                      void* stream) {
  if (M < 0 || N < 0 || K < 0) return DQ4_ERR_N;
  if (in_dtype != DQ4_OUT_F16 && in_dtype != DQ4_OUT_BF16) return DQ4_ERR_DTYPE;
  if (N > 0 && K > INT64_MAX / N) return DQ4_ERR_N;
  if (int st = validate(N * K, blocksize, nested_blocksize, true, out_dtype)) return st;
  if (M == 0 || N == 0) return DQ4_OK;
  if (K == 0 || K % kBK != 0 || M > INT32_MAX || N > INT32_MAX || K > INT32_MAX)
    return DQ4_ERR_N;
  if (!X || !packed || !scale_codes || !nested_absmax || !scale_codebook || !value_codebook ||
      !Y)
    return DQ4_ERR_NULL;
  if (misaligned(X, 16) || misaligned(packed, 16) || misaligned(nested_absmax, 4) ||
      misaligned(scale_codebook, 4) || misaligned(value_codebook, 4) ||
      misaligned(Y, out_itemsize(out_dtype)) || misaligned(bad, 4))
    return DQ4_ERR_ALIGN;
  int dev = 0, sms = 0;
  if (int st = current_device(&dev, &sms)) return st;
  EncodeTiled encode = tensor_map_encoder();
  if (!encode) return fail_cuda(DQ4_ERR_LAUNCH, cudaErrorNotSupported);

  const int bx = pick_bx(M, N, sms);
  const int64_t tiles_x = (M + bx - 1) / bx, tiles_w = (N + kBW - 1) / kBW;
  if (tiles_x * tiles_w > INT32_MAX) return DQ4_ERR_N;
  const cuuint32_t estride[2] = {1, 1};
  // X as a 2-D tensor (K fastest, M rows): 64 x bx boxes, 128-byte swizzle, rows past M
  // read as zero
  CUtensorMap tx;
  const cuuint64_t xdim[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
  const cuuint64_t xstride[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t xbox[2] = {kBK, static_cast<cuuint32_t>(bx)};
  CUresult cr = encode(&tx,
                       in_dtype == DQ4_OUT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                       2, const_cast<void*>(X), xdim, xstride, xbox, estride,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return fail_cuda(DQ4_ERR_LAUNCH, cudaErrorInvalidValue);
  // the packed weight as N rows of K / 2 bytes: 32 x 128 boxes, unswizzled
  CUtensorMap tw;
  const cuuint64_t wdim[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(N)};
  const cuuint64_t wstride[1] = {static_cast<cuuint64_t>(K / 2)};
  const cuuint32_t wbox[2] = {kBK / 2, kBW};
  cr = encode(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(packed), wdim,
              wstride, wbox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (cr != CUDA_SUCCESS) return fail_cuda(DQ4_ERR_LAUNCH, cudaErrorInvalidValue);

  LinArgs p;
  p.w = make_args(packed, scale_codes, nested_absmax, scale_codebook, value_codebook, offset,
                  N * K, blocksize, nested_blocksize, nullptr);
  p.Y = Y;
  p.M = M;
  p.N = N;
  p.K = K;
  p.bad = bad;
  p.out_dtype = out_dtype;
  p.tiles_x = static_cast<int>(tiles_x);
  const auto st = static_cast<cudaStream_t>(stream);
  const int64_t grid = tiles_x * tiles_w;
  return in_dtype == DQ4_OUT_BF16 ? launch_bx<true>(bx, tx, tw, p, grid, st, dev)
                                  : launch_bx<false>(bx, tx, tw, p, grid, st, dev);
}

}  // extern "C"

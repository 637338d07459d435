// Row-blocked dequantization fused into a tcgen05 GEMM with FP32 accuracy:
// dq4_nested_out_prod, dst[cols, ncols] = W^T G, W the FP32 dequantization of a rows x cols
// nested 4-bit weight (dq4_nested's values, row-major) and G a rows x ncols FP32 matrix, the
// sum running over W's rows.  Source: "cuda: out_prod dequantizes a 2D weight in row blocks"
// (llama.cpp pull request #4), section "What": the weight's row blocks go through the same
// F32 dequantization and a GEMM accumulates them into dst block after block, so the whole
// dequantized weight never exists at once.  Here the row blocks are 64-row stages decoded
// inside the GEMM kernel, so no dequantized block is written either.
//
// FP32 accuracy on the BF16 tensor cores: an FP32 value x splits exactly into three BF16
// terms x = x0 + x1 + x2 (x0 = x with its low 16 bits cleared, x1 likewise for x - x0,
// x2 = x - x0 - x1, which has at most 8 significant bits).  dst accumulates in FP32 the six
// products W_i G_j with i + j <= 2; the three dropped ones are below 2^-24 of W G.  With G
// holding a single 1 per column, dst holds W's values exactly (their three terms sum back
// exactly), which pins the in-kernel decoding bit for bit.
//
// A CTA owns 128 columns of W (the MMA's M side, TMEM lanes) and NB <= 128 columns of G (its
// N side) over a range of rows (K); the ranges split the rows so that the CTAs fill the SMs.
// Seventeen warps:
//  * warps 0..15, two groups of eight taking alternate 64-row stages, each group with its
//    own stage slot.  A group first stages the stage's inputs in shared memory (G's rows, and
//    per row of W's tile its packed bytes, scale codes and absmax, by cp.async, all in flight
//    at once) and computes each row's nested scales (separately rounded FP32 multiply and
//    add).  Then a thread decodes W column c0 + t over half the stage's rows (warps w and
//    w + 4 share a TMEM lane quadrant; nibble, FP32 product with the row's scale) into the
//    three BF16 terms, two rows per 32-bit TMEM column, written to the slot's A planes in
//    TMEM, and splits half the stage's rows of one G column into three BF16 planes,
//    transposed to the K-major 128-byte-swizzled layout of the MMA's B operand in shared
//    memory.  Every 8 stages (a chain) the threads add the accumulator into running FP32 sums
//    they hold in registers (the tensor pipe's accumulation loses up to about an ulp per MMA,
//    so chains stay short), and after the last chain they store the sums to the CTA's
//    output tile (dst, or the partial tile of their row range);
//  * warp 16 allocates the TMEM; its lane 0 issues the 24 MMAs of a stage (4 K steps of 16 x
//    6 products, A from TMEM, B from shared memory) into the chain's accumulator buffer (two
//    alternate) and commits the slot back.
// With several row ranges, a second kernel adds the partial tiles in range order
// (deterministic).  Waits on mbarriers are bounded; a wait that runs out counts into *bad
// and the CTA leaves its loops, waits for its MMAs and frees its TMEM.
#include "common.cuh"
#include "tcgen05.cuh"
#include "tmap.cuh"

#include <atomic>

namespace dq4d {
namespace {

constexpr int kOpM = 128;       // W columns per CTA = MMA M = TMEM lanes
constexpr int kOpK = 64;        // rows per stage: 64 BF16 = one 128-byte swizzle row
constexpr int kOpPlanes = 3;    // BF16 terms of an FP32 value
constexpr int kOpGroups = 2;    // producer groups, each with one stage slot
// Stages accumulated in one TMEM accumulator (a chain) before the producers add it into
// their running FP32 sums.  The tensor pipe's FP32 accumulation loses up to about an ulp
// of the accumulator per MMA, so a chain as long as the whole row range would cost
// accuracy on long sums (3e-4 relative at 50000 rows in one chain, measured); chains of
// 8 stages (192 MMAs) keep the error at a few 1e-6.
constexpr int kOpChain = 8;
constexpr int kOpGroupWarps = 8;  // warps per producer group (two per TMEM lane quadrant)
constexpr int kOpGroupThreads = 32 * kOpGroupWarps;
constexpr int kOpMmaWarp = kOpGroups * kOpGroupWarps;
constexpr int kOpThreads = 32 * (kOpMmaWarp + 1);
constexpr uint32_t kOpTmemCols = 512;
constexpr uint32_t kOpATmem = 256;  // the A planes' first TMEM column (the accumulator: 0..NB-1)
constexpr int kOpAPlaneCols = kOpK / 2;                       // 32-bit columns of one A plane
constexpr int kOpASlotCols = kOpPlanes * kOpAPlaneCols;       // 96
static_assert(kOpATmem + kOpGroups * kOpASlotCols <= kOpTmemCols, "A slots fit TMEM");
// The six products W_i G_j (i + j <= 2), smallest first.
__device__ constexpr int kOpPassW[6] = {2, 1, 0, 1, 0, 0};
__device__ constexpr int kOpPassG[6] = {0, 1, 2, 0, 1, 0};

template <int NB, bool kTma>
struct OpSmem {
  static_assert(NB == 16 || NB == 32 || NB == 64 || NB == 128, "N tile");
  static constexpr int kPlane = NB * 128;  // one B plane: NB rows (G columns) x 64 BF16
  static constexpr int kSlot = kOpPlanes * kPlane;
  // A group's staging of one stage's inputs: the G rows (kOpK x NB FP32), and per row of W's
  // tile its packed bytes (17 aligned words by cp.async: 128 nibbles from any start; with
  // kTma one 64-byte TMA box row, the rows starting on 32-value boundaries), scale codes
  // (2 aligned words: at most 5 blocks of >= 32 values) and absmax (8 aligned floats: at
  // most 5 groups)
  static constexpr int kGRowBytes = NB * 4;
  static constexpr int kWRowBytes = kTma ? 64 : 68, kCRowBytes = 8, kARowBytes = 32;
  static constexpr int kGOff = 0;
  static constexpr int kWOff = kGOff + kOpK * kGRowBytes;
  static constexpr int kCOff = kWOff + kOpK * kWRowBytes;
  static constexpr int kAOff = kCOff + kOpK * kCRowBytes;
  // then the row's nested scales, one per block it touches (at most 5), from block
  // (first block) on
  static constexpr int kSOff = kAOff + kOpK * kARowBytes;
  static constexpr int kSRowBytes = 32;
  // (1024-byte aligned: TMA boxes land at its start)
  static constexpr int kStage = (kSOff + kOpK * kSRowBytes + 1023) / 1024 * 1024;
  static constexpr int kStageOff = kOpGroups * kSlot;
  static constexpr int kBarOff = kStageOff + kOpGroups * kStage;
  // accumulator buffers in TMEM (columns b NB ..): two when they fit beside the A slots, so
  // a chain is added into the output while the next one accumulates
  static constexpr int kAccBufs = 2;
  static_assert(kAccBufs * NB <= int(kOpATmem), "accumulators fit before the A slots");
  // full and empty per slot; acc_full and acc_empty per accumulator buffer; acc_done; the
  // TMA staging's completion per group
  static constexpr int kBars = 2 * kOpGroups + 2 * kAccBufs + 1 + kOpGroups;
  static constexpr int kUsed = kBarOff + 8 * kBars + 1024;  // + alignment slack
  // more than half an SM's shared memory: one CTA per SM, so the 512-column TMEM
  // allocation never waits for another CTA
  static constexpr int kBytes = kUsed > 118 * 1024 ? kUsed : 118 * 1024;
  static_assert(kBytes + 1280 <= 227 * 1024, "shared memory budget");
};

struct OpArgs {
  Args w;                 // the nested weight, n = rows * cols values
  const float* G;         // rows x ncols
  float* out;             // dst (one row range) or the partial tiles [ranges][cols][ncols]
  int64_t rows, cols, ncols;
  int64_t rows_per_range;  // a multiple of kOpK
  int tiles_c;            // W-column tiles (blockIdx.x = tile_j * tiles_c + tile_c)
  int g_vec4;             // G's rows start 16-byte aligned (ncols % 4 == 0, G aligned)
  // every row of W starts on an 8-value word and meets the scale blocks at the same column
  // offsets (cols % 8 == 0, and cols % blocksize == 0 or blocksize % cols == 0)
  int rows_alike;
  int* bad;               // optional device counter of timed-out waits
};

// Asynchronous 4- and 16-byte copies from global to shared memory (cp.async), their
// commit and the wait for all of a thread's copies.
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ uint32_t ld_shared_u8(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

// Word wi (4 bytes from 4 wi) of a byte array of `size` bytes into shared memory at dst:
// an asynchronous copy when it lies inside the array, its bytes one by one when it straddles
// the end, nothing past it (those bytes are never read).
__device__ __forceinline__ void stage_word(uint32_t dst, const uint8_t* base, int64_t wi,
                                           int64_t size) {
  const int64_t b = 4 * wi;
  if (b + 4 <= size) {
    cp_async4(dst, base + b);
  } else if (b < size) {
    uint32_t v = 0;
    for (int k = 0; k < 4 && b + k < size; ++k) v |= uint32_t(__ldg(base + b + k)) << (8 * k);
    asm volatile("st.shared.b32 [%0], %1;" :: "r"(dst), "r"(v) : "memory");
  }
}

// The high 16 bits of two FP32 words, a's in the low half: two BF16 values (each word
// exactly a BF16 value) in one 32-bit TMEM column or shared-memory word.
__device__ __forceinline__ uint32_t hi_pair(uint32_t a, uint32_t b) {
  return __byte_perm(a, b, 0x7632);
}

// x = t0 + t1 + t2 exactly, each term a BF16 value kept in an FP32 word.
__device__ __forceinline__ void split3(float x, uint32_t& t0, uint32_t& t1, uint32_t& t2) {
  const uint32_t u = __float_as_uint(x);
  t0 = u & 0xFFFF0000u;
  const float r = __fsub_rn(x, __uint_as_float(t0));  // exact: x's low 16 significand bits
  t1 = __float_as_uint(r) & 0xFFFF0000u;
  t2 = __float_as_uint(__fsub_rn(r, __uint_as_float(t1)));  // exact, at most 8 bits
}

template <int NB, bool kTma>
__global__ void __launch_bounds__(kOpThreads, 1)
    dq4_outprod_kernel(const __grid_constant__ CUtensorMap tm_g,
                       const __grid_constant__ CUtensorMap tm_w, const OpArgs p) {
  using S = OpSmem<NB, kTma>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ float s_scb[256];
  __shared__ float s_vcb[16];
  __shared__ uint32_t s_tmem;
  __shared__ volatile int s_abort;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(base);
  const uint32_t bar0 = sbase + S::kBarOff;
  auto full = [&](int s) { return bar0 + 8 * s; };                 // a group's stage written
  auto empty = [&](int s) { return bar0 + 8 * (kOpGroups + s); };  // its MMAs completed
  constexpr int kAccBufs = S::kAccBufs;
  // acc_full(b): the chain in buffer b is final; acc_empty(b): both groups added it out
  auto acc_full = [&](int b) { return bar0 + 8 * (2 * kOpGroups + b); };
  auto acc_empty = [&](int b) { return bar0 + 8 * (2 * kOpGroups + kAccBufs + b); };
  const uint32_t acc_done = bar0 + 8 * (2 * kOpGroups + 2 * kAccBufs);
  // staged(g): the TMA boxes of group g's current stage landed (kTma)
  auto staged = [&](int g) { return bar0 + 8 * (2 * kOpGroups + 2 * kAccBufs + 1 + g); };
  volatile int* abort_flag = &s_abort;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto fail = [&]() {
    *abort_flag = 1;
    if (p.bad) atomicAdd(p.bad, 1);
  };

  const int tile_c = int(blockIdx.x) % p.tiles_c, tile_j = int(blockIdx.x) / p.tiles_c;
  const int64_t c0 = int64_t(tile_c) * kOpM, j0 = int64_t(tile_j) * NB;
  const int64_t r_begin = int64_t(blockIdx.y) * p.rows_per_range;
  const int64_t r_end = min(p.rows, r_begin + p.rows_per_range);
  const int nst = r_end > r_begin ? int((r_end - r_begin + kOpK - 1) / kOpK) : 0;

  if (warp == kOpMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(&s_tmem)), "r"(kOpTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    if (lane == 0) {
      for (int s = 0; s < kOpGroups; ++s) {
        mbar_init(full(s), kOpGroupWarps);  // the group's warps
        mbar_init(empty(s), 1);
      }
      for (int b = 0; b < kAccBufs; ++b) {
        mbar_init(acc_full(b), 1);
        mbar_init(acc_empty(b), kOpMmaWarp);  // every producer warp
      }
      mbar_init(acc_done, 1);
      for (int g = 0; g < kOpGroups; ++g) mbar_init(staged(g), 1);
      *abort_flag = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      if (kTma) {
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tm_g)));
        asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tm_w)));
      }
    }
  } else if (tid < 256) {
    static_assert(kOpMmaWarp * 32 >= 256, "the producers load the scale codebook");
    s_scb[tid] = __ldg(p.w.scb + tid);
    if (tid < 16) s_vcb[tid] = __ldg(p.w.vcb + tid);
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = s_tmem;

  if (warp == kOpMmaWarp) {
    if (lane == 0) {
      // ---- 4 K steps x 6 products per stage; chain k (stages k kOpChain ..) accumulates in
      // buffer k % kAccBufs, which the producers must have added out for chain k - kAccBufs
      const uint32_t idesc = instr_desc_f16<kOpM, NB>(true);
      for (int l = 0; l < nst; ++l) {
        const int slot = l & 1, k = l / kOpChain, b = k % kAccBufs;
        const bool chain_first = l % kOpChain == 0;
        const bool chain_last = l % kOpChain == kOpChain - 1 || l == nst - 1;
        if (*abort_flag || !mbar_wait(full(slot), uint32_t(l >> 1) & 1u) ||
            (chain_first && k >= kAccBufs &&
             !mbar_wait(acc_empty(b), uint32_t(k / kAccBufs - 1) & 1u))) {
          if (!*abort_flag) fail();
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t d = tmem + b * NB;
        const uint32_t a_slot = tmem + kOpATmem + slot * kOpASlotCols;
        const uint32_t b_slot = sbase + slot * S::kSlot;
#pragma unroll
        for (int ks = 0; ks < kOpK / 16; ++ks) {
#pragma unroll
          for (int q = 0; q < 6; ++q) {
            const uint32_t a = a_slot + kOpPassW[q] * kOpAPlaneCols + ks * 8;
            const uint64_t db = smem_desc(b_slot + kOpPassG[q] * S::kPlane + ks * 32);
            const uint32_t acc = (chain_first && ks == 0 && q == 0) ? 0u : 1u;
            asm volatile(
                "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
                :: "r"(d), "r"(a), "l"(db), "r"(idesc), "r"(acc));
          }
        }
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
            :: "r"(empty(slot)) : "memory");
        if (chain_last)
          asm volatile(
              "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
              :: "r"(acc_full(b)) : "memory");
      }
      // tracks every MMA issued above: no MMA still writes TMEM when it is freed
      asm volatile(
          "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
          :: "r"(acc_done) : "memory");
      mbar_wait(acc_done, 0);
    }
  } else {
    // ---- producers: group g takes stages g, g + 2, .. into slot g
    // warp gw of group g: TMEM lane quadrant quad = gw % 4, row half hf = gw / 4 (warps gw
    // and gw + 4 take the first and last 32 rows of a stage for the same W columns)
    const int group = warp / kOpGroupWarps, gw = warp % kOpGroupWarps;
    const int quad = gw & 3, hf = gw >> 2;
    const int t = quad * 32 + lane;     // this thread's W column (TMEM lane)
    const int tg = gw * 32 + lane;      // its index in the group
    const int64_t c = c0 + t;
    const bool c_ok = c < p.cols;
    const float offset = p.w.offset;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(quad * 32) << 16) + kOpATmem +
                            group * kOpASlotCols;
    const uint32_t b_slot = sbase + group * S::kSlot;
    // Chain k added into this thread's share of the running FP32 sum (round to nearest, in
    // chain order): warp w reads TMEM lanes 32 (w % 4) .. (W columns c), a quarter of the
    // NB accumulator columns (G columns j; the group's half, split between the quadrant's
    // two warps, one of them alone when the half is 8 columns).  Both groups add chain k
    // before the MMAs reuse its buffer.  The sums go to the CTA's output tile (dst, or its
    // row range's partial tile) once, after the last chain.
    constexpr int kHalfN = NB / 2;
    constexpr int kQuarterN = kHalfN >= 16 ? kHalfN / 2 : kHalfN;
    const int jb = group * kHalfN + hf * kQuarterN;
    const bool reads = hf * kQuarterN < kHalfN;  // warp-uniform
    float run[kQuarterN];
#pragma unroll
    for (int e = 0; e < kQuarterN; ++e) run[e] = 0.f;
    auto flush = [&](int k) -> bool {
      const int b = k % kAccBufs;
      const bool got = __all_sync(0xFFFFFFFFu, !*abort_flag &&
                                                   mbar_wait(acc_full(b), uint32_t(k / kAccBufs) & 1u) &&
                                                   !*abort_flag);
      if (!got) {
        if (lane == 0 && !*abort_flag) fail();
        return false;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      if (reads) {
#pragma unroll
        for (int cc = 0; cc < kQuarterN; cc += 8) {
          uint32_t v[8];
          tmem_ld<8>(tmem + (static_cast<uint32_t>(quad * 32) << 16) + b * NB + jb + cc, v);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            run[cc + e] = k == 0 ? __uint_as_float(v[e]) : __fadd_rn(run[cc + e], __uint_as_float(v[e]));
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(acc_empty(b));
      return true;
    };
    int flushed = 0;  // chains this group has added out
    const int nchains = (nst + kOpChain - 1) / kOpChain;
    // This group's staging: its threads (tg = t) copy a stage's inputs in, one barrier of the
    // group's 128 threads (named barrier 1 + group) later every thread reads any of them.
    const uint32_t stg = sbase + S::kStageOff + group * S::kStage;
    auto group_bar = [&]() {
      asm volatile("bar.sync %0, %1;" :: "r"(1 + group), "n"(kOpGroupThreads) : "memory");
    };
    // the same barrier, returning whether any of the group's threads passed `mine` true
    auto group_bar_any = [&](bool mine) -> bool {
      uint32_t any;
      asm volatile(
          "{\n.reg .pred p, q;\nsetp.ne.u32 q, %1, 0;\n"
          "bar.red.or.pred p, %2, %3, q;\nselp.u32 %0, 1, 0, p;\n}"
          : "=r"(any) : "r"(mine ? 1u : 0u), "r"(1 + group), "n"(kOpGroupThreads) : "memory");
      return any != 0;
    };
    const int64_t npk = (p.w.n + 1) / 2, nblk = (p.w.n + (int64_t(1) << p.w.log2_bs) - 1) >>
                                               p.w.log2_bs;
    const int64_t ngrp = (nblk + (int64_t(1) << p.w.log2_nbs) - 1) >> p.w.log2_nbs;
    bool tma_pending = false;  // (thread tg 0) a stage's boxes are in flight, not yet waited for
    int tma_l = 0;             // (thread tg 0) the local stage they belong to
    auto stage_in = [&](int64_t r0) {
      // G rows r0 .. r0 + 63, columns j0 .. j0 + NB - 1 (rows and columns past the ends are
      // left alone, or with kTma zero-filled past the matrix: a whole stage of rows reads
      // them only into dst columns that are never stored, a partial one selects zeros); with
      // kTma also W's packed rows, one box each, completing on staged(group)
      if constexpr (kTma) {
        if (tg == 0) {
          mbar_expect(staged(group), kOpK * S::kGRowBytes + kOpK * S::kWRowBytes);
          tma_load_2d(stg + S::kGOff, reinterpret_cast<uint64_t>(&tm_g), int(j0), int(r0),
                      staged(group));
          tma_load_2d(stg + S::kWOff, reinterpret_cast<uint64_t>(&tm_w), int(c0 / 2), int(r0),
                      staged(group));
          tma_pending = true;
        }
      } else if (p.g_vec4) {
        for (int q = tg; q < kOpK * NB / 4; q += kOpGroupThreads) {
          const int rr = q / (NB / 4), jq = q - rr * (NB / 4);
          const int64_t r = r0 + rr, j = j0 + 4 * jq;
          if (r < r_end && j < p.ncols)
            cp_async16(stg + S::kGOff + rr * S::kGRowBytes + 16 * jq, p.G + r * p.ncols + j);
        }
      } else {
        for (int q = tg; q < kOpK * NB; q += kOpGroupThreads) {
          const int rr = q / NB, jl = q - rr * NB;
          const int64_t r = r0 + rr, j = j0 + jl;
          if (r < r_end && j < p.ncols)
            cp_async4(stg + S::kGOff + rr * S::kGRowBytes + 4 * jl, p.G + r * p.ncols + j);
        }
      }
      // per row of W's tile: packed bytes, scale codes and absmax, from aligned words; four
      // threads per row (packed words 0..5, 6..11, 12..16; the codes and the absmax)
      {
        static_assert(kOpGroupThreads == 4 * kOpK, "four staging threads per row");
        const int rr = tg >> 2, part = tg & 3;
        const int64_t r = r0 + rr;
        if (r < r_end) {
          const int64_t i0 = r * p.cols + c0;  // the tile row's first value
          const int64_t b0 = i0 >> p.w.log2_bs;
          const uint32_t wrow = stg + S::kWOff + rr * S::kWRowBytes;
          if (kTma) {  // the codes and two halves of the absmax words, one part each
            const int64_t a0 = (b0 >> p.w.log2_nbs) & ~int64_t(3);
            if (part == 0) {
              for (int k = 0; k < 2; ++k)
                stage_word(stg + S::kCOff + rr * S::kCRowBytes + 4 * k, p.w.codes,
                           (b0 >> 2) + k, nblk);
            } else if (part < 3) {
              for (int k = 4 * (part - 1); k < 4 * part; ++k)
                if (a0 + k < ngrp)
                  cp_async4(stg + S::kAOff + rr * S::kARowBytes + 4 * k, p.w.absmax + a0 + k);
            }
          } else if (part < 3) {
            for (int k = part * 6; k < (part < 2 ? part * 6 + 6 : 17); ++k)
              stage_word(wrow + 4 * k, p.w.packed, (i0 >> 3) + k, npk);
          } else {
            for (int k = 0; k < 2; ++k)
              stage_word(stg + S::kCOff + rr * S::kCRowBytes + 4 * k, p.w.codes, (b0 >> 2) + k,
                         nblk);
            const int64_t a0 = (b0 >> p.w.log2_nbs) & ~int64_t(3);
            for (int k = 0; k < 8; ++k)
              if (a0 + k < ngrp)
                cp_async4(stg + S::kAOff + rr * S::kARowBytes + 4 * k, p.w.absmax + a0 + k);
          }
        }
      }
      cp_async_commit();
    };
    bool ok = true;
    for (int l = group; l < nst && ok; l += kOpGroups) {
      const int64_t r0 = r_begin + int64_t(l) * kOpK;
      group_bar();  // every thread of the group is done with the previous stage's staging
      stage_in(r0);
      if (kTma) tma_l = l;
      // the chains before that of stage l - 2 (whose slot this stage reuses): added out one
      // chain after they completed, so the MMAs, which need a buffer back kAccBufs chains
      // later, find it free (the MMAs of those chains were issued: their stages are decoded)
      bool wok = true;  // this warp's waits of this stage (warp-uniform)
      for (const int need = (l >= kOpGroups ? (l - kOpGroups) / kOpChain : 0) - 1;
           wok && flushed <= need; ++flushed)
        wok = flush(flushed);
      if (wok && l >= kOpGroups) {  // the MMAs of this slot's previous stage completed
        wok = __all_sync(0xFFFFFFFFu,
                         !*abort_flag && mbar_wait(empty(group), uint32_t((l >> 1) - 1) & 1u));
        if (wok)
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        else if (lane == 0 && !*abort_flag)
          fail();
      }
      cp_async_wait_all();
      if (kTma && wok) {  // the stage's boxes landed (every thread acquires them)
        wok = __all_sync(0xFFFFFFFFu, mbar_wait(staged(group), uint32_t(l >> 1) & 1u));
        if (tg == 0 && wok) tma_pending = false;
        if (!wok && lane == 0 && !*abort_flag) fail();
      }
      // every thread's copies landed: the group's barrier, which also ORs the warps' failed
      // waits, so the group's warps leave their loop together (a warp that left alone would
      // leave the others waiting at the next group barrier)
      if (group_bar_any(!wok)) {
        ok = false;
        break;
      }
      // each row's nested scales (separately rounded FP32 multiply and add), for the blocks
      // b0 + k it touches: 64 rows x 5 blocks over the group's threads
      for (int q = tg; q < kOpK * 5; q += kOpGroupThreads) {
        const int rr = q / 5, k = q - rr * 5;
        const int64_t r = r0 + rr;
        if (r >= r_end) continue;
        const int64_t b0 = (r * p.cols + c0) >> p.w.log2_bs, b = b0 + k;
        if (b >= nblk) continue;
        const uint32_t code = ld_shared_u8(stg + S::kCOff + rr * S::kCRowBytes +
                                           uint32_t(b - ((b0 >> 2) << 2)));
        const float am = ld_shared_f32(
            stg + S::kAOff + rr * S::kARowBytes +
            4 * uint32_t((b >> p.w.log2_nbs) - ((b0 >> p.w.log2_nbs) & ~int64_t(3))));
        asm volatile("st.shared.f32 [%0], %1;"
                     :: "r"(stg + S::kSOff + rr * S::kSRowBytes + 4 * k),
                        "f"(__fadd_rn(__fmul_rn(s_scb[code], am), offset)) : "memory");
      }
      group_bar();  // the scales are in
      // W column c over this warp's 32 rows of the stage, 16 rows (8 TMEM columns per
      // plane) at a time:
      // with m8 = the row's first value's offset in its aligned 8-value word and mb = its
      // offset in its block, value c0 + t sits in byte (m8 + t) / 2 of the staged words and
      // in block (mb + t) >> log2 blocksize of the row's scales.  The staged bytes and scales
      // are read with plain loads (no shared-memory store comes between them and the
      // barrier above), so the compiler may issue a batch's loads together.
      const uint8_t* st_p = base + (stg - sbase);
      const int rows_left = r_end - r0 < kOpK ? int(r_end - r0) : kOpK;
      const uint32_t i0s = uint32_t(r0 * p.cols + c0);  // low bits suffice
      const uint32_t cols32 = uint32_t(p.cols), bs_mask = (1u << p.w.log2_bs) - 1u;
      // A whole stage of alike rows: value t of every row sits at byte t / 2 of its staged
      // word run (c0 and the rows start on 8-value words) and in the same slot of its scales,
      // so the row loop needs no per-row index arithmetic.  Columns past cols then decode
      // staged bytes of no meaning, into TMEM lanes whose sums are never stored.
      const bool fast = p.rows_alike && rows_left == kOpK;  // uniform across the group
      const uint8_t* w_t = st_p + S::kWOff + (t >> 1);
      const uint32_t nib_shift = (t & 1) ? 0u : 4u;
      const float* s_t = reinterpret_cast<const float*>(st_p + S::kSOff) +
                         (p.cols % (int64_t(1) << p.w.log2_bs) == 0
                              ? (((uint32_t(c0) & bs_mask) + uint32_t(t)) >> p.w.log2_bs)
                              : 0u);
#pragma unroll 1
      for (int h = 2 * hf; h < 2 * hf + 2; ++h) {
        float v[16];
        if (fast) {
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int rr = h * 16 + q;
            const uint32_t nib = (uint32_t(w_t[rr * S::kWRowBytes]) >> nib_shift) & 0xFu;
            v[q] = __fmul_rn(s_vcb[nib], s_t[rr * (S::kSRowBytes / 4)]);
          }
        } else {
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const int rr = h * 16 + q;
            const uint32_t i0lo = i0s + uint32_t(rr) * cols32;
            const uint32_t m8 = (i0lo & 7u) + uint32_t(t);
            const uint32_t mb = (i0lo & bs_mask) + uint32_t(t);
            const uint32_t byte = st_p[S::kWOff + rr * S::kWRowBytes + (m8 >> 1)];
            const uint32_t nib = (m8 & 1u) ? (byte & 0xFu) : (byte >> 4);
            const float sc = *reinterpret_cast<const float*>(
                st_p + S::kSOff + rr * S::kSRowBytes + 4 * (mb >> p.w.log2_bs));
            v[q] = (c_ok && rr < rows_left) ? __fmul_rn(s_vcb[nib], sc) : 0.f;
          }
        }
        uint32_t t0[8], t1[8], t2[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          uint32_t e0[2], e1[2], e2[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) split3(v[2 * k + e], e0[e], e1[e], e2[e]);
          t0[k] = hi_pair(e0[0], e0[1]);
          t1[k] = hi_pair(e1[0], e1[1]);
          t2[k] = hi_pair(e2[0], e2[1]);
        }
        tmem_st<8>(t_lane + 0 * kOpAPlaneCols + h * 8, t0);
        tmem_st<8>(t_lane + 1 * kOpAPlaneCols + h * 8, t1);
        tmem_st<8>(t_lane + 2 * kOpAPlaneCols + h * 8, t2);
      }
      // G column j0 + jl over kGChunks of the stage's 8 chunks of 8 rows (thread tg: column
      // tg % NB, chunks kGChunks (tg / NB) ..; every thread of the group takes a share when
      // NB >= 32), split and transposed: plane row jl = the G column, 64 BF16 of K = 128
      // bytes, 16-byte chunk w stored at w ^ (jl & 7) within the 1024-byte group of 8 rows.
      // A chunk's 8 values are loaded before its plane stores.
      {
        constexpr int kTpc = kOpGroupThreads / NB < 8 ? kOpGroupThreads / NB : 8;
        constexpr int kGChunks = 8 / kTpc;
        if (tg < NB * kTpc) {
          const int jl = tg % NB, w0 = (tg / NB) * kGChunks;
          const bool j_ok = j0 + jl < p.ncols;
          const uint32_t row = b_slot + (jl >> 3) * 1024 + (jl & 7) * 128;
          const float* gp = reinterpret_cast<const float*>(st_p + S::kGOff) + jl;
          constexpr int kBatch = kGChunks < 2 ? kGChunks : 2;  // chunks loaded together
#pragma unroll
          for (int wb = 0; wb < kGChunks; wb += kBatch) {
          float g[8 * kBatch];
#pragma unroll
          for (int q = 0; q < 8 * kBatch; ++q) {
            const int rr = 8 * (w0 + wb) + q;
            const float x = gp[rr * (S::kGRowBytes / 4)];
            // (a whole stage keeps columns past ncols as staged: they feed only dst
            // columns that are never stored)
            g[q] = (rows_left == kOpK || (j_ok && rr < rows_left)) ? x : 0.f;
          }
#pragma unroll
          for (int wq = 0; wq < kBatch; ++wq) {
            const int w = w0 + wb + wq;
            uint32_t q0[4], q1[4], q2[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              uint32_t e0[2], e1[2], e2[2];
#pragma unroll
              for (int e = 0; e < 2; ++e) split3(g[8 * wq + 2 * k + e], e0[e], e1[e], e2[e]);
              q0[k] = hi_pair(e0[0], e0[1]);
              q1[k] = hi_pair(e1[0], e1[1]);
              q2[k] = hi_pair(e2[0], e2[1]);
            }
            const uint32_t off = row + ((w ^ (jl & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                         :: "r"(off), "r"(q0[0]), "r"(q0[1]), "r"(q0[2]), "r"(q0[3]) : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                         :: "r"(off + S::kPlane), "r"(q1[0]), "r"(q1[1]), "r"(q1[2]), "r"(q1[3])
                         : "memory");
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                         :: "r"(off + 2 * S::kPlane), "r"(q2[0]), "r"(q2[1]), "r"(q2[2]),
                            "r"(q2[3]) : "memory");
          }
          }
        }
      }
      // the B planes (generic writes) visible to the MMAs (async proxy), the A planes'
      // TMEM stores complete, then the group's warps arrive
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(full(group));
    }
    // boxes still in flight after a failed wait land before the CTA leaves
    if (kTma && tma_pending) mbar_wait(staged(group), uint32_t(tma_l >> 1) & 1u);
    // the remaining chains, the last one after the last stage; then the sums out
    for (; ok && flushed < nchains; ++flushed) ok = flush(flushed);
    if (ok && reads && c_ok) {
      float* o = p.out + int64_t(blockIdx.y) * p.cols * p.ncols + c * p.ncols + j0 + jb;
#pragma unroll
      for (int e = 0; e < kQuarterN; ++e)
        if (j0 + jb + e < p.ncols) o[e] = run[e];
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == kOpMmaWarp) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(tmem), "r"(kOpTmemCols));
  }
}

// dst[i] = the sum of part[s][i] over the row ranges s, in range order.
__global__ void outprod_reduce_kernel(const float* __restrict__ part, int ranges,
                                      int64_t count, float* __restrict__ dst) {
  for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < count;
       i += int64_t(gridDim.x) * blockDim.x) {
    float acc = __ldg(part + i);
    for (int s = 1; s < ranges; ++s) acc = __fadd_rn(acc, __ldg(part + int64_t(s) * count + i));
    dst[i] = acc;
  }
}

template <int NB, bool kTma>
int launch_outprod(const CUtensorMap& tm_g, const CUtensorMap& tm_w, const OpArgs& a, int tiles,
                   int ranges, cudaStream_t st, int dev) {
  using S = OpSmem<NB, kTma>;
  static std::atomic<int> configured[kMaxDevices];
  if (dev >= 0 && dev < kMaxDevices && !configured[dev].load()) {
    const cudaError_t e = cudaFuncSetAttribute(
        dq4_outprod_kernel<NB, kTma>, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes);
    if (e != cudaSuccess) return fail_cuda(DQ4_ERR_LAUNCH, e);
    configured[dev].store(1);
  }
  dq4_outprod_kernel<NB, kTma>
      <<<dim3(unsigned(tiles), unsigned(ranges)), kOpThreads, S::kBytes, st>>>(tm_g, tm_w, a);
  return check_launch();
}

// The tensor maps of the TMA staging: G as rows x ncols FP32 (NB x 64 boxes) and the packed
// weight as rows x cols / 2 bytes (64 x 64 boxes: 128 values of 64 rows), both unswizzled
// and zero-filled past the matrix.  False when the shape or the pointers do not allow them
// (then the kernel stages by cp.async).
bool outprod_tensor_maps(const uint8_t* packed, const float* G, int64_t rows, int64_t cols,
                         int64_t ncols, int nb, bool rows_alike, CUtensorMap* tm_g,
                         CUtensorMap* tm_w) {
  if (!rows_alike || cols % 32 != 0 || ncols % 4 != 0 || misaligned(G, 16) ||
      misaligned(packed, 16) || rows >= (int64_t(1) << 31) || ncols >= (int64_t(1) << 31) ||
      cols >= (int64_t(1) << 32))
    return false;
  EncodeTiled encode = tensor_map_encoder();
  if (!encode) return false;
  const cuuint32_t estride[2] = {1, 1};
  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(ncols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(ncols) * 4};
  const cuuint32_t gbox[2] = {static_cast<cuuint32_t>(nb), static_cast<cuuint32_t>(kOpK)};
  if (encode(tm_g, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(G), gdim, gstride, gbox,
             estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  const cuuint64_t wdim[2] = {static_cast<cuuint64_t>(cols / 2), static_cast<cuuint64_t>(rows)};
  const cuuint64_t wstride[1] = {static_cast<cuuint64_t>(cols / 2)};
  const cuuint32_t wbox[2] = {static_cast<cuuint32_t>(kOpM / 2), static_cast<cuuint32_t>(kOpK)};
  return encode(tm_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(packed), wdim,
                wstride, wbox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// How a problem runs: the G-column tile width, the tiles, and the row ranges.
struct OpPlan {
  int nb = 16;
  int64_t tiles_c = 0, tiles = 0;
  int64_t ranges = 1, rows_per_range = 0;
  int64_t ws_bytes = 0;  // the partial tiles of ranges > 1
};

// Row ranges fill the SMs in one wave (one CTA per SM), each of whole 64-row stages; the
// partial tiles must fit `budget` bytes (a budget below two ranges' worth gives one range,
// written straight to dst).
OpPlan plan_outprod(int64_t rows, int64_t cols, int64_t ncols, int sms, int64_t budget) {
  OpPlan pl;
  while (pl.nb < 128 && pl.nb < ncols) pl.nb *= 2;
  pl.tiles_c = (cols + kOpM - 1) / kOpM;
  pl.tiles = pl.tiles_c * ((ncols + pl.nb - 1) / pl.nb);
  const int64_t stages = (rows + kOpK - 1) / kOpK;
  int64_t want = pl.tiles >= sms ? 1 : sms / pl.tiles;
  if (want > stages) want = stages;
  if (want > 65535) want = 65535;
  const int64_t tile_bytes = cols * ncols * 4;
  const int64_t fit = tile_bytes > 0 ? budget / tile_bytes : 0;
  if (want > fit) want = fit;
  if (want < 2) want = 1;
  const int64_t per = (stages + want - 1) / want;  // stages per range
  pl.rows_per_range = per * kOpK;
  pl.ranges = stages > 0 ? (stages + per - 1) / per : 1;
  pl.ws_bytes = pl.ranges > 1 ? pl.ranges * tile_bytes : 0;
  return pl;
}

}  // namespace
}  // namespace dq4d

using namespace dq4d;

extern "C" {

int dq4_nested_out_prod(const uint8_t* packed, const uint8_t* scale_codes,
                        const float* nested_absmax, const float* scale_codebook,
                        const float* value_codebook, float offset, int64_t rows, int64_t cols,
                        int32_t blocksize, int32_t nested_blocksize, const float* G,
                        int64_t ncols, float* dst, float* workspace, int64_t workspace_bytes,
                        int* bad, void* stream) {
  if (rows < 0 || cols < 0 || ncols < 0 || workspace_bytes < 0) return DQ4_ERR_N;
  if (cols > 0 && rows > INT64_MAX / cols) return DQ4_ERR_N;
  if (ncols > 0 && cols > INT64_MAX / 4 / ncols) return DQ4_ERR_N;
  const int64_t n = rows * cols;
  if (int st = validate(n, blocksize, nested_blocksize, true, DQ4_OUT_F32)) return st;
  if (cols == 0 || ncols == 0) return DQ4_OK;
  if (!dst) return DQ4_ERR_NULL;
  if (misaligned(dst, 4) || misaligned(bad, 4)) return DQ4_ERR_ALIGN;
  const auto st = static_cast<cudaStream_t>(stream);
  if (rows == 0) {  // an empty sum
    const cudaError_t e = cudaMemsetAsync(dst, 0, size_t(cols) * size_t(ncols) * 4, st);
    return e == cudaSuccess ? DQ4_OK : fail_cuda(DQ4_ERR_LAUNCH, e);
  }
  if (!packed || !scale_codes || !nested_absmax || !scale_codebook || !value_codebook || !G)
    return DQ4_ERR_NULL;
  if (misaligned(packed, 4) || misaligned(scale_codes, 4) || misaligned(nested_absmax, 4) ||
      misaligned(scale_codebook, 4) || misaligned(value_codebook, 4) || misaligned(G, 4) ||
      misaligned(workspace, 4))
    return DQ4_ERR_ALIGN;
  int dev = 0, sms = 0;
  if (int s = current_device(&dev, &sms)) return s;
  const OpPlan pl = plan_outprod(rows, cols, ncols, sms, workspace ? workspace_bytes : 0);
  if (pl.tiles > INT32_MAX) return DQ4_ERR_N;
  OpArgs a;
  a.w = make_args(packed, scale_codes, nested_absmax, scale_codebook, value_codebook, offset, n,
                  blocksize, nested_blocksize, nullptr);
  a.G = G;
  a.out = pl.ranges > 1 ? workspace : dst;
  a.rows = rows;
  a.cols = cols;
  a.ncols = ncols;
  a.rows_per_range = pl.rows_per_range;
  a.tiles_c = int(pl.tiles_c);
  a.g_vec4 = (ncols % 4 == 0 && !misaligned(G, 16)) ? 1 : 0;
  a.rows_alike = (cols % 8 == 0 && (cols % blocksize == 0 || blocksize % cols == 0)) ? 1 : 0;
  a.bad = bad;
  CUtensorMap tm_g, tm_w;
  std::memset(&tm_g, 0, sizeof tm_g);
  std::memset(&tm_w, 0, sizeof tm_w);
  const bool tma =
      outprod_tensor_maps(packed, G, rows, cols, ncols, pl.nb, a.rows_alike != 0, &tm_g, &tm_w);
  const int T = int(pl.tiles), R = int(pl.ranges);
  int status;
  switch (pl.nb * 2 + (tma ? 1 : 0)) {
    case 32: status = launch_outprod<16, false>(tm_g, tm_w, a, T, R, st, dev); break;
    case 33: status = launch_outprod<16, true>(tm_g, tm_w, a, T, R, st, dev); break;
    case 64: status = launch_outprod<32, false>(tm_g, tm_w, a, T, R, st, dev); break;
    case 65: status = launch_outprod<32, true>(tm_g, tm_w, a, T, R, st, dev); break;
    case 128: status = launch_outprod<64, false>(tm_g, tm_w, a, T, R, st, dev); break;
    case 129: status = launch_outprod<64, true>(tm_g, tm_w, a, T, R, st, dev); break;
    case 256: status = launch_outprod<128, false>(tm_g, tm_w, a, T, R, st, dev); break;
    default: status = launch_outprod<128, true>(tm_g, tm_w, a, T, R, st, dev); break;
  }
  if (status || pl.ranges == 1) return status;
  const int64_t count = cols * ncols;
  int64_t grid = (count + 255) / 256;
  if (grid > int64_t(sms) * 8) grid = int64_t(sms) * 8;
  outprod_reduce_kernel<<<unsigned(grid), 256, 0, st>>>(workspace, int(pl.ranges), count, dst);
  return check_launch();
}

int64_t dq4_nested_out_prod_workspace_bytes(int64_t rows, int64_t cols, int64_t ncols) {
  if (rows <= 0 || cols <= 0 || ncols <= 0) return 0;
  if (rows > INT64_MAX / cols || cols > INT64_MAX / 4 / ncols) return 0;
  int dev = 0, sms = 0;
  if (current_device(&dev, &sms) != DQ4_OK) return -DQ4_ERR_DEVICE;
  return plan_outprod(rows, cols, ncols, sms, INT64_MAX).ws_bytes;
}

}  // extern "C"

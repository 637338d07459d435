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
// The work is the (tile, weight stage) units, tile-major; with a caller
// workspace and tiles that would not fill the SMs in whole rounds, one CTA runs
// per SM on an equal share of the units, a run that may cross tile boundaries.
// Each tile piece (segment) accumulates on its own in TMEM; whole tiles are
// stored at once, and a tile shared by several CTAs is summed from their FP32
// partials, in K order, by the last of them to finish (no CTA waits for
// another).
// Warps 0..7 dequantize, then 1 or 2 MMA-issuing warps (I, below), then the two TMA
// warps: 12 warps for narrow tiles (BX <= 64), 11 for wide ones.
//  * warp 8 + I (lane 0): streams the packed weight rows of each stage's tile with
//    TMA into a ring of raw stages (four 128-row x 64-value boxes, 4 KB each,
//    32-byte swizzled), as far ahead as the ring allows, once the dequantizing
//    warps have issued their first scale-code loads (which would otherwise queue
//    behind these copies in DRAM);
//  * warp 9 + I (lane 0): streams the activation tiles (BX rows x 64 K per K step,
//    128-byte swizzle, rows past M zero-filled) into their own ring, a whole
//    stage per slot for narrow tiles;
//  * warps 0..7, two groups of four that take alternate weight stages (so one
//    group's barrier polls overlap the other's arithmetic): warp w owns TMEM
//    lanes 32 (w % 4) .. (the weight rows), a thread one row.  Per 64-value K
//    step it computes the nested scales of its row's two 32-value halves
//    (separately rounded FP32 multiply and add; a stage's scale codes come in
//    one aligned load when the shape allows, loaded two own stages ahead and
//    unpacked only when their stage is decoded) and the 64 values (both values
//    of a packed byte from one 8-byte load of a byte-indexed codebook pair
//    table in shared memory, which these warps build at the start; FP32
//    products, RN to BF16 / FP16), and writes them to the weight ring in TMEM
//    with one tcgen05.st; afterwards
//    warps 0..7 run the epilogue: tcgen05.ld of each segment's accumulator,
//    conversion, stores of Y (or of a partial tile, and the shared tiles' sums);
//  * warps 8 .. 8 + I - 1: warp 8 allocates the TMEM; lane 0 of each issues
//    tcgen05.mma (A = weights from TMEM, B = activations from shared memory,
//    M = 128, N = BX, K = 16) and commits the weight and activation slots back to
//    their producers.  A tcgen05.mma holds its issuing thread about 120 cycles
//    whatever N is, so a single issuer would pace narrow tiles; with I = 2, issuer
//    i takes the stages producer group i decodes, into accumulators of its own,
//    and the read-out adds the two partial sums in a fixed order.
// Every W value is computed exactly as dq4_nested does, so the GEMM consumes
// the same operand bits as "dequantize, then F.linear".  Waits on mbarriers
// are bounded; a wait that runs out counts into *bad, raises a CTA-wide abort
// flag, and the CTA drains its copies and MMAs, frees its TMEM and returns.
#include "common.cuh"
#include "tcgen05.cuh"
#include "tmap.cuh"

#include <mutex>

namespace dq4d {
namespace {

#ifndef DQ4_LIN_PWARPS
#define DQ4_LIN_PWARPS 8  // dequantizing warps per CTA: 8 or 16
#endif
#ifndef DQ4_LIN_GROUPS
#define DQ4_LIN_GROUPS 2  // producer groups taking turns on weight stages (<= the ring depth)
#endif
constexpr int kProducerWarps = DQ4_LIN_PWARPS;
constexpr int kGroups = DQ4_LIN_GROUPS;
constexpr int kGroupWarps = kProducerWarps / kGroups;  // warps writing one weight stage
static_assert(kProducerWarps == 8 || kProducerWarps == 16, "8 or 16 producer warps");
static_assert(kGroups == 1 || kGroups == 2 || kGroups == 4, "1, 2 or 4 producer groups");
static_assert(kGroupWarps == 4 || kGroupWarps == 8 || kGroupWarps == 16, "whole quadrants");
constexpr int kTPR = kGroupWarps / 4;              // producer threads per weight row
constexpr int kWords = 8 / kTPR;                   // packed 32-bit words per thread and K step
constexpr int kHalves = kWords >= 8 ? 2 : 1;       // 32-value halves per thread and K step
constexpr int kMmaWarp = kProducerWarps;           // the first MMA warp; also allocates TMEM
// MMA-issuing warps.  A tcgen05.mma holds its issuing thread about 120 cycles whatever its N
// (measured on GB300 for N = 16 .. 128, A from TMEM or shared memory), while two issuing
// threads in different warps overlap: narrow tiles, whose MMAs carry few FLOPs, issue from
// two threads, each into accumulators of its own.
__host__ __device__ constexpr int kIssOf(int bx) { return bx <= 64 ? 2 : 1; }
__host__ __device__ constexpr int kRawWarpOf(int bx) { return kProducerWarps + kIssOf(bx); }
__host__ __device__ constexpr int kXWarpOf(int bx) { return kProducerWarps + kIssOf(bx) + 1; }
__host__ __device__ constexpr int kThreadsOf(int bx) {
  return 32 * (kProducerWarps + kIssOf(bx) + 2);
}
constexpr int kBW = 128;           // weight rows per CTA = MMA M = TMEM lanes
constexpr int kBK = 64;            // 64 16-bit values = one 128-byte swizzle row
constexpr int kRawBytes = kBW * kBK / 2;  // one raw stage: 128 rows x 32 packed bytes
// Instruction descriptor of this kernel's MMAs: M = 128 weight rows, N = BX.
template <int BX>
__device__ __forceinline__ uint32_t instr_desc(bool bf16) {
  return instr_desc_f16<kBW, BX>(bf16);
}

// Named barrier 1 over the 256 epilogue threads, AND-reducing a predicate.
__device__ __forceinline__ bool bar_and_256(bool v) {
  uint32_t r;
  asm volatile(
      "{\n.reg .pred p, q;\nsetp.ne.u32 p, %1, 0;\nbar.red.and.pred q, 1, 256, p;\n"
      "selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r) : "r"(static_cast<uint32_t>(v)) : "memory");
  return r != 0;
}

// (a * s, b * s) for the FP32 pair ab = {a, b} (a in the low word), each product
// rounded to nearest FP32 on its own: one packed f32x2 multiply, never contracted.
__device__ __forceinline__ void mul2_rn64(uint64_t ab, uint64_t s2, float& x, float& y) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(ab), "l"(s2));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(r));
}

struct LinArgs {
  Args w;          // the nested 4-bit weight (n = N * K values, row-major N x K)
  void* Y;
  int64_t M, N, K;
  int* bad;        // optional device counter of timed-out waits
  int out_dtype;
  int tiles_x;     // activation-row tiles of Y
  // bytes of scale codes one weight stage (64 kSub values of a row) spans, when those
  // codes form one aligned window with one absmax group (else 0: one load per K step)
  int code_window;
  // The work is units = tiles x stages, tile-major (tile t = tile_w * tiles_x + tile_x).
  // With whole != 0 there is one CTA per tile, CTA c taking tile c whole.  Otherwise
  // CTA c takes units c units / ctas .. (c + 1) units / ctas - 1 (units < 2^32, ctas <
  // 2^16), a run of stages that may cross tile boundaries: its first and last segments
  // may be parts of tiles that other CTAs share; those go to ws_part as FP32 partial
  // tiles, and the last CTA to arrive at such a tile (ws_count) sums its parts in K
  // order.
  int whole;
  int ctas;
  uint32_t units;
  uint32_t units_q, units_r;  // units / ctas, units % ctas
  float* ws_part;  // [ctas][2][BX][128]: CTA c's partial first (0) and last (1) segments
  int* ws_count;   // [ctas]: arrivals at the shared tile whose last part CTA c holds
};

// First unit of CTA c under the split work division: c units / ctas, in 32-bit
// arithmetic (c (units % ctas) < ctas^2 < 2^32).
__host__ __device__ __forceinline__ uint32_t split_begin(uint32_t c, const LinArgs& p) {
  return c * p.units_q + c * p.units_r / uint32_t(p.ctas);
}

// The dequantized weights (the MMA's A operand) live in TMEM, after the FP32
// accumulators: a ring of kAS weight stages of kSub 64-value K steps (32 columns each:
// 64 16-bit values per lane = weight row).  Producers write them with tcgen05.st, so
// shared memory only carries the activation ring (B operand, TMA) and the raw packed
// weight ring (TMA), both as deep as the budget allows.  A weight stage spans kSub K
// steps, so the per-stage barrier work of the producers is shared by 32 * kSub values
// per thread.
#ifndef DQ4_LIN_SUB
#define DQ4_LIN_SUB 4
#endif
constexpr int kSub = DQ4_LIN_SUB;         // 64-value K steps per weight stage
constexpr uint32_t kTmemCols = 512;       // the whole TMEM of the SM
// Accumulator buffers per MMA issuer: two for the narrowest tiles (a segment accumulates
// while the previous one is read out), one of BX columns otherwise.  Issuer i's buffer b
// is columns (i kAcc + b) BX ..; all of them lie in columns 0 .. kATmem(BX) - 1, the weight
// ring in the rest: kAS(BX) stages.
__host__ __device__ constexpr int kAccOf(int bx) { return bx <= 32 ? 2 : 1; }
__host__ __device__ constexpr uint32_t kATmem(int bx) { return bx <= 128 ? 128u : 256u; }
__host__ __device__ constexpr int kASOf(int bx) {
  return int((kTmemCols - kATmem(bx)) / 32) / kSub;
}
template <int BX>
struct LinSmem {
  static constexpr int kAS = kASOf(BX);              // weight stages in TMEM
  static constexpr int kAcc = kAccOf(BX);            // accumulator buffers per issuer
  static constexpr int kIss = kIssOf(BX);            // MMA-issuing threads
  static_assert(kAS >= 2, "double-buffered weight ring");
  static_assert(kIss * kAcc * BX <= int(kATmem(BX)), "accumulators fit before the weight ring");
  // mbarrier waits test a phase's parity, so a waiter must never be two phases ahead
  // of the barrier.  A group at stage i waits for the MMAs of stage i - kAS and knows,
  // from its previous wait, that those of stage i - kGroups - kAS completed (MMAs
  // complete in order): kAS >= kGroups keeps it at most one phase ahead.
  static_assert(kAS >= kGroups, "no producer group runs two weight phases ahead");
  static_assert(kATmem(BX) + kAS * kSub * 32 <= kTmemCols, "weight ring fits TMEM");
  static constexpr int kRawSlot = kSub * kRawBytes;
  static constexpr int kB = BX * kBK * 2;           // one K step of activations
  // K steps per activation slot: a whole stage for narrow tiles (one wait and one
  // release per stage for an MMA thread, and stage l's slot is l % kXS), one K step for
  // wide ones
  static constexpr int kXSub = BX <= 64 ? kSub : 1;
  static_assert(kIss == 1 || kXSub == kSub, "several issuers take whole-stage slots");
  static constexpr int kXSlot = kXSub * kB;
  static constexpr int kXS = BX <= 64 ? 3 : BX == 128 ? 6 : 4;  // slots
  // The codebook as a byte-indexed pair table: entry b holds (vcb[b >> 4], vcb[b & 15]),
  // the two values of a packed byte, as 8 bytes, replicated 16 times so that lane l reads
  // copy l % 16: each half warp's 8-byte loads then fall in 16 distinct bank pairs
  // whatever bytes its lanes decode.  Entry b copy g sits at (16 b + g) * 8.
  static constexpr int kTabBytes = 256 * 16 * 8;
  // raw weight stages: what the activation ring and the table leave of a 224 KB budget,
  // at most 16
  static constexpr int kRawFit = (224 * 1024 - kTabBytes - kXS * kXSlot) / kRawSlot;
  // A group waits for the raw load of its stage i; the load into the same slot before it
  // (stage i - kRawS) must be known complete, which holds when that stage is the group's
  // own: kRawS a multiple of kGroups (TMA loads need not complete in issue order).
  static constexpr int kRawS = (kRawFit < 16 ? kRawFit : 16) / kGroups * kGroups;
  static_assert(kRawS >= 4, "raw ring too shallow");
  static constexpr int kXOff = 0;
  static constexpr int kRawOff = kXOff + kXS * kXSlot;
  static constexpr int kTabOff = kRawOff + kRawS * kRawSlot;
  static constexpr int kBarOff = kTabOff + kTabBytes;
  // full_w, empty_a per weight stage; full_x, empty_x per activation stage;
  // raw_full, raw_empty per raw stage; acc_full, acc_empty per accumulator buffer (shared
  // by the issuers); acc_done
  static constexpr int kBars = 2 * kAS + 2 * kXS + 2 * kRawS + 2 * kAcc + 1;
  static constexpr int kBytes = kBarOff + 8 * kBars + 1024;  // + alignment slack
  // with the kernel's static shared memory (the scale codebook and a few words)
  static_assert(kBytes + 1280 <= 227 * 1024, "shared memory budget");
  // more than half an SM's shared memory: one CTA per SM, so the 512-column TMEM
  // allocation never waits for another CTA
  static_assert(kBytes > 116 * 1024, "one CTA per SM");
  static_assert(kB % 1024 == 0, "swizzle atoms stay 1024-byte aligned");
};

// Slot and phase parity of a ring position, advanced without division.
template <int kDepth>
struct RingPos {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next() {
    if (++slot == kDepth) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

#if DQ4_PDL && DQ4_L2_PREFETCH
constexpr int kLinPrefetch = 4;  // local weight stages prefetched before the setup
// Thread t of the dequantizing warps asks L2 for row t % 128 of every (t / 128)-th of the
// first n_pf local stages (the first first_seg of them in the tile at weight row n0a, the
// rest in the next tile, at n0b, from its stage 0), and the first group also for the
// rows' scale-code and absmax lines.  Not inlined: it runs once, before the setup, and
// stays out of the main loop's register allocation.
__device__ __noinline__ void linear_prefetch(const LinArgs& p, int64_t n0a, int64_t n0b,
                                             int stage0, int first_seg, int n_pf,
                                             int st_count) {
  constexpr int kRowGroups = kProducerWarps * 32 / kBW;
  const int row = threadIdx.x & (kBW - 1);
  for (int j = threadIdx.x / kBW; j < n_pf; j += kRowGroups) {
    const bool first = j < first_seg;
    const int64_t n = (first ? n0a : n0b) + row;
    const int stage = first ? stage0 + j : j - first_seg;
    if (n >= p.N || stage >= st_count) continue;  // (a third tile is not prefetched)
    const int64_t i = n * p.K + int64_t(stage) * kSub * kBK;  // the stage's first value
    asm volatile("prefetch.global.L2 [%0];" :: "l"(p.w.packed + (i >> 1)));
    if (j < kRowGroups) {
      const int64_t b = i >> p.w.log2_bs;
      asm volatile("prefetch.global.L2 [%0];" :: "l"(p.w.codes + b));
      asm volatile("prefetch.global.L2 [%0];" :: "l"(p.w.absmax + (b >> p.w.log2_nbs)));
    }
  }
}
#endif

template <int BX, bool kBF16>
__global__ void __launch_bounds__(kThreadsOf(BX), 1)
    dq4_linear_kernel(const __grid_constant__ CUtensorMap tmap_x,
                      const __grid_constant__ CUtensorMap tmap_w, const LinArgs p) {
  using S = LinSmem<BX>;
  constexpr int kAS = S::kAS, kXS = S::kXS, kRawS = S::kRawS, kAcc = S::kAcc, kIss = S::kIss;
  constexpr int kRawWarp = kRawWarpOf(BX), kXWarp = kXWarpOf(BX);
  constexpr uint32_t kATmemCol = kATmem(BX);
  constexpr int kOut = kBF16 ? DQ4_OUT_BF16 : DQ4_OUT_F16;
  constexpr unsigned kFull = 0xFFFFFFFFu;
  extern __shared__ uint8_t smem_raw[];
  __shared__ float s_scb[256];
  __shared__ uint32_t s_tmem;          // TMEM base address from tcgen05.alloc
  __shared__ volatile int s_abort;     // set when any wait of the CTA ran out
  __shared__ int s_last[2];            // this CTA completes its first / last shared tile
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(base);
  const uint32_t bar0 = sbase + S::kBarOff;
  auto full_w = [&](int s) { return bar0 + 8 * s; };              // producer warps
  auto empty_a = [&](int s) { return bar0 + 8 * (kAS + s); };     // MMAs reading it done
  auto full_x = [&](int s) { return bar0 + 8 * (2 * kAS + s); };  // activation TMA
  auto empty_x = [&](int s) { return bar0 + 8 * (2 * kAS + kXS + s); };
  auto raw_full = [&](int s) { return bar0 + 8 * (2 * kAS + 2 * kXS + s); };
  auto raw_empty = [&](int s) { return bar0 + 8 * (2 * kAS + 2 * kXS + kRawS + s); };
  // acc_full(b): the segment in accumulator buffer b is final (one arrival per issuer);
  // acc_empty(b): read out; acc_done: every MMA done (one arrival per issuer)
  auto acc_full = [&](int b) { return bar0 + 8 * (2 * kAS + 2 * kXS + 2 * kRawS + b); };
  auto acc_empty = [&](int b) { return acc_full(kAcc + b); };
  const uint32_t acc_done = acc_full(2 * kAcc);
  volatile int* abort_flag = &s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int kt_count = int(p.K / kBK);                    // 64-value K steps
  const int st_count = (kt_count + kSub - 1) / kSub;      // weight stages per tile
  // this CTA's units u0 .. u1 - 1 (tile-major), local stages l = 0 .. nl - 1: segment s
  // is the part in tile t0 + s, from local stage seg_start(s) on (no 64-bit division)
  int64_t u0, u1, t0;
  int stage0, nseg;
  if (p.whole) {
    t0 = blockIdx.x;
    u0 = t0 * st_count;
    u1 = u0 + st_count;
    stage0 = 0;
    nseg = 1;
  } else {
    const uint32_t a = split_begin(blockIdx.x, p), b = split_begin(blockIdx.x + 1, p);
    const uint32_t ta = a / uint32_t(st_count);
    u0 = a;
    u1 = b;
    t0 = ta;
    stage0 = int(a - ta * uint32_t(st_count));
    nseg = int((b - 1) / uint32_t(st_count) - ta) + 1;
  }
  const int nl = int(u1 - u0);
  auto seg_start = [&](int sg) { return sg == 0 ? 0 : sg * st_count - stage0; };
  // where a local stage sits: its segment, its stage within the tile, and the tile's first
  // weight row and activation row (advanced without division but at tile boundaries)
  struct Cursor {
    int seg, stage;
    int64_t n0, m0;
  };
  auto set_origin = [&](Cursor& c) {
    const uint32_t t = uint32_t(t0 + c.seg), tw = t / uint32_t(p.tiles_x);
    c.n0 = int64_t(tw) * kBW;
    c.m0 = int64_t(t - tw * uint32_t(p.tiles_x)) * BX;
  };
  auto cursor_at = [&](int l) {
    Cursor c;
    c.seg = (stage0 + l) / st_count;
    c.stage = stage0 + l - c.seg * st_count;
    set_origin(c);
    return c;
  };
  auto advance = [&](Cursor& c, int k) {
    c.stage += k;
    if (c.stage >= st_count) {
      do {
        c.stage -= st_count;
        ++c.seg;
      } while (c.stage >= st_count);
      set_origin(c);
    }
  };
  auto fail = [&]() {
    *abort_flag = 1;
    if (p.bad) atomicAdd(p.bad, 1);
  };

#if DQ4_PDL && DQ4_L2_PREFETCH
  // Before the setup and griddepcontrol.wait: the dequantizing threads ask L2 for the
  // packed weight lines of this CTA's first kLinPrefetch local stages (thread t: row
  // t % 128 of every (t / 128)-th stage) and for the rows' scale-code and absmax lines, so
  // the first stages' DRAM reads overlap the setup.  A prefetch returns nothing to the
  // thread and L2 is the point of coherence, so no value read after the wait changes.
  // (narrow tiles only: measured at N = 11008, K = 4096, M = 16 18.6 -> 17.4 us, M = 32
  // unchanged, M = 64 and up unchanged or up to 1 % slower)
  if (BX <= 32 && warp < kProducerWarps) {
    const int n_pf = nl < kLinPrefetch ? nl : kLinPrefetch;
    // the stages' tiles: the run's first segment, then (at most) the next tile
    const int first_seg = st_count - stage0;  // local stages left in the first tile
    const uint32_t ta = uint32_t(t0), tb = uint32_t(t0 + 1);
    linear_prefetch(p, int64_t(ta / uint32_t(p.tiles_x)) * kBW,
                    int64_t(tb / uint32_t(p.tiles_x)) * kBW, stage0, first_seg, n_pf,
                    st_count);
  }
#endif
  // The setup below touches no global memory (the tensor maps are kernel parameters), so
  // under programmatic dependent launch it overlaps the previous kernel in the stream;
  // every global read comes after griddepcontrol.wait.  Two CTAs of this kernel never
  // share an SM (each takes more than half its shared memory), so when the previous
  // kernel is this one the TMEM is free; after another kernel that holds TMEM on this SM,
  // the allocation waits until that kernel releases it.
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(&s_tmem)), "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    if (lane == 0) {
      for (int s = 0; s < kAS; ++s) {
        mbar_init(full_w(s), kGroupWarps);
        mbar_init(empty_a(s), 1);
      }
      for (int s = 0; s < kXS; ++s) {
        mbar_init(full_x(s), 1);
        mbar_init(empty_x(s), 1);
      }
      for (int s = 0; s < kRawS; ++s) {
        mbar_init(raw_full(s), 1);
        mbar_init(raw_empty(s), kGroupWarps);
      }
      for (int g = 0; g < kAcc; ++g) {
        mbar_init(acc_full(g), kIss);
        mbar_init(acc_empty(g), 8);  // the 8 epilogue warps
      }
      mbar_init(acc_done, kIss);
      *abort_flag = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmap_x)));
      asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmap_w)));
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = s_tmem;
#if DQ4_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
#endif

  if (warp == kRawWarp) {
    // the weight copies start once the producers issued their first stages' code loads,
    // which would otherwise queue behind the copies in DRAM (named barrier 3)
    asm volatile("bar.sync 3, %0;" :: "n"(kProducerWarps * 32 + 32) : "memory");
    if (lane == 0) {
      // ---- packed weight rows of each local stage's tile: kSub boxes of 128 rows x 32
      // bytes (64 values) per stage, 32-byte swizzled, each in its own 4 KB
      const uint64_t tw = reinterpret_cast<uint64_t>(&tmap_w);
      RingPos<kRawS> pos;
      Cursor cs = cursor_at(0);
      int l = 0;
      for (; l < nl; ++l, pos.next(), advance(cs, 1)) {
        if (l >= kRawS) {
          if (*abort_flag) break;
          if (!mbar_wait(raw_empty(pos.slot), pos.phase ^ 1u)) {
            fail();
            break;
          }
        }
        const int ns = min(kSub, kt_count - cs.stage * kSub);
        mbar_expect(raw_full(pos.slot), ns * kRawBytes);
        for (int sub = 0; sub < ns; ++sub)
          tma_load_2d(sbase + S::kRawOff + pos.slot * S::kRawSlot + sub * kRawBytes, tw,
                      (cs.stage * kSub + sub) * (kBK / 2), int(cs.n0), raw_full(pos.slot));
      }
      if (*abort_flag)  // copies still in flight land before the CTA leaves
        for (int j = l - 1; j >= 0 && j >= l - kRawS; --j)
          mbar_wait(raw_full(j % kRawS), (j / kRawS) & 1);
    }
  } else if (warp == kXWarp) {
    if (lane == 0) {
      // ---- activation rows of each local stage's tile, kXSub 64-value K steps per slot
      constexpr int kXSub = S::kXSub;
      const uint64_t tx = reinterpret_cast<uint64_t>(&tmap_x);
      RingPos<kXS> pos;
      int q = 0;  // slots requested
      bool stop = false;
      Cursor cs = cursor_at(0);
      for (int l = 0; l < nl && !stop; ++l, advance(cs, 1)) {
        const int ns = min(kSub, kt_count - cs.stage * kSub);
        for (int sub = 0; sub < ns; sub += kXSub, ++q, pos.next()) {
          if (q >= kXS) {
            if (*abort_flag || !mbar_wait(empty_x(pos.slot), pos.phase ^ 1u)) {
              if (!*abort_flag) fail();
              stop = true;
              break;
            }
          }
          const int cnt = min(kXSub, ns - sub);
          mbar_expect(full_x(pos.slot), cnt * S::kB);
          for (int i = 0; i < cnt; ++i)
            tma_load_2d(sbase + S::kXOff + pos.slot * S::kXSlot + i * S::kB, tx,
                        (cs.stage * kSub + sub + i) * kBK, int(cs.m0), full_x(pos.slot));
        }
      }
      if (*abort_flag)
        for (int j = q - 1; j >= 0 && j >= q - kXS; --j)
          mbar_wait(full_x(j % kXS), (j / kXS) & 1);
    }
  } else if (warp >= kMmaWarp && warp < kMmaWarp + kIss) {
    if (lane == 0) {
      if constexpr (kIss == 1) {
        // ---- the MMA issue: local stage l reads its weight slot (l % kAS) and its
        // activation slots (one per stage for narrow tiles, one per K step otherwise),
        // accumulating into its segment's accumulator (columns buf * BX ..), which the
        // segment kAcc back must have left; each slot is released when its MMAs complete
        const uint32_t idesc = instr_desc<BX>(kBF16);
        RingPos<kAS> apos;
        RingPos<kXS> xpos;
        Cursor cs = cursor_at(0);
        bool stop = false, first = true;  // first: the stage opens its segment
        int committed = 0;  // segments whose accumulator was committed
        for (int l = 0; l < nl && !stop; ++l, apos.next(), advance(cs, 1)) {
          // the weight stage and (with whole-stage activation slots) its activations, polled
          // together first
          const bool ready = !*abort_flag &&
                             (S::kXSub == kSub
                                  ? mbar_try2(full_w(apos.slot), apos.phase, full_x(xpos.slot),
                                              xpos.phase)
                                  : mbar_try(full_w(apos.slot), apos.phase));
          if (!ready && (*abort_flag || !mbar_wait(full_w(apos.slot), apos.phase))) {
            if (!*abort_flag) fail();
            break;
          }
          const int buf = kAcc == 1 ? 0 : (cs.seg & 1);
          if (first && cs.seg >= kAcc &&
              (*abort_flag ||
               !mbar_wait(acc_empty(buf), uint32_t(cs.seg / kAcc - 1) & 1u))) {
            if (!*abort_flag) fail();
            break;
          }
          const int ns = min(kSub, kt_count - cs.stage * kSub);
          const uint32_t d_tmem = tmem + buf * BX;
          for (int sub = 0; sub < ns; ++sub) {
            const int xi = sub % S::kXSub;  // K step within the activation slot
            if (xi == 0 && !(ready && sub == 0 && S::kXSub == kSub) &&
                !mbar_wait(full_x(xpos.slot), xpos.phase)) {
              fail();
              stop = true;
              break;
            }
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            // weights (M side) from TMEM: 8 columns per 16-value K slice
            const uint32_t a_tmem = tmem + kATmemCol + (apos.slot * kSub + sub) * 32;
            const uint32_t b_addr = sbase + S::kXOff + xpos.slot * S::kXSlot + xi * S::kB;
  #pragma unroll
            for (int ks = 0; ks < kBK / 16; ++ks) {
              const uint64_t db = smem_desc(b_addr + ks * 32);
              const uint32_t acc = (first && sub == 0 && ks == 0) ? 0u : 1u;
              asm volatile(
                  "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                  "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
                  :: "r"(d_tmem), "r"(a_tmem + ks * 8), "l"(db), "r"(idesc), "r"(acc));
            }
            if (xi == S::kXSub - 1 || sub == ns - 1) {  // the slot's last K step
              asm volatile(
                  "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                  :: "r"(empty_x(xpos.slot)) : "memory");
              xpos.next();
            }
          }
          if (stop) break;
          asm volatile(
              "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
              :: "r"(empty_a(apos.slot)) : "memory");
          first = cs.stage == st_count - 1 || l == nl - 1;  // the segment's last stage
          if (first) {
            asm volatile(
                "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                :: "r"(acc_full(buf)) : "memory");
            ++committed;
          }
        }
        // after a failure, release the epilogue's next wait on each accumulator
        for (int k = 0; k < kAcc && committed < nseg; ++k, ++committed)
          asm volatile(
              "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
              :: "r"(acc_full(kAcc == 1 ? 0 : (committed & 1))) : "memory");
        // tracks every MMA issued above: no MMA still writes TMEM when it is freed below
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
            :: "r"(acc_done) : "memory");
        mbar_wait(acc_done, 0);
      } else {
        // ---- several issuers: issuer iss issues local stages iss, iss + kIss, .. (the stages
        // producer group iss decodes) into its own accumulator buffers, columns
        // (iss kAcc + buf) BX ..; stage l reads weight slot l % kAS and the whole-stage
        // activation slot l % kXS.  Each issuer arrives once per segment on the segment's
        // acc_full, having issued its MMAs of that segment (if any); the read-out adds the
        // issuers' partial sums.  An issuer takes a buffer, and arrives on its acc_full, only
        // after the read-out of the segment kAcc back (acc_empty), so the phases of a
        // buffer's barriers never mix segments.
        const int iss = warp - kMmaWarp;
        const uint32_t idesc = instr_desc<BX>(kBF16);
        bool stop = false;
        int my_seg = 0;     // segments before my_seg have this issuer's acc_full arrival
        int open_seg = -1;  // the segment this issuer holds a buffer for
        auto buf_of = [&](int sg) { return kAcc == 1 ? 0 : (sg & 1); };
        auto acquire = [&](int sg) {  // segment sg's buffer was read out for segment sg - kAcc
          if (sg < kAcc) return true;
          if (*abort_flag) return false;
          if (mbar_wait(acc_empty(buf_of(sg)), uint32_t(sg / kAcc - 1) & 1u)) return true;
          fail();
          return false;
        };
        auto close = [&](int sg) {  // arrives once this issuer's MMAs so far completed
          asm volatile(
              "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
              :: "r"(acc_full(buf_of(sg))) : "memory");
        };
        Cursor cs = cursor_at(iss);
        for (int l = iss; l < nl; l += kIss, advance(cs, kIss)) {
          for (; my_seg < cs.seg; ++my_seg) {  // segments with no stage of this issuer
            if (!acquire(my_seg)) {
              stop = true;
              break;
            }
            close(my_seg);
          }
          if (stop) break;
          const int aslot = l % kAS, xslot = l % kXS;
          const uint32_t aph = uint32_t(l / kAS) & 1u, xph = uint32_t(l / kXS) & 1u;
          const bool ready =
              !*abort_flag && mbar_try2(full_w(aslot), aph, full_x(xslot), xph);
          if (!ready && (*abort_flag || !mbar_wait(full_w(aslot), aph) ||
                         !mbar_wait(full_x(xslot), xph))) {
            if (!*abort_flag) fail();
            stop = true;
            break;
          }
          const bool first = open_seg != cs.seg;  // this issuer's first stage of the segment
          if (first) {
            if (!acquire(cs.seg)) {
              stop = true;
              break;
            }
            open_seg = cs.seg;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const int ns = min(kSub, kt_count - cs.stage * kSub);
          const uint32_t d_tmem = tmem + (iss * kAcc + buf_of(cs.seg)) * BX;
          for (int sub = 0; sub < ns; ++sub) {
            const uint32_t a_tmem = tmem + kATmemCol + (aslot * kSub + sub) * 32;
            const uint32_t b_addr = sbase + S::kXOff + xslot * S::kXSlot + sub * S::kB;
#pragma unroll
            for (int ks = 0; ks < kBK / 16; ++ks) {
              const uint64_t db = smem_desc(b_addr + ks * 32);
              const uint32_t acc = (first && sub == 0 && ks == 0) ? 0u : 1u;
              asm volatile(
                  "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                  "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
                  :: "r"(d_tmem), "r"(a_tmem + ks * 8), "l"(db), "r"(idesc), "r"(acc));
            }
          }
          asm volatile(
              "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
              :: "r"(empty_x(xslot)) : "memory");
          asm volatile(
              "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
              :: "r"(empty_a(aslot)) : "memory");
          // this issuer's last stage of the segment: the segment ends before its next stage
          Cursor cn = cs;
          advance(cn, kIss);
          if (l + kIss >= nl || cn.seg != cs.seg) {
            close(cs.seg);
            my_seg = cs.seg + 1;
          }
        }
        if (!stop) {
          for (; my_seg < nseg; ++my_seg) {  // trailing segments with no stage of this issuer
            if (!acquire(my_seg)) {
              stop = true;
              break;
            }
            close(my_seg);
          }
        }
        // after a failure, release the epilogue's next wait on each buffer
        for (int k = 0; stop && k < kAcc && my_seg < nseg; ++k, ++my_seg) close(my_seg);
        // tracks every MMA this issuer issued: no MMA still writes TMEM when it is freed
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
            :: "r"(acc_done) : "memory");
        mbar_wait(acc_done, 0);
      }
    }
  } else {
    // The codebooks, loaded first (their latency overlaps the first stages' code loads
    // below); the scale codebook goes to shared memory, the value codebook becomes the
    // pair table after those loads are issued.
    static_assert(kProducerWarps * 32 >= 256, "the producers load the scale codebook");
    const float scb_v = tid < 256 ? __ldg(p.w.scb + tid) : 0.f;
    const float vcb_v = __ldg(p.w.vcb + (lane & 15));
    // ---- dequantize.  Producer group `group` (kGroupWarps warps) takes local stages
    // group, group + kGroups, ...; within it, warp w writes TMEM lanes 32 (w % 4) ..
    // (weight row r = 32 (w % 4) + lane of the stage's tile) and values 8 kWords h ..
    // 8 kWords (h + 1) - 1 of every 64-value K step, h = (w % kGroupWarps) / 4.
    // kHalves 32-value halves per K step each lie in one block (blocksize >= 32).
    const int gw = warp % kGroupWarps, group = warp / kGroupWarps;
    const int quad = gw & 3, h = gw >> 2;
    const int r = quad * 32 + lane;
    const float offset = p.w.offset;
    const uint32_t t_row = tmem + (static_cast<uint32_t>(quad * 32) << 16) + kATmemCol +
                           4 * kWords * h;  // this warp's lanes, its columns of a K step
    // The scale codes / absmax of the stage at cursor cs (local stage l) for this thread's
    // row.  With an aligned code window the stage's codes arrive in one load (w) and its
    // absmax in another (m), unpacked into c / a only when the stage is decoded: nothing
    // consumes a load in the iteration that issues it, so no warp waits on one.  Otherwise
    // the codes and absmax are loaded per K step straight into c / a.
    auto fetch = [&](int l, const Cursor& cs, uint32_t (&c)[kSub][kHalves],
                     float (&a)[kSub][kHalves], uint64_t& w, float& m) {
      w = 0;
      m = 0.f;
#pragma unroll
      for (int sub = 0; sub < kSub; ++sub)
#pragma unroll
        for (int hh = 0; hh < kHalves; ++hh) {
          c[sub][hh] = 0;
          a[sub][hh] = 0.f;
        }
      if (l >= nl || cs.n0 + r >= p.N) return;
      const int j0 = cs.stage * kSub;
      const int64_t idx0 = (cs.n0 + r) * p.K + 8 * kWords * h;  // this thread's first value
      if (p.code_window != 0) {
        const int64_t b00 = (idx0 - 8 * kWords * h + int64_t(j0) * kBK) >> p.w.log2_bs;
        const uint8_t* cp = p.w.codes + b00;
        switch (p.code_window) {
          case 8: w = __ldg(reinterpret_cast<const unsigned long long*>(cp)); break;
          case 4: w = __ldg(reinterpret_cast<const unsigned int*>(cp)); break;
          case 2: w = __ldg(reinterpret_cast<const unsigned short*>(cp)); break;
          default: w = __ldg(cp); break;
        }
        m = __ldg(p.w.absmax + (b00 >> p.w.log2_nbs));
        return;
      }
#pragma unroll
      for (int sub = 0; sub < kSub; ++sub)
#pragma unroll
        for (int hh = 0; hh < kHalves; ++hh) {
          const int j = j0 + sub;
          if (j < kt_count) {
            const int64_t b = (idx0 + int64_t(j) * kBK + 32 * hh) >> p.w.log2_bs;
            c[sub][hh] = __ldg(p.w.codes + b);
            a[sub][hh] = __ldg(p.w.absmax + (b >> p.w.log2_nbs));
          }
        }
    };
    // a window-loaded stage's codes and absmax, per K step and 32-value half
    auto unpack = [&](uint64_t w, float m, uint32_t (&c)[kSub][kHalves],
                      float (&a)[kSub][kHalves]) {
      if (p.code_window == 0) return;
#pragma unroll
      for (int sub = 0; sub < kSub; ++sub)
#pragma unroll
        for (int hh = 0; hh < kHalves; ++hh) {
          const int off = (kBK * sub + 32 * hh + 8 * kWords * h) >> p.w.log2_bs;
          c[sub][hh] = static_cast<uint32_t>(w >> (8 * off)) & 0xFFu;  // off < window
          a[sub][hh] = m;
        }
    };
    // ---- read-out of segment ds (warps 0..7; named barrier 1 over their 256 threads):
    // warps w and w + 4 read TMEM lanes 32 (w % 4) .. (weight rows = columns of Y), each
    // half of the BX accumulator columns (activation rows).  A whole tile goes to Y; a
    // shared one to this CTA's partial slot, and the last CTA to arrive at the tile sums
    // its parts into Y.
    constexpr int kHalf = BX / 2;
    constexpr int kChunk = kHalf < 32 ? kHalf : 32;  // columns per step of the parts' sum
    constexpr int kBatch = kChunk <= 8 ? 4 : kChunk <= 16 ? 2 : 1;  // parts loaded at once
    // accumulator columns per TMEM read (one wait); 8 when partial sums of several issuers
    // are added (two reads live at once)
    constexpr int kLd = (kHalf < 32 || kIss > 1) ? 8 : 32;
    const int eq = warp & 3, c_begin = ((warp >> 2) & 1) * kHalf;
    auto store_y = [&](int64_t m, int64_t ny, float f) {
      const int64_t o = m * p.N + ny;  // a warp writes 32 consecutive columns of row m
      if (p.out_dtype == DQ4_OUT_F32) {
        static_cast<float*>(p.Y)[o] = f;
      } else if (p.out_dtype == DQ4_OUT_BF16) {
        static_cast<__nv_bfloat16*>(p.Y)[o] = __float2bfloat16_rn(f);
      } else {
        static_cast<__half*>(p.Y)[o] = __float2half_rn(f);
      }
    };
    bool failed = false;
    // where segment ds sits: its tile, the tile's first activation row for this warp's half
    // of the columns, this lane's column of Y, and whether the segment is the whole tile
    struct SegAt {
      int64_t t, m0, ny;
      bool whole;
    };
    auto seg_at = [&](int ds) {
      SegAt g;
      g.t = t0 + ds;
      const uint32_t tw = uint32_t(g.t) / uint32_t(p.tiles_x);
      g.m0 = int64_t(uint32_t(g.t) - tw * uint32_t(p.tiles_x)) * BX + c_begin;
      g.ny = int64_t(tw) * kBW + eq * 32 + lane;
      g.whole = (ds > 0 || stage0 == 0) && (ds < nseg - 1 || u1 == (g.t + 1) * st_count);
      return g;
    };
    // a shared tile's parts are those of CTAs c_first .. c_last, in K order (found by
    // stepping from this CTA: a tile has few parts); c_last holds the tile's last part,
    // which no other shared tile ends in
    auto parts_of = [&](int64_t t, uint32_t& c_first, uint32_t& c_last) {
      const uint32_t t_lo = uint32_t(t) * uint32_t(st_count), t_hi = t_lo + st_count;
      c_first = blockIdx.x;
      c_last = blockIdx.x;
      while (split_begin(c_first, p) > t_lo) --c_first;
      while (split_begin(c_last + 1, p) < t_hi) ++c_last;
    };
    // ---- read-out of segments d0 .. d1 - 1 (warps 0..7; named barrier 1 over their 256
    // threads).  Whole tiles go to Y.  A shared tile goes to this CTA's partial slot (0 for
    // its first segment, 1 for its last: only those two can be shared), and the CTA
    // arrives at the counters of all its shared tiles in one round (one barrier, fence and
    // atomic each); the last of a tile's CTAs to arrive sums its parts into Y.
    auto drain = [&](int d0, int d1) {
      if (warp >= 8) return;
      int nshared = 0;
      int shared_seg[2] = {0, 0};
      for (int ds = d0; ds < d1; ++ds) {
        const int buf = kAcc == 1 ? 0 : (ds & 1);
        const bool mine = !failed && !*abort_flag &&
                          mbar_wait(acc_full(buf), uint32_t(ds / kAcc) & 1u) && !*abort_flag;
        if (!bar_and_256(mine)) {  // the same verdict in all 256 threads
          failed = true;
          return;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const SegAt g = seg_at(ds);
        const uint32_t t_acc = tmem + (static_cast<uint32_t>(eq * 32) << 16) + buf * BX +
                               c_begin;
        // kLd accumulator columns from c on: with several issuers, the sum of the partial
        // sums of those that issued a stage of the segment (local stages sa .. sb - 1), in
        // issuer order (deterministic)
        const int sa = seg_start(ds), sb = ds < nseg - 1 ? seg_start(ds + 1) : nl;
        auto read_acc = [&](int c, uint32_t(&v)[kLd]) {
          if constexpr (kIss == 1) {
            tmem_ld(t_acc + c, v);
          } else {
            bool any = false;
#pragma unroll
            for (int i = 0; i < kIss; ++i) {
              if (sa + (i - sa % kIss + kIss) % kIss >= sb) continue;  // no stage of issuer i
              uint32_t w[kLd];
              tmem_ld(t_acc + i * kAcc * BX + c, w);
#pragma unroll
              for (int j = 0; j < kLd; ++j)
                v[j] = any ? __float_as_uint(
                                 __fadd_rn(__uint_as_float(v[j]), __uint_as_float(w[j])))
                           : w[j];
              any = true;
            }
          }
        };
        if (g.whole) {
#pragma unroll 1
          for (int c = 0; c < kHalf; c += kLd) {
            if (g.m0 + c >= p.M) break;  // warp-uniform
            uint32_t v[kLd];
            read_acc(c, v);
            if (g.ny >= p.N) continue;
#pragma unroll
            for (int j = 0; j < kLd; ++j) {
              if (g.m0 + c + j >= p.M) break;
              store_y(g.m0 + c + j, g.ny, __uint_as_float(v[j]));
            }
          }
        } else {
          float* part = p.ws_part +
                        ((int64_t(blockIdx.x) * 2 + (ds == 0 ? 0 : 1)) * BX + c_begin) * kBW +
                        eq * 32 + lane;
#pragma unroll 1
          for (int c = 0; c < kHalf; c += kLd) {
            uint32_t v[kLd];
            read_acc(c, v);
#pragma unroll
            for (int j = 0; j < kLd; ++j) part[(c + j) * kBW] = __uint_as_float(v[j]);
          }
          shared_seg[nshared++] = ds;
        }
        // after its TMEM loads of the segment the warp hands the accumulator back
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(acc_empty(buf));
      }
      if (nshared == 0) return;
      // the barrier orders every thread's partials before thread 0's release (cumulative),
      // which the counters carry; the last arriver's acquire takes the others' partials, and
      // the second barrier hands them to its threads.  Both counters' atomics are in flight
      // at once.
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (tid == 0) {
        uint32_t cf0, cl0, cf1 = 0, cl1 = 0;
        parts_of(t0 + shared_seg[0], cf0, cl0);
        if (nshared > 1) parts_of(t0 + shared_seg[1], cf1, cl1);
        const int o0 = atomic_add_acq_rel(p.ws_count + cl0, 1);
        const int o1 = nshared > 1 ? atomic_add_acq_rel(p.ws_count + cl1, 1) : 0;
        s_last[0] = o0 == int(cl0 - cf0);
        s_last[1] = nshared > 1 && o1 == int(cl1 - cf1);
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
      for (int k = 0; k < nshared; ++k) {
        if (!s_last[k]) continue;
        const SegAt g = seg_at(shared_seg[k]);
        uint32_t c_first, c_last;
        parts_of(g.t, c_first, c_last);
        // part q is CTA c_first + q's first segment (slot 0), except that the tile may be
        // the last segment (slot 1) of CTA c_first, when that CTA began in an earlier tile
        const int slot0 = split_begin(c_first, p) < uint32_t(g.t) * uint32_t(st_count) ? 1 : 0;
        const int nparts = int(c_last - c_first + 1);
        auto part_of = [&](int q) {
          return p.ws_part +
                 ((int64_t(c_first + q) * 2 + (q == 0 ? slot0 : 0)) * BX + c_begin) * kBW +
                 eq * 32 + lane;
        };
#pragma unroll 1
        for (int c = 0; c < kHalf; c += kChunk) {
          // the loads of kBatch parts at a time before their sums (independent loads
          // overlap), parts added in K order, part 0 first
          float acc[kChunk];
#pragma unroll 1
          for (int q0 = 0; q0 < nparts; q0 += kBatch) {
            float x[kBatch][kChunk];
#pragma unroll
            for (int qq = 0; qq < kBatch; ++qq) {
              if (q0 + qq >= nparts) break;
              const float* src = part_of(q0 + qq) + c * kBW;
#pragma unroll
              for (int j = 0; j < kChunk; ++j) x[qq][j] = __ldcg(src + j * kBW);
            }
#pragma unroll
            for (int qq = 0; qq < kBatch; ++qq) {
              if (q0 + qq >= nparts) break;
#pragma unroll
              for (int j = 0; j < kChunk; ++j)
                acc[j] = q0 + qq == 0 ? x[qq][j] : __fadd_rn(acc[j], x[qq][j]);
            }
          }
          if (g.ny < p.N) {
#pragma unroll
            for (int j = 0; j < kChunk; ++j) {
              if (g.m0 + c + j >= p.M) break;
              store_y(g.m0 + c + j, g.ny, acc[j]);
            }
          }
        }
        if (tid == 0) p.ws_count[c_last] = 0;  // ready for the next call
      }
    };

    // the codes / absmax of this group's next two stages, rotated every stage (no
    // unrolling over stages: the loop body stays small enough for the instruction cache)
    uint32_t cA[kSub][kHalves], cB[kSub][kHalves];
    float aA[kSub][kHalves], aB[kSub][kHalves];
    uint64_t wA, wB;
    float mA, mB;
    Cursor cur = cursor_at(group);            // stage l
    Cursor pf = cursor_at(group + kGroups);   // stage l + 2 kGroups, once advanced below
    fetch(group, cur, cA, aA, wA, mA);
    fetch(group + kGroups, pf, cB, aB, wB, mB);
    advance(pf, kGroups);
    asm volatile("bar.arrive 3, %0;" :: "n"(kProducerWarps * 32 + 32) : "memory");
    // The pair table, built by the producer warps alone while the TMA warps start their
    // copies and the loads above are in flight: the entries' values by shuffle (entry b
    // copy g = word 16 b + g holds vcb[b >> 4], vcb[b & 15]); named barrier 2 over the
    // producer threads orders it and the scale codebook before their first lookup.
    if (tid < 256) s_scb[tid] = scb_v;
    for (int i = tid; i < 256 * 16; i += kProducerWarps * 32) {
      const int b = i >> 4;
      float2 e;
      e.x = __shfl_sync(kFull, vcb_v, b >> 4);
      e.y = __shfl_sync(kFull, vcb_v, b & 15);
      *reinterpret_cast<float2*>(base + S::kTabOff + 8 * i) = e;
    }
    asm volatile("bar.sync 2, %0;" :: "n"(kProducerWarps * 32) : "memory");
    RingPos<kAS> apos;
    RingPos<kRawS> rpos;
    for (int g = 0; g < group; ++g) {  // this group's first stage
      apos.next();
      rpos.next();
    }
    bool timed_out = false;
    int next_drain = 0;  // the next segment to read out
    // this lane's copy of the pair table: entry b at tab + 128 b
    const uint32_t tab = sbase + S::kTabOff + (lane & 15) * 8;
    const int flip = (r >> 2) & 1;  // the raw boxes' 32-byte swizzle for this row
    // Segment d is read out kAS stages into segment d + 1 (before the first stage whose
    // weight slot waits for MMAs that may need its accumulator buffer back; the MMAs then
    // have those kAS stages queued when they get it), the last one after the last stage.
    // Reading a CTA's first segment out early lets the CTAs that share its tile finish
    // that tile without it, so each CTA completes at most one tile at its end.  Narrow
    // tiles whose segments all have accumulator buffers of their own read every segment
    // out after the last stage instead: the MMAs never wait for a buffer then, and the
    // decoding warps do not stop mid-run (measured at N = 11008, K = 4096: M = 16 17.5 ->
    // 16.5 us, M = 32 18.4 -> 17.3 us).
    // The stage loop runs up to the next read-out, so the read-out code stays out of it.
    constexpr bool kNarrow = BX <= 32;
    const bool drain_at_end = kNarrow && nseg <= kAcc;
    int l = group;  // this group's next local stage
    int lim = 0;    // the stages before the next read-out
    for (;;) {
      lim = drain_at_end || next_drain >= nseg - 1
                ? nl
                : min(nl, seg_start(next_drain + 1) + kAS);
      for (; l < lim; l += kGroups) {  // local stage l
        unpack(wA, mA, cA, aA);  // loaded an iteration ago
        float sc[kSub][kHalves];
  #pragma unroll
        for (int sub = 0; sub < kSub; ++sub)
  #pragma unroll
          for (int hh = 0; hh < kHalves; ++hh) {  // two roundings, never an FMA
            sc[sub][hh] = __fadd_rn(__fmul_rn(s_scb[cA[sub][hh]], aA[sub][hh]), offset);
            cA[sub][hh] = cB[sub][hh];
            aA[sub][hh] = aB[sub][hh];
          }
        wA = wB;
        mA = mB;
        fetch(l + 2 * kGroups, pf, cB, aB, wB, mB);
        advance(pf, kGroups);
        // the raw stage has landed and the MMAs that read this weight slot last completed
        // (the first kAS stages have nothing to wait for: their empty phase reads as done)
        bool ok = !*abort_flag &&
                  (mbar_try2(raw_full(rpos.slot), rpos.phase, empty_a(apos.slot),
                             l >= kAS ? apos.phase ^ 1u : 1u) ||
                   (mbar_wait(raw_full(rpos.slot), rpos.phase) &&
                    (l < kAS || mbar_wait(empty_a(apos.slot), apos.phase ^ 1u))));
        if (!__all_sync(kFull, ok)) {  // warp-uniform, so the warp stays converged
          timed_out = failed = true;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const int ns = min(kSub, kt_count - cur.stage * kSub);
        // rows are 32 bytes apart in each raw box, whose 32-byte swizzle stores the 16-byte
        // chunk c of row r at chunk c ^ ((r >> 2) & 1): the 8 rows a quarter warp reads then
        // fill all 32 banks
        const uint32_t raw_row = sbase + S::kRawOff + rpos.slot * S::kRawSlot + r * 32;
        const uint32_t t_stage = t_row + apos.slot * kSub * 32;
  #pragma unroll 1
        for (int sub = 0; sub < ns; ++sub) {
          // this K step's scales, picked by selects rather than a register-array index
          uint64_t sc2[kHalves];
  #pragma unroll
          for (int hh = 0; hh < kHalves; ++hh) {
            float v = sc[0][hh];
  #pragma unroll
            for (int k = 1; k < kSub; ++k) v = sub == k ? sc[k][hh] : v;
            asm("mov.b64 %0, {%1, %1};" : "=l"(sc2[hh]) : "f"(v));
          }
          uint32_t wd[kWords];
          const uint32_t row = raw_row + sub * kRawBytes;
  #pragma unroll
          for (int v = 0; v < (kWords + 3) / 4; ++v) {
            const int chunk = (kWords * h) / 4 + v;  // logical 16-byte chunk of the row
            const uint32_t src = row + (((chunk ^ flip) & 1) << 4) + ((kWords * h) % 4) * 4;
            if constexpr (kWords >= 4) {
              const uint4 w4 = lds_v4(src);
              wd[4 * v] = w4.x, wd[4 * v + 1] = w4.y, wd[4 * v + 2] = w4.z, wd[4 * v + 3] = w4.w;
            } else {
              const uint2 w2 = lds_v2(src);
              wd[0] = w2.x, wd[1] = w2.y;
            }
          }
          uint32_t o[4 * kWords];  // 8 values per word, two per 32-bit TMEM column
  #pragma unroll
          for (int e = 0; e < kWords; ++e) {
  #pragma unroll
            for (int j = 0; j < 4; ++j) {
              // byte j's pair (earlier value = high nibble, later = low nibble)
              const uint32_t byte = __byte_perm(wd[e], 0, 0x4440 + j);
              float v0, v1;
              mul2_rn64(lds_b64(tab + (byte << 7)), sc2[e / 4 < kHalves ? e / 4 : 0], v0, v1);
              o[4 * e + j] = pack2<kOut>(v0, v1);
            }
          }
          // rows past N hold finite values (zero codes, zero-filled nibbles) and only feed
          // accumulator lanes that are never stored
          tmem_st<4 * kWords>(t_stage + sub * 32, o);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(full_w(apos.slot));
          mbar_arrive(raw_empty(rpos.slot));
        }
  #pragma unroll
        for (int g = 0; g < kGroups; ++g) {
          apos.next();
          rpos.next();
        }
        advance(cur, kGroups);
      }
      if (timed_out) {
        if (lane == 0) fail();
        timed_out = false;
      }
      // every segment is read out, failed or not (each read-out takes all epilogue threads)
      if (next_drain >= nseg) break;
      drain(next_drain, next_drain + 1);
      ++next_drain;
      if (failed) l = nl;  // no more stages
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(tmem), "r"(kTmemCols));
  }
}

// ------------------------------------------------------------- host side
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
  cfg.blockDim = dim3(kThreadsOf(BX));
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
  kernel<<<static_cast<unsigned>(grid), kThreadsOf(BX), S::kBytes, stream>>>(tx, tw, p);
  return check_launch();
#endif
}

// How a problem runs: the activation-tile width BX, the CTAs and the workspace.
struct LinPlan {
  int bx = 16;
  int64_t tiles_x = 0, tiles = 0;
  int st_count = 0;
  int ctas = 0;                          // == tiles: one CTA per tile, each whole
  int64_t count_bytes = 0, ws_bytes = 0;  // a split's counters and whole workspace
};

// Plans by estimated time, in units of 1/800 of a weight stage: a stage of BX columns
// costs 640 + BX (dequantization with the shared-memory reads it contends for, and the
// MMAs), a CTA about 2400 more (pipeline fill, drain and read-out), and a split CTA the
// partial tiles' stores and sums, about 1600 + 15 BX (two FP32 partials of 128 x BX each
// go out and come back, at the end of the run when every SM does the same) plus, for
// BX >= 128, 12 BX per CTA beyond two sharing a tile (its last arriver sums that many
// partials of 64 KB or more: with 4 to 17 sharers such splits lost to whole tiles at
// N = K = 4096, M = 128 .. 512 and at N <= 1024, and with 2 they won by 12 to 25 % at
// N = 9856; narrower tiles' partials are small, and their splits kept winning), and a
// read-out per tile boundary it crosses: hidden with two accumulator buffers per issuer,
// about 400 with one buffer and one issuer, and 2000 with one buffer for each of two
// issuers (both wait at the boundary; measured at BX = 64, where whole tiles win).  The
// widths tried are the powers of two from 16 up to the first one >= M.  With split false
// only whole-tile plans count.
LinPlan plan_linear(int64_t M, int64_t N, int64_t K, int sms, bool split) {
  LinPlan best;
  int64_t best_cost = INT64_MAX;
  const int st_count = int((K / kBK + kSub - 1) / kSub);
  for (int bx = 16; bx <= 256; bx *= 2) {
    LinPlan pl;
    pl.bx = bx;
    pl.st_count = st_count;
    pl.tiles_x = (M + bx - 1) / bx;
    pl.tiles = pl.tiles_x * ((N + kBW - 1) / kBW);
    const int64_t units = pl.tiles * st_count;
    const int64_t stage_cost = 640 + bx;
    // one CTA per tile, rounds of sms at a time
    const int64_t rounds = (pl.tiles + sms - 1) / sms;
    int64_t cost = rounds * (st_count * stage_cost + 2400);
    pl.ctas = int(pl.tiles < INT32_MAX ? pl.tiles : INT32_MAX);
    // one CTA per SM, an equal share of the units each (the kernel's unit arithmetic is
    // 32-bit: units < 2^32, sms < 2^16)
    if (split && units >= sms && units <= int64_t(UINT32_MAX) && sms < 65536) {
      const int64_t per_cta = (units + sms - 1) / sms;
      const int64_t crossings = (per_cta + st_count - 1) / st_count;
      // CTAs sharing a tile, whose 128 x BX FP32 partials its last arriver sums
      const int64_t parts = (st_count + per_cta - 1) / per_cta + 1;
      const int64_t split_cost =
          per_cta * stage_cost + 2400 + 1600 + 15 * bx +
          (bx >= 128 && parts > 2 ? 12 * bx * (parts - 2) : 0) +
          (kAccOf(bx) == 1 ? (kIssOf(bx) > 1 ? 2000 : 400) * crossings : 0);
      if (split_cost < cost) {
        cost = split_cost;
        pl.ctas = sms;
        // the counters come first and sit at the same offsets for every problem on this
        // device (one per CTA, at most one per SM), so a workspace reused across problems
        // never reads another problem's partial tiles as counters
        pl.count_bytes = (int64_t(sms) * 4 + 255) / 256 * 256;
        pl.ws_bytes = pl.count_bytes + int64_t(sms) * 2 * bx * kBW * 4;
      }
    }
    if (cost < best_cost) {
      best_cost = cost;
      best = pl;
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
                      int32_t nested_blocksize, int32_t out_dtype, void* Y, void* workspace,
                      int64_t workspace_bytes, int* bad, void* stream) {
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
      misaligned(Y, out_itemsize(out_dtype)) || misaligned(bad, 4) || misaligned(workspace, 256))
    return DQ4_ERR_ALIGN;
  int dev = 0, sms = 0;
  if (int st = current_device(&dev, &sms)) return st;
  EncodeTiled encode = tensor_map_encoder();
  if (!encode) return fail_cuda(DQ4_ERR_LAUNCH, cudaErrorNotSupported);

  // a split needs the workspace; without one large enough, every CTA takes a whole tile
  LinPlan pl = plan_linear(M, N, K, sms, true);
  if (pl.ws_bytes > 0 && (!workspace || workspace_bytes < pl.ws_bytes))
    pl = plan_linear(M, N, K, sms, false);
  if (pl.tiles > INT32_MAX) return DQ4_ERR_N;
  const int bx = pl.bx;
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
  // the packed weight as N rows of K / 2 bytes: 32 x 128 boxes, 32-byte swizzle
  CUtensorMap tw;
  const cuuint64_t wdim[2] = {static_cast<cuuint64_t>(K / 2), static_cast<cuuint64_t>(N)};
  const cuuint64_t wstride[1] = {static_cast<cuuint64_t>(K / 2)};
  const cuuint32_t wbox[2] = {kBK / 2, kBW};
  cr = encode(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(packed), wdim,
              wstride, wbox, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_32B,
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
  p.tiles_x = static_cast<int>(pl.tiles_x);
  const bool split = pl.ws_bytes > 0;
  p.whole = split ? 0 : 1;
  p.ctas = pl.ctas;
  p.units = split ? uint32_t(pl.tiles * pl.st_count) : 0;
  p.units_q = split ? p.units / uint32_t(pl.ctas) : 0;
  p.units_r = split ? p.units % uint32_t(pl.ctas) : 0;
  p.ws_count = split ? static_cast<int*>(workspace) : nullptr;
  p.ws_part = split ? reinterpret_cast<float*>(static_cast<char*>(workspace) + pl.count_bytes)
                    : nullptr;
  {
    // a stage covers 64 kSub values of a row, starting at a multiple of that when K is
    // one; its codes are then blocks b00 .. b00 + window - 1 with b00 a multiple of the
    // window, all in one absmax group when the window is at most nested_blocksize
    const int64_t span = int64_t(kBK) * kSub;
    int64_t window = span / blocksize;
    if (window < 1) window = 1;
    p.code_window = (K % span == 0 && window <= nested_blocksize && window <= 8 &&
                     !misaligned(scale_codes, static_cast<int>(window)))
                        ? static_cast<int>(window)
                        : 0;
  }
  const auto st = static_cast<cudaStream_t>(stream);
  const int64_t grid = pl.ctas;
  return in_dtype == DQ4_OUT_BF16 ? launch_bx<true>(bx, tx, tw, p, grid, st, dev)
                                  : launch_bx<false>(bx, tx, tw, p, grid, st, dev);
}

int64_t dq4_nested_linear_workspace_bytes(int64_t M, int64_t N, int64_t K) {
  if (M <= 0 || N <= 0 || K <= 0 || K % kBK != 0 || M > INT32_MAX || N > INT32_MAX ||
      K > INT32_MAX)
    return 0;
  int dev = 0, sms = 0;
  if (current_device(&dev, &sms) != DQ4_OK) return -DQ4_ERR_DEVICE;
  return plan_linear(M, N, K, sms, true).ws_bytes;
}

}  // extern "C"

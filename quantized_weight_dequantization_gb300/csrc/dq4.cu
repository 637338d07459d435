// Blockwise 4-bit dequantization with nested (double-quantized) scales for
// GB300 (sm_103a): the kernels and the C-ABI entry points declared in
// include/dq4.h.
//
// Operation: "Fuse nested scale reconstruction into SM103 4-bit
// dequantization" (bitsandbytes issue #21), section "Proposed experiment":
//   scale = scale_codebook[scale_code] * nested_absmax[nested_group] + offset
//   value = decode_4bit(packed_value) * scale
// with the multiply and the add of the scale rounded separately (section
// "Correctness requirements").  __fmul_rn / __fadd_rn are never contracted
// into an FMA, and the library is also compiled with -fmad=false.
//
// Design (a streaming, HBM-bound map; no tensor cores):
//  * A warp owns a tile of 32*U consecutive "words" (U = 8).  A word is the
//    packed data of 16 output bytes: 8 values (4 packed bytes) for FP16/BF16
//    output, 4 values (2 packed bytes) for FP32.  Lane l handles words
//    tile + 32k + l, so each packed load and each 16-byte output store of a
//    warp covers one contiguous, fully used span.
//  * The grid covers the whole array, one tile per warp: the hardware hands
//    out CTAs in index order, so the addresses in flight at any time form one
//    compact window moving through HBM.  (On GB300 this beats a persistent
//    grid-stride loop by ~13% for this 1:4 read:write stream.)  Only if the
//    grid would exceed the launch limit do warps loop over several tiles,
//    loading the next tile before decoding the current one.
//  * blocksize >= 32 is a power of two, so a word never straddles two outer
//    blocks.  The tile's blocks are consecutive; lane j rebuilds the scale of
//    the tile's blocks j, j+32, ... and each word takes its scale by a warp
//    shuffle: one scale code, one nested absmax and one codebook lookup per
//    block, never an FP32 scale array.
//  * The 16-entry value codebook sits in shared memory (banks 0..15, so the
//    data-dependent lookups of a warp never conflict); the 256-entry scale
//    codebook too.
//  * Packed loads and output stores use the streaming (evict-first) cache
//    hint: every byte is touched once.
//  * Launched with programmatic dependent launch: CTAs of a launch may be
//    scheduled while the previous kernel in the stream finishes, and wait
//    for its completion (griddepcontrol.wait) before touching memory.
//  * Values after the last whole word (fewer than one word, including an
//    odd padding nibble) are written one by one by CTA 0.  Unaligned
//    `packed` / `out` pointers take a per-value kernel with the same math.
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include <cublas_v2.h>  // types only: cuBLAS is reached through dlopen / dlsym
#include <dlfcn.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <utility>

#include "dq4.h"

namespace {

#ifndef DQ4_THREADS
#define DQ4_THREADS 256
#endif
constexpr int kThreads = DQ4_THREADS;
constexpr int kWarpsPerCta = kThreads / 32;
constexpr int kMaxDevices = 64;
constexpr int64_t kMaxGrid = 2147483647;  // gridDim.x limit
constexpr int kAbiVersion = 1;

thread_local int t_last_cuda_error = 0;

// ------------------------------------------------------------------ args
struct Args {
  const uint8_t* packed;
  const uint8_t* codes;   // scale codes (nested form only)
  const float* absmax;    // nested absmax (nested form) or per-block absmax
  const float* scb;       // scale codebook (nested form only)
  const float* vcb;       // value codebook
  void* out;
  int64_t n;
  int64_t first;  // per-value kernel: output i is the value first + i (0 elsewhere)
  int64_t nblocks;
  float offset;
  int log2_bs;
  int log2_nbs;
};

template <int OUT>
struct Traits;
template <>
struct Traits<DQ4_OUT_F16> {
  using Word = uint32_t;
  static constexpr int kLog2Vals = 3;
};
template <>
struct Traits<DQ4_OUT_BF16> {
  using Word = uint32_t;
  static constexpr int kLog2Vals = 3;
};
template <>
struct Traits<DQ4_OUT_F32> {
  using Word = uint16_t;
  static constexpr int kLog2Vals = 2;
};

// Words per lane per warp tile (tunable at build time).  A tile of 32*U
// words touches at most 32*U >> log2(words per block) outer blocks; each
// lane rebuilds J = ceil(that / 32) of their scales.
#ifndef DQ4_U_HALF
#define DQ4_U_HALF 8
#endif
#ifndef DQ4_U_F32
#define DQ4_U_F32 8
#endif
// 1: a warp loads its next tile before it decodes the current one.
#ifndef DQ4_PREFETCH
#define DQ4_PREFETCH 1
#endif
// packed-word loads: 0 streaming (ld.global.cs), 1 read-only non-coherent (ld.global.nc)
#ifndef DQ4_LD_HINT
#define DQ4_LD_HINT 0
#endif
// output stores: 0 streaming (st.global.cs), 1 default write-back
#ifndef DQ4_ST_HINT
#define DQ4_ST_HINT 0
#endif
// 0: one tile per warp over the whole array; k > 0: at most k CTAs per SM
// (a persistent grid-stride loop)
#ifndef DQ4_CTAS_PER_SM
#define DQ4_CTAS_PER_SM 0
#endif

// 1: a warp issues its first tile's loads before the CTA stages the
// codebooks (measured ~1% slower on GB300, so off).
#ifndef DQ4_EARLY_LOADS
#define DQ4_EARLY_LOADS 0
#endif
// 1: launch the tile kernel with programmatic stream serialization: its CTAs
// may be scheduled while the previous kernel in the stream drains its last
// wave, and wait (griddepcontrol.wait) for that kernel's completion before
// any memory access, so stream order is kept.  Worth 2-18% on GB300 for
// back-to-back launches (most on small arrays).
#ifndef DQ4_PDL
#define DQ4_PDL 1
#endif

template <int OUT>
struct Tile {
  static constexpr int U = (OUT == DQ4_OUT_F32) ? DQ4_U_F32 : DQ4_U_HALF;
  static constexpr int kWshiftMin = 5 - Traits<OUT>::kLog2Vals;  // blocksize >= 32
  static constexpr int kBlocksMax = (32 * U) >> kWshiftMin;
  static constexpr int J = kBlocksMax > 32 ? kBlocksMax / 32 : 1;
  static_assert(J <= 4, "at most four scale registers per lane");
};

// ------------------------------------------------------------- device math
__device__ __forceinline__ float nested_scale(const Args& a, const float* s_scb, int64_t b) {
  const float A = __ldg(a.absmax + (b >> a.log2_nbs));
  const float c = s_scb[__ldg(a.codes + b)];
  return __fadd_rn(__fmul_rn(c, A), a.offset);  // two roundings, never an FMA
}

template <bool NESTED>
__device__ __forceinline__ float block_scale(const Args& a, const float* s_scb, int64_t b) {
  if constexpr (NESTED) {
    return nested_scale(a, s_scb, b);
  } else {
    return __ldg(a.absmax + b);
  }
}

template <int OUT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  uint32_t u;
  if constexpr (OUT == DQ4_OUT_F16) {
    const __half2 h = __floats2half2_rn(lo, hi);
    memcpy(&u, &h, sizeof u);
  } else {
    const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    memcpy(&u, &h, sizeof u);
  }
  return u;
}

// 16 output bytes from one packed word and its block's scale.
template <int OUT>
__device__ __forceinline__ uint4 decode_word(typename Traits<OUT>::Word w, float s,
                                             const float* vcb) {
  uint32_t r[4];
  if constexpr (OUT == DQ4_OUT_F32) {
#pragma unroll
    for (int j = 0; j < 2; ++j) {  // byte j -> values 2j (high nibble), 2j+1 (low)
      const uint32_t byte = (uint32_t(w) >> (8 * j)) & 0xFFu;
      r[2 * j] = __float_as_uint(__fmul_rn(vcb[byte >> 4], s));
      r[2 * j + 1] = __float_as_uint(__fmul_rn(vcb[byte & 0xFu], s));
    }
  } else {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint32_t byte = (w >> (8 * j)) & 0xFFu;
      r[j] = pack2<OUT>(__fmul_rn(vcb[byte >> 4], s), __fmul_rn(vcb[byte & 0xFu], s));
    }
  }
  return make_uint4(r[0], r[1], r[2], r[3]);
}

template <bool NESTED>
__device__ __forceinline__ float value_at(const Args& a, const float* s_scb, const float* s_vcb,
                                          int64_t i) {
  const uint32_t byte = a.packed[i >> 1];
  const uint32_t nib = (i & 1) ? (byte & 0xFu) : (byte >> 4);
  return __fmul_rn(s_vcb[nib], block_scale<NESTED>(a, s_scb, i >> a.log2_bs));
}

template <int OUT>
__device__ __forceinline__ void store_one(void* out, int64_t i, float v) {
  if constexpr (OUT == DQ4_OUT_F16) {
    static_cast<__half*>(out)[i] = __float2half_rn(v);
  } else if constexpr (OUT == DQ4_OUT_BF16) {
    static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
  } else {
    static_cast<float*>(out)[i] = v;
  }
}

template <bool NESTED>
__device__ __forceinline__ void stage_codebooks(const Args& a, float* s_vcb, float* s_scb) {
  if (threadIdx.x < 16) s_vcb[threadIdx.x] = __ldg(a.vcb + threadIdx.x);
  if constexpr (NESTED) {
    for (int k = threadIdx.x; k < 256; k += blockDim.x) s_scb[k] = __ldg(a.scb + k);
  }
  __syncthreads();
}

// ---------------------------------------------------------------- kernels
template <typename Word>
__device__ __forceinline__ Word load_word(const Word* p) {
#if DQ4_LD_HINT == 0
  return __ldcs(p);
#else
  return __ldg(p);
#endif
}

__device__ __forceinline__ void store_16(uint4* p, uint4 v) {
#if DQ4_ST_HINT == 0
  __stcs(p, v);
#else
  *p = v;
#endif
}

// Registers of one warp tile: U packed words per lane, and the raw scale
// inputs (code, absmax) of up to J blocks per lane.
template <int OUT>
struct TileRegs {
  typename Traits<OUT>::Word w[Tile<OUT>::U];
  uint32_t code[Tile<OUT>::J];
  float am[Tile<OUT>::J];
};

template <int OUT, bool NESTED>
__device__ __forceinline__ void load_tile(const Args& a, int64_t base, int64_t n_words, int wshift,
                                          int lane, TileRegs<OUT>& r) {
  using Word = typename Traits<OUT>::Word;
  constexpr int U = Tile<OUT>::U;
  constexpr int64_t kTile = 32 * U;
  const Word* pw = reinterpret_cast<const Word*>(a.packed);
#pragma unroll
  for (int k = 0; k < U; ++k) {
    const int64_t wi = base + k * 32 + lane;
    r.w[k] = wi < n_words ? load_word(pw + wi) : Word(0);
  }
  const int64_t b0 = base >> wshift;
  const int64_t b_last = ((base + kTile < n_words ? base + kTile : n_words) - 1) >> wshift;
#pragma unroll
  for (int j = 0; j < Tile<OUT>::J; ++j) {
    const int64_t b = b0 + lane + 32 * j;
    r.code[j] = 0;
    r.am[j] = 0.f;
    if (b <= b_last) {
      if constexpr (NESTED) {
        r.code[j] = __ldg(a.codes + b);
        r.am[j] = __ldg(a.absmax + (b >> a.log2_nbs));
      } else {
        r.am[j] = __ldg(a.absmax + b);
      }
    }
  }
}

template <int OUT, bool NESTED>
__device__ __forceinline__ void decode_tile(const Args& a, int64_t base, int64_t n_words,
                                            int wshift, int lane, const TileRegs<OUT>& r,
                                            const float* s_scb, const float* s_vcb) {
  constexpr int U = Tile<OUT>::U;
  constexpr int J = Tile<OUT>::J;
  float sc[J];
#pragma unroll
  for (int j = 0; j < J; ++j) {
    if constexpr (NESTED) {
      sc[j] = __fadd_rn(__fmul_rn(s_scb[r.code[j]], r.am[j]), a.offset);  // never an FMA
    } else {
      sc[j] = r.am[j];
    }
  }
  uint4* po = reinterpret_cast<uint4*>(a.out);
  const int64_t b0 = base >> wshift;
#pragma unroll
  for (int k = 0; k < U; ++k) {
    const int64_t wi = base + k * 32 + lane;
    const int idx = int((wi >> wshift) - b0);  // the word's block within the tile
    // idx >> 5 == k >> wshift for every lane, so the register choice is warp-uniform
    float src = sc[0];
#pragma unroll
    for (int j = 1; j < J; ++j)
      if ((k >> wshift) == j) src = sc[j];
    const float s = __shfl_sync(0xffffffffu, src, idx & 31);
    if (wi < n_words) store_16(po + wi, decode_word<OUT>(r.w[k], s, s_vcb));
  }
}

template <int OUT, bool NESTED>
__global__ void __launch_bounds__(kThreads) dq4_vec_kernel(const Args a) {
  using T = Traits<OUT>;
  constexpr int64_t kTile = 32 * Tile<OUT>::U;
  __shared__ float s_vcb[16];
  __shared__ float s_scb[NESTED ? 256 : 1];
#if DQ4_PDL
  // No global memory is touched before the previous grid in the stream has
  // completed; dependents may be scheduled once every CTA here has started.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
#endif

  const int64_t n_words = a.n >> T::kLog2Vals;
  const int wshift = a.log2_bs - T::kLog2Vals;  // log2(words per outer block)
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t stride = ((int64_t(gridDim.x) * kThreads) >> 5) * kTile;

  int64_t base = warp * kTile;
  const bool active = base < n_words;  // warp-uniform
  TileRegs<OUT> cur;
#if DQ4_EARLY_LOADS
  if (active) load_tile<OUT, NESTED>(a, base, n_words, wshift, lane, cur);
  stage_codebooks<NESTED>(a, s_vcb, s_scb);
#else
  stage_codebooks<NESTED>(a, s_vcb, s_scb);
  if (active) load_tile<OUT, NESTED>(a, base, n_words, wshift, lane, cur);
#endif
  if (active) {
    for (;;) {
      const int64_t next = base + stride;
      const bool more = next < n_words;  // warp-uniform
#if DQ4_PREFETCH
      TileRegs<OUT> nxt;
      if (more) load_tile<OUT, NESTED>(a, next, n_words, wshift, lane, nxt);
      decode_tile<OUT, NESTED>(a, base, n_words, wshift, lane, cur, s_scb, s_vcb);
      if (!more) break;
      cur = nxt;
#else
      decode_tile<OUT, NESTED>(a, base, n_words, wshift, lane, cur, s_scb, s_vcb);
      if (!more) break;
      load_tile<OUT, NESTED>(a, next, n_words, wshift, lane, cur);
#endif
      base = next;
    }
  }

  // fewer than one word of values remains after the last whole word
  const int64_t tail0 = n_words << T::kLog2Vals;
  if (blockIdx.x == 0 && tail0 + threadIdx.x < a.n) {
    const int64_t i = tail0 + threadIdx.x;
    store_one<OUT>(a.out, i, value_at<NESTED>(a, s_scb, s_vcb, i));
  }
}

// ------------------------------------------------------ transposed output
// The flat values are the row-major rows x cols weight W; the output is W^T
// row-major: element (r, c) of W goes to out[c * rows + r].
// A warp owns a tile of 64 rows x 64 columns of W, and lane p owns the rows
// r0 + 2p and r0 + 2p + 1 of it: it reads the 32-byte packed segment of each
// of its two rows (two 16-byte loads per row) and decodes 8 columns at a
// time.  For every column c the warp then holds the whole 64-value output
// segment out[c * rows + r0 .. + 64), and lane p writes its pair (rows 2p,
// 2p + 1) with one 4-byte store (8 bytes for FP32): 128 B (256 B)
// contiguous per warp store instruction, with no shared-memory staging.
// Tiles are walked in column-major order (consecutive warps go down a
// column band), so consecutive warps extend the same output rows.
// kLoadVec: cols % 32 == 0 and `packed` 16-byte aligned (every row segment
// is two aligned 16-byte loads); otherwise values are read one by one.
// kStoreVec: rows is even and `out` is aligned to two elements (pair
// stores); otherwise elements are stored one by one.
constexpr int kTR = 64;  // warp-tile rows of W
constexpr int kTC = 64;  // warp-tile columns of W

template <int OUT>
__device__ __forceinline__ uint32_t out_bits(float v) {
  if constexpr (OUT == DQ4_OUT_F16) {
    return __half_as_ushort(__float2half_rn(v));
  } else if constexpr (OUT == DQ4_OUT_BF16) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
  } else {
    return __float_as_uint(v);
  }
}

// Store the values of rows (r, r + 1) at column c of W into W^T.
// `o` is the element index of (r, c) in W^T: c * rows + r.
template <int OUT, bool kStoreVec>
__device__ __forceinline__ void store_pair(void* out, int64_t o, float v0, float v1, bool has0,
                                           bool has1) {
  if constexpr (OUT == DQ4_OUT_F32) {
    if (kStoreVec && has1) {
      __stcs(reinterpret_cast<uint2*>(static_cast<float*>(out) + o),
             make_uint2(__float_as_uint(v0), __float_as_uint(v1)));
    } else {
      if (has0) static_cast<float*>(out)[o] = v0;
      if (has1) static_cast<float*>(out)[o + 1] = v1;
    }
  } else {
    if (kStoreVec && has1) {
      __stcs(reinterpret_cast<unsigned int*>(static_cast<uint16_t*>(out) + o),
             pack2<OUT>(v0, v1));  // one conversion for the pair; row r at the lower address
    } else {
      if (has0) static_cast<uint16_t*>(out)[o] = uint16_t(out_bits<OUT>(v0));
      if (has1) static_cast<uint16_t*>(out)[o + 1] = uint16_t(out_bits<OUT>(v1));
    }
  }
}

// Staged form (cols % 32 == 0, `packed` 16-byte aligned).  A CTA owns 128 rows
// x 256 columns of W: its packed bytes (128 B per row, whole cache lines) and
// the scales of its 32-value row segments are first loaded cooperatively and
// coalesced into shared memory; then each warp decodes one 64 x 64 warp tile
// from shared memory and stores it as above.  CTAs are walked in column-major
// order.
constexpr int kSR = 128;                 // CTA tile rows
constexpr int kSC = 256;                 // CTA tile columns (128 packed bytes per row)
constexpr int kSRowBytes = kSC / 2;      // smem row: 8 chunks of 16 B, XOR-swizzled
constexpr int kSSeg = kSC / 32;          // 32-value scale segments per row

// 16-byte chunk `ch` of staged row `rr` sits at chunk position ch ^ key(rr):
// lanes reading rows 2p (and 2p + 1) of 8 consecutive p then hit 8 distinct
// chunk positions, i.e. all 32 banks.
__device__ __forceinline__ int swz(int rr, int ch) { return ch ^ ((rr >> 1) & 7); }

// minimum resident CTAs per SM the staged transposed kernel is compiled for
#ifndef DQ4_T_MIN_CTAS
#define DQ4_T_MIN_CTAS 8
#endif

template <int OUT, bool kStoreVec>
__global__ void __launch_bounds__(kThreads, DQ4_T_MIN_CTAS)
    dq4_transposed_kernel(const Args a, int64_t rows, int64_t cols, uint32_t tiles_r) {
  __shared__ float s_vcb[16];
  __shared__ float s_scb[256];
  __shared__ __align__(16) uint8_t s_pk[kSR][kSRowBytes];
  __shared__ __align__(8) float s_sc[kSSeg][kSR];  // [segment][row]: a lane's 2 rows are a float2
#if DQ4_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
#endif
  if (threadIdx.x < 16) s_vcb[threadIdx.x] = __ldg(a.vcb + threadIdx.x);
  for (int k = threadIdx.x; k < 256; k += kThreads) s_scb[k] = __ldg(a.scb + k);
  const int64_t r0 = int64_t(blockIdx.x % tiles_r) * kSR;  // column-major CTA order
  const int64_t c0 = int64_t(blockIdx.x / tiles_r) * kSC;

  // packed rows: 8 x 16 B per row; a warp reads 4 whole rows per instruction
#pragma unroll
  for (int k = 0; k < kSR * 8 / kThreads; ++k) {
    const int id = threadIdx.x + kThreads * k;
    const int rr = id >> 3, ch = id & 7;
    const int64_t r = r0 + rr, c = c0 + 32 * ch;
    uint4 v = make_uint4(0, 0, 0, 0);
    if (r < rows && c < cols)
      v = __ldcs(reinterpret_cast<const uint4*>(a.packed + ((r * cols + c) >> 1)));
    *reinterpret_cast<uint4*>(&s_pk[rr][16 * swz(rr, ch)]) = v;
  }
  __syncthreads();  // codebooks staged
  // scales of the 32-value segments (bs >= 32 and cols % 32 == 0: one block each)
#pragma unroll
  for (int k = 0; k < kSR * kSSeg / kThreads; ++k) {
    const int id = threadIdx.x + kThreads * k;
    const int rr = id / kSSeg, q = id % kSSeg;
    const int64_t r = r0 + rr, c = c0 + 32 * q;
    s_sc[q][rr] = (r < rows && c < cols) ? nested_scale(a, s_scb, (r * cols + c) >> a.log2_bs)
                                         : 0.f;
  }
  __syncthreads();

  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wr = 64 * (w >> 2);  // warp tile: rows wr .. +64, columns wc .. +64 of the CTA tile
  const int wc = 64 * (w & 3);
  const int64_t ra = r0 + wr + 2 * lane;  // this lane's rows: ra, ra + 1
  const bool has0 = ra < rows, has1 = ra + 1 < rows;
  if (!has0) return;
  const int64_t cbase = c0 + wc;
  const int ncol = int(cols - cbase < 64 ? cols - cbase : 64);
  if (ncol <= 0) return;
  const int lr = wr + 2 * lane;  // local row of ra
  int64_t o = cbase * rows + ra;  // W^T index of (ra, column); advances by rows per column
#pragma unroll
  for (int q = 0; q < 2; ++q) {
    if (32 * q >= ncol) break;
    const int ch = wc / 32 + q;  // 16-byte chunk of this 32-column half
    const uint4 s0 = *reinterpret_cast<const uint4*>(&s_pk[lr][16 * swz(lr, ch)]);
    const uint4 s1 = *reinterpret_cast<const uint4*>(&s_pk[lr + 1][16 * swz(lr + 1, ch)]);
    const float2 scp = *reinterpret_cast<const float2*>(&s_sc[ch][lr]);
    const float sc0 = scp.x, sc1 = scp.y;
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // packed word k: 8 columns
      const uint32_t w0 = k == 0 ? s0.x : k == 1 ? s0.y : k == 2 ? s0.z : s0.w;
      const uint32_t w1 = k == 0 ? s1.x : k == 1 ? s1.y : k == 2 ? s1.z : s1.w;
#pragma unroll
      for (int j = 0; j < 8; ++j) {  // value j of a word: byte j/2, high nibble first
        const int sh = 8 * (j >> 1) + ((j & 1) ? 0 : 4);
        const float v0 = __fmul_rn(s_vcb[(w0 >> sh) & 0xFu], sc0);
        const float v1 = __fmul_rn(s_vcb[(w1 >> sh) & 0xFu], sc1);
        store_pair<OUT, kStoreVec>(a.out, o, v0, v1, has0, has1);
        o += rows;
      }
    }
  }
}

// Per-value form for other shapes: a warp owns 64 rows x 64 columns, lane p
// the rows r0 + 2p and r0 + 2p + 1, read value by value.
template <int OUT, bool kStoreVec>
__global__ void __launch_bounds__(kThreads)
    dq4_transposed_any_kernel(const Args a, int64_t rows, int64_t cols, uint32_t tiles_r,
                              uint32_t n_tiles) {
  __shared__ float s_vcb[16];
  __shared__ float s_scb[256];
#if DQ4_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
#endif
  stage_codebooks<true>(a, s_vcb, s_scb);
  const uint32_t t = blockIdx.x * uint32_t(kWarpsPerCta) + (threadIdx.x >> 5);
  if (t >= n_tiles) return;
  const int lane = threadIdx.x & 31;
  const int64_t r0 = int64_t(t % tiles_r) * kTR;  // column-major tile order
  const int64_t c0 = int64_t(t / tiles_r) * kTC;
  const int64_t ra = r0 + 2 * lane;
  const bool has0 = ra < rows, has1 = ra + 1 < rows;
  if (!has0) return;
  const int ncol = int(cols - c0 < kTC ? cols - c0 : kTC);
  // each row's scale is rebuilt only when the row crosses into a new block
  const int64_t i0 = ra * cols + c0, i1 = i0 + cols;
  int64_t b0 = -1, b1 = -1;
  float sc0 = 0.f, sc1 = 0.f;
  int64_t o = c0 * rows + ra;
  for (int cc = 0; cc < ncol; ++cc) {
    const int64_t ia = i0 + cc, ib = i1 + cc;
    if ((ia >> a.log2_bs) != b0) { b0 = ia >> a.log2_bs; sc0 = nested_scale(a, s_scb, b0); }
    const uint32_t ba = a.packed[ia >> 1];
    const float v0 = __fmul_rn(s_vcb[(ia & 1) ? (ba & 0xFu) : (ba >> 4)], sc0);
    float v1 = 0.f;
    if (has1) {
      if ((ib >> a.log2_bs) != b1) { b1 = ib >> a.log2_bs; sc1 = nested_scale(a, s_scb, b1); }
      const uint32_t bb = a.packed[ib >> 1];
      v1 = __fmul_rn(s_vcb[(ib & 1) ? (bb & 0xFu) : (bb >> 4)], sc1);
    }
    store_pair<OUT, kStoreVec>(a.out, o, v0, v1, has0, has1);
    o += rows;
  }
}

// ------------------------------------- LLM.int8 correction-operand preparation
// "Fuse LLM.int8 correction operand preparation into one CUDA kernel"
// (bitsandbytes issue #16), sections "Summary", "Bounded method" and "Exact
// correctness oracle", in one launch over two output regions:
//   subA[m][l] = A[m][cols[l]]                                   (16-bit copy)
//   subB[l][n] = RN16(RN32(RN32(CB[n][cols[l]] * SCB[n]) * RN32(1/127)))
// CTAs [0, ctas_a) fill subA: each covers kAElems consecutive elements of
// the row-major M x L array, lanes walking l, so stores are contiguous.  CTAs
// [ctas_a, ...) fill subB: each covers kBN consecutive n (two per thread:
// both SCB values in one 8-byte load, both results in one 4-byte store) and
// kBL consecutive l; per l a warp stores 128 contiguous bytes of subB.  The
// CB reads are a column gather (one byte of each of two rows per l); a
// thread issues all kBL * 2 of them before using any.  Column indices are
// bounds-checked: an index outside [0, K) reads nothing, yields 0 and is
// counted once into *bad (if given).
constexpr int kAElems = 2048;  // subA elements per CTA
constexpr int kBN = 2 * kThreads;  // subB: n per CTA
constexpr int kBL = 4;             // subB: l per CTA

struct PrepArgs {
  const uint16_t* A;
  const int8_t* CB;
  const float* SCB;
  const int64_t* cols;
  uint16_t* subA;
  uint16_t* subB;
  int* bad;
  int64_t M, N, K, L;
  int64_t ctas_a;
  int64_t l_chunks;
  bool count_in_a;  // bad indices are counted once: in the subA region if M > 0
};

__device__ __forceinline__ bool col_ok(int64_t c, int64_t K) { return c >= 0 && c < K; }

template <bool kPairStore>
__global__ void __launch_bounds__(kThreads) int8_prep_kernel(const PrepArgs p) {
#if DQ4_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
#endif
  const int64_t bid = blockIdx.x;
  if (bid < p.ctas_a) {
    // ---- subA: a contiguous run of the row-major M x L array
    const int64_t e0 = bid * kAElems;
    const int64_t total = p.M * p.L;
    for (int k = 0; k < kAElems / kThreads; ++k) {
      const int64_t e = e0 + k * kThreads + threadIdx.x;
      if (e >= total) break;
      const int64_t m = e / p.L, l = e - m * p.L;
      const int64_t c = __ldg(p.cols + l);
      uint16_t v = 0;
      if (col_ok(c, p.K)) {
        v = __ldg(p.A + m * p.K + c);
      } else if (p.bad && p.count_in_a && m == 0) {
        atomicAdd(p.bad, 1);
      }
      p.subA[e] = v;
    }
    return;
  }
  // ---- subB: kBN consecutive n x kBL consecutive l
  const int64_t b = bid - p.ctas_a;
  const int64_t l0 = (b % p.l_chunks) * kBL;
  const int64_t n0 = (b / p.l_chunks) * kBN + 2 * threadIdx.x;
  if (n0 >= p.N) return;
  const bool two = n0 + 1 < p.N;
  const float recip127 = __fdiv_rn(1.0f, 127.0f);  // the FP32 constant RN32(1/127)
  float s0, s1 = 0.f;
  if (kPairStore && two) {
    const float2 sp = __ldg(reinterpret_cast<const float2*>(p.SCB + n0));
    s0 = sp.x;
    s1 = sp.y;
  } else {
    s0 = __ldg(p.SCB + n0);
    if (two) s1 = __ldg(p.SCB + n0 + 1);
  }
  int8_t c0[kBL], c1[kBL];
  bool ok[kBL];
#pragma unroll
  for (int j = 0; j < kBL; ++j) {
    const int64_t l = l0 + j;
    c0[j] = 0;
    c1[j] = 0;
    ok[j] = false;
    if (l < p.L) {
      const int64_t c = __ldg(p.cols + l);
      ok[j] = col_ok(c, p.K);
      if (ok[j]) {
        c0[j] = __ldg(p.CB + n0 * p.K + c);
        if (two) c1[j] = __ldg(p.CB + (n0 + 1) * p.K + c);
      } else if (p.bad && !p.count_in_a && n0 == 0) {
        atomicAdd(p.bad, 1);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < kBL; ++j) {
    const int64_t l = l0 + j;
    if (l >= p.L) break;
    // RN32(CB * SCB) then a separately rounded RN32(t1 * (1/127)), then RN16
    const float v0 = ok[j] ? __fmul_rn(__fmul_rn(float(c0[j]), s0), recip127) : 0.f;
    const float v1 = ok[j] ? __fmul_rn(__fmul_rn(float(c1[j]), s1), recip127) : 0.f;
    uint16_t* dst = p.subB + l * p.N + n0;
    if (kPairStore && two) {
      const __half2 h = __floats2half2_rn(v0, v1);
      uint32_t u;
      memcpy(&u, &h, sizeof u);
      __stcs(reinterpret_cast<unsigned int*>(dst), u);
    } else {
      dst[0] = __half_as_ushort(__float2half_rn(v0));
      if (two) dst[1] = __half_as_ushort(__float2half_rn(v1));
    }
  }
}

template <int OUT, bool NESTED>
__global__ void __launch_bounds__(kThreads) dq4_scalar_kernel(const Args a) {
  __shared__ float s_vcb[16];
  __shared__ float s_scb[NESTED ? 256 : 1];
  stage_codebooks<NESTED>(a, s_vcb, s_scb);
  const int64_t stride = int64_t(gridDim.x) * kThreads;
  for (int64_t i = int64_t(blockIdx.x) * kThreads + threadIdx.x; i < a.n; i += stride)
    store_one<OUT>(a.out, i, value_at<NESTED>(a, s_scb, s_vcb, a.first + i));
}

// Unfused step 1: FP32 scale buffer from the codes (no offset yet).
__global__ void __launch_bounds__(kThreads)
    scale_codes_kernel(const uint8_t* codes, const float* nested_absmax, const float* scb,
                       int64_t nblocks, int log2_nbs, float* scales) {
  const int64_t stride = int64_t(gridDim.x) * kThreads;
  for (int64_t b = int64_t(blockIdx.x) * kThreads + threadIdx.x; b < nblocks; b += stride)
    scales[b] = __fmul_rn(__ldg(scb + __ldg(codes + b)), __ldg(nested_absmax + (b >> log2_nbs)));
}

// Unfused step 2: the offset as a separate elementwise pass.
__global__ void __launch_bounds__(kThreads)
    add_offset_kernel(float* scales, int64_t nblocks, float offset) {
  const int64_t stride = int64_t(gridDim.x) * kThreads;
  for (int64_t b = int64_t(blockIdx.x) * kThreads + threadIdx.x; b < nblocks; b += stride)
    scales[b] = __fadd_rn(scales[b], offset);
}

// ------------------------------------------------------------- host side
struct DeviceCache {
  std::atomic<int> sms{0};
  std::atomic<int> cc{0};
};
DeviceCache g_devices[kMaxDevices];

int fail_cuda(int status, cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return status;
}

// Current device's SM count, after checking that it is compute capability 10.3.
int current_device(int* dev_out, int* sms_out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(DQ4_ERR_DEVICE, e);
  int cc = 0, sms = 0;
  if (dev >= 0 && dev < kMaxDevices) {
    cc = g_devices[dev].cc.load(std::memory_order_relaxed);
    sms = g_devices[dev].sms.load(std::memory_order_relaxed);
  }
  if (cc == 0 || sms == 0) {
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return fail_cuda(DQ4_ERR_DEVICE, e);
    cc = major * 10 + minor;
    if (dev >= 0 && dev < kMaxDevices) {
      g_devices[dev].cc.store(cc, std::memory_order_relaxed);
      g_devices[dev].sms.store(sms, std::memory_order_relaxed);
    }
  }
  if (cc != 103) return fail_cuda(DQ4_ERR_ARCH, cudaErrorNoKernelImageForDevice);
  *dev_out = dev;
  *sms_out = sms;
  return DQ4_OK;
}

// Resident CTAs per SM of `kernel`, cached per device.
template <typename Kernel>
int ctas_per_sm(Kernel kernel, int dev, std::atomic<int>* cache) {
  int occ = (dev >= 0 && dev < kMaxDevices) ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (occ > 0) return occ;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, 0) != cudaSuccess ||
      occ < 1) {
    cudaGetLastError();
    occ = 1;
  }
  if (dev >= 0 && dev < kMaxDevices) cache[dev].store(occ, std::memory_order_relaxed);
  return occ;
}

int check_launch() {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(DQ4_ERR_LAUNCH, e);
  return DQ4_OK;
}

// Launch `kernel` on `stream`, with programmatic stream serialization when
// DQ4_PDL is on (the kernel then waits with griddepcontrol.wait before it
// touches memory).
template <typename... KArgs, typename... Actual>
int launch_kernel(void (*kernel)(KArgs...), int64_t grid, cudaStream_t stream,
                  Actual&&... args) {
#if DQ4_PDL
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t le = cudaLaunchKernelEx(&cfg, kernel, std::forward<Actual>(args)...);
  if (le != cudaSuccess) {
    cudaGetLastError();
    return fail_cuda(DQ4_ERR_LAUNCH, le);
  }
  return DQ4_OK;
#else
  kernel<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(std::forward<Actual>(args)...);
  return check_launch();
#endif
}

template <int OUT, bool NESTED>
int launch_dq4(const Args& a, cudaStream_t stream) {
  int dev = 0, sms = 0;
  if (int st = current_device(&dev, &sms)) return st;
  using Word = typename Traits<OUT>::Word;
  const bool vec = (reinterpret_cast<uintptr_t>(a.packed) % sizeof(Word) == 0) &&
                   (reinterpret_cast<uintptr_t>(a.out) % 16 == 0);
  if (vec) {
    const int64_t n_words = a.n >> Traits<OUT>::kLog2Vals;
    const int64_t tiles = (n_words + 32 * Tile<OUT>::U - 1) / (32 * Tile<OUT>::U);
    int64_t grid = (tiles + kWarpsPerCta - 1) / kWarpsPerCta;
    const int64_t cap = DQ4_CTAS_PER_SM > 0 ? int64_t(sms) * DQ4_CTAS_PER_SM : kMaxGrid;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    return launch_kernel(dq4_vec_kernel<OUT, NESTED>, grid, stream, a);
  } else {
    static std::atomic<int> occ_cache[kMaxDevices];
    auto kernel = dq4_scalar_kernel<OUT, NESTED>;
    int64_t grid = (a.n + kThreads - 1) / kThreads;
    const int64_t cap = int64_t(sms) * ctas_per_sm(kernel, dev, occ_cache);
    if (grid > cap) grid = cap;
    kernel<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(a);
  }
  return check_launch();
}

template <bool NESTED>
int dispatch_dtype(const Args& a, int32_t out_dtype, cudaStream_t stream) {
  switch (out_dtype) {
    case DQ4_OUT_F16: return launch_dq4<DQ4_OUT_F16, NESTED>(a, stream);
    case DQ4_OUT_BF16: return launch_dq4<DQ4_OUT_BF16, NESTED>(a, stream);
    case DQ4_OUT_F32: return launch_dq4<DQ4_OUT_F32, NESTED>(a, stream);
    default: return DQ4_ERR_DTYPE;
  }
}

template <int OUT>
int launch_transposed(const Args& a, int64_t rows, int64_t cols, cudaStream_t stream) {
  int dev = 0, sms = 0;
  if (int st = current_device(&dev, &sms)) return st;
  constexpr uintptr_t osz = (OUT == DQ4_OUT_F32) ? 4 : 2;
  const bool sv = rows % 2 == 0 && reinterpret_cast<uintptr_t>(a.out) % (2 * osz) == 0;
  if (cols % 32 == 0 && reinterpret_cast<uintptr_t>(a.packed) % 16 == 0) {
    const int64_t tiles_r = (rows + kSR - 1) / kSR;
    const int64_t grid = tiles_r * ((cols + kSC - 1) / kSC);
    if (grid > int64_t(UINT32_MAX)) return DQ4_ERR_N;  // 32-bit tile ids
    const uint32_t tr = uint32_t(tiles_r);
    if (sv) return launch_kernel(dq4_transposed_kernel<OUT, true>, grid, stream, a, rows, cols, tr);
    return launch_kernel(dq4_transposed_kernel<OUT, false>, grid, stream, a, rows, cols, tr);
  }
  const int64_t tiles_r = (rows + kTR - 1) / kTR;
  const int64_t n_tiles = tiles_r * ((cols + kTC - 1) / kTC);
  if (n_tiles > int64_t(UINT32_MAX) - kWarpsPerCta) return DQ4_ERR_N;  // 32-bit tile ids
  const int64_t grid = (n_tiles + kWarpsPerCta - 1) / kWarpsPerCta;
  const uint32_t tr = uint32_t(tiles_r), nt = uint32_t(n_tiles);
  if (sv) return launch_kernel(dq4_transposed_any_kernel<OUT, true>, grid, stream, a, rows, cols, tr, nt);
  return launch_kernel(dq4_transposed_any_kernel<OUT, false>, grid, stream, a, rows, cols, tr, nt);
}

bool is_pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }

int log2_exact(int64_t v) {
  int r = 0;
  while ((int64_t(1) << r) < v) ++r;
  return r;
}

bool misaligned(const void* p, uintptr_t align) {
  return reinterpret_cast<uintptr_t>(p) % align != 0;
}

int out_itemsize(int32_t out_dtype) { return out_dtype == DQ4_OUT_F32 ? 4 : 2; }

// Checks shared by every entry point, in a fixed order; n == 0 returns
// DQ4_OK before any pointer is looked at.
int validate(int64_t n, int32_t blocksize, int32_t nested_blocksize, bool nested,
             int32_t out_dtype) {
  if (n < 0) return DQ4_ERR_N;
  if (!is_pow2(blocksize) || blocksize < 32 || blocksize > 4096) return DQ4_ERR_BLOCKSIZE;
  if (nested && !is_pow2(nested_blocksize)) return DQ4_ERR_NESTED_BLOCKSIZE;
  if (out_dtype != DQ4_OUT_F16 && out_dtype != DQ4_OUT_BF16 && out_dtype != DQ4_OUT_F32)
    return DQ4_ERR_DTYPE;
  return DQ4_OK;
}

Args make_args(const uint8_t* packed, const uint8_t* codes, const float* absmax,
               const float* scb, const float* vcb, float offset, int64_t n, int32_t blocksize,
               int32_t nested_blocksize, void* out) {
  Args a;
  a.packed = packed;
  a.codes = codes;
  a.absmax = absmax;
  a.scb = scb;
  a.vcb = vcb;
  a.out = out;
  a.n = n;
  a.first = 0;
  a.nblocks = (n + blocksize - 1) / blocksize;
  a.offset = offset;
  a.log2_bs = log2_exact(blocksize);
  a.log2_nbs = log2_exact(nested_blocksize);
  return a;
}

}  // namespace

// ------------------------------------------------------------ C-ABI
extern "C" {

int dq4_abi_version(void) { return kAbiVersion; }

int dq4_nested(const uint8_t* packed, const uint8_t* scale_codes, const float* nested_absmax,
               const float* scale_codebook, const float* value_codebook, float offset,
               int64_t n, int32_t blocksize, int32_t nested_blocksize, int32_t out_dtype,
               void* out, void* stream) {
  if (int st = validate(n, blocksize, nested_blocksize, true, out_dtype)) return st;
  if (n == 0) return DQ4_OK;
  if (!packed || !scale_codes || !nested_absmax || !scale_codebook || !value_codebook || !out)
    return DQ4_ERR_NULL;
  if (misaligned(nested_absmax, 4) || misaligned(scale_codebook, 4) ||
      misaligned(value_codebook, 4) || misaligned(out, out_itemsize(out_dtype)))
    return DQ4_ERR_ALIGN;
  const Args a = make_args(packed, scale_codes, nested_absmax, scale_codebook, value_codebook,
                           offset, n, blocksize, nested_blocksize, out);
  return dispatch_dtype<true>(a, out_dtype, static_cast<cudaStream_t>(stream));
}

int dq4_nested_transposed(const uint8_t* packed, const uint8_t* scale_codes,
                          const float* nested_absmax, const float* scale_codebook,
                          const float* value_codebook, float offset, int64_t rows,
                          int64_t cols, int32_t blocksize, int32_t nested_blocksize,
                          int32_t out_dtype, void* out, void* stream) {
  if (rows < 0 || cols < 0) return DQ4_ERR_N;
  if (cols > 0 && rows > INT64_MAX / cols) return DQ4_ERR_N;
  const int64_t n = rows * cols;
  if (int st = validate(n, blocksize, nested_blocksize, true, out_dtype)) return st;
  if (n == 0) return DQ4_OK;
  if (!packed || !scale_codes || !nested_absmax || !scale_codebook || !value_codebook || !out)
    return DQ4_ERR_NULL;
  if (misaligned(nested_absmax, 4) || misaligned(scale_codebook, 4) ||
      misaligned(value_codebook, 4) || misaligned(out, out_itemsize(out_dtype)))
    return DQ4_ERR_ALIGN;
  const Args a = make_args(packed, scale_codes, nested_absmax, scale_codebook, value_codebook,
                           offset, n, blocksize, nested_blocksize, out);
  const auto st = static_cast<cudaStream_t>(stream);
  switch (out_dtype) {
    case DQ4_OUT_F16: return launch_transposed<DQ4_OUT_F16>(a, rows, cols, st);
    case DQ4_OUT_BF16: return launch_transposed<DQ4_OUT_BF16>(a, rows, cols, st);
    default: return launch_transposed<DQ4_OUT_F32>(a, rows, cols, st);
  }
}

int dq4(const uint8_t* packed, const float* absmax, const float* value_codebook, int64_t n,
        int32_t blocksize, int32_t out_dtype, void* out, void* stream) {
  if (int st = validate(n, blocksize, 1, false, out_dtype)) return st;
  if (n == 0) return DQ4_OK;
  if (!packed || !absmax || !value_codebook || !out) return DQ4_ERR_NULL;
  if (misaligned(absmax, 4) || misaligned(value_codebook, 4) ||
      misaligned(out, out_itemsize(out_dtype)))
    return DQ4_ERR_ALIGN;
  const Args a = make_args(packed, nullptr, absmax, nullptr, value_codebook, 0.f, n, blocksize,
                           1, out);
  return dispatch_dtype<false>(a, out_dtype, static_cast<cudaStream_t>(stream));
}

int dq4_nested_unfused(const uint8_t* packed, const uint8_t* scale_codes,
                       const float* nested_absmax, const float* scale_codebook,
                       const float* value_codebook, float offset, int64_t n,
                       int32_t blocksize, int32_t nested_blocksize, int32_t out_dtype,
                       void* out, float* scale_scratch, void* stream) {
  if (int st = validate(n, blocksize, nested_blocksize, true, out_dtype)) return st;
  if (n == 0) return DQ4_OK;
  if (!packed || !scale_codes || !nested_absmax || !scale_codebook || !value_codebook || !out ||
      !scale_scratch)
    return DQ4_ERR_NULL;
  if (misaligned(nested_absmax, 4) || misaligned(scale_codebook, 4) ||
      misaligned(value_codebook, 4) || misaligned(scale_scratch, 4) ||
      misaligned(out, out_itemsize(out_dtype)))
    return DQ4_ERR_ALIGN;
  int dev = 0, sms = 0;
  if (int st = current_device(&dev, &sms)) return st;
  const auto st = static_cast<cudaStream_t>(stream);
  const int64_t nblocks = (n + blocksize - 1) / blocksize;
  int64_t grid = (nblocks + kThreads - 1) / kThreads;
  if (grid > int64_t(sms) * 8) grid = int64_t(sms) * 8;
  scale_codes_kernel<<<static_cast<unsigned>(grid), kThreads, 0, st>>>(
      scale_codes, nested_absmax, scale_codebook, nblocks, log2_exact(nested_blocksize),
      scale_scratch);
  if (int e = check_launch()) return e;
  add_offset_kernel<<<static_cast<unsigned>(grid), kThreads, 0, st>>>(scale_scratch, nblocks,
                                                                       offset);
  if (int e = check_launch()) return e;
  return dq4(packed, scale_scratch, value_codebook, n, blocksize, out_dtype, out, stream);
}

int dq4_int8_correction_prep(const uint16_t* A, const int8_t* CB, const float* SCB,
                             const int64_t* cols, int64_t M, int64_t N, int64_t K, int64_t L,
                             uint16_t* subA, uint16_t* subB, int* bad_cols, void* stream) {
  if (M < 0 || N < 0 || K < 0 || L < 0) return DQ4_ERR_N;
  if (L == 0 || (M == 0 && N == 0)) return DQ4_OK;
  if (K == 0) return DQ4_ERR_N;
  if (M > 0 && L > INT64_MAX / M) return DQ4_ERR_N;
  if (N > 0 && K > INT64_MAX / N) return DQ4_ERR_N;
  if (!cols || (M > 0 && (!A || !subA)) || (N > 0 && (!CB || !SCB || !subB))) return DQ4_ERR_NULL;
  if (misaligned(cols, 8) || misaligned(SCB, 4) || misaligned(A, 2) || misaligned(subA, 2) ||
      misaligned(subB, 2) || misaligned(bad_cols, 4))
    return DQ4_ERR_ALIGN;
  int dev = 0, sms = 0;
  if (int st = current_device(&dev, &sms)) return st;
  PrepArgs p;
  p.A = A;
  p.CB = CB;
  p.SCB = SCB;
  p.cols = cols;
  p.subA = subA;
  p.subB = subB;
  p.bad = bad_cols;
  p.M = M;
  p.N = N;
  p.K = K;
  p.L = L;
  p.ctas_a = (M * L + kAElems - 1) / kAElems;
  p.l_chunks = (L + kBL - 1) / kBL;
  p.count_in_a = M > 0;
  const int64_t ctas_b = N > 0 ? ((N + kBN - 1) / kBN) * p.l_chunks : 0;
  const int64_t grid = p.ctas_a + ctas_b;
  if (grid > kMaxGrid) return DQ4_ERR_N;
  const bool pair = N % 2 == 0 && reinterpret_cast<uintptr_t>(subB) % 4 == 0 &&
                    reinterpret_cast<uintptr_t>(SCB) % 8 == 0;
  const auto st = static_cast<cudaStream_t>(stream);
  if (pair) return launch_kernel(int8_prep_kernel<true>, grid, st, p);
  return launch_kernel(int8_prep_kernel<false>, grid, st, p);
}

}  // extern "C"

// --------------------------------------------- row-blocked dequant + GEMM
namespace {

using CublasSetStream = cublasStatus_t (*)(cublasHandle_t, cudaStream_t);
using CublasGemmEx = cublasStatus_t (*)(cublasHandle_t, cublasOperation_t, cublasOperation_t,
                                        int, int, int, const void*, const void*, cudaDataType,
                                        int, const void*, cudaDataType, int, const void*, void*,
                                        cudaDataType, int, cublasComputeType_t,
                                        cublasGemmAlgo_t);
struct CublasApi {
  CublasSetStream set_stream = nullptr;
  CublasGemmEx gemm = nullptr;
};

// The cuBLAS already loaded in the process (the one the caller's handle
// belongs to), else the system's; resolved once.
const CublasApi* cublas_api() {
  static std::once_flag once;
  static CublasApi api;
  std::call_once(once, [] {
    void* h = dlopen("libcublas.so.13", RTLD_NOW | RTLD_NOLOAD);
    if (!h) h = dlopen("libcublas.so.13", RTLD_NOW);
    if (!h) h = dlopen("libcublas.so", RTLD_NOW);
    if (!h) return;
    api.set_stream = reinterpret_cast<CublasSetStream>(dlsym(h, "cublasSetStream_v2"));
    api.gemm = reinterpret_cast<CublasGemmEx>(dlsym(h, "cublasGemmEx"));
  });
  return (api.set_stream && api.gemm) ? &api : nullptr;
}

int64_t gcd64(int64_t x, int64_t y) {
  while (y) {
    const int64_t t = x % y;
    x = y;
    y = t;
  }
  return x;
}

// FP32 values [first, first + count) of the flat problem, one by one (for
// row blocks that do not start on a nested-group boundary).
int launch_range_f32(Args a, int64_t first, int64_t count, float* out, cudaStream_t stream) {
  int dev = 0, sms = 0;
  if (int st = current_device(&dev, &sms)) return st;
  a.first = first;
  a.n = count;
  a.out = out;
  static std::atomic<int> occ_cache[kMaxDevices];
  auto kernel = dq4_scalar_kernel<DQ4_OUT_F32, true>;
  int64_t grid = (count + kThreads - 1) / kThreads;
  const int64_t cap = int64_t(sms) * ctas_per_sm(kernel, dev, occ_cache);
  if (grid > cap) grid = cap;
  kernel<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(a);
  return check_launch();
}

}  // namespace

extern "C" {

int dq4_nested_out_prod(const uint8_t* packed, const uint8_t* scale_codes,
                        const float* nested_absmax, const float* scale_codebook,
                        const float* value_codebook, float offset, int64_t rows, int64_t cols,
                        int32_t blocksize, int32_t nested_blocksize, const float* G,
                        int64_t ncols, float* dst, float* transient, int64_t transient_bytes,
                        void* cublas_handle, void* stream) {
  if (rows < 0 || cols < 0 || ncols < 0) return DQ4_ERR_N;
  if (cols > 0 && rows > INT64_MAX / cols) return DQ4_ERR_N;
  const int64_t n = rows * cols;
  if (int st = validate(n, blocksize, nested_blocksize, true, DQ4_OUT_F32)) return st;
  if (cols == 0 || ncols == 0) return DQ4_OK;
  if (cols > INT32_MAX || ncols > INT32_MAX) return DQ4_ERR_N;  // cuBLAS dimensions
  if (!dst) return DQ4_ERR_NULL;
  if (misaligned(dst, 4)) return DQ4_ERR_ALIGN;
  const auto st = static_cast<cudaStream_t>(stream);
  if (rows == 0) {  // an empty sum
    const cudaError_t e = cudaMemsetAsync(dst, 0, size_t(cols) * size_t(ncols) * 4, st);
    return e == cudaSuccess ? DQ4_OK : fail_cuda(DQ4_ERR_LAUNCH, e);
  }
  if (!packed || !scale_codes || !nested_absmax || !scale_codebook || !value_codebook || !G ||
      !transient || !cublas_handle)
    return DQ4_ERR_NULL;
  if (misaligned(nested_absmax, 4) || misaligned(scale_codebook, 4) ||
      misaligned(value_codebook, 4) || misaligned(G, 4) || misaligned(transient, 4))
    return DQ4_ERR_ALIGN;
  const int64_t row_bytes = cols * 4;
  if (transient_bytes < row_bytes) return DQ4_ERR_TOO_LARGE;  // at least one row
  int64_t rb = transient_bytes / row_bytes;
  if (rb > rows) rb = rows;
  if (rb > INT32_MAX) rb = INT32_MAX;
  // keep block starts on nested-group boundaries when the budget allows it,
  // so every block takes the vector path
  const int64_t unit = int64_t(blocksize) * nested_blocksize;
  const int64_t ralign = unit / gcd64(cols % unit ? cols % unit : unit, unit);
  if (rb >= ralign) rb -= rb % ralign;
  const CublasApi* cb = cublas_api();
  if (!cb) return DQ4_ERR_CUBLAS;
  const auto h = static_cast<cublasHandle_t>(cublas_handle);
  if (cb->set_stream(h, st) != CUBLAS_STATUS_SUCCESS) return DQ4_ERR_CUBLAS;
  Args base = make_args(packed, scale_codes, nested_absmax, scale_codebook, value_codebook,
                        offset, n, blocksize, nested_blocksize, transient);
  for (int64_t r0 = 0; r0 < rows; r0 += rb) {
    const int64_t nr = rows - r0 < rb ? rows - r0 : rb;
    const int64_t first = r0 * cols, count = nr * cols;
    int status;
    if (first % unit == 0) {
      status = dq4_nested(packed + first / 2, scale_codes + first / blocksize,
                          nested_absmax + first / unit, scale_codebook, value_codebook, offset,
                          count, blocksize, nested_blocksize, DQ4_OUT_F32, transient, stream);
    } else {
      status = launch_range_f32(base, first, count, transient, st);
    }
    if (status) return status;
    // dst (cols x ncols, row-major) += W_blk^T (cols x nr) * G_blk (nr x ncols); in
    // cuBLAS's column-major terms: dst^T = G_blk^T * W_blk
    const float alpha = 1.f, beta = r0 == 0 ? 0.f : 1.f;
    const cublasStatus_t cs =
        cb->gemm(h, CUBLAS_OP_N, CUBLAS_OP_T, int(ncols), int(cols), int(nr), &alpha,
                 G + r0 * ncols, CUDA_R_32F, int(ncols), transient, CUDA_R_32F, int(cols), &beta,
                 dst, CUDA_R_32F, int(ncols), CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
    if (cs != CUBLAS_STATUS_SUCCESS) return DQ4_ERR_CUBLAS;
  }
  return DQ4_OK;
}

const char* dq4_status_string(int status) {
  switch (status) {
    case DQ4_OK: return "ok";
    case DQ4_ERR_NULL: return "a required pointer is NULL";
    case DQ4_ERR_N: return "n (or rows, cols) is negative or too large";
    case DQ4_ERR_BLOCKSIZE: return "blocksize must be a power of two in [32, 4096]";
    case DQ4_ERR_NESTED_BLOCKSIZE: return "nested_blocksize must be a power of two >= 1";
    case DQ4_ERR_DTYPE: return "out_dtype must be DQ4_OUT_F16, DQ4_OUT_BF16 or DQ4_OUT_F32";
    case DQ4_ERR_ALIGN: return "a float array or the output is misaligned for its type";
    case DQ4_ERR_DEVICE: return "the current CUDA device could not be queried";
    case DQ4_ERR_ARCH: return "the current device is not compute capability 10.3 (GB300)";
    case DQ4_ERR_LAUNCH: return "the CUDA runtime reported an error at kernel launch";
    case DQ4_ERR_TOO_LARGE:
      return "the problem needs more scratch than given (DQ4_STATIC_SCRATCH_BLOCKS for the "
             "static array; one row of W for a transient buffer)";
    case DQ4_ERR_CUBLAS: return "cuBLAS could not be loaded or reported an error";
    default: return "unknown status";
  }
}

int dq4_last_cuda_error(void) { return t_last_cuda_error; }

}  // extern "C"

// ------------------------------------------------ allocation-free variant
// The FP32 scale scratch of the unfused sequence, as a fixed array in the
// library, for callers that may not allocate device memory.  Host code
// must not use the symbol itself as a pointer (on the host it only names
// the array); its device address is looked up once per device.
namespace {

static __device__ __align__(256) float g_static_scale_scratch[DQ4_STATIC_SCRATCH_BLOCKS];

std::atomic<float*> g_static_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device `dev`.
int static_scratch_address(int dev, float** out) {
  if (dev < 0 || dev >= kMaxDevices) return fail_cuda(DQ4_ERR_DEVICE, cudaErrorInvalidDevice);
  float* ptr = g_static_scratch_addr[dev].load(std::memory_order_acquire);
  if (ptr == nullptr) {
    void* addr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&addr, g_static_scale_scratch);
    if (e != cudaSuccess || addr == nullptr)
      return fail_cuda(DQ4_ERR_DEVICE, e != cudaSuccess ? e : cudaErrorInvalidSymbol);
    ptr = static_cast<float*>(addr);
    g_static_scratch_addr[dev].store(ptr, std::memory_order_release);
  }
  *out = ptr;
  return DQ4_OK;
}

}  // namespace

extern "C" int dq4_nested_unfused_static(const uint8_t* packed, const uint8_t* scale_codes,
                                         const float* nested_absmax, const float* scale_codebook,
                                         const float* value_codebook, float offset, int64_t n,
                                         int32_t blocksize, int32_t nested_blocksize,
                                         int32_t out_dtype, void* out, void* stream) {
  if (int st = validate(n, blocksize, nested_blocksize, true, out_dtype)) return st;
  if (n == 0) return DQ4_OK;
  if ((n + blocksize - 1) / blocksize > int64_t(DQ4_STATIC_SCRATCH_BLOCKS))
    return DQ4_ERR_TOO_LARGE;
  if (!packed || !scale_codes || !nested_absmax || !scale_codebook || !value_codebook || !out)
    return DQ4_ERR_NULL;
  int dev = 0, sms = 0;
  if (int st = current_device(&dev, &sms)) return st;
  float* scratch = nullptr;
  if (int st = static_scratch_address(dev, &scratch)) return st;
  return dq4_nested_unfused(packed, scale_codes, nested_absmax, scale_codebook, value_codebook,
                            offset, n, blocksize, nested_blocksize, out_dtype, out, scratch,
                            stream);
}

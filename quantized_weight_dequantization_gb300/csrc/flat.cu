// The flat dequantization path of the dq4 library: dq4_nested (fused, one
// launch), dq4 (non-nested), dq4_nested_unfused (the three-launch sequence)
// and dq4_nested_unfused_static, plus the per-value kernel.
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
//    for its completion (griddepcontrol.wait) before reading or writing
//    memory.  In grids of up to 8 waves each warp first asks L2 for its first
//    tile's lines (prefetch.global.L2, which returns nothing and so changes no
//    value read after the wait), so its DRAM reads start during the previous
//    kernel's tail and the codebook staging.
//  * Values after the last whole word (fewer than one word, including an
//    odd padding nibble) are written one by one by CTA 0.  Unaligned
//    `packed` / `out` pointers take a per-value kernel with the same math.
#include "common.cuh"

namespace dq4d {

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
  const int64_t n_words = a.n >> T::kLog2Vals;
  const int wshift = a.log2_bs - T::kLog2Vals;  // log2(words per outer block)
  const int lane = threadIdx.x & 31;
  const int64_t warp = (int64_t(blockIdx.x) * kThreads + threadIdx.x) >> 5;
  const int64_t stride = ((int64_t(gridDim.x) * kThreads) >> 5) * kTile;
#if DQ4_PDL
#if DQ4_L2_PREFETCH
  // A prefetch returns nothing to the thread and L2 is the point of coherence, so asking
  // for these lines before the previous grid completes changes no value this kernel
  // reads; it only starts their DRAM reads early.  One lane per 128-byte line of the
  // tile's packed words, one for its first scale codes and one for its first absmax.
  // (The host sets prefetch_ctas to the grid for small grids and to 0 for large ones.)
  if (blockIdx.x < a.prefetch_ctas) {
    using Word = typename T::Word;
    constexpr int kLines = int(kTile * sizeof(Word) / 128);
    const int64_t base0 = warp * kTile;
    if (base0 < n_words) {
      const char* pk = reinterpret_cast<const char*>(a.packed) + base0 * int64_t(sizeof(Word));
      const int64_t bytes = (n_words - base0) * int64_t(sizeof(Word));
      const int64_t b0 = base0 >> wshift;
      if (lane < kLines && int64_t(lane) * 128 < bytes) {
        asm volatile("prefetch.global.L2 [%0];" :: "l"(pk + lane * 128));
      } else if (NESTED && lane == kLines) {
        asm volatile("prefetch.global.L2 [%0];" :: "l"(a.codes + b0));
      } else if (lane == kLines + 1) {
        asm volatile("prefetch.global.L2 [%0];" :: "l"(a.absmax + (NESTED ? b0 >> a.log2_nbs : b0)));
      }
    }
  }
#endif
  // No global memory is read or written before the previous grid in the stream has
  // completed; dependents may be scheduled once every CTA here has started.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
#endif

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
    static std::atomic<int> vec_occ[kMaxDevices];
    Args b = a;
    const int64_t wave = int64_t(sms) * ctas_per_sm(dq4_vec_kernel<OUT, NESTED>, dev, vec_occ);
    b.prefetch_ctas = grid <= int64_t(DQ4_PREFETCH_WAVES) * wave ? grid : 0;
    return launch_kernel(dq4_vec_kernel<OUT, NESTED>, grid, stream, b);
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

}  // namespace dq4d

using namespace dq4d;

extern "C" {

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

// Shared definitions of the dq4 library (GB300, sm_103a): build-time tuning
// knobs, the kernel argument block, the per-value arithmetic of nested 4-bit
// dequantization, and host-side launch helpers.  Every translation unit of
// the library includes this header; the entry points are declared in dq4.h.
//
// Operation: "Fuse nested scale reconstruction into SM103 4-bit
// dequantization" (bitsandbytes issue #21), section "Proposed experiment":
//   scale = scale_codebook[scale_code] * nested_absmax[nested_group] + offset
//   value = decode_4bit(packed_value) * scale
// with the multiply and the add of the scale rounded separately (section
// "Correctness requirements").  __fmul_rn / __fadd_rn are never contracted
// into an FMA, and the library is also compiled with -fmad=false.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <utility>

#include "dq4.h"

namespace dq4d {

#ifndef DQ4_THREADS
#define DQ4_THREADS 256
#endif
constexpr int kThreads = DQ4_THREADS;
constexpr int kWarpsPerCta = kThreads / 32;
constexpr int kMaxDevices = 64;
constexpr int64_t kMaxGrid = 2147483647;  // gridDim.x limit


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
  int64_t prefetch_ctas;  // tile kernel: CTAs below this index prefetch their first tile
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
// 1: before griddepcontrol.wait, a warp asks L2 for the lines of its first tile (packed
// words, scale codes, absmax) with prefetch.global.L2, so their DRAM reads start while
// the previous kernel drains and while the CTA stages its codebooks.  Done by every CTA
// of grids of at most DQ4_PREFETCH_WAVES waves of resident CTAs and by none of larger
// ones, where the ramp is amortised and the extra instructions cost ~0.4 % (measured on
// GB300: 42 MB 8.25 -> 7.86 us, 113 MB 18.36 -> 17.69 us, 591 MB 87.1 -> 87.5 us).
#ifndef DQ4_L2_PREFETCH
#define DQ4_L2_PREFETCH 1
#endif
#ifndef DQ4_PREFETCH_WAVES
#define DQ4_PREFETCH_WAVES 8
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

// ------------------------------------------------------------- host side
// (defined in host.cu)
int fail_cuda(int status, cudaError_t e);
// Current device's SM count, after checking that it is compute capability 10.3.
int current_device(int* dev_out, int* sms_out);
int check_launch();
bool is_pow2(int64_t v);
int log2_exact(int64_t v);
bool misaligned(const void* p, uintptr_t align);
int out_itemsize(int32_t out_dtype);
// Checks shared by every entry point, in a fixed order; n == 0 returns
// DQ4_OK before any pointer is looked at.
int validate(int64_t n, int32_t blocksize, int32_t nested_blocksize, bool nested,
             int32_t out_dtype);
Args make_args(const uint8_t* packed, const uint8_t* codes, const float* absmax,
               const float* scb, const float* vcb, float offset, int64_t n, int32_t blocksize,
               int32_t nested_blocksize, void* out);
// (defined in flat.cu) FP32 values [first, first + count) of the flat
// problem `a`, one by one, into `out`.
int launch_range_f32(Args a, int64_t first, int64_t count, float* out, cudaStream_t stream);

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

}  // namespace dq4d

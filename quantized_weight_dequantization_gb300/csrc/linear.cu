// Nested 4-bit dequantization fused into a tcgen05 GEMM: dq4_nested_linear,
// Y[M, N] = X[M, K] * W[N, K]^T with W given as nested 4-bit codes (the
// rows x cols = N x K weight that dq4_nested would expand) and never written
// out.  This is the dequantize-plus-linear shape of "Fuse nested scale
// reconstruction into SM103 4-bit dequantization" (bitsandbytes issue #21,
// sections "Problem" and "B300 evidence plan": the fallback that rebuilds the
// scales, materialises the whole weight and calls F.linear), done without the
// weight.
//
// A CTA computes a 128 x BN tile of Y with 9 warps:
//  * warp 8 (control): allocates BN TMEM columns; lane 0 loads the X tiles
//    (128 rows x 64 K, BF16/FP16) with TMA into a kStages-deep shared ring
//    (128-byte swizzle; rows past M are zero-filled), and issues the
//    tcgen05.mma (M = 128, N = BN, K = 16; A and B from shared memory, the
//    FP32 accumulator in TMEM), committing each stage back to the producers;
//  * warps 0..7 (256 threads): dequantize the W tile of each stage (BN rows x
//    64 K) from packed nibbles into the same ring, in the K-major 128-byte
//    swizzled layout the MMA reads, then run the epilogue: tcgen05.ld of the
//    accumulator rows (warp w reads TMEM lanes 32 (w % 4) ..), conversion to
//    the output type and the stores of Y.
// Every W value is computed exactly as dq4_nested does (separately rounded
// FP32 multiply and add for the scale, FP32 product, RN to BF16 / FP16), so
// the GEMM consumes the same operand bits as "dequantize, then F.linear".
// Waits on mbarriers are bounded; a wait that runs out counts into *bad and
// the CTA stops issuing work, frees its TMEM and returns.
#include "common.cuh"

#include <cuda.h>  // CUtensorMap and its enums (the encoder is reached through the runtime)

#include <mutex>

namespace dq4d {
namespace {

constexpr int kLinThreads = 288;  // 8 dequant/epilogue warps + 1 control warp
constexpr int kProducers = 256;
constexpr int kBM = 128;
constexpr int kBK = 64;            // 64 16-bit values = one 128-byte swizzle row
constexpr int kStages = 4;
constexpr uint32_t kWaitLimit = 1u << 26;

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
// both FP16, both K-major, M = 128, N = BN.
template <int BN>
__device__ __forceinline__ uint32_t instr_desc(bool bf16) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) |
         (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(kBM >> 4) << 24);
}

__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (uint32_t it = 0; it < kWaitLimit; ++it) {
    uint32_t done;
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done) : "r"(bar), "r"(parity) : "memory");
    if (done) return true;
  }
  return false;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,"
      "%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

struct LinArgs {
  Args w;          // the nested 4-bit weight (n = N * K values, row-major N x K)
  void* Y;
  int64_t M, N, K;
  int* bad;        // optional device counter of timed-out waits
  int out_dtype;
  int tiles_n;     // column tiles of Y
};

template <int BN, bool kBF16>
struct LinSmem {
  static constexpr int kA = kBM * kBK * 2;   // bytes of an A stage
  static constexpr int kB = BN * kBK * 2;    // bytes of a B stage
  static constexpr int kStage = kA + kB;
  static constexpr int kBarOff = kStages * kStage;
  static constexpr int kBytes = kBarOff + 256 + 1024;  // + barriers, slot, alignment slack
};

// Byte offset of 16-byte chunk `ch` of row `r` in a K-major 128-byte-swizzled tile.
__device__ __forceinline__ int swz128(int r, int ch) {
  return (r >> 3) * 1024 + (r & 7) * 128 + ((ch ^ (r & 7)) << 4);
}

template <int BN, bool kBF16>
__global__ void __launch_bounds__(kLinThreads, 1)
    dq4_linear_kernel(const __grid_constant__ CUtensorMap tmap_x, const LinArgs p) {
  using S = LinSmem<BN, kBF16>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ float s_vcb[16];
  __shared__ float s_scb[256];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(base);
  const uint32_t bar0 = sbase + S::kBarOff;                 // full_a[s]: 8 bytes each
  auto full_a = [&](int s) { return bar0 + 8 * s; };
  auto full_b = [&](int s) { return bar0 + 8 * (kStages + s); };
  auto empty = [&](int s) { return bar0 + 8 * (2 * kStages + s); };
  const uint32_t acc_full = bar0 + 8 * (3 * kStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base + S::kBarOff + 8 * (3 * kStages + 1));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile_m = blockIdx.x / p.tiles_n, tile_n = blockIdx.x % p.tiles_n;
  const int64_t m0 = int64_t(tile_m) * kBM, n0 = int64_t(tile_n) * BN;
  const int kt_count = int(p.K / kBK);

#if DQ4_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
#endif
  if (tid < 16) s_vcb[tid] = __ldg(p.w.vcb + tid);
  for (int k = tid; k < 256; k += kLinThreads) s_scb[k] = __ldg(p.w.scb + k);
  if (warp == 8) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(tmem_slot)), "r"(BN));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    if (lane == 0) {
      for (int s = 0; s < kStages; ++s) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(full_a(s)));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(full_b(s)), "r"(kProducers));
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(empty(s)));
      }
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(acc_full));
      *abort_flag = 0;
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmap_x)));
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;
  bool failed = false;

  if (warp == 8) {
    if (lane == 0) {
      // ---- TMA for X and the MMA issue, one thread
      const bool bf16 = kBF16;
      const uint32_t idesc = instr_desc<BN>(bf16);
      const uint64_t tmap_ptr = reinterpret_cast<uint64_t>(&tmap_x);
      int issued = 0;  // X tiles requested
      const int lookahead = kt_count < kStages ? kt_count : kStages;
      auto load_x = [&](int tile) {  // X tile `tile` into its stage
        const int st = tile % kStages;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                     :: "r"(full_a(st)), "r"(S::kA) : "memory");
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%2, %3}], [%4];"
            :: "r"(sbase + st * S::kStage), "l"(tmap_ptr), "r"(tile * kBK), "r"(int(m0)),
               "r"(full_a(st)) : "memory");
      };
      for (; issued < lookahead; ++issued) load_x(issued);
      for (int kt = 0; kt < kt_count && !failed; ++kt) {
        const int s = kt % kStages;
        const uint32_t par = (kt / kStages) & 1;
        if (!mbar_wait(full_a(s), par) || !mbar_wait(full_b(s), par)) {
          failed = true;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t a_addr = sbase + s * S::kStage;
        const uint32_t b_addr = a_addr + S::kA;
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
            :: "r"(empty(s)) : "memory");
        // while these MMAs run, refill the stage the previous tile used (its MMAs,
        // issued earlier, complete first)
        if (kt >= 1 && issued < kt_count) {
          const int prev = kt - 1;
          if (!mbar_wait(empty(prev % kStages), (prev / kStages) & 1)) {
            failed = true;
            break;
          }
          load_x(issued);
          ++issued;
        }
      }
      if (!failed) {
        asm volatile(
            "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
            :: "r"(acc_full) : "memory");
      } else {
        *abort_flag = 1;
        if (p.bad) atomicAdd(p.bad, 1);
      }
    }
  } else {
    // ---- dequantize the W tiles (BN rows x 64 K per stage), then the epilogue
    constexpr int kChunks = BN * (kBK / 8) / kProducers;  // 8-value chunks per thread per stage
    const float offset = p.w.offset;
    for (int kt = 0; kt < kt_count; ++kt) {
      const int s = kt % kStages;
      if (kt >= kStages) {
        // the stage is free once the MMAs of round kt / kStages - 1 completed
        if (*abort_flag || !mbar_wait(empty(s), ((kt / kStages) - 1) & 1)) {
          failed = true;
          break;
        }
      }
      uint8_t* sB = base + s * S::kStage + S::kA;
      const int64_t k0 = int64_t(kt) * kBK;
#pragma unroll
      for (int j = 0; j < kChunks; ++j) {
        const int c = tid + kProducers * j;
        const int r = c >> 3, ch = c & 7;
        const int64_t n = n0 + r;
        uint4 q = make_uint4(0, 0, 0, 0);
        if (n < p.N) {
          // 8 values of row n at K offset k0 + 8 ch: one aligned packed word, one block
          const int64_t i0 = n * p.K + k0 + 8 * ch;
          const uint32_t wd = __ldg(reinterpret_cast<const uint32_t*>(p.w.packed) + (i0 >> 3));
          const int64_t b = i0 >> p.w.log2_bs;
          const float sc = __fadd_rn(__fmul_rn(s_scb[__ldg(p.w.codes + b)],
                                               __ldg(p.w.absmax + (b >> p.w.log2_nbs))),
                                     offset);
          uint32_t h[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t byte = (wd >> (8 * e)) & 0xFFu;
            h[e] = pack2<kBF16 ? DQ4_OUT_BF16 : DQ4_OUT_F16>(__fmul_rn(s_vcb[byte >> 4], sc),
                                                             __fmul_rn(s_vcb[byte & 0xFu], sc));
          }
          q = make_uint4(h[0], h[1], h[2], h[3]);
        }
        *reinterpret_cast<uint4*>(sB + swz128(r, ch)) = q;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive(full_b(s));
    }
    // epilogue: warps w and w + 4 share TMEM lane quadrant w % 4; each takes half the columns
    if (!failed && !*abort_flag && mbar_wait(acc_full, 0)) {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int quad = warp & 3;
      const int64_t row = m0 + quad * 32 + lane;
      const int c_begin = (warp >> 2) * (BN / 2);
#pragma unroll 1
      for (int cb = c_begin; cb < c_begin + BN / 2; cb += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + (static_cast<uint32_t>(quad * 32) << 16) + cb, v);
        const int64_t col0 = n0 + cb;
        if (row >= p.M) continue;
        const int64_t ncol = p.N - col0 < 32 ? p.N - col0 : 32;
        if (ncol <= 0) continue;
        const int64_t o = row * p.N + col0;
        const int osz = p.out_dtype == DQ4_OUT_F32 ? 4 : 2;
        if (ncol == 32 && (reinterpret_cast<uintptr_t>(p.Y) + o * osz) % 16 == 0) {
          uint4* y4 = reinterpret_cast<uint4*>(static_cast<char*>(p.Y) + o * osz);
          if (p.out_dtype == DQ4_OUT_F32) {
#pragma unroll
            for (int e = 0; e < 8; ++e)
              y4[e] = make_uint4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
          } else if (p.out_dtype == DQ4_OUT_BF16) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              y4[e] = make_uint4(
                  pack2<DQ4_OUT_BF16>(__uint_as_float(v[8 * e]), __uint_as_float(v[8 * e + 1])),
                  pack2<DQ4_OUT_BF16>(__uint_as_float(v[8 * e + 2]), __uint_as_float(v[8 * e + 3])),
                  pack2<DQ4_OUT_BF16>(__uint_as_float(v[8 * e + 4]), __uint_as_float(v[8 * e + 5])),
                  pack2<DQ4_OUT_BF16>(__uint_as_float(v[8 * e + 6]), __uint_as_float(v[8 * e + 7])));
          } else {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              y4[e] = make_uint4(
                  pack2<DQ4_OUT_F16>(__uint_as_float(v[8 * e]), __uint_as_float(v[8 * e + 1])),
                  pack2<DQ4_OUT_F16>(__uint_as_float(v[8 * e + 2]), __uint_as_float(v[8 * e + 3])),
                  pack2<DQ4_OUT_F16>(__uint_as_float(v[8 * e + 4]), __uint_as_float(v[8 * e + 5])),
                  pack2<DQ4_OUT_F16>(__uint_as_float(v[8 * e + 6]), __uint_as_float(v[8 * e + 7])));
          }
          continue;
        }
        // a ragged or unaligned chunk: element by element (static register indices)
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          if (e >= ncol) break;
          const float f = __uint_as_float(v[e]);
          if (p.out_dtype == DQ4_OUT_F32) {
            static_cast<float*>(p.Y)[o + e] = f;
          } else if (p.out_dtype == DQ4_OUT_BF16) {
            static_cast<__nv_bfloat16*>(p.Y)[o + e] = __float2bfloat16_rn(f);
          } else {
            static_cast<__half*>(p.Y)[o + e] = __float2half_rn(f);
          }
        }
      }
    } else if (tid == 0 && p.bad) {
      atomicAdd(p.bad, 1);
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 8)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(tmem), "r"(BN));
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

template <int BN, bool kBF16>
int launch_linear(const CUtensorMap& tmap, const LinArgs& p, cudaStream_t stream, int dev) {
  using S = LinSmem<BN, kBF16>;
  auto kernel = dq4_linear_kernel<BN, kBF16>;
  static std::atomic<int> configured[kMaxDevices];
  if (dev >= 0 && dev < kMaxDevices && !configured[dev].load()) {
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S::kBytes);
    if (e != cudaSuccess) return fail_cuda(DQ4_ERR_LAUNCH, e);
    configured[dev].store(1);
  }
  const int64_t grid = int64_t(p.tiles_n) * ((p.M + kBM - 1) / kBM);
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
  const cudaError_t le = cudaLaunchKernelEx(&cfg, kernel, tmap, p);
  if (le != cudaSuccess) {
    cudaGetLastError();
    return fail_cuda(DQ4_ERR_LAUNCH, le);
  }
  return DQ4_OK;
#else
  kernel<<<static_cast<unsigned>(grid), kLinThreads, S::kBytes, stream>>>(tmap, p);
  return check_launch();
#endif
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
  if (K == 0 || K % kBK != 0 || M > INT32_MAX || K > INT32_MAX) return DQ4_ERR_N;
  if (!X || !packed || !scale_codes || !nested_absmax || !scale_codebook || !value_codebook ||
      !Y)
    return DQ4_ERR_NULL;
  if (misaligned(X, 16) || misaligned(packed, 4) || misaligned(nested_absmax, 4) ||
      misaligned(scale_codebook, 4) || misaligned(value_codebook, 4) ||
      misaligned(Y, out_itemsize(out_dtype)) || misaligned(bad, 4))
    return DQ4_ERR_ALIGN;
  int dev = 0, sms = 0;
  if (int st = current_device(&dev, &sms)) return st;
  EncodeTiled encode = tensor_map_encoder();
  if (!encode) return fail_cuda(DQ4_ERR_LAUNCH, cudaErrorNotSupported);

  // X as a 2-D tensor (K fastest, M rows): 64 x 128 boxes, 128-byte swizzle
  CUtensorMap tmap;
  const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
  const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(K) * 2};
  const cuuint32_t box[2] = {kBK, kBM};
  const cuuint32_t estride[2] = {1, 1};
  const CUresult cr = encode(&tmap,
                             in_dtype == DQ4_OUT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                      : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                             2, const_cast<void*>(X), gdim, gstride, box, estride,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
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
  const auto st = static_cast<cudaStream_t>(stream);
  // 256-column tiles when they still give at least one wave of CTAs; else 128
  const int64_t tiles_m = (M + kBM - 1) / kBM;
  const bool wide = ((N + 255) / 256) * tiles_m >= sms;
  const int bn = wide ? 256 : 128;
  const int64_t tiles_n = (N + bn - 1) / bn;
  if (tiles_n * tiles_m > INT32_MAX) return DQ4_ERR_N;
  p.tiles_n = static_cast<int>(tiles_n);
  if (in_dtype == DQ4_OUT_BF16)
    return wide ? launch_linear<256, true>(tmap, p, st, dev)
                : launch_linear<128, true>(tmap, p, st, dev);
  return wide ? launch_linear<256, false>(tmap, p, st, dev)
              : launch_linear<128, false>(tmap, p, st, dev);
}

}  // extern "C"

// LLM.int8 correction-operand preparation: dq4_int8_correction_prep.
#include "common.cuh"

namespace dq4d {

// ------------------------------------- LLM.int8 correction-operand preparation
// "Fuse LLM.int8 correction operand preparation into one CUDA kernel"
// (bitsandbytes issue #16), sections "Summary", "Bounded method" and "Exact
// correctness oracle", in one launch over two output regions:
//   subA[m][l] = A[m][cols[l]]                                   (16-bit copy)
//   subB[l][n] = RN16(RN32(RN32(CB[n][cols[l]] * SCB[n]) * RN32(1/127)))
// CTAs [0, ctas_a) fill subA: each covers a_per * kThreads consecutive elements
// of the row-major M x L array, lanes walking l, so stores are contiguous.  A
// thread's elements are a chain of dependent loads (index, then A), so a_per
// is as small as filling the SMs once allows (1 .. 8): small M x L spreads over
// many CTAs, large M x L keeps its gathers paced against the subB ones.  CTAs
// [ctas_a, ...) fill subB: each covers kBN consecutive n (two per thread:
// both SCB values in one 8-byte load, both results in one 4-byte store) and
// kBL consecutive l; per l a warp stores 128 contiguous bytes of subB.  The
// CB reads are a column gather (one byte of each of two rows per l); a
// thread issues all kBL * 2 of them before using any.  Column indices are
// bounds-checked: an index outside [0, K) reads nothing, yields 0 and is
// counted once into *bad (if given).
constexpr int kAMaxPer = 8;  // most subA elements per thread
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
  int a_per;  // subA elements per thread
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
    const int64_t e0 = bid * p.a_per * kThreads;
    const int64_t total = p.M * p.L;
    for (int k = 0; k < p.a_per; ++k) {
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

}  // namespace dq4d

using namespace dq4d;

extern "C" {

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
  {
    const int64_t per = (M * L + int64_t(kThreads) * sms - 1) / (int64_t(kThreads) * sms);
    p.a_per = int(per < 1 ? 1 : per > kAMaxPer ? kAMaxPer : per);
  }
  p.ctas_a = (M * L + int64_t(p.a_per) * kThreads - 1) / (int64_t(p.a_per) * kThreads);
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

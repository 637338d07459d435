// Row-blocked dequantization feeding cuBLAS GEMMs: dq4_nested_out_prod.
#include "common.cuh"

#include <cublas_v2.h>  // types only: cuBLAS is reached through dlopen / dlsym
#include <dlfcn.h>

#include <mutex>

namespace dq4d {
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

}  // namespace
}  // namespace dq4d

using namespace dq4d;

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

}  // extern "C"

// Host-side utilities of the dq4 library: the per-device property cache,
// argument validation, status strings and the C-ABI helpers.
#include "common.cuh"

namespace dq4d {

namespace {
thread_local int t_last_cuda_error = 0;
struct DeviceCache {
  std::atomic<int> sms{0};
  std::atomic<int> cc{0};
};
DeviceCache g_devices[kMaxDevices];

}  // namespace

int fail_cuda(int status, cudaError_t e) {
  t_last_cuda_error = static_cast<int>(e);
  return status;
}

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
int check_launch() {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail_cuda(DQ4_ERR_LAUNCH, e);
  return DQ4_OK;
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
  a.prefetch_ctas = 0;
  return a;
}

}  // namespace dq4d

using namespace dq4d;

extern "C" {

// incremented on any change of a signature in dq4.h (2: dq4_nested_linear's workspace)
constexpr int kAbiVersion = 3;
int dq4_abi_version(void) { return kAbiVersion; }

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
    case DQ4_ERR_CUBLAS: return "reserved (no entry point calls cuBLAS)";
    default: return "unknown status";
  }
}

int dq4_last_cuda_error(void) { return t_last_cuda_error; }

}  // extern "C"

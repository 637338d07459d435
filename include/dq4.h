/*
 * dq4 — blockwise 4-bit weight dequantization with nested (double-quantized)
 * scales, fused into one pass, for NVIDIA GB300 (compute capability 10.3).
 *
 * The operation ("Fuse nested scale reconstruction into SM103 4-bit
 * dequantization", bitsandbytes issue #21, sections "Problem", "Proposed
 * experiment" and "Correctness requirements"):
 *
 *   for i in [0, n):
 *     nib   = high nibble of packed[i/2] if i is even, else its low nibble
 *     b     = i / blocksize                  (outer block: one scale code)
 *     g     = b / nested_blocksize           (nested group of scale codes)
 *     scale = RN32( RN32(scale_codebook[scale_codes[b]] * nested_absmax[g]) + offset )
 *     v     = RN32( value_codebook[nib] * scale )
 *     out[i] = RN_out(v)          (IEEE round-to-nearest-even; FP32 stores v)
 *
 * The FP32 multiply and add of the scale are rounded separately (never a
 * fused multiply-add) so that the result is bit-identical to the unfused
 * sequence "dequantize scale codes to FP32, add the offset, dequantize the
 * values" of section "Problem".  No FP32 scale tensor is materialised by
 * dq4_nested.  Subnormals are kept (no flush to zero); FP16 overflow gives
 * +-infinity.  Every output bit is deterministic.
 *
 * Conventions shared by every entry point
 *  - All array pointers are DEVICE pointers (global memory of the current
 *    device), owned by the caller.  The library never allocates, frees or
 *    synchronizes; inputs are never modified.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *    stream).  Work is enqueued on it and the call returns immediately;
 *    ordering with other work on that stream is the stream's order.
 *  - The return value is a status code (DQ4_OK = 0 means enqueued).  On any
 *    error nothing has been enqueued, except DQ4_ERR_LAUNCH, which reports
 *    the CUDA runtime's error right after a launch (dq4_last_cuda_error()
 *    gives the cudaError_t).
 *  - n == 0 is a successful no-op (pointers may then be NULL).
 *  - blocksize: a power of two in [32, 4096].  nested_blocksize: a power of
 *    two >= 1 (256 is the standard nested layout).
 *  - Alignment: float arrays 4-byte aligned; `out` aligned to its element
 *    size.  Fastest path: `packed` 4-byte aligned and `out` 16-byte aligned
 *    (any cudaMalloc / PyTorch allocation is); other alignments run a
 *    per-element path with the same results.
 *  - Calls from several host threads are safe; the library keeps only a
 *    per-device cache of device properties (and, for
 *    dq4_nested_unfused_static, one static scratch array per device).
 */
#ifndef DQ4_H
#define DQ4_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Output element types (out_dtype). */
#define DQ4_OUT_F16 0  /* IEEE binary16, 2 bytes per value */
#define DQ4_OUT_BF16 1 /* bfloat16, 2 bytes per value */
#define DQ4_OUT_F32 2  /* IEEE binary32, 4 bytes per value */

/* Status codes. */
#define DQ4_OK 0
#define DQ4_ERR_NULL 1             /* a required pointer is NULL while n > 0 */
#define DQ4_ERR_N 2                /* n < 0 (or rows, cols < 0 / rows * cols too large) */
#define DQ4_ERR_BLOCKSIZE 3        /* blocksize not a power of two in [32, 4096] */
#define DQ4_ERR_NESTED_BLOCKSIZE 4 /* nested_blocksize not a power of two >= 1 */
#define DQ4_ERR_DTYPE 5            /* out_dtype not one of DQ4_OUT_* */
#define DQ4_ERR_ALIGN 6            /* a float array or `out` misaligned for its type */
#define DQ4_ERR_DEVICE 7           /* no current CUDA device could be queried */
#define DQ4_ERR_ARCH 8             /* current device is not compute capability 10.3 */
#define DQ4_ERR_LAUNCH 9           /* the CUDA runtime reported an error at launch */
#define DQ4_ERR_TOO_LARGE 10       /* more scratch needed than given (the static array) */
#define DQ4_ERR_CUBLAS 11          /* reserved: no entry point calls cuBLAS any more */

/* Version of this interface (incremented on any change of a signature). */
int dq4_abi_version(void);

/*
 * Fused nested dequantization: one kernel launch.
 *   packed           uint8[ceil(n/2)]  two 4-bit codes per byte, even index in the
 *                                      high nibble; for odd n the low nibble of the
 *                                      last byte is padding and is ignored
 *   scale_codes      uint8[NB]         NB = ceil(n / blocksize), one code per block
 *   nested_absmax    float[NG]         NG = ceil(NB / nested_blocksize)
 *   scale_codebook   float[256]        decodes a scale code
 *   value_codebook   float[16]         decodes a 4-bit code (decode_4bit)
 *   offset           scalar FP32 added to every rebuilt scale
 *   n                number of values
 *   out_dtype        DQ4_OUT_F16 / DQ4_OUT_BF16 / DQ4_OUT_F32
 *   out              n elements of out_dtype, flat (the weight's row-major order)
 * Formula: issue #21, section "Proposed experiment"; rounding: section
 * "Correctness requirements".
 */
int dq4_nested(const uint8_t* packed, const uint8_t* scale_codes, const float* nested_absmax,
               const float* scale_codebook, const float* value_codebook, float offset,
               int64_t n, int32_t blocksize, int32_t nested_blocksize, int32_t out_dtype,
               void* out, void* stream);

/*
 * Fused nested dequantization with transposed output: one kernel launch.
 * The n = rows * cols values are the row-major rows x cols weight W (value
 * i = W[i / cols][i % cols], exactly as dq4_nested reads them), and `out`
 * receives W^T row-major (cols x rows): value (r, c) goes to
 * out[c * rows + r].  Arguments and per-value arithmetic are those of
 * dq4_nested; rows and cols must be >= 0 and rows * cols must fit in
 * int64 (DQ4_ERR_N otherwise).  Source: issue #21, section "Correctness
 * requirements", which lists the op's transposed-output behaviour among
 * the cases that must stay bitwise identical.  Fastest when cols % 32 == 0
 * and `packed` is 16-byte aligned, and, for 16-bit output, rows % 4 == 0
 * with `out` 8-byte aligned (8-byte stores of four rows); any other shape
 * or alignment takes a second kernel, with the same results, that stages
 * each row's bytes from any nibble and stores element by element.
 */
int dq4_nested_transposed(const uint8_t* packed, const uint8_t* scale_codes,
                          const float* nested_absmax, const float* scale_codebook,
                          const float* value_codebook, float offset, int64_t rows,
                          int64_t cols, int32_t blocksize, int32_t nested_blocksize,
                          int32_t out_dtype, void* out, void* stream);

/*
 * Non-nested dequantization (a plain FP32 absmax per block): one launch.
 *   out[i] = RN_out( RN32( value_codebook[nib_i] * absmax[i / blocksize] ) )
 * absmax is float[ceil(n / blocksize)].  This is the third step of the
 * unfused sequence (issue #21, section "Problem", step 3) and the non-nested
 * state of section "Proposed experiment".
 */
int dq4(const uint8_t* packed, const float* absmax, const float* value_codebook, int64_t n,
        int32_t blocksize, int32_t out_dtype, void* out, void* stream);

/*
 * The unfused sequence of issue #21, section "Problem", as three launches on
 * `stream`, kept for comparison with the fused kernel:
 *   1. scale_scratch[b] = RN32(scale_codebook[scale_codes[b]] * nested_absmax[g])
 *   2. scale_scratch[b] = RN32(scale_scratch[b] + offset)
 *   3. dq4(packed, scale_scratch, ...)
 * scale_scratch is a caller-owned device float[ceil(n / blocksize)], fully
 * overwritten; it holds the FP32 scales afterwards.  The output is
 * bit-identical to dq4_nested.
 */
int dq4_nested_unfused(const uint8_t* packed, const uint8_t* scale_codes,
                       const float* nested_absmax, const float* scale_codebook,
                       const float* value_codebook, float offset, int64_t n,
                       int32_t blocksize, int32_t nested_blocksize, int32_t out_dtype,
                       void* out, float* scale_scratch, void* stream);

/*
 * The unfused sequence of dq4_nested_unfused, for callers that cannot
 * allocate device memory.  Some callers may not call cudaMalloc / cudaFree
 * at all: a serving loop that reserves all device memory when it starts
 * and forbids allocation afterwards (cudaMalloc and cudaFree can
 * synchronize the device and stall every other stream), a runtime whose
 * memory is handed out only by its own pool, or an allocator's own hook,
 * which must not re-enter the allocator.  This entry point allocates
 * nothing: the FP32 scale scratch is a fixed array inside the library.
 * No source page has a counterpart of this entry point; it only repackages
 * the unfused sequence above.
 *
 * Arguments, layout and results are those of dq4_nested_unfused, without
 * `scale_scratch`; the output is bit-identical.
 *   - Limit: ceil(n / blocksize) <= DQ4_STATIC_SCRATCH_BLOCKS outer blocks
 *     (16 MiB of FP32 scratch); a larger problem returns DQ4_ERR_TOO_LARGE
 *     before anything is enqueued.
 *   - The scratch is a file-scope __device__ array, so every GPU on which
 *     the library's kernels are loaded holds those 16 MiB until the
 *     process exits.
 *   - The first call on each device looks up the array's device address
 *     (once per device, with that device current).  Make that first call
 *     before any stream capture begins.  The address is kept until the
 *     process exits; after cudaDeviceReset the array may be loaded at
 *     another address, so calls after a reset of the device are not
 *     supported.
 *   - All calls share the one array, and each call overwrites the part it
 *     uses before reading it (nothing has to start at zero).  Calls that
 *     overlap on the GPU (on different streams, or from different host
 *     threads without ordering) race on it: order them on one stream.
 */
#define DQ4_STATIC_SCRATCH_BLOCKS 4194304
int dq4_nested_unfused_static(const uint8_t* packed, const uint8_t* scale_codes,
                              const float* nested_absmax, const float* scale_codebook,
                              const float* value_codebook, float offset, int64_t n,
                              int32_t blocksize, int32_t nested_blocksize, int32_t out_dtype,
                              void* out, void* stream);

/*
 * LLM.int8 correction-operand preparation in one launch.  Source: "Fuse
 * LLM.int8 correction operand preparation into one CUDA kernel"
 * (bitsandbytes issue #16), sections "Summary", "Bounded method" and
 * "Exact correctness oracle":
 *   subA[m][l] = A[m][cols[l]]                      (16-bit copy, bit for bit)
 *   subB[l][n] = RN16( RN32( RN32(CB[n][cols[l]] * SCB[n]) * RN32(1/127) ) )
 *   A        uint16[M][K]  16-bit activations (FP16 or BF16 bits), row-major
 *   CB       int8[N][K]    int8 weights, row-major
 *   SCB      float[N]      per-row statistics
 *   cols     int64[L]      outlier column indices; repeats allowed
 *   subA     uint16[M][L]  written row-major (the gather of A's columns)
 *   subB     uint16[L][N]  FP16, written row-major (the transposed dequantized
 *                          columns, the layout the correction GEMM consumes)
 *   bad_cols optional device int (NULL to skip): incremented once per index
 *            outside [0, K); such an index reads nothing and yields zeros.
 * L == 0 (no outliers) is a successful no-op.  M, N, K, L >= 0 and K >= 1
 * when L > 0 (DQ4_ERR_N otherwise).  Pointers aligned to their element
 * types (DQ4_ERR_ALIGN).  Fastest when N is even and subB 4-byte / SCB
 * 8-byte aligned.
 */
int dq4_int8_correction_prep(const uint16_t* A, const int8_t* CB, const float* SCB,
                             const int64_t* cols, int64_t M, int64_t N, int64_t K, int64_t L,
                             uint16_t* subA, uint16_t* subB, int* bad_cols, void* stream);

/*
 * Row-blocked dequantization fused into a GEMM:
 *   dst = W^T * G       W = the FP32 dequantization of the rows x cols weight
 * (dq4_nested's values read row-major), G a rows x ncols FP32 matrix, dst a
 * cols x ncols FP32 matrix, all row-major.  The sum runs over W's rows in
 * blocks of 64 rows, each dequantized inside the GEMM kernel (the whole
 * dequantized weight never exists, nor does any dequantized block in device
 * memory).  Source: "cuda: out_prod dequantizes a 2D weight in row blocks"
 * (llama.cpp pull request #4), section "What" (the weight's row blocks
 * dequantized through the F32 converter and accumulated into dst block
 * after block, with a bounded transient).
 *
 * Accuracy: each FP32 operand is split exactly into three BF16 terms and the
 * tensor cores accumulate in FP32 the six products whose terms total at most
 * 2 (the three dropped ones are below 2^-24 of each product), so dst carries
 * FP32 accuracy.  A G with a single 1 per column returns W's values exactly.
 *   workspace        optional device float buffer of workspace_bytes: the
 *                    rows are cut into row ranges that run on separate SMs
 *                    (as many as fill the GPU and whose cols x ncols FP32
 *                    partial tiles fit the buffer); a second kernel then
 *                    adds the partial tiles in range order, so the result is
 *                    deterministic.  NULL or too small: one row range,
 *                    written straight to dst.
 *                    dq4_nested_out_prod_workspace_bytes gives the size that
 *                    fills the current device.
 *   bad              optional device int: incremented when a wait inside the
 *                    kernel timed out (the result is then invalid)
 * rows == 0 zero-fills dst; cols == 0 or ncols == 0 is a no-op.
 * Requires a CC 10.3 device; every pointer 4-byte aligned (packed and
 * scale_codes included: they are staged in 4-byte words), else
 * DQ4_ERR_ALIGN.
 */
int dq4_nested_out_prod(const uint8_t* packed, const uint8_t* scale_codes,
                        const float* nested_absmax, const float* scale_codebook,
                        const float* value_codebook, float offset, int64_t rows, int64_t cols,
                        int32_t blocksize, int32_t nested_blocksize, const float* G,
                        int64_t ncols, float* dst, float* workspace, int64_t workspace_bytes,
                        int* bad, void* stream);

/*
 * The workspace bytes dq4_nested_out_prod uses to spread an (rows, cols,
 * ncols) problem over the current device's SMs (0 when one row range fills
 * them; negative DQ4_ERR_DEVICE if there is no usable device).
 */
int64_t dq4_nested_out_prod_workspace_bytes(int64_t rows, int64_t cols, int64_t ncols);

/*
 * Nested 4-bit dequantization fused into a tensor-core GEMM (one launch):
 *   Y = X * W^T       X: M x K (BF16 or FP16, in_dtype), W: the N x K weight
 * whose n = N * K values (row-major) are given as nested 4-bit codes exactly
 * as for dq4_nested; W is decoded stage by stage into tensor memory, where
 * the MMAs read it as their A operand (the same operand bits dq4_nested
 * writes for in_dtype), and never materialised in device memory.  Y is
 * M x N row-major in out_dtype; the accumulation is FP32 (tcgen05, sm_103a).
 * Source: "Fuse nested scale reconstruction into SM103 4-bit dequantization"
 * (bitsandbytes issue #21), sections "Problem" and "B300 evidence plan" (the
 * dequantize-plus-linear fallback, which rebuilds the scales, materialises
 * the weight and calls F.linear).
 *   in_dtype   DQ4_OUT_F16 or DQ4_OUT_BF16 (X's type; W is decoded to it)
 *   K          a positive multiple of 64; M, N >= 0 (M, N, K <= INT32_MAX)
 *   X, packed  16-byte aligned (both are read by TMA)
 *   workspace  optional device memory (NULL to skip), 256-byte aligned, of
 *              workspace_bytes bytes, zero-filled before its first use.  When
 *              dq4_nested_linear_workspace_bytes(M, N, K) is nonzero (the tiles
 *              would not fill the SMs in whole rounds and sharing them is
 *              expected to be faster) and workspace_bytes is at least that,
 *              one CTA runs per SM on an equal share of the (tile, K stage)
 *              units: partial FP32 tiles meet in the workspace and are summed
 *              in K order (deterministic).  Its size is bounded by the SM
 *              count, not the problem.  A completed call leaves its counters
 *              zero again, so it can be reused by later calls of any shape in
 *              the same stream (not by concurrent calls).  Without it each
 *              tile runs on one CTA; the result is the same up to FP32
 *              summation order.
 *   bad        optional device int (NULL to skip): incremented by each part
 *              of a CTA that stopped because a bounded wait ran out (never
 *              expected; nonzero means Y is incomplete and the workspace must
 *              be zero-filled again before its next use)
 * DQ4_ERR_N for K not a multiple of 64; DQ4_ERR_ALIGN for a misaligned X,
 * packed or workspace.
 */
int dq4_nested_linear(const void* X, int32_t in_dtype, const uint8_t* packed,
                      const uint8_t* scale_codes, const float* nested_absmax,
                      const float* scale_codebook, const float* value_codebook, float offset,
                      int64_t M, int64_t N, int64_t K, int32_t blocksize,
                      int32_t nested_blocksize, int32_t out_dtype, void* Y, void* workspace,
                      int64_t workspace_bytes, int* bad, void* stream);

/*
 * The workspace bytes dq4_nested_linear uses for an M x K by N x K problem on
 * the current device (0 when it would not use one); -DQ4_ERR_DEVICE without a
 * CC 10.3 device.  Shapes dq4_nested_linear rejects give 0.
 */
int64_t dq4_nested_linear_workspace_bytes(int64_t M, int64_t N, int64_t K);

/*
 * The fused path (dq4_nested's values, bit for bit) from host arrays to a
 * host array: the inputs go to the device, the output comes back, chunk by
 * chunk, with the copies of one chunk overlapping the kernel and the copies
 * of the others.  Source: "Fuse nested scale reconstruction into SM103 4-bit
 * dequantization" (bitsandbytes issue #21), section "Proposed experiment".
 *   packed .. value_codebook   HOST arrays laid out as for dq4_nested
 *                              (page-locked, for the copies to overlap)
 *   out                        HOST array of n elements of out_dtype
 *   scratch                    DEVICE memory, 256-byte aligned, of
 *                              scratch_bytes >= dq4_nested_host_scratch_bytes
 *                              (a smaller scratch takes smaller chunks, down
 *                              to one nested group; below that,
 *                              DQ4_ERR_TOO_LARGE)
 * The call is ordered in `stream`: it starts after the work already enqueued
 * there and the work enqueued after it sees `out` complete.  The host arrays
 * must stay valid until then.  Chunks start on nested-group boundaries, so a
 * chunk's scale codes and absmax are its own.  Each copy is one
 * cudaMemcpyAsync; two internal streams per device carry them.
 */
int dq4_nested_host(const uint8_t* packed, const uint8_t* scale_codes,
                    const float* nested_absmax, const float* scale_codebook,
                    const float* value_codebook, float offset, int64_t n, int32_t blocksize,
                    int32_t nested_blocksize, int32_t out_dtype, void* out, void* scratch,
                    int64_t scratch_bytes, void* stream);

/* Device scratch bytes for dq4_nested_host's default chunk (at most 2^24
 * values, whole nested groups); 0 for invalid arguments or n == 0. */
int64_t dq4_nested_host_scratch_bytes(int64_t n, int32_t blocksize, int32_t nested_blocksize,
                                      int32_t out_dtype);

/* A static, human-readable string for a status code (never NULL). */
const char* dq4_status_string(int status);

/* The cudaError_t behind the last DQ4_ERR_LAUNCH / DQ4_ERR_DEVICE /
 * DQ4_ERR_ARCH returned on the calling thread (0 if none). */
int dq4_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* DQ4_H */

// Host-to-host form of the fused path: dq4_nested_host.  The inputs and the
// output are host arrays (page-locked for the copies to overlap); the values
// are those dq4_nested computes ("Fuse nested scale reconstruction into SM103
// 4-bit dequantization", bitsandbytes issue #21, section "Proposed
// experiment").  The work runs in chunks of whole nested groups through two
// device buffers in the caller's scratch, so a chunk's scale codes and absmax
// are its own:
//   copy-in stream : inputs of chunk i   -> buffer i % 2 (after chunk i - 2's
//                    output left it)
//   caller's stream: dq4_nested on chunk i (after its inputs landed)
//   copy-out stream: output of chunk i   -> host (after its kernel)
// so the copies of one chunk overlap the kernel and the copies of the others.
// Each copy is one cudaMemcpyAsync.  The call is ordered in the caller's
// stream: it starts after the work already there and ends before the work
// enqueued after it.
#include "common.cuh"

#include <mutex>

namespace dq4d {
namespace {

// a chunk holds this many values unless the scratch or the problem is smaller
// (2^23 and 2^24 measure alike for a 470 MB output; 2^22 is slower, and a second copy-out
// stream gains nothing: the device-to-host link is the bound)
constexpr int64_t kChunkTarget = int64_t(1) << 24;

int64_t align256(int64_t b) { return (b + 255) / 256 * 256; }

int64_t out_size(int32_t out_dtype) { return out_dtype == DQ4_OUT_F32 ? 4 : 2; }

// device bytes of one buffer for a chunk of c values (a multiple of blocksize)
int64_t buffer_bytes(int64_t c, int32_t bs, int32_t nbs, int32_t out_dtype) {
  const int64_t blocks = (c + bs - 1) / bs;
  return align256((c + 1) / 2) + align256(blocks) + align256(4 * ((blocks + nbs - 1) / nbs)) +
         align256(c * out_size(out_dtype));
}

constexpr int64_t kCodebookBytes = 256 * 4 + 256;  // scale codebook (1 KB), value codebook

// the chunk size for n values: whole nested groups, at most kChunkTarget values
int64_t chunk_values(int64_t n, int32_t bs, int32_t nbs) {
  const int64_t group = int64_t(bs) * nbs;
  int64_t c = kChunkTarget / group * group;
  if (c < group) c = group;
  const int64_t whole = (n + group - 1) / group * group;
  return c < whole ? c : whole;
}

struct PipeStreams {
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, in_done[2] = {}, kern_done[2] = {}, out_done[2] = {};
  bool ready = false;
};

std::mutex g_pipe_mutex;  // held while a call enqueues (the streams and events are shared)
PipeStreams g_pipe[kMaxDevices];

int pipe_streams(int dev, PipeStreams** ps) {
  PipeStreams& p = g_pipe[dev];
  if (!p.ready) {
    cudaError_t e = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.start, cudaEventDisableTiming);
    for (int b = 0; b < 2 && e == cudaSuccess; ++b) {
      e = cudaEventCreateWithFlags(&p.in_done[b], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.kern_done[b], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p.out_done[b], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) return fail_cuda(DQ4_ERR_LAUNCH, e);
    p.ready = true;
  }
  *ps = &p;
  return DQ4_OK;
}

}  // namespace
}  // namespace dq4d

using namespace dq4d;

extern "C" {

int64_t dq4_nested_host_scratch_bytes(int64_t n, int32_t blocksize, int32_t nested_blocksize,
                                      int32_t out_dtype) {
  if (validate(n, blocksize, nested_blocksize, true, out_dtype) != DQ4_OK || n <= 0) return 0;
  const int64_t c = chunk_values(n, blocksize, nested_blocksize);
  return 2 * buffer_bytes(c, blocksize, nested_blocksize, out_dtype) + kCodebookBytes;
}

int dq4_nested_host(const uint8_t* packed, const uint8_t* scale_codes,
                    const float* nested_absmax, const float* scale_codebook,
                    const float* value_codebook, float offset, int64_t n, int32_t blocksize,
                    int32_t nested_blocksize, int32_t out_dtype, void* out, void* scratch,
                    int64_t scratch_bytes, void* stream) {
  if (int st = validate(n, blocksize, nested_blocksize, true, out_dtype)) return st;
  if (n == 0) return DQ4_OK;
  if (!packed || !scale_codes || !nested_absmax || !scale_codebook || !value_codebook || !out ||
      !scratch)
    return DQ4_ERR_NULL;
  if (misaligned(scratch, 256)) return DQ4_ERR_ALIGN;
  const int64_t group = int64_t(blocksize) * nested_blocksize;
  // the largest chunk (whole groups, at most the default) two buffers of the scratch hold
  int64_t c = chunk_values(n, blocksize, nested_blocksize);
  while (c > group && 2 * buffer_bytes(c, blocksize, nested_blocksize, out_dtype) +
                              kCodebookBytes > scratch_bytes)
    c -= group;
  if (2 * buffer_bytes(c, blocksize, nested_blocksize, out_dtype) + kCodebookBytes >
      scratch_bytes)
    return DQ4_ERR_TOO_LARGE;
  int dev = 0, sms = 0;
  if (int st = current_device(&dev, &sms)) return st;

  std::lock_guard<std::mutex> lock(g_pipe_mutex);
  PipeStreams* ps = nullptr;
  if (int st = pipe_streams(dev, &ps)) return st;
  const auto caller = static_cast<cudaStream_t>(stream);
  const int64_t osz = out_size(out_dtype);
  // scratch: codebooks, then two buffers of [packed | codes | absmax | out]
  char* base = static_cast<char*>(scratch);
  float* scb_d = reinterpret_cast<float*>(base);
  float* vcb_d = reinterpret_cast<float*>(base + 1024);
  const int64_t buf = buffer_bytes(c, blocksize, nested_blocksize, out_dtype);
  const int64_t blocks_c = (c + blocksize - 1) / blocksize;
  const int64_t off_codes = align256((c + 1) / 2);
  const int64_t off_absmax = off_codes + align256(blocks_c);
  const int64_t off_out = off_absmax + align256(4 * ((blocks_c + nested_blocksize - 1) /
                                                     nested_blocksize));
  auto check = [&](cudaError_t e) { return e == cudaSuccess ? DQ4_OK : fail_cuda(DQ4_ERR_LAUNCH, e); };

  // start after the caller's earlier work; codebooks first on the copy-in stream
  if (int st = check(cudaEventRecord(ps->start, caller))) return st;
  if (int st = check(cudaStreamWaitEvent(ps->in, ps->start, 0))) return st;
  if (int st = check(cudaStreamWaitEvent(ps->out, ps->start, 0))) return st;
  if (int st = check(cudaMemcpyAsync(scb_d, scale_codebook, 256 * 4, cudaMemcpyHostToDevice,
                                     ps->in)))
    return st;
  if (int st = check(cudaMemcpyAsync(vcb_d, value_codebook, 16 * 4, cudaMemcpyHostToDevice,
                                     ps->in)))
    return st;
  int last = 0;
  for (int64_t i0 = 0, i = 0; i0 < n; i0 += c, ++i) {
    const int b = int(i & 1);
    last = b;
    const int64_t cn = n - i0 < c ? n - i0 : c;                    // values of this chunk
    const int64_t b0 = i0 / blocksize, g0 = b0 / nested_blocksize;  // i0: whole groups
    const int64_t nb = ((i0 + cn - 1) / blocksize + 1) - b0;
    const int64_t ng = ((b0 + nb - 1) / nested_blocksize + 1) - g0;
    // buffer b: packed | codes | absmax | out, each sized for a full chunk (buffer_bytes)
    char* p = base + kCodebookBytes + b * buf;
    uint8_t* packed_d = reinterpret_cast<uint8_t*>(p);
    uint8_t* codes_d = reinterpret_cast<uint8_t*>(p + off_codes);
    float* absmax_d = reinterpret_cast<float*>(p + off_absmax);
    char* out_d = p + off_out;
    // inputs of this chunk, once the buffer's previous output has left
    if (i >= 2)
      if (int st = check(cudaStreamWaitEvent(ps->in, ps->out_done[b], 0))) return st;
    if (int st = check(cudaMemcpyAsync(packed_d, packed + i0 / 2, (i0 + cn + 1) / 2 - i0 / 2,
                                       cudaMemcpyHostToDevice, ps->in)))
      return st;
    if (int st = check(cudaMemcpyAsync(codes_d, scale_codes + b0, nb, cudaMemcpyHostToDevice,
                                       ps->in)))
      return st;
    if (int st = check(cudaMemcpyAsync(absmax_d, nested_absmax + g0, ng * 4,
                                       cudaMemcpyHostToDevice, ps->in)))
      return st;
    if (int st = check(cudaEventRecord(ps->in_done[b], ps->in))) return st;
    // the chunk's dequantization in the caller's stream
    if (int st = check(cudaStreamWaitEvent(caller, ps->in_done[b], 0))) return st;
    if (int st = dq4_nested(packed_d, codes_d, absmax_d, scb_d, vcb_d, offset, cn, blocksize,
                            nested_blocksize, out_dtype, out_d, caller))
      return st;
    if (int st = check(cudaEventRecord(ps->kern_done[b], caller))) return st;
    // its output back to the host
    if (int st = check(cudaStreamWaitEvent(ps->out, ps->kern_done[b], 0))) return st;
    if (int st = check(cudaMemcpyAsync(static_cast<char*>(out) + i0 * osz, out_d, cn * osz,
                                       cudaMemcpyDeviceToHost, ps->out)))
      return st;
    if (int st = check(cudaEventRecord(ps->out_done[b], ps->out))) return st;
  }
  // the call ends in the caller's stream (the copy-out stream runs in order, so its last
  // copy covers the earlier ones)
  return check(cudaStreamWaitEvent(caller, ps->out_done[last], 0));
}

}  // extern "C"

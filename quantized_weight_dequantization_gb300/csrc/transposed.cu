// Transposed-output path of the dq4 library: dq4_nested_transposed.
#include "common.cuh"

namespace dq4d {

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
// That is the staged form below (cols % 32 == 0 and `packed` 16-byte aligned,
// every row segment two aligned 16-byte chunks); kStoreVec: rows is even and
// `out` is aligned to two elements (pair stores), otherwise elements are
// stored one by one.  Other shapes take the odd-shape staged form further
// down.

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

// (a * sa, b * sb), each product rounded to nearest FP32 on its own (one packed f32x2
// multiply; no contraction, so the bits equal two __fmul_rn).
__device__ __forceinline__ void mul2_pair(float a, float b, uint64_t s2, float& x, float& y) {
  uint64_t ab, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ab) : "f"(a), "f"(b));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(ab), "l"(s2));
  asm("mov.b64 {%0, %1}, %2;" : "=f"(x), "=f"(y) : "l"(r));
}

// The FP32 word at shared-memory byte address `addr`.
__device__ __forceinline__ float lds_f32_t(uint32_t addr) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
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
// x 256 columns of W: the scale codes and absmax of its 32-value row segments
// are loaded into registers first, then its packed bytes (128 B per row, whole
// cache lines) cooperatively and coalesced into shared memory, so both round
// trips overlap; after one barrier the threads turn their codes into the
// segments' scales in shared memory, and after another each warp decodes one
// 64 x 64 warp tile from shared memory and stores it as above.  CTAs are walked
// in column-major order.
constexpr int kSR = 128;                 // CTA tile rows
constexpr int kSC = 256;                 // CTA tile columns (128 packed bytes per row)
constexpr int kSRowBytes = kSC / 2;      // smem row: 8 chunks of 16 B, XOR-swizzled
constexpr int kSSeg = kSC / 32;          // 32-value scale segments per row

// 16-byte chunk `ch` of staged row `rr` sits at chunk position ch ^ key(rr):
// lanes reading rows 2p (and 2p + 1) of 8 consecutive p then hit 8 distinct
// chunk positions, i.e. all 32 banks.
__device__ __forceinline__ int swz(int rr, int ch) { return ch ^ ((rr >> 1) & 7); }

// Resident CTAs per SM the staged transposed kernel is compiled for: 8 (32 registers a
// thread, the full 64 warps) by default.  The four-row form is also built for 6 (40
// registers): a grid of more than one but at most 1.5 waves of 8 CTAs per SM runs as 1.3 to
// 2 waves of 6 instead of a full wave and a thin second one, which measured faster there
// (GB300, FP16/BF16, 4096 x 11008 and 11008 x 4096: 21.5 -> 20.7 us; 4096 x 12288: 23.9 ->
// 22.4 us; at exactly one wave, at 1.74 waves and from 2.5 waves on, and for grids under
// one wave, 8 per SM was as fast or faster).
constexpr int kTMinCtas = 8;
constexpr int kTMinCtasWide = 6;

// kQuad (16-bit output, rows % 4 == 0, out 8-byte aligned): lanes 2q and 2q + 1 hold rows
// 4q .. 4q + 3 of the tile between them; per two columns they swap one packed pair, so each
// writes 8 bytes (4 rows) of one column: half the store instructions of pair stores.
template <int OUT, bool kStoreVec, bool kQuad = false, int kMinCtas = kTMinCtas>
__global__ void __launch_bounds__(kThreads, kMinCtas)
    dq4_transposed_kernel(const Args a, int64_t rows, int64_t cols, uint32_t tiles_r) {
  __shared__ float s_vcb[16];
  __shared__ float s_scb[256];
  __shared__ __align__(16) uint8_t s_pk[kSR][kSRowBytes];
  // [segment][row]: a lane's 2 rows are one float2; the 4-float pad puts a warp's
  // 8 segments x 4 rows of stores in 32 distinct banks
  __shared__ __align__(8) float s_sc[kSSeg][kSR + 4];
#if DQ4_PDL
#if DQ4_L2_PREFETCH
  // (as in the flat kernel) L2 prefetches of the tile's lines before the wait: thread t
  // of the first kSR asks for row r0 + t's packed bytes and absmax, thread kSR + t for its
  // scale codes.  A prefetch returns nothing, so no value read after the wait changes.
  if (blockIdx.x < a.prefetch_ctas) {
    const int t = threadIdx.x & (kSR - 1);
    const int64_t r = int64_t(blockIdx.x % tiles_r) * kSR + t;
    if (r < rows) {
      const int64_t i = r * cols + int64_t(blockIdx.x / tiles_r) * kSC;
      if (threadIdx.x < kSR) {
        asm volatile("prefetch.global.L2 [%0];" :: "l"(a.packed + (i >> 1)));
        asm volatile("prefetch.global.L2 [%0];"
                     :: "l"(a.absmax + ((i >> a.log2_bs) >> a.log2_nbs)));
      } else {
        asm volatile("prefetch.global.L2 [%0];" :: "l"(a.codes + (i >> a.log2_bs)));
      }
    }
  }
#endif
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
#endif
  if (threadIdx.x < 16) s_vcb[threadIdx.x] = __ldg(a.vcb + threadIdx.x);
  for (int k = threadIdx.x; k < 256; k += kThreads) s_scb[k] = __ldg(a.scb + k);
  const int64_t r0 = int64_t(blockIdx.x % tiles_r) * kSR;  // column-major CTA order
  const int64_t c0 = int64_t(blockIdx.x / tiles_r) * kSC;

  // the scale inputs of the 32-value segments first, so their loads overlap the packed rows'
  constexpr int kScPer = kSR * kSSeg / kThreads;
  uint32_t sc_code[kScPer];
  float sc_am[kScPer];
#pragma unroll
  for (int k = 0; k < kScPer; ++k) {
    const int id = threadIdx.x + kThreads * k;
    const int rr = id / kSSeg, q = id % kSSeg;
    const int64_t r = r0 + rr, c = c0 + 32 * q;
    sc_code[k] = 0;
    sc_am[k] = 0.f;
    if (r < rows && c < cols) {
      const int64_t b = (r * cols + c) >> a.log2_bs;
      sc_code[k] = __ldg(a.codes + b);
      sc_am[k] = __ldg(a.absmax + (b >> a.log2_nbs));
    }
  }
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
  for (int k = 0; k < kScPer; ++k) {
    const int id = threadIdx.x + kThreads * k;
    const int rr = id / kSSeg, q = id % kSSeg;  // a warp: 4 rows x 8 segments (codes coalesced)
    // (segments past the edges get a scale of no meaning: their values are never stored)
    s_sc[q][rr] = __fadd_rn(__fmul_rn(s_scb[sc_code[k]], sc_am[k]), a.offset);
  }
  __syncthreads();

  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wr = 64 * (w >> 2);  // warp tile: rows wr .. +64, columns wc .. +64 of the CTA tile
  const int wc = 64 * (w & 3);
  const int64_t ra = r0 + wr + 2 * lane;  // this lane's rows: ra, ra + 1
  const bool has0 = ra < rows, has1 = ra + 1 < rows;
  // (the quad path keeps every lane for its shuffles: a pair's rows are valid together)
  if (!kQuad && !has0) return;
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
    uint64_t sc2;  // (scale of row ra, scale of row ra + 1)
    asm("mov.b64 %0, {%1, %2};" : "=l"(sc2) : "f"(scp.x), "f"(scp.y));
    const uint32_t vcb = static_cast<uint32_t>(__cvta_generic_to_shared(s_vcb));
#pragma unroll
    for (int k = 0; k < 4; ++k) {  // packed word k: 8 columns
      const uint32_t w0 = k == 0 ? s0.x : k == 1 ? s0.y : k == 2 ? s0.z : s0.w;
      const uint32_t w1 = k == 0 ? s1.x : k == 1 ? s1.y : k == 2 ? s1.z : s1.w;
      // nibble * 4 (the byte offset of its codebook entry) in each byte: the high
      // nibbles (values 0, 2, 4, 6 of the word) and the low ones (1, 3, 5, 7)
      const uint32_t h0 = (w0 >> 2) & 0x3C3C3C3Cu, l0 = (w0 << 2) & 0x3C3C3C3Cu;
      const uint32_t h1 = (w1 >> 2) & 0x3C3C3C3Cu, l1 = (w1 << 2) & 0x3C3C3C3Cu;
      if constexpr (kQuad) {
        const bool odd = lane & 1;
#pragma unroll
        for (int j = 0; j < 8; j += 2) {  // columns j (high nibbles) and j + 1 (low)
          const uint32_t sel = 0x4440u + (j >> 1);
          float v0, v1, u0, u1;
          mul2_pair(lds_f32_t(vcb + __byte_perm(h0, 0, sel)),
                    lds_f32_t(vcb + __byte_perm(h1, 0, sel)), sc2, v0, v1);
          mul2_pair(lds_f32_t(vcb + __byte_perm(l0, 0, sel)),
                    lds_f32_t(vcb + __byte_perm(l1, 0, sel)), sc2, u0, u1);
          const uint32_t pj = pack2<OUT>(v0, v1), pj1 = pack2<OUT>(u0, u1);
          const uint32_t got = __shfl_xor_sync(0xffffffffu, odd ? pj : pj1, 1);
          // even lane: column j, rows ra .. ra + 3; odd lane: column j + 1, rows ra - 2 .. ra + 1
          const uint2 val = odd ? make_uint2(got, pj1) : make_uint2(pj, got);
          const int64_t at = odd ? o + rows - 2 : o;
          if (has0) __stcs(reinterpret_cast<uint2*>(static_cast<uint16_t*>(a.out) + at), val);
          o += 2 * rows;
        }
      } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {  // value j of a word: byte j/2, high nibble first
        const uint32_t sel = 0x4440u + (j >> 1);
        const float a0 = lds_f32_t(vcb + __byte_perm((j & 1) ? l0 : h0, 0, sel));
        const float a1 = lds_f32_t(vcb + __byte_perm((j & 1) ? l1 : h1, 0, sel));
        float v0, v1;
        mul2_pair(a0, a1, sc2, v0, v1);
        store_pair<OUT, kStoreVec>(a.out, o, v0, v1, has0, has1);
        o += rows;
      }
      }
    }
  }
}

// Values n .. n + 7 of a staged row (n counted in value order from the row's first staged
// byte), one per nibble, value n + k at bits 4k: the two words holding them, each byte's two
// nibbles swapped (the high nibble is the even value), shifted down to value n.
__device__ __forceinline__ uint32_t nibbles8(const uint32_t* w, uint32_t n) {
  const uint32_t i = n >> 3;
  uint64_t v = (uint64_t(w[i + 1]) << 32) | w[i];
  v = ((v >> 4) & 0x0F0F0F0F0F0F0F0Full) | ((v << 4) & 0xF0F0F0F0F0F0F0F0ull);
  return uint32_t(v >> (4 * (n & 7u)));
}

// Staged form for any other shape (cols % 32 != 0 or `packed` not 16-byte aligned): the
// same 128 x 256 CTA tile and 64 x 64 warp tiles as the staged form.  A row of the tile
// starts at any nibble and may cross several scale blocks, so the CTA stages, per row, the
// packed bytes that hold its (at most 256) values, and the scales of the (at most 9) blocks
// they touch.  Warp w stages rows 16 w .. 16 w + 15: with `packed` 4-byte aligned, the 34
// aligned words that hold a row's bytes (129 bytes cover 256 nibbles from an odd start,
// plus up to 3 bytes before them), every load of its rows in flight together; otherwise
// byte by byte.  Lane p then decodes rows p and p + 32 of its warp tile (not 2p, 2p + 1),
// eight columns at a time: their nibbles from two staged words (nibbles8) and the scales of
// the at most two blocks they fall in.  With staged rows 35 words apart its 32 lanes read 32
// banks, and each store instruction writes 32 consecutive elements of W^T (element stores:
// rows and columns of any parity).
constexpr int kOddRowWords = 34;
constexpr int kOddRowStride = 4 * 35;  // bytes between staged rows (35 words: odd)
constexpr int kOddSeg = kSC / 32 + 1;  // blocks of >= 32 values a 256-value row run touches

template <int OUT>
__global__ void __launch_bounds__(kThreads)
    dq4_transposed_any_kernel(const Args a, int64_t rows, int64_t cols, uint32_t tiles_r) {
  __shared__ float s_vcb[16];
  __shared__ float s_scb[256];
  __shared__ __align__(16) uint8_t s_pk[kSR][kOddRowStride];
  __shared__ float s_sc[kSR][kOddSeg];
#if DQ4_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
#endif
  if (threadIdx.x < 16) s_vcb[threadIdx.x] = __ldg(a.vcb + threadIdx.x);
  for (int k = threadIdx.x; k < 256; k += kThreads) s_scb[k] = __ldg(a.scb + k);
  const int64_t r0 = int64_t(blockIdx.x % tiles_r) * kSR;  // column-major CTA order
  const int64_t c0 = int64_t(blockIdx.x / tiles_r) * kSC;
  const int nv = int(cols - c0 < kSC ? cols - c0 : kSC);  // values of a row in the tile
  const int64_t n_bytes = (a.n + 1) >> 1;
  // the scale codes and absmax of the blocks each row touches, into registers first
  constexpr int kScPer = (kSR * kOddSeg + kThreads - 1) / kThreads;
  uint32_t sc_code[kScPer];
  float sc_am[kScPer];
#pragma unroll
  for (int k = 0; k < kScPer; ++k) {
    const int id = threadIdx.x + kThreads * k;
    const int rr = id / kOddSeg, q = id - rr * kOddSeg;
    const int64_t r = r0 + rr;
    sc_code[k] = 0;
    sc_am[k] = 0.f;
    if (rr < kSR && r < rows) {
      const int64_t i0 = r * cols + c0;
      const int64_t b = (i0 >> a.log2_bs) + q;
      if (b <= (i0 + nv - 1) >> a.log2_bs) {
        sc_code[k] = __ldg(a.codes + b);
        sc_am[k] = __ldg(a.absmax + (b >> a.log2_nbs));
      }
    }
  }
  // the packed bytes of each row's values: staged byte k of row rr is byte
  // ((i0 >> 1) & ~3) + k of the array (word aligned; byte (i0 >> 1) + k with byte loads)
  {
    const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kRowsPerWarp = kSR / kWarpsPerCta;
    const bool words = (reinterpret_cast<uintptr_t>(a.packed) & 3) == 0;  // CTA-uniform
    if (words) {
      const uint32_t* pw = reinterpret_cast<const uint32_t*>(a.packed);
      const int64_t full_words = n_bytes >> 2;  // words wholly inside the array
#pragma unroll 4
      for (int q = 0; q < kRowsPerWarp; ++q) {
        const int rr = w * kRowsPerWarp + q;
        const int64_t r = r0 + rr;
        const int64_t w0 = r < rows ? ((r * cols + c0) >> 1) >> 2 : 0;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int j = lane + 32 * h;
          if (j >= kOddRowWords) break;
          const int64_t wi = w0 + j;
          uint32_t v = 0;
          if (r < rows) {
            if (wi < full_words) {
              v = __ldcs(pw + wi);
            } else {  // the array's last, partial word
              for (int e = 0; e < 4 && 4 * wi + e < n_bytes; ++e)
                v |= uint32_t(a.packed[4 * wi + e]) << (8 * e);
            }
          }
          reinterpret_cast<uint32_t*>(s_pk[rr])[j] = v;
        }
      }
    } else {
#pragma unroll 2
      for (int q = 0; q < kRowsPerWarp; ++q) {
        const int rr = w * kRowsPerWarp + q;
        const int64_t r = r0 + rr;
        const int64_t b0 = r < rows ? (r * cols + c0) >> 1 : 0;
        constexpr int kBytes = 4 * kOddRowWords;
        uint8_t v[(kBytes + 31) / 32];
#pragma unroll
        for (int h = 0; h < (kBytes + 31) / 32; ++h) {
          const int k = lane + 32 * h;
          v[h] = (k < kBytes && r < rows && b0 + k < n_bytes) ? __ldcs(a.packed + b0 + k)
                                                             : uint8_t(0);
        }
#pragma unroll
        for (int h = 0; h < (kBytes + 31) / 32; ++h) {
          const int k = lane + 32 * h;
          if (k < kBytes) s_pk[rr][k] = v[h];
        }
      }
    }
  }
  __syncthreads();  // codebooks staged
#pragma unroll
  for (int k = 0; k < kScPer; ++k) {
    const int id = threadIdx.x + kThreads * k;
    const int rr = id / kOddSeg, q = id - rr * kOddSeg;
    // (blocks past a row's values get a scale of no meaning: no value reads it)
    if (rr < kSR) s_sc[rr][q] = __fadd_rn(__fmul_rn(s_scb[sc_code[k]], sc_am[k]), a.offset);
  }
  __syncthreads();

  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wr = 64 * (w >> 2);  // warp tile: rows wr .. +64, columns wc .. +64 of the CTA tile
  const int wc = 64 * (w & 3);
  const int la = wr + lane, lb = la + 32;  // this lane's rows of the CTA tile
  const int64_t ra = r0 + la, rb = r0 + lb;
  const bool has0 = ra < rows, has1 = rb < rows;
  if (!has0) return;
  const int ncol = nv - wc < 64 ? nv - wc : 64;
  if (ncol <= 0) return;
  // per row: the nibble position of column 0 in the staged row (value order from the staged
  // run's first byte: 8 x that word's index plus the first value's place in it) and the first
  // value's offset in its block; column c of the tile is then nibble n + c of the staged row
  // and block ((m + c) >> log2 bs) of the row's staged scales
  const bool words = (reinterpret_cast<uintptr_t>(a.packed) & 3) == 0;
  const uint32_t bs_mask = (1u << a.log2_bs) - 1u, pmask = words ? 7u : 1u;
  const int64_t i0a = ra * cols + c0, i0b = rb * cols + c0;
  const uint32_t pa = uint32_t(i0a) & pmask, pb = uint32_t(i0b) & pmask;
  const uint32_t ma = uint32_t(i0a) & bs_mask, mb = uint32_t(i0b) & bs_mask;
  const uint32_t* wa = reinterpret_cast<const uint32_t*>(s_pk[la]);
  const uint32_t* wb = reinterpret_cast<const uint32_t*>(s_pk[lb]);
  const float* sca = s_sc[la];
  const float* scb = s_sc[lb];
  int64_t o = (c0 + wc) * rows + ra;  // W^T index of (ra, column); advances by rows
  // eight columns at a time: their nibbles from two staged words, and the scales of the (at
  // most two: blocks hold >= 32 values) blocks they fall in
#pragma unroll 1
  for (int cc = 0; cc < ncol; cc += 8) {
    const uint32_t c = uint32_t(wc + cc);
    const uint32_t xa = nibbles8(wa, pa + c), xb = nibbles8(wb, pb + c);
    const uint32_t qa = (ma + c) >> a.log2_bs, qb = (mb + c) >> a.log2_bs;
    // columns left in the block of column c (>= 1); the next block's index is clamped to
    // the staged ones (a row's 256 values touch at most kOddSeg blocks)
    const uint32_t ta = (bs_mask + 1u) - ((ma + c) & bs_mask);
    const uint32_t tb = (bs_mask + 1u) - ((mb + c) & bs_mask);
    const float sa0 = sca[qa], sa1 = sca[min(qa + 1u, uint32_t(kOddSeg - 1))];
    const float sb0 = scb[qb], sb1 = scb[min(qb + 1u, uint32_t(kOddSeg - 1))];
    const int kn = ncol - cc < 8 ? ncol - cc : 8;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (k < kn) {
        store_one<OUT>(a.out, o, __fmul_rn(s_vcb[(xa >> (4 * k)) & 0xFu],
                                           uint32_t(k) < ta ? sa0 : sa1));
        if (has1)
          store_one<OUT>(a.out, o + 32, __fmul_rn(s_vcb[(xb >> (4 * k)) & 0xFu],
                                                  uint32_t(k) < tb ? sb0 : sb1));
      }
      o += rows;
    }
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
    const bool quad = OUT != DQ4_OUT_F32 && rows % 4 == 0 &&
                      reinterpret_cast<uintptr_t>(a.out) % 8 == 0;
    // every CTA prefetches in grids of at most DQ4_PREFETCH_WAVES waves, none in larger
    // ones, and only for 16-bit output: with FP32 output a wave writes more than L2 holds
    // and the prefetch measured slower (8192 x 8192: 49.3 -> 51.6 us; FP16 28672 x 8192:
    // 100.2 -> 97.0 us, 4096 x 4096: 10.7 -> 9.5 us)
    static std::atomic<int> occ_cache[kMaxDevices];
    static std::atomic<int> occ_cache_wide[kMaxDevices];
    Args b = a;
    const int64_t wave =
        int64_t(sms) * ctas_per_sm(dq4_transposed_kernel<OUT, true, true>, dev, occ_cache);
    b.prefetch_ctas =
        OUT != DQ4_OUT_F32 && grid <= int64_t(DQ4_PREFETCH_WAVES) * wave ? grid : 0;
    if (quad && grid > wave && 2 * grid <= 3 * wave) {  // (1, 1.5] waves of 8 CTAs per SM
      constexpr auto kWide = dq4_transposed_kernel<OUT, true, true, kTMinCtasWide>;
      const int64_t wave6 = int64_t(sms) * ctas_per_sm(kWide, dev, occ_cache_wide);
      b.prefetch_ctas = grid <= int64_t(DQ4_PREFETCH_WAVES) * wave6 ? grid : 0;
      return launch_kernel(kWide, grid, stream, b, rows, cols, tr);
    }
    if (quad)
      return launch_kernel(dq4_transposed_kernel<OUT, true, true>, grid, stream, b, rows, cols, tr);
    if (sv) return launch_kernel(dq4_transposed_kernel<OUT, true>, grid, stream, b, rows, cols, tr);
    return launch_kernel(dq4_transposed_kernel<OUT, false>, grid, stream, b, rows, cols, tr);
  }
  const int64_t tiles_r = (rows + kSR - 1) / kSR;
  const int64_t grid = tiles_r * ((cols + kSC - 1) / kSC);  // one CTA per 128 x 256 tile
  if (grid > int64_t(UINT32_MAX)) return DQ4_ERR_N;        // 32-bit tile ids
  return launch_kernel(dq4_transposed_any_kernel<OUT>, grid, stream, a, rows, cols,
                       uint32_t(tiles_r));
}

}  // namespace dq4d

using namespace dq4d;

extern "C" {

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

}  // extern "C"

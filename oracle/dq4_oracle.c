/*
 * Plain scalar CPU oracle for blockwise 4-bit dequantization with nested
 * (double-quantized) scales.  TEST INFRASTRUCTURE ONLY: the tests, the smoke
 * check and the CPU-baseline leg of the benchmark load it; the product path
 * never does.  It shares no code with the CUDA library.
 *
 * Source: "Fuse nested scale reconstruction into SM103 4-bit dequantization"
 * (bitsandbytes issue #21), sections "Problem" and "Proposed experiment":
 *
 *     scale = scale_codebook[scale_code] * nested_absmax[nested_group] + offset
 *     value = decode_4bit(packed_value) * scale
 *
 * and section "Correctness requirements": the FP32 multiply and the FP32 add
 * of the scale are rounded separately (no contraction).  This file must be
 * compiled with -ffp-contract=off (the builder in oracle/__init__.py does),
 * and each rounding is its own statement.
 *
 * Readings where the page is silent (each one is listed in the design notes):
 *   - two values per byte, the even index in the HIGH nibble; for odd n the
 *     low nibble of the last byte is padding and is never read;
 *   - block b = i / blocksize, nested group g = b / nested_blocksize (groups
 *     of scale codes);
 *   - decode_4bit(k) = value_codebook[k];
 *   - the value product is an FP32 product (one rounding), which is then
 *     rounded to FP16 / BF16 with IEEE round-to-nearest-even, subnormals
 *     kept, overflow to infinity.
 */
#include <stdint.h>
#include <string.h>

#define ORACLE_OUT_F16 0
#define ORACLE_OUT_BF16 1
#define ORACLE_OUT_F32 2

/* ------------------------------------------------------------------------
 * IEEE-754 round-to-nearest-even from binary32 to a narrower binary format
 * with p significand bits (hidden bit included), exponent bias `bias`.
 * Written from the definition: |x| = m * 2^E exactly; the quantum of the
 * result is 2^Q with Q = max(floor(log2|x|), emin) - (p - 1); the integer
 * m * 2^(E - Q) is rounded half-to-even; a carry to 2^p renormalises; an
 * exponent above emax becomes infinity.
 * ---------------------------------------------------------------------- */
static int bit_length_u64(uint64_t v) {
    int b = 0;
    while (v) { b++; v >>= 1; }
    return b;
}

static uint16_t round_f32_to_narrow(float x, int p, int bias, int exp_bits) {
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    const uint16_t sign = (uint16_t)((u >> 31) << 15);
    const uint32_t e32 = (u >> 23) & 0xFFu;
    const uint32_t f32 = u & 0x7FFFFFu;
    const int emax = bias;           /* largest unbiased exponent */
    const int emin = 1 - bias;       /* smallest normal exponent */
    const uint16_t exp_all_ones = (uint16_t)(((1u << exp_bits) - 1u) << (p - 1));

    if (e32 == 0xFFu) {
        if (f32 == 0) return (uint16_t)(sign | exp_all_ones);                 /* +-inf */
        return (uint16_t)(sign | exp_all_ones | (1u << (p - 2)));             /* quiet NaN */
    }
    uint64_t m;
    int E;
    if (e32 == 0) { m = f32; E = -149; }                 /* binary32 subnormal or zero */
    else { m = f32 | 0x800000u; E = (int)e32 - 150; }
    if (m == 0) return sign;                             /* +-0 */

    const int L = E + bit_length_u64(m) - 1;             /* floor(log2 |x|) */
    int Q = (L > emin ? L : emin) - (p - 1);
    const int s = Q - E;                                 /* bits dropped */
    uint64_t R;
    if (s <= 0) {
        R = m << (-s);                                   /* exact, no rounding needed */
    } else if (s > 60) {
        R = 0;                                           /* far below half a quantum */
    } else {
        R = m >> s;
        const uint64_t rem = m & ((1ull << s) - 1ull);
        const uint64_t half = 1ull << (s - 1);
        if (rem > half || (rem == half && (R & 1ull))) R++;
    }
    if (R == (1ull << p)) { R >>= 1; Q++; }              /* rounding carried */
    if (R == 0) return sign;
    if (R < (1ull << (p - 1))) return (uint16_t)(sign | R);   /* subnormal result */
    const int field = Q + (p - 1) + bias;
    if (Q + (p - 1) > emax) return (uint16_t)(sign | exp_all_ones);  /* overflow */
    return (uint16_t)(sign | ((uint32_t)field << (p - 1)) | (uint32_t)(R - (1ull << (p - 1))));
}

uint16_t oracle_f32_to_f16(float x) { return round_f32_to_narrow(x, 11, 15, 5); }
uint16_t oracle_f32_to_bf16(float x) { return round_f32_to_narrow(x, 8, 127, 8); }

void oracle_f32_to_f16_array(const float* x, uint16_t* y, int64_t count) {
    for (int64_t i = 0; i < count; i++) y[i] = oracle_f32_to_f16(x[i]);
}

void oracle_f32_to_bf16_array(const float* x, uint16_t* y, int64_t count) {
    for (int64_t i = 0; i < count; i++) y[i] = oracle_f32_to_bf16(x[i]);
}

/* Every binary32 bit pattern u in [first, first + count) converted, for the
 * exhaustive pins of the two converters. */
void oracle_convert_bit_range(uint32_t first, int64_t count, int to_bf16, uint16_t* y) {
    for (int64_t k = 0; k < count; k++) {
        uint32_t u = first + (uint32_t)k;
        float x;
        memcpy(&x, &u, sizeof x);
        y[k] = to_bf16 ? oracle_f32_to_bf16(x) : oracle_f32_to_f16(x);
    }
}

/* ------------------------------------------------------------------------
 * The method.
 * ---------------------------------------------------------------------- */

/* The 4-bit code of value i: high nibble of byte i/2 for even i, low for odd. */
static int nibble_of(const uint8_t* packed, int64_t i) {
    const uint8_t byte = packed[i / 2];
    return (i % 2 == 0) ? (byte >> 4) : (byte & 0x0F);
}

/* scale = scale_codebook[code] * nested_absmax[g] + offset, two FP32 roundings. */
float oracle_nested_scale(uint8_t code, float nested_absmax_g, const float* scale_codebook,
                          float offset) {
    const float product = scale_codebook[code] * nested_absmax_g;  /* RN32(product) */
    const float scale = product + offset;                          /* RN32(sum) */
    return scale;
}

static void store_value(void* out, int64_t i, float v, int out_dtype) {
    if (out_dtype == ORACLE_OUT_F16) {
        ((uint16_t*)out)[i] = oracle_f32_to_f16(v);
    } else if (out_dtype == ORACLE_OUT_BF16) {
        ((uint16_t*)out)[i] = oracle_f32_to_bf16(v);
    } else {
        ((float*)out)[i] = v;
    }
}

/* Fused nested dequantization of n values (the definition, value by value). */
void oracle_dq4_nested(const uint8_t* packed, const uint8_t* scale_codes,
                       const float* nested_absmax, const float* scale_codebook,
                       const float* value_codebook, float offset, int64_t n,
                       int64_t blocksize, int64_t nested_blocksize, int out_dtype, void* out) {
    for (int64_t i = 0; i < n; i++) {
        const int64_t b = i / blocksize;
        const int64_t g = b / nested_blocksize;
        const float scale = oracle_nested_scale(scale_codes[b], nested_absmax[g],
                                                scale_codebook, offset);
        const float v = value_codebook[nibble_of(packed, i)] * scale;   /* RN32(product) */
        store_value(out, i, v, out_dtype);
    }
}

/* Transposed output: the flat values are the row-major rows x cols weight W
 * (value i = W[i / cols][i % cols]); out holds W^T row-major, so element
 * (r, c) of W goes to out[c * rows + r].  Same per-value arithmetic. */
void oracle_dq4_nested_transposed(const uint8_t* packed, const uint8_t* scale_codes,
                                  const float* nested_absmax, const float* scale_codebook,
                                  const float* value_codebook, float offset, int64_t rows,
                                  int64_t cols, int64_t blocksize, int64_t nested_blocksize,
                                  int out_dtype, void* out) {
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t c = 0; c < cols; c++) {
            const int64_t i = r * cols + c;
            const int64_t b = i / blocksize;
            const int64_t g = b / nested_blocksize;
            const float scale = oracle_nested_scale(scale_codes[b], nested_absmax[g],
                                                    scale_codebook, offset);
            const float v = value_codebook[nibble_of(packed, i)] * scale;
            store_value(out, c * rows + r, v, out_dtype);
        }
    }
}

/* Non-nested dequantization: the per-block FP32 absmax is given directly. */
void oracle_dq4(const uint8_t* packed, const float* absmax, const float* value_codebook,
                int64_t n, int64_t blocksize, int out_dtype, void* out) {
    for (int64_t i = 0; i < n; i++) {
        const float v = value_codebook[nibble_of(packed, i)] * absmax[i / blocksize];
        store_value(out, i, v, out_dtype);
    }
}

/* The unfused sequence's first two steps: the FP32 per-block scale buffer. */
void oracle_nested_scales(const uint8_t* scale_codes, const float* nested_absmax,
                          const float* scale_codebook, float offset, int64_t nblocks,
                          int64_t nested_blocksize, float* scales) {
    for (int64_t b = 0; b < nblocks; b++)
        scales[b] = oracle_nested_scale(scale_codes[b], nested_absmax[b / nested_blocksize],
                                        scale_codebook, offset);
}

/* ------------------------------------------------------------------------
 * LLM.int8 correction-operand preparation: "Fuse LLM.int8 correction
 * operand preparation into one CUDA kernel" (bitsandbytes issue #16),
 * sections "Summary", "Bounded method" and "Exact correctness oracle":
 *   subA[m][l] = A[m][cols[l]]                               (raw 16-bit copy)
 *   subB[l][n] = RN16( RN32( RN32(CB[n][cols[l]] * SCB[n]) * RN32(1/127) ) )
 * A is M x K (16-bit elements), CB is N x K int8, SCB has N FP32 entries,
 * cols has L column indices in [0, K) (repeats allowed).  The reciprocal-127
 * constant is the FP32 quotient 1/127 rounded once.
 * ---------------------------------------------------------------------- */
void oracle_int8_correction_prep(const uint16_t* A, const int8_t* CB, const float* SCB,
                                 const int64_t* cols, int64_t M, int64_t N, int64_t K,
                                 int64_t L, uint16_t* subA, uint16_t* subB) {
    const float recip127 = 1.0f / 127.0f;
    for (int64_t m = 0; m < M; m++)
        for (int64_t l = 0; l < L; l++)
            subA[m * L + l] = A[m * K + cols[l]];
    for (int64_t l = 0; l < L; l++) {
        for (int64_t n = 0; n < N; n++) {
            const float t1 = (float)CB[n * K + cols[l]] * SCB[n];   /* RN32(CB * SCB) */
            const float t2 = t1 * recip127;                         /* RN32(t1 * 1/127) */
            subB[l * N + n] = oracle_f32_to_f16(t2);
        }
    }
}

/*
 * Oracle for the GGML Q4_0 x f32 quantized matmul, the Q4_0 -> f32 dequant,
 * and the Q8_0 dequant and quantize.
 *
 * TEST INFRASTRUCTURE ONLY.  This plain, single-threaded C99 code exists to
 * check the CUDA library.  Only the test suite, the smoke check and the CPU
 * baseline leg of the bench may load it; the product path never does.  It
 * shares no source with the CUDA library (no headers, helpers or tables).
 *
 * What it follows ("fuel-vulkan-kernels — quantized (GGML) kernel contracts",
 * fuel-dispatch 0.20.71, kernel-contracts/vulkan/quantized.fkc.md):
 *   - section "dequant_q4_0": an 18-byte block holds an f16 scale d followed
 *     by 16 bytes of 4-bit quants, one nibble per element; each element is
 *     (nibble - 8) * d, the nibble unsigned 0..15;
 *   - sections "qmatvec_q4_0" and "matmul_q4_0_tiled": C[m][n] is the sum over
 *     k of A[m][k] * dequant(W)[n][k], with W a row-major [N][K/32] block
 *     stream and K a multiple of 32.
 *   - section "dequant_q8_0": a 34-byte block holds an f16 scale d followed by
 *     32 signed 8-bit quants; each element is qs * d;
 *   - section "quantize_q8_0": per 32-element block, d = max|x| / 127, the
 *     block stores f16(d) and qs = round(x / d);
 *   - the GEMV fused with a preceding activation quantization ("act-quant
 *     fusion" in "vulkan: shader and sequencing efficiency backlog"): the
 *     product above with A replaced by dequant_q8_0(quantize_q8_0(A)).
 * Element j (0..15) of a Q4_0 block sits in the low nibble of quant byte j and
 * element j+16 in its high nibble; d is little-endian IEEE binary16 in the
 * block's first two bytes.  Sums are taken in fp64 in ascending k.
 *
 * Readings where the quantize section leaves a step open (the CUDA library
 * takes the same ones): the block arithmetic is f32 (the source is f32);
 * max|x| ignores NaN elements; d = max|x| / 127 is one correctly rounded f32
 * division; the stored scale is d narrowed to binary16 with round-to-nearest-
 * even (overflow to infinity); qs = round(x / d) uses that f32 d, one
 * correctly rounded f32 division, rounding halfway cases away from zero, then
 * clamped to [-127, 127] (this binds only when d is an f32 subnormal); qs = 0
 * where d is 0 or x / d is NaN.
 *
 * Every function here is pinned by the CPU tests (exhaustive f16 decode,
 * hand-built blocks, closed forms, brute force), none is "parity unpinned".
 */
#ifndef QM_ORACLE_H
#define QM_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_Q4_0_BLOCK_BYTES 18
#define ORACLE_Q4_0_BLOCK_ELEMS 32
#define ORACLE_Q8_0_BLOCK_BYTES 34

/* IEEE 754 binary16 bit pattern -> double (exact; NaN keeps only its class). */
double oracle_f16_to_double(uint16_t h);

/* Same conversion over an array (used by the exhaustive decoder test). */
void oracle_f16_to_double_array(const uint16_t* h, int64_t n, double* out);

/* A float -> IEEE 754 binary16 bit pattern, round to nearest, ties to even;
 * too large -> infinity; NaN -> a quiet NaN of the same sign.  Over an array. */
void oracle_float_to_f16_array(const float* x, int64_t n, uint16_t* out);

/* out[32*b + j] = (float)((nibble_j(b) - 8) * d(b)) for b < n_blocks. */
void oracle_dequant_q4_0(const uint8_t* wq, int64_t n_blocks, float* out);

/* out[32*b + j] = (float)(qs_j(b) * d(b)) for b < n_blocks (exact). */
void oracle_dequant_q8_0(const uint8_t* blob, int64_t n_blocks, float* out);

/* x[32*b + j] for b < n_blocks -> n_blocks Q8_0 blocks in blob, following the
 * readings above. */
void oracle_quantize_q8_0(const float* x, int64_t n_blocks, uint8_t* blob);

/* Full product: C[m*N+n] = sum_k A[m*K+k] * W[n][k] in fp64, ascending k;
 * S[m*N+n] = sum_k |A[m*K+k] * W[n][k]| (the tolerance scale).  S may be NULL.
 * Returns 0, or -1 if K is not a multiple of 32 or a size is negative. */
int oracle_matmul_q4_0(const float* A, const uint8_t* wq, int64_t M, int64_t N,
                       int64_t K, double* C, double* S);

/* The same sum for `count` chosen entries (m_idx[i], n_idx[i]) only, for
 * sampled checks at sizes where the full product is too slow.  S may be NULL.
 * Returns 0, or -1 on a bad size or an index out of range. */
int oracle_matmul_q4_0_entries(const float* A, const uint8_t* wq, int64_t M,
                               int64_t N, int64_t K, const int64_t* m_idx,
                               const int64_t* n_idx, int64_t count, double* C,
                               double* S);

/* C = A' x dequant(W)^T with A' = dequant_q8_0(quantize_q8_0(A)) row by row:
 * the product of the GEMV fused with a preceding activation quantization.  S
 * is the absolute sum with A'.  Returns 0, -1 on a bad size, -2 if scratch
 * memory could not be had. */
int oracle_matmul_q4_0_q8act(const float* A, const uint8_t* wq, int64_t M, int64_t N,
                             int64_t K, double* C, double* S);

/* The same at the (m_idx[i], n_idx[i]) entries only. */
int oracle_matmul_q4_0_q8act_entries(const float* A, const uint8_t* wq, int64_t M,
                                     int64_t N, int64_t K, const int64_t* m_idx,
                                     const int64_t* n_idx, int64_t count, double* C,
                                     double* S);

#ifdef __cplusplus
}
#endif

#endif /* QM_ORACLE_H */

/*
 * Oracle for the GGML Q4_0 x f32 quantized matmul and the Q8_0 dequant and
 * quantize — TEST INFRASTRUCTURE ONLY.
 * See qm_oracle.h for what it follows and who may use it.  Plain loops, fp64,
 * single-threaded, no blocking or reordering: a reader can check each line
 * against the definitions in the kernel-contract page
 * ("fuel-vulkan-kernels — quantized (GGML) kernel contracts").
 */
#include "qm_oracle.h"

#include <math.h>
#include <stddef.h>
#include <stdlib.h>

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 *   exponent 0      -> subnormal, value = fraction * 2^-24
 *   exponent 1..30  -> normal,    value = (1 + fraction/1024) * 2^(exponent-15)
 *   exponent 31     -> infinity (fraction 0) or NaN (fraction != 0)        */
double oracle_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int exponent = (h >> 10) & 0x1F;
    int fraction = h & 0x3FF;
    double magnitude;

    if (exponent == 0) {
        magnitude = ldexp((double)fraction, -24);
    } else if (exponent == 31) {
        magnitude = (fraction == 0) ? INFINITY : NAN;
    } else {
        magnitude = ldexp(1.0 + (double)fraction / 1024.0, exponent - 15);
    }
    return sign ? -magnitude : magnitude;
}

void oracle_f16_to_double_array(const uint16_t* h, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_to_double(h[i]);
}

/* binary16 from a value, by the definition: find the power of two 2^e below
 * |x|; normals (e >= -14) keep 11 significant bits, i.e. a quantum of
 * 2^(e-10); smaller values are multiples of 2^-24.  |x| / quantum is exact in
 * double, and nearbyint rounds it to the nearest integer, ties to even (the
 * default rounding mode).  Rounding up to 2^11 quanta moves to the next
 * exponent.  The largest finite binary16 is 65504; halfway to the next step
 * (65520) and beyond round to infinity. */
static uint16_t float_to_f16(float xf)
{
    double x = (double)xf;
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    double a = fabs(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7E00u);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u);
    if (a < ldexp(1.0, -14)) {
        double m = nearbyint(a / ldexp(1.0, -24));  /* 0 .. 1024; 1024 is 2^-14 */
        return (uint16_t)(sign | (uint16_t)m);
    }
    int e = 0;
    frexp(a, &e);
    e -= 1;  /* a in [2^e, 2^(e+1)) */
    double m = nearbyint(a / ldexp(1.0, e - 10));  /* 1024 .. 2048 */
    if (m == 2048.0) {
        m = 1024.0;
        e += 1;
    }
    return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)(m - 1024.0));
}

void oracle_float_to_f16_array(const float* x, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = float_to_f16(x[i]);
}

/* The block's scale d: bytes 0 and 1, little-endian binary16. */
static double block_scale(const uint8_t* block)
{
    uint16_t bits = (uint16_t)(block[0] | ((uint16_t)block[1] << 8));
    return oracle_f16_to_double(bits);
}

/* The unsigned 4-bit quant of element j (0..31): the quant bytes start at
 * block offset 2; element j < 16 is the low nibble of quant byte j, element
 * j >= 16 the high nibble of quant byte j - 16. */
static int block_nibble(const uint8_t* block, int j)
{
    const uint8_t* qs = block + 2;
    if (j < 16) return qs[j] & 0x0F;
    return (qs[j - 16] >> 4) & 0x0F;
}

/* Dequantized weight W[n][k] of a row-major [N][K/32] block stream, exact in
 * double: (nibble - 8) has at most 4 significant bits, d at most 11. */
static double weight_at(const uint8_t* wq, int64_t K, int64_t n, int64_t k)
{
    int64_t blocks_per_row = K / ORACLE_Q4_0_BLOCK_ELEMS;
    int64_t b = k / ORACLE_Q4_0_BLOCK_ELEMS;
    int j = (int)(k % ORACLE_Q4_0_BLOCK_ELEMS);
    const uint8_t* block = wq + (n * blocks_per_row + b) * ORACLE_Q4_0_BLOCK_BYTES;
    return (double)(block_nibble(block, j) - 8) * block_scale(block);
}

void oracle_dequant_q4_0(const uint8_t* wq, int64_t n_blocks, float* out)
{
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t b = 0; b < n_blocks; ++b) {
        const uint8_t* block = wq + b * ORACLE_Q4_0_BLOCK_BYTES;
        double d = block_scale(block);
        for (int j = 0; j < ORACLE_Q4_0_BLOCK_ELEMS; ++j) {
            double x = (double)(block_nibble(block, j) - 8) * d;
            out[b * ORACLE_Q4_0_BLOCK_ELEMS + j] = (float)x;
        }
    }
}

/* Q8_0 dequant: quant j is the signed byte at block offset 2 + j. */
void oracle_dequant_q8_0(const uint8_t* blob, int64_t n_blocks, float* out)
{
    for (int64_t b = 0; b < n_blocks; ++b) {
        const uint8_t* block = blob + b * ORACLE_Q8_0_BLOCK_BYTES;
        double d = block_scale(block);
        for (int j = 0; j < ORACLE_Q4_0_BLOCK_ELEMS; ++j) {
            int qs = (int)(int8_t)block[2 + j];
            out[b * ORACLE_Q4_0_BLOCK_ELEMS + j] = (float)((double)qs * d);
        }
    }
}

/* Q8_0 quantize, one block at a time, in the steps of the quantize section
 * (readings in qm_oracle.h). */
void oracle_quantize_q8_0(const float* x, int64_t n_blocks, uint8_t* blob)
{
    for (int64_t b = 0; b < n_blocks; ++b) {
        const float* xb = x + b * ORACLE_Q4_0_BLOCK_ELEMS;
        uint8_t* block = blob + b * ORACLE_Q8_0_BLOCK_BYTES;
        /* max |x| over the block; a NaN never compares greater */
        float amax = 0.0f;
        for (int j = 0; j < ORACLE_Q4_0_BLOCK_ELEMS; ++j) {
            float a = fabsf(xb[j]);
            if (a > amax) amax = a;
        }
        float d = amax / 127.0f;
        uint16_t bits = float_to_f16(d);
        block[0] = (uint8_t)(bits & 0xFF);
        block[1] = (uint8_t)(bits >> 8);
        for (int j = 0; j < ORACLE_Q4_0_BLOCK_ELEMS; ++j) {
            int q = 0;
            if (d != 0.0f) {
                float t = xb[j] / d;
                if (!isnan(t)) {
                    double r = round((double)t);  /* halfway cases away from zero */
                    if (r > 127.0) r = 127.0;
                    if (r < -127.0) r = -127.0;
                    q = (int)r;
                }
            }
            block[2 + j] = (uint8_t)(int8_t)q;
        }
    }
}

static int sizes_ok(int64_t M, int64_t N, int64_t K)
{
    return M >= 0 && N >= 0 && K >= 0 && (K % ORACLE_Q4_0_BLOCK_ELEMS) == 0;
}

/* One output entry: the fp64 sum over ascending k and its absolute sum. */
static void entry(const float* A, const uint8_t* wq, int64_t K, int64_t m,
                  int64_t n, double* c_out, double* s_out)
{
    double c = 0.0;
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        double product = (double)A[m * K + k] * weight_at(wq, K, n, k);
        c += product;
        s += fabs(product);
    }
    *c_out = c;
    if (s_out) *s_out = s;
}

int oracle_matmul_q4_0(const float* A, const uint8_t* wq, int64_t M, int64_t N,
                       int64_t K, double* C, double* S)
{
    if (!sizes_ok(M, N, K)) return -1;
    /* Entries are independent; a build with OpenMP (the multi-core CPU
     * baseline) shares them out over threads, each still summed by entry()
     * alone, so the result is the same bit for bit. */
#ifdef _OPENMP
#pragma omp parallel for collapse(2) schedule(static)
#endif
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            entry(A, wq, K, m, n, &C[m * N + n], S ? &S[m * N + n] : NULL);
        }
    }
    return 0;
}

int oracle_matmul_q4_0_entries(const float* A, const uint8_t* wq, int64_t M,
                               int64_t N, int64_t K, const int64_t* m_idx,
                               const int64_t* n_idx, int64_t count, double* C,
                               double* S)
{
    if (!sizes_ok(M, N, K) || count < 0) return -1;
    for (int64_t i = 0; i < count; ++i) {
        if (m_idx[i] < 0 || m_idx[i] >= M || n_idx[i] < 0 || n_idx[i] >= N) return -1;
    }
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < count; ++i) {
        entry(A, wq, K, m_idx[i], n_idx[i], &C[i], S ? &S[i] : NULL);
    }
    return 0;
}

/* The product with the activations quantized first (the GEMV fused with a
 * preceding activation quantization, as the efficiency backlog page
 * "vulkan: shader and sequencing efficiency backlog" lists it): each row of A
 * goes through quantize_q8_0 and back through dequant_q8_0, and the result
 * A' enters the same fp64 product as oracle_matmul_q4_0, S being the absolute
 * sum with A'.  Nothing else: the three steps are the functions above. */
static int dequantized_row(const float* A, int64_t K, int64_t m, uint8_t* q8, float* row)
{
    oracle_quantize_q8_0(A + m * K, K / ORACLE_Q4_0_BLOCK_ELEMS, q8);
    oracle_dequant_q8_0(q8, K / ORACLE_Q4_0_BLOCK_ELEMS, row);
    return 0;
}

int oracle_matmul_q4_0_q8act(const float* A, const uint8_t* wq, int64_t M, int64_t N,
                             int64_t K, double* C, double* S)
{
    if (!sizes_ok(M, N, K)) return -1;
    int64_t nb = K / ORACLE_Q4_0_BLOCK_ELEMS;
    uint8_t* q8 = (uint8_t*)malloc((size_t)(nb > 0 ? nb : 1) * ORACLE_Q8_0_BLOCK_BYTES);
    float* rows = (float*)malloc((size_t)(M * K > 0 ? M * K : 1) * sizeof(float));
    if (!q8 || !rows) {
        free(q8);
        free(rows);
        return -2;
    }
    for (int64_t m = 0; m < M; ++m) dequantized_row(A, K, m, q8, rows + m * K);
#ifdef _OPENMP
#pragma omp parallel for collapse(2) schedule(static)
#endif
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            entry(rows, wq, K, m, n, &C[m * N + n], S ? &S[m * N + n] : NULL);
        }
    }
    free(q8);
    free(rows);
    return 0;
}

int oracle_matmul_q4_0_q8act_entries(const float* A, const uint8_t* wq, int64_t M,
                                     int64_t N, int64_t K, const int64_t* m_idx,
                                     const int64_t* n_idx, int64_t count, double* C,
                                     double* S)
{
    if (!sizes_ok(M, N, K) || count < 0) return -1;
    for (int64_t i = 0; i < count; ++i) {
        if (m_idx[i] < 0 || m_idx[i] >= M || n_idx[i] < 0 || n_idx[i] >= N) return -1;
    }
    int64_t nb = K / ORACLE_Q4_0_BLOCK_ELEMS;
    uint8_t* q8 = (uint8_t*)malloc((size_t)(nb > 0 ? nb : 1) * ORACLE_Q8_0_BLOCK_BYTES);
    float* rows = (float*)malloc((size_t)(M * K > 0 ? M * K : 1) * sizeof(float));
    if (!q8 || !rows) {
        free(q8);
        free(rows);
        return -2;
    }
    for (int64_t m = 0; m < M; ++m) dequantized_row(A, K, m, q8, rows + m * K);
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < count; ++i) {
        entry(rows, wq, K, m_idx[i], n_idx[i], &C[i], S ? &S[i] : NULL);
    }
    free(q8);
    free(rows);
    return 0;
}

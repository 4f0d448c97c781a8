// Decode-regime GEMV on tensor cores: C[m][n] = sum_k A[m][k] * W[n][k] for
// M = 1..8 rows of f32 activations against a Q4_0 weight stream (sections
// "qmatvec_q4_0" and "matmul_q4_0_tiled" of "fuel-vulkan-kernels — quantized
// (GGML) kernel contracts": element j < 16 of a block is the low nibble of
// quant byte j, element j + 16 its high nibble, value (nibble - 8) * d).
//
// Arithmetic.  Each block's 32 products go through mma.sync m16n8k16 with
// bf16 operands and f32 accumulation:
//   * A operand (16 x 16) = 16 weight rows x 16 k of (q - 8), exact in bf16.
//   * B operand (16 x 8) = activation pieces: hi = bf16(a), lo = bf16(a - hi),
//     so |a - hi - lo| <= 2^-17 |a| and every product is exact in f32.  For
//     M <= 4 one MMA per k-step carries hi pieces in columns 0..M-1 and lo
//     pieces in columns M..2M-1; for M > 4 a second MMA adds the lo pieces.
//   * The block's MMA result is scaled once by its row's d in f32.  A row
//     whose total comes out infinite or NaN is recomputed element by element
//     (a non-finite d times q = 8 must give NaN, as the definition does).
//
// Data movement.  A "unit" is 8 blocks of one row (144 bytes, 256 k); a "row
// group" is 16 rows (one MMA tile); a "row block" is rps row groups.  A CTA
// (one per SM) owns a range of row blocks for one range of units (a K split).
// A producer warp streams stages through a ring in shared memory with TMA: a
// stage is one row block x c consecutive units, as c boxes of [16 rps rows]
// [144 B] (the 144-byte row stride keeps the per-lane 4-byte loads on
// distinct banks).  The W = rps * c consumer warps take one tile (16 rows x 1
// unit) each from every stage, in stage order, so a warp can never run two
// phases ahead of a stage's barrier.  Warp w always takes row group w % rps
// and unit column w / rps, so it accumulates its rows over every c-th unit of
// the row block; the c partial sums of a row group meet in shared memory
// (fixed column order) when the row block ends.  Consecutive stages walk a
// row block's units in order, so each row's bytes are read front to back by
// one CTA.  The activations of the CTA's K range arrive once (TMA, f32) and
// are rewritten in place as B fragments.
//
// Loads.  Lane (g, t) of a warp holds rows g and g + 8 of the tile and needs 4
// quant bytes of each per block.  A block pair is 36 bytes = 9 aligned words:
// the odd block's quants are words 5..8 (lane t takes word 5 + t); the even
// block's are misaligned by 2, so lanes t < 3 take words 1..3 (quant bytes
// 2..13) and lane 3 joins the halves of words 0 and 4 (bytes 0, 1, 14, 15).
// The order of k inside an MMA is free as long as A and B agree, so the B
// fragments are built in that same lane order.  Word 0 carries the even
// block's d, word 4 the odd block's.
//
// Launch.  Launched with programmatic stream serialization: the kernel lets
// its dependents start at once, and before its own wait it only initialises
// barriers and asks L2 for its first stages of weights (a hint that cannot
// return stale data); every read of A or the weights into the SM, and every
// write, comes after griddepcontrol.wait.
//
// Split K.  With S > 1 ranges (S = 2, 4 or 8) the S CTAs of a row-block range
// form a thread-block cluster: each keeps its row groups' partial sums in its
// own shared memory and, after a bounded mbarrier handshake, adds a share of
// the row groups over all S CTAs in range order through distributed shared
// memory and writes C, so results do not depend on timing and nothing is
// written outside C.  The allocation-free entry point (qm_matmul_q4_0_noalloc)
// instead meets the partial sums in its fixed scratch array, where the last of
// the S CTAs to arrive adds them in range order; it leaves the counters at zero.
#include <algorithm>
#include <mutex>

#include "qm_device.cuh"
#include "qm_internal.h"

namespace qm {

__device__ unsigned int g_gemv_tc_error = 0;

namespace {

constexpr int kUnitBytes = 144;
constexpr int kUnitElems = 256;
// Rows of one warp tile: 16 for the MMA consumer, 32 (one per lane) for the
// packed FP32 consumer.
__host__ __device__ constexpr int group_rows(bool packed) { return packed ? 32 : 16; }
// Consumer warps at most (the MMA consumer needs more registers per thread).
// (The integer consumer keeps more values per lane as M grows: fewer warps,
// so that the CTA's warps, counted in fours, leave it more registers.)
__host__ __device__ constexpr int max_warps(bool packed, int M = 1, bool q8 = false) {
    return !packed ? 16 : !q8 ? 24 : M == 1 ? 24 : M == 2 ? 22 : 14;
}
// Threads of a CTA at most: the consumers and the producer warp.
__host__ __device__ constexpr int max_threads(bool packed, int M = 1, bool q8 = false) {
    return (max_warps(packed, M, q8) + 1) * 32;
}
constexpr int kMaxStages = 12;
constexpr int kMaxSplits = 16;
// One warp's partial sums at the end of a row block: group rows x 8 columns.
__host__ __device__ constexpr int slot_floats(bool packed) { return group_rows(packed) * 8; }

struct TcPlan {
    const uint8_t* wq;  // the weight stream (read directly only by the exact fix-up)
    int N;
    int64_t K;
    int U;          // units per row
    int RG;         // row groups, ceil(N / 16)
    int S;          // K ranges; range s is units [s U / S, (s + 1) U / S)
    int rps;        // row groups per row block
    int c;          // units per stage (rps * c tiles)
    int hs;         // warps per tile: 1 (whole unit) or 2 (half a unit each)
    int rbpc;       // row blocks per CTA
    int nu_max;     // units in the largest K range
    int stages;     // ring depth
    int cl;         // 1: the S K ranges add up through a cluster (no scratch)
    float* part;    // [RG][S][M][16] split partial sums (S > 1, cl = 0)
    unsigned* ctr;  // [RG] arrival counters (S > 1, cl = 0), zero between launches
};

__device__ __forceinline__ uint32_t lds_u32(const uint8_t* p) {
    return *reinterpret_cast<const uint32_t*>(p);
}

// D = A x B (C = 0) and D += A x B, m16n8k16, bf16 in, f32 out.
__device__ __forceinline__ void mma_first(float d[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%10, %10, %10, %10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
}
__device__ __forceinline__ void mma_acc(float d[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (q - 8) as bf16 pairs from a quant word Q holding quant bytes (b0, b1, b2,
// b3), b0 lowest: R0 = low nibbles of (b0, b2), R1 = high nibbles of (b0, b2),
// R2 = low nibbles of (b1, b3), R3 = high nibbles of (b1, b3), the first of
// each pair in the low half.  A nibble under the bf16 exponent of 128 reads as
// 128 + q; subtracting 136 leaves q - 8, both steps exact.
__device__ __forceinline__ void decode_bf16(uint32_t Q, uint32_t R[4]) {
    constexpr uint32_t kMagic = 0x43004300u;  // bf16 128.0 in both halves
    const uint32_t r[4] = {(Q & 0x000F000Fu) | kMagic, ((Q >> 4) & 0x000F000Fu) | kMagic,
                           ((Q >> 8) & 0x000F000Fu) | kMagic, ((Q >> 12) & 0x000F000Fu) | kMagic};
    const __nv_bfloat162 bias = __floats2bfloat162_rn(-136.0f, -136.0f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const __nv_bfloat162 v = __hadd2(*reinterpret_cast<const __nv_bfloat162*>(&r[i]), bias);
        R[i] = *reinterpret_cast<const uint32_t*>(&v);
    }
}

// Quant bytes (b0, b2) of lane quarter t in a block of the given parity (the
// word layout above); k-step h of the block pairs elements (b0 + h, b2 + h)
// in the fragment's first k pair and (b0 + h + 16, b2 + h + 16) in its second.
__device__ __forceinline__ void lane_bytes(int t, int odd, int& b0, int& b2) {
    if (odd) {
        b0 = 4 * t;
        b2 = 4 * t + 2;
    } else if (t < 3) {
        b0 = 4 * t + 2;
        b2 = 4 * t + 4;
    } else {
        b0 = 0;
        b2 = 14;
    }
}

template <int M>
__host__ __device__ constexpr int tc_sets() { return M <= 4 ? 1 : 2; }

// Fragment columns a lane group reads: 2M (one set) or M per set.
template <int M>
__host__ __device__ constexpr int frag_cols() { return tc_sets<M>() == 1 ? 2 * M : M; }

// Rewrite one unit of staged activations, f32 [M][256] as the TMA box lands,
// into the unit's B fragments in place (the two take the same M KB).  Entry
// (uint2) for block kb, k-step h, set p, column col < frag_cols, quarter t:
// ((((kb * 2 + h) * P + p) * frag_cols + col) * 4 + t).  One set: columns
// 0..M-1 = hi pieces of rows 0..M-1, M..2M-1 = lo pieces.  Two sets: set 0 hi,
// set 1 lo, column = row.  A warp reads its 2M (hi, lo) groups of 4 values
// into registers, syncs, and overwrites.  The pieces are formed two at a
// time (packed bf16x2 conversions; lo from one packed FMA x - hi, exact), which
// halves the work of the conversion pipe; a value whose hi or lo is not
// finite makes its rows' totals not finite, and the epilogue recomputes those
// rows element by element.
template <int M>
__device__ __forceinline__ void build_fragments(uint8_t* unit, int lane) {
    constexpr int kPer = 2 * M;  // (kb, h, row, t) groups per lane
    const float* f = reinterpret_cast<const float*>(unit);
    float x[kPer][4];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int idx = lane + 32 * i;
        const int t = idx & 3;
        const int m = (idx >> 2) % M;
        const int kbh = idx / (4 * M);
        const int kb = kbh >> 1;
        const int h = kbh & 1;
        int b0, b2;
        lane_bytes(t, kb & 1, b0, b2);
        const float* row = f + m * kUnitElems + kb * kBlockElems;
        x[i][0] = row[b0 + h];
        x[i][1] = row[b2 + h];
        x[i][2] = row[b0 + h + 16];
        x[i][3] = row[b2 + h + 16];
    }
    __syncwarp();
    uint2* out = reinterpret_cast<uint2*>(unit);
    constexpr int P = tc_sets<M>();
    constexpr int NC = frag_cols<M>();
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int idx = lane + 32 * i;
        const int t = idx & 3;
        const int m = (idx >> 2) % M;
        const int kbh = idx / (4 * M);
        uint32_t hw[2], lw[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const __nv_bfloat162 hb = __floats2bfloat162_rn(x[i][2 * e], x[i][2 * e + 1]);
            hw[e] = *reinterpret_cast<const uint32_t*>(&hb);
            const float2 rest = __ffma2_rn(make_float2(__uint_as_float(hw[e] << 16), __uint_as_float(hw[e] & 0xFFFF0000u)),
                                           make_float2(-1.0f, -1.0f), make_float2(x[i][2 * e], x[i][2 * e + 1]));
            const __nv_bfloat162 lb = __floats2bfloat162_rn(rest.x, rest.y);
            lw[e] = *reinterpret_cast<const uint32_t*>(&lb);
        }
        const uint2 vh = make_uint2(hw[0], hw[1]);
        const uint2 vl = make_uint2(lw[0], lw[1]);
        if constexpr (P == 1) {
            out[(kbh * NC + m) * 4 + t] = vh;
            out[(kbh * NC + M + m) * 4 + t] = vl;
        } else {
            out[((kbh * 2 + 0) * NC + m) * 4 + t] = vh;
            out[((kbh * 2 + 1) * NC + m) * 4 + t] = vl;
        }
    }
}

// One block of a tile: quant words Qa (row g) and Qb (row g + 8), scales da,
// db, fragments F of block kb (entries of k-step 0 first).  Lane group g
// reads fragment column gc = g mod frag_cols: columns past frag_cols only
// repeat earlier ones, and their results are never read.
template <int M>
__device__ __forceinline__ void block_mma(uint32_t Qa, uint32_t Qb, float da, float db,
                                          const uint2* F, int gc, int t, float acc[4]) {
    constexpr int P = tc_sets<M>();
    constexpr int NC = frag_cols<M>();
    uint32_t ra[4], rb[4];
    decode_bf16(Qa, ra);
    decode_bf16(Qb, rb);
    uint2 b[2][P];
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int p = 0; p < P; ++p)
            b[h][p] = F[((h * P + p) * NC + gc) * 4 + t];
    float D[4];
    mma_first(D, ra[0], rb[0], ra[1], rb[1], b[0][0].x, b[0][0].y);
    if constexpr (P == 2) mma_acc(D, ra[0], rb[0], ra[1], rb[1], b[0][1].x, b[0][1].y);
    mma_acc(D, ra[2], rb[2], ra[3], rb[3], b[1][0].x, b[1][0].y);
    if constexpr (P == 2) mma_acc(D, ra[2], rb[2], ra[3], rb[3], b[1][1].x, b[1][1].y);
    acc[0] = fmaf(da, D[0], acc[0]);
    acc[1] = fmaf(da, D[1], acc[1]);
    acc[2] = fmaf(db, D[2], acc[2]);
    acc[3] = fmaf(db, D[3], acc[3]);
}

// NP block pairs of a tile from pair pp0 on (a whole unit: NP = 4, pp0 = 0;
// half h of it: NP = 2, pp0 = 2h): rows r0 (row g) and r1 (row g + 8) of a
// unit in shared memory, the unit's fragments F.
template <int M, int NP>
__device__ __forceinline__ void pairs_mma(const uint8_t* r0, const uint8_t* r1, const uint2* F, int pp0,
                                          int gc, int t, uint32_t xoff, uint32_t sel, float acc[4]) {
    constexpr int kEntriesPerBlock = 2 * tc_sets<M>() * frag_cols<M>() * 4;
    const uint32_t yoff = 20 + 4 * t;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
        const int pp = pp0 + i;
        const uint8_t* a = r0 + 36 * pp;
        const uint8_t* b = r1 + 36 * pp;
        const uint32_t w0a = lds_u32(a), w4a = lds_u32(a + 16), xa = lds_u32(a + xoff),
                       ya = lds_u32(a + yoff);
        const uint32_t w0b = lds_u32(b), w4b = lds_u32(b + 16), xb = lds_u32(b + xoff),
                       yb = lds_u32(b + yoff);
        const float dea = f16_bits_to_float(w0a & 0xFFFFu), doa = f16_bits_to_float(w4a >> 16);
        const float deb = f16_bits_to_float(w0b & 0xFFFFu), dob = f16_bits_to_float(w4b >> 16);
        block_mma<M>(__byte_perm(xa, w4a, sel), __byte_perm(xb, w4b, sel), dea, deb,
                     F + (2 * pp) * kEntriesPerBlock, gc, t, acc);
        block_mma<M>(ya, yb, doa, dob, F + (2 * pp + 1) * kEntriesPerBlock, gc, t, acc);
    }
}

// ---------------------------------------------------------------------------
// Packed FP32 consumer (lane = row): a lane reads half of its row's 144-byte
// unit (72 bytes, two block pairs) with four 16-byte loads and one 8-byte load
// (rows 144 bytes apart put the 8 lanes of a quarter-warp on distinct bank
// quads) and realigns the even blocks' quants with byte permutes.  Each nibble
// q goes into bits 16..19 of a word whose top byte is 0x43, which reads as the
// float 128 + q; one packed FMA per pair, x * d - 136 d, then gives (q - 8) * d
// exactly (136 d and (q - 8) d have at most 19 significant bits), and a second
// packed FMA (fma.rn.f32x2) adds its product with the activation into the
// row's sums.  A non-finite d makes the row's total non-finite, which the
// epilogue recomputes element by element.

// Selectors of __byte_perm(v, 0x43000000, s): byte i of v into bits 16..23,
// 0x43 into the top byte, zeros below.
constexpr uint32_t kPkHigh = 0x43000000u;
__host__ __device__ constexpr uint32_t pk_sel(int i) { return 0x7044u | (static_cast<uint32_t>(i) << 8); }

// One block: quant words q (elements j and j + 16 in byte j of the 16), its
// d pair and bias pair (-136 d), activations a (f32 [M][256] at the block).
template <int M>
__device__ __forceinline__ void block_dot_pk(const float* a, const uint32_t q[4], float2 d2, float2 b2,
                                             float2 (&s)[M][2]) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint32_t lo = q[w] & 0x0F0F0F0Fu;         // elements 4w .. 4w+3
        const uint32_t hi = (q[w] >> 4) & 0x0F0F0F0Fu;  // elements 16+4w .. 16+4w+3
        float2 v[4];
        v[0] = __ffma2_rn(make_float2(__uint_as_float(__byte_perm(lo, kPkHigh, pk_sel(0))),
                                      __uint_as_float(__byte_perm(lo, kPkHigh, pk_sel(1)))), d2, b2);
        v[1] = __ffma2_rn(make_float2(__uint_as_float(__byte_perm(lo, kPkHigh, pk_sel(2))),
                                      __uint_as_float(__byte_perm(lo, kPkHigh, pk_sel(3)))), d2, b2);
        v[2] = __ffma2_rn(make_float2(__uint_as_float(__byte_perm(hi, kPkHigh, pk_sel(0))),
                                      __uint_as_float(__byte_perm(hi, kPkHigh, pk_sel(1)))), d2, b2);
        v[3] = __ffma2_rn(make_float2(__uint_as_float(__byte_perm(hi, kPkHigh, pk_sel(2))),
                                      __uint_as_float(__byte_perm(hi, kPkHigh, pk_sel(3)))), d2, b2);
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const float4 al = *reinterpret_cast<const float4*>(a + m * kUnitElems + 4 * w);
            const float4 ah = *reinterpret_cast<const float4*>(a + m * kUnitElems + 16 + 4 * w);
            s[m][0] = __ffma2_rn(make_float2(al.x, al.y), v[0], s[m][0]);
            s[m][1] = __ffma2_rn(make_float2(al.z, al.w), v[1], s[m][1]);
            s[m][0] = __ffma2_rn(make_float2(ah.x, ah.y), v[2], s[m][0]);
            s[m][1] = __ffma2_rn(make_float2(ah.z, ah.w), v[3], s[m][1]);
        }
    }
}

__device__ __forceinline__ void pk_scale(uint32_t bits16, float2& d2, float2& b2) {
    const float d = f16_bits_to_float(bits16);
    const float b = -136.0f * d;
    d2 = make_float2(d, d);
    b2 = make_float2(b, b);
}

// A whole unit (8 blocks, nine 16-byte loads) of this lane's row against the
// unit's activations a (f32 [M][256] in shared memory).  acc holds the row's
// sums as two float pairs per activation row.
template <int M>
__device__ __forceinline__ void unit_dot_pk(const uint8_t* row, const float* a, float (&acc)[4 * M]) {
    uint32_t w[36];
#pragma unroll
    for (int i = 0; i < 9; ++i) {
        const uint4 v = reinterpret_cast<const uint4*>(row)[i];
        w[4 * i + 0] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
    float2 s[M][2];
#pragma unroll
    for (int m = 0; m < M; ++m) {
        s[m][0] = make_float2(acc[4 * m + 0], acc[4 * m + 1]);
        s[m][1] = make_float2(acc[4 * m + 2], acc[4 * m + 3]);
    }
#pragma unroll
    for (int pp = 0; pp < 4; ++pp) {
        const uint32_t* Wp = w + 9 * pp;
        float2 d2, b2;
        const uint32_t qa[4] = {__byte_perm(Wp[0], Wp[1], 0x5432u), __byte_perm(Wp[1], Wp[2], 0x5432u),
                                __byte_perm(Wp[2], Wp[3], 0x5432u), __byte_perm(Wp[3], Wp[4], 0x5432u)};
        pk_scale(Wp[0] & 0xFFFFu, d2, b2);
        block_dot_pk<M>(a + 64 * pp, qa, d2, b2, s);
        const uint32_t qb[4] = {Wp[5], Wp[6], Wp[7], Wp[8]};
        pk_scale(Wp[4] >> 16, d2, b2);
        block_dot_pk<M>(a + 64 * pp + 32, qb, d2, b2, s);
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
        acc[4 * m + 0] = s[m][0].x;
        acc[4 * m + 1] = s[m][0].y;
        acc[4 * m + 2] = s[m][1].x;
        acc[4 * m + 3] = s[m][1].y;
    }
}

// Half h of a unit (blocks 4h .. 4h + 3), as above.
template <int M>
__device__ __forceinline__ void half_dot_pk(const uint8_t* row, int h, const float* a, float (&acc)[4 * M]) {
    uint32_t w[18];
    if (h == 0) {  // bytes 0 .. 71: 16-byte loads first
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = reinterpret_cast<const uint4*>(row)[i];
            w[4 * i + 0] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
        const uint2 v = *reinterpret_cast<const uint2*>(row + 64);
        w[16] = v.x;
        w[17] = v.y;
    } else {  // bytes 72 .. 143: 16-byte loads from byte 80
        const uint2 v = *reinterpret_cast<const uint2*>(row + 72);
        w[0] = v.x;
        w[1] = v.y;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 u = reinterpret_cast<const uint4*>(row + 80)[i];
            w[2 + 4 * i + 0] = u.x;
            w[2 + 4 * i + 1] = u.y;
            w[2 + 4 * i + 2] = u.z;
            w[2 + 4 * i + 3] = u.w;
        }
    }
    float2 s[M][2];
#pragma unroll
    for (int m = 0; m < M; ++m) {
        s[m][0] = make_float2(acc[4 * m + 0], acc[4 * m + 1]);
        s[m][1] = make_float2(acc[4 * m + 2], acc[4 * m + 3]);
    }
    const float* ah = a + 128 * h;
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
        const uint32_t* Wp = w + 9 * pp;
        float2 d2, b2;
        // Even block: d in the low half of word 0, quants at bytes 2..17.
        const uint32_t qa[4] = {__byte_perm(Wp[0], Wp[1], 0x5432u), __byte_perm(Wp[1], Wp[2], 0x5432u),
                                __byte_perm(Wp[2], Wp[3], 0x5432u), __byte_perm(Wp[3], Wp[4], 0x5432u)};
        pk_scale(Wp[0] & 0xFFFFu, d2, b2);
        block_dot_pk<M>(ah + 64 * pp, qa, d2, b2, s);
        // Odd block: d in the high half of word 4, quants in words 5..8.
        const uint32_t qb[4] = {Wp[5], Wp[6], Wp[7], Wp[8]};
        pk_scale(Wp[4] >> 16, d2, b2);
        block_dot_pk<M>(ah + 64 * pp + 32, qb, d2, b2, s);
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
        acc[4 * m + 0] = s[m][0].x;
        acc[4 * m + 1] = s[m][0].y;
        acc[4 * m + 2] = s[m][1].x;
        acc[4 * m + 3] = s[m][1].y;
    }
}

// ---------------------------------------------------------------------------
// Integer consumer with the activations quantized to Q8_0 first (the GEMV
// fused with a preceding activation quantization: "act-quant fusion" in
// "vulkan: shader and sequencing efficiency backlog"; quantization as in
// section "quantize_q8_0" of "fuel-vulkan-kernels — quantized (GGML) kernel
// contracts").  The product is A' x dequant(W)^T with A' = dequant_q8_0(
// quantize_q8_0(A)), and per block of 32 it factors exactly:
//     sum_j A'_j W_j = (d_a d_w) * (sum_j q_j qs_j - 8 sum_j qs_j),
// q the weight nibbles 0..15, qs the activation quants, d_a and d_w the two
// binary16 scales.  The integer sums are exact (dp4a on the nibbles as
// unsigned bytes against the signed quants; 8 sum qs, the block's "row sum",
// is computed once per activation block for all N rows), d_a d_w is exact in
// f32 (two 11-bit significands), and |sum| <= 32 * 8 * 127 is exact too, so a
// block adds to its row's sum with one rounding.  A row whose total comes out
// infinite or NaN (a non-finite scale) is recomputed element by element from
// A' and W, as the definition does it.

// One block (index bi of 8 in the unit): quant words q (elements j and
// j + 16 in byte j of the 16), the weight scale dw, the unit's quantized
// activations au.
template <int M>
__device__ __forceinline__ void block_dot_q8(const uint8_t* au, int bi, const uint32_t q[4], float dw,
                                             float (&acc)[4 * M]) {
    uint32_t lo[4], hi[4];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        lo[w] = q[w] & 0x0F0F0F0Fu;         // elements 4w .. 4w+3
        hi[w] = (q[w] >> 4) & 0x0F0F0F0Fu;  // elements 16+4w .. 16+4w+3
    }
    const float* dq = reinterpret_cast<const float*>(au + M * kUnitElems);
    const int* sq = reinterpret_cast<const int*>(au + M * kUnitElems + M * 32);
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const int4* qa = reinterpret_cast<const int4*>(au + m * kUnitElems + bi * 32);
        const int4 a0 = qa[0], a1 = qa[1];
        int s = __dp4a(static_cast<int>(lo[0]), a0.x, 0);
        s = __dp4a(static_cast<int>(lo[1]), a0.y, s);
        s = __dp4a(static_cast<int>(lo[2]), a0.z, s);
        s = __dp4a(static_cast<int>(lo[3]), a0.w, s);
        s = __dp4a(static_cast<int>(hi[0]), a1.x, s);
        s = __dp4a(static_cast<int>(hi[1]), a1.y, s);
        s = __dp4a(static_cast<int>(hi[2]), a1.z, s);
        s = __dp4a(static_cast<int>(hi[3]), a1.w, s);
        // Independent sums per row: four for M <= 2, two above (registers).
        float& a = acc[4 * m + (M <= 2 ? (bi & 3) : (bi & 1))];
        a = fmaf(dw * dq[m * 8 + bi], static_cast<float>(s - sq[m * 8 + bi]), a);
    }
}

// Half h of a unit (blocks 4h .. 4h + 3) of this lane's row, 72 bytes
// realigned as for the packed consumer, against the unit's quantized
// activations au.
template <int M>
__device__ __forceinline__ void half_dot_q8(const uint8_t* row, int h, const uint8_t* au, float (&acc)[4 * M]) {
    uint32_t w[18];
    if (h == 0) {  // bytes 0 .. 71: 16-byte loads first
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 v = reinterpret_cast<const uint4*>(row)[i];
            w[4 * i + 0] = v.x;
            w[4 * i + 1] = v.y;
            w[4 * i + 2] = v.z;
            w[4 * i + 3] = v.w;
        }
        const uint2 v = *reinterpret_cast<const uint2*>(row + 64);
        w[16] = v.x;
        w[17] = v.y;
    } else {  // bytes 72 .. 143: 16-byte loads from byte 80
        const uint2 v = *reinterpret_cast<const uint2*>(row + 72);
        w[0] = v.x;
        w[1] = v.y;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 u = reinterpret_cast<const uint4*>(row + 80)[i];
            w[2 + 4 * i + 0] = u.x;
            w[2 + 4 * i + 1] = u.y;
            w[2 + 4 * i + 2] = u.z;
            w[2 + 4 * i + 3] = u.w;
        }
    }
#pragma unroll
    for (int pp = 0; pp < 2; ++pp) {
        const uint32_t* Wp = w + 9 * pp;
        const uint32_t qa[4] = {__byte_perm(Wp[0], Wp[1], 0x5432u), __byte_perm(Wp[1], Wp[2], 0x5432u),
                                __byte_perm(Wp[2], Wp[3], 0x5432u), __byte_perm(Wp[3], Wp[4], 0x5432u)};
        block_dot_q8<M>(au, 4 * h + 2 * pp, qa, f16_bits_to_float(Wp[0] & 0xFFFFu), acc);
        const uint32_t qb[4] = {Wp[5], Wp[6], Wp[7], Wp[8]};
        block_dot_q8<M>(au, 4 * h + 2 * pp + 1, qb, f16_bits_to_float(Wp[4] >> 16), acc);
    }
}

// Exact row sum over nblocks blocks from the quantized activations of the
// CTA's units (frag: unit j at frag + j M KB), element by element: A'_k =
// qs_k d_a exactly in f32, then the product with (q - 8) d_w, as the
// definition does it (a non-finite scale times a zero weight gives NaN).
template <int M>
__device__ __noinline__ float row_range_exact_q8(const uint8_t* row_blocks, int nblocks, const uint8_t* frag,
                                                 int m) {
    float s = 0.f;
    for (int b = 0; b < nblocks; ++b) {
        const uint8_t* au = frag + (b >> 3) * (M * 1024);
        const int bi = b & 7;
        const float da = reinterpret_cast<const float*>(au + M * kUnitElems)[m * 8 + bi];
        const int8_t* qs = reinterpret_cast<const int8_t*>(au + m * kUnitElems + bi * 32);
        const uint8_t* blk = row_blocks + kBlockBytes * b;
        const float d = f16_bits_to_float(static_cast<uint32_t>(blk[0]) | (static_cast<uint32_t>(blk[1]) << 8));
        for (int j = 0; j < kBlockElems; ++j) {
            const uint32_t byte = blk[2 + (j & 15)];
            const uint32_t nib = (j < 16) ? (byte & 0xFu) : (byte >> 4);
            s = fmaf(static_cast<float>(qs[j]) * da, magic_minus8(nib | kMagicBits) * d, s);
        }
    }
    return s;
}

template <int M, bool kPk, bool kQ8 = false>
__global__ void __launch_bounds__(max_threads(kPk, M, kQ8), 1)
    gemv_q4_0_tc(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap amap,
                 const float* __restrict__ A, float* __restrict__ C, const TcPlan p) {
    constexpr int kRows = group_rows(kPk);
    constexpr int kSlot = slot_floats(kPk);
    const int W = p.rps * p.c * p.hs;
    extern __shared__ __align__(128) uint8_t smem[];
    // ring [stages][c boxes][kRows rps rows][144 B] | activations [nu_max][M KB]
    // (B fragments for the MMA consumer, f32 for the packed one) | partial-sum
    // slots [2][W][kRows][8] f32 | the CTA's split partial sums [rbpc][rps]
    // [M][kRows] f32 (cluster split only) | full[stages] | empty[stages] |
    // a_bar | red_bar[2] (cluster split: partial sums written, partial sums
    // read)
    const int box_bytes = p.rps * kRows * kUnitBytes;
    const int stage_bytes = p.c * box_bytes;
    uint8_t* ring = smem;
    uint8_t* frag = smem + p.stages * stage_bytes;
    float* slots = reinterpret_cast<float*>(frag + p.nu_max * M * 1024);
    float* cpart = slots + 2 * W * kSlot;
    uint64_t* full = reinterpret_cast<uint64_t*>(cpart + (p.cl ? p.rbpc * p.rps * M * kRows : 0));
    uint64_t* empty = full + p.stages;
    uint64_t* a_bar = empty + p.stages;
    uint64_t* red_bar = a_bar + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = static_cast<int>(blockIdx.x) % p.S;
    const int u0 = static_cast<int>(static_cast<int64_t>(split) * p.U / p.S);
    const int nu = static_cast<int>(static_cast<int64_t>(split + 1) * p.U / p.S) - u0;
    const int RB = (p.RG + p.rps - 1) / p.rps;
    const int rb0 = (static_cast<int>(blockIdx.x) / p.S) * p.rbpc;
    const int nrb = max(0, min(p.rbpc, RB - rb0));
    const int spr = (nu + p.c - 1) / p.c;  // stages per row block
    const int nst = nrb * spr;

    grid_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], W);  // every consumer warp, once per stage
        }
        mbar_init(a_bar, 1);
        mbar_init(&red_bar[0], p.S);  // one arrival per CTA of the cluster
        mbar_init(&red_bar[1], p.S);
        fence_barrier_init();
    }
    __syncthreads();
    // Cluster launches: every CTA's barriers are initialised before any CTA
    // can arrive on them remotely.
    if (p.cl) cluster_sync_all();

    if (warp == W) {
        if (lane == 0 && nst > 0) {
            prefetch_tensormap(&wmap);
            prefetch_tensormap(&amap);
            const int rows_per_block = p.rps * kRows;
            // Warm L2 with the first stage before waiting on earlier kernels;
            // more would compete with their last reads and with the
            // activations, which can only be read after the wait.
            const int warm = 1;
            {
                int sc = 0, row = rb0 * rows_per_block;
                for (int s = 0; s < warm; ++s) {
                    for (int ul = 0; ul < p.c; ++ul) {
                        const int j = sc * p.c + ul;
                        if (j < nu) tma_prefetch_l2_3d(&wmap, 0, u0 + j, row);
                    }
                    if (++sc == spr) {
                        sc = 0;
                        row += rows_per_block;
                    }
                }
            }
            grid_dependency_wait();
            // The CTA's activations: one [M][256] f32 box per unit.
            mbar_arrive_expect_tx(a_bar, static_cast<uint32_t>(nu) * M * 1024);
            for (int j = 0; j < nu; ++j)
                tma_load_2d(frag + j * M * 1024, &amap, (u0 + j) * kUnitElems, 0, a_bar);
            int sc = 0, row = rb0 * rows_per_block, st = 0;
            uint32_t phase = 0;
            for (int s = 0; s < nst; ++s) {
                if (s >= p.stages && !mbar_wait_bounded(&empty[st], phase ^ 1u, &g_gemv_tc_error))
                    break;
                const int nbox = min(p.c, nu - sc * p.c);
                mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(nbox * box_bytes));
                for (int ul = 0; ul < nbox; ++ul)
                    tma_load_3d(ring + st * stage_bytes + ul * box_bytes, &wmap, 0,
                                u0 + sc * p.c + ul, row, &full[st]);
                if (++sc == spr) {
                    sc = 0;
                    row += rows_per_block;
                }
                if (++st == p.stages) {
                    st = 0;
                    phase ^= 1u;
                }
            }
        }
        return;
    }

    grid_dependency_wait();
    if (nst == 0) return;  // no consumer of this CTA reaches a barrier
    bool ok = mbar_wait_bounded(a_bar, 0, &g_gemv_tc_error);
    if constexpr (!kPk) {
        if (ok) {
            for (int j = warp; j < nu; j += W) build_fragments<M>(frag + j * M * 1024, lane);
        }
    } else if constexpr (kQ8) {
        if (ok) {
            for (int j = warp; j < nu; j += W) quantize_unit_q8<M>(frag + j * M * 1024, lane);
        }
    }
    named_barrier_sync(1, W * 32);

    const int g = lane >> 2;
    const int t = lane & 3;
    const int gc = g % frag_cols<M>();
    // Warp (ul * rps + rgl) * hs + h takes half h of its tile when hs = 2.
    const int h = warp % p.hs;
    const int rgl = (warp / p.hs) % p.rps;  // row group within the row block
    const int ul = warp / (p.hs * p.rps);   // unit column within a stage
    const uint32_t xoff = (t < 3) ? 4u + 4u * t : 0u;
    const uint32_t sel = (t < 3) ? 0x3210u : 0x5432u;
    const uint2* F = reinterpret_cast<const uint2*>(frag);
    // MMA consumer: rows g and g + 8 of the 16-row tile; packed consumer: row lane.
    const uint8_t* tile0 =
        ring + ul * box_bytes + (rgl * kRows + (kPk ? lane : g)) * kUnitBytes;
    constexpr int kAcc = 4 * (kPk ? M : 1);
    float acc[kAcc];
#pragma unroll
    for (int i = 0; i < kAcc; ++i) acc[i] = 0.f;
    int st = 0;
    uint32_t phase = 0;

    for (int rbi = 0; rbi < nrb; ++rbi) {
        for (int sc = 0; sc < spr; ++sc) {
            const int j = sc * p.c + ul;  // unit within the CTA's K range
            if (ok) ok = mbar_wait_bounded(&full[st], phase, &g_gemv_tc_error);
            if (ok && j < nu) {
                const uint8_t* r0 = tile0 + st * stage_bytes;
                const float* aj = reinterpret_cast<const float*>(frag + j * M * 1024);
                const uint2* Fj = F + j * (M * 128);
                if constexpr (kQ8) {
                    // (The planner gives the lane-per-row consumers half units: hs = 2.)
                    half_dot_q8<M>(r0, h, frag + j * M * 1024, acc);
                } else if constexpr (kPk) {
                    if (p.hs == 1) unit_dot_pk<M>(r0, aj, acc);
                    else half_dot_pk<M>(r0, h, aj, acc);
                } else {
                    pairs_mma<M, 4>(r0, r0 + 8 * kUnitBytes, Fj, 0, gc, t, xoff, sel, acc);  // hs = 1
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
            if (++st == p.stages) {
                st = 0;
                phase ^= 1u;
            }
        }

        // Row block done: partial sums to shared memory; the warp of unit
        // column 0 (half 0) adds its row group's c * hs slots (column order)
        // and takes one row per lane.  Slots alternate between row blocks, so
        // one barrier per row block keeps a slot from being rewritten before
        // it is read.
        float* slot = slots + ((rbi & 1) * W + warp) * kSlot;
        if constexpr (kPk) {
#pragma unroll
            for (int m = 0; m < M; ++m)
                slot[lane * 8 + m] = (acc[4 * m] + acc[4 * m + 1]) + (acc[4 * m + 2] + acc[4 * m + 3]);
        } else {
            reinterpret_cast<float2*>(slot)[g * 4 + t] = make_float2(acc[0], acc[1]);
            reinterpret_cast<float2*>(slot)[(g + 8) * 4 + t] = make_float2(acc[2], acc[3]);
        }
#pragma unroll
        for (int i = 0; i < kAcc; ++i) acc[i] = 0.f;
        if (W > p.rps) {
            named_barrier_sync(1, W * 32);
        } else {
            __syncwarp();
        }
        if (ul != 0 || h != 0) continue;
        const int rg = (rb0 + rbi) * p.rps + rgl;
        const int r = lane & (kRows - 1);
        const int row = rg * kRows + r;
        float tot[M];
#pragma unroll
        for (int m = 0; m < M; ++m) tot[m] = 0.f;
        for (int u = 0; u < p.c; ++u) {
            for (int hh = 0; hh < p.hs; ++hh) {
                const float* su =
                    slots + ((rbi & 1) * W + (u * p.rps + rgl) * p.hs + hh) * kSlot + r * 8;
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    tot[m] += su[m];
                    if constexpr (!kPk && tc_sets<M>() == 1) tot[m] += su[M + m];
                }
            }
        }
        if (rg >= p.RG) continue;  // whole warp: a row group past the matrix
        const bool mine = lane < kRows && row < p.N;
        if (mine) {
            const uint8_t* row_blocks =
                p.wq + (static_cast<int64_t>(row) * p.U + u0) * kUnitBytes;
#pragma unroll
            for (int m = 0; m < M; ++m) {
                if (!isfinite(tot[m])) {
                    if constexpr (kQ8)
                        tot[m] = row_range_exact_q8<M>(row_blocks, nu * 8, frag, m);
                    else
                        tot[m] = row_range_exact(row_blocks, nu * 8,
                                                 A + m * p.K + static_cast<int64_t>(u0) * kUnitElems);
                }
            }
        }
        if (p.S == 1) {
            if (mine) {
#pragma unroll
                for (int m = 0; m < M; ++m) C[static_cast<int64_t>(m) * p.N + row] = tot[m];
            }
        } else if (lane < kRows) {
            float* part = p.cl ? cpart + (rbi * p.rps + rgl) * (M * kRows)
                               : p.part + (static_cast<int64_t>(rg) * p.S + split) * (M * kRows);
#pragma unroll
            for (int m = 0; m < M; ++m) part[m * kRows + lane] = tot[m];
        }
    }
    if (p.S == 1) return;
    if (p.cl) {
        // Split K through the cluster (ranks in range order).  Every consumer
        // warp comes here, whatever its waits returned, so the arrivals come
        // on every path.  Row group i of the CTA's row blocks (i = rbi * rps +
        // rgl) is added up by rank i % S, one warp per row group, over the S
        // CTAs' partial sums in rank order.
        asm volatile("fence.acq_rel.cluster;" ::: "memory");
        named_barrier_sync(1, W * 32);
        if (threadIdx.x == 0) {
            for (int r = 0; r < p.S; ++r)
                mbar_arrive_cluster(mapa_shared(smem_addr(&red_bar[0]), static_cast<uint32_t>(r)));
        }
        const uint32_t rank = cluster_ctarank();
        if (mbar_wait_cluster_bounded(&red_bar[0], 0, &g_gemv_tc_error)) {
            const uint32_t cbase = smem_addr(cpart);
            for (int i = static_cast<int>(rank) + p.S * warp; i < nrb * p.rps; i += p.S * W) {
                const int rg = rb0 * p.rps + i;
                const int row = rg * kRows + lane;
                if (rg >= p.RG || lane >= kRows || row >= p.N) continue;
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    const uint32_t off = static_cast<uint32_t>(((i * M + m) * kRows + lane) * 4);
                    float v = 0.f;
                    for (int r = 0; r < p.S; ++r) v += ld_dsmem_f32(mapa_shared(cbase + off, static_cast<uint32_t>(r)));
                    C[static_cast<int64_t>(m) * p.N + row] = v;
                }
            }
        }
        // No CTA leaves while another may still read its partial sums.
        named_barrier_sync(1, W * 32);
        if (threadIdx.x == 0) {
            for (int r = 0; r < p.S; ++r)
                mbar_arrive_cluster(mapa_shared(smem_addr(&red_bar[1]), static_cast<uint32_t>(r)));
        }
        mbar_wait_cluster_bounded(&red_bar[1], 0, &g_gemv_tc_error);
        return;
    }
    if (ul != 0 || h != 0) return;

    // Split K: one fence for all of this warp's partial sums, then its
    // arrivals; the last of the S arrivals at a row group adds the partials
    // in range order.  (Fencing once here rather than after every row block
    // keeps the fence's wait out of the streaming loop.)
    __threadfence();
    __syncwarp();
    for (int rbi = 0; rbi < nrb; ++rbi) {
        const int rg = (rb0 + rbi) * p.rps + rgl;
        if (rg >= p.RG) break;
        unsigned old = 0;
        if (lane == 0) old = atomicAdd(&p.ctr[rg], 1u);
        old = __shfl_sync(0xFFFFFFFFu, old, 0);
        if (old != static_cast<unsigned>(p.S - 1)) continue;
        __threadfence();
        const int row = rg * kRows + lane;
        if (lane < kRows && row < p.N) {
            const float* base = p.part + static_cast<int64_t>(rg) * p.S * (M * kRows);
#pragma unroll
            for (int m = 0; m < M; ++m) {
                float v = 0.f;
                for (int q = 0; q < p.S; ++q)
                    v += __ldcg(base + q * (M * kRows) + m * kRows + lane);
                C[static_cast<int64_t>(m) * p.N + row] = v;
            }
        }
        __syncwarp();
        if (lane == 0) atomicExch(&p.ctr[rg], 0u);
    }
}

// Shared memory of one CTA: W consumer warps, stages of `tiles` tiles,
// cpart floats of split partial sums (cluster split).
int64_t tc_smem_bytes(int M, bool packed, int W, int tiles, int stages, int nu_max, int64_t cpart) {
    return static_cast<int64_t>(stages) * tiles * group_rows(packed) * kUnitBytes +
           static_cast<int64_t>(nu_max) * M * 1024 + 2LL * W * slot_floats(packed) * 4 + cpart * 4 +
           (2LL * stages + 3) * 8;
}

// Largest cluster split's partial sums in one CTA (floats): keeps the ring
// deep where a split is worth taking.
constexpr int64_t kMaxClusterPartFloats = 8192;

// Relative rate of one SM with W consumer warps (more warps hide more of the
// shared-memory, barrier and arithmetic latency; past 16 measured no gain).
double warp_efficiency(int W) {
    return W >= 16 ? 1.0 : W >= 14 ? 0.96 : W >= 12 ? 0.92 : W >= 10 ? 0.86 : 0.8;
}

// Best stage shape with hs warps a tile (rps row groups x c units, W = rps c
// hs consumer warps) and S (K ranges) for one CTA per SM.  The K ranges add
// up through a cluster when `fit` is given (S = 2, 4 or 8; fit[0..2] clusters
// of 2, 4 and 8 CTAs can be resident at once, and the split's clusters must
// all be), otherwise through the scratch `ws`.  The cost is the
// largest per-CTA tile count (idle tile slots included) over the warp
// efficiency, with charges for split-K partial sums (their bytes against the
// weight bytes, plus a little per split), for short K ranges (a CTA that reads
// few bytes of each row leaves DRAM pages to be reopened by others), for a
// shallow ring, and for cross-warp reductions at more than one row block per
// CTA.  Returns the cost (infinite when nothing fits).
double plan_tc_hs(int M, bool packed, bool q8, int hs, int64_t N, int64_t K, const DeviceInfo& dev,
                  const Workspace* ws, const int* fit, TcPlan* out, int* grid, int* smem) {
    const int kRows = group_rows(packed);
    const int U = static_cast<int>(K / kUnitElems);
    const int64_t RG = (N + kRows - 1) / kRows;
    const int P = dev.sm_count;
    double best = 1e300;
    for (int W = std::min(max_warps(packed, M, q8), 16 * hs); W >= 8; --W) {
        if (W % hs != 0) continue;
        const int tiles = W / hs;
        for (int c = 1; c <= tiles; ++c) {
            if (tiles % c != 0) continue;
            const int rps = tiles / c;
            if (rps * kRows > 256) continue;  // TMA box height
            const int64_t RB = (RG + rps - 1) / rps;
            for (int S = 1; S <= kMaxSplits && S <= U; ++S) {
                const bool cl = S > 1 && fit != nullptr;
                int64_t Gs = std::max(1, P / S);
                if (cl) {
                    if (S != 2 && S != 4 && S != 8) continue;
                    Gs = std::min<int64_t>(Gs, fit[S == 2 ? 0 : S == 4 ? 1 : 2]);
                    if (Gs < 1) continue;
                } else if (S > 1 && (!ws || RG * S * M * kRows > static_cast<int64_t>(ws->part_floats) ||
                                     RG > static_cast<int64_t>(ws->ctr_count))) {
                    continue;
                }
                const int nu_max = (U + S - 1) / S;
                const int64_t rbpc = (RB + Gs - 1) / Gs;
                const int64_t g_used = (RB + rbpc - 1) / rbpc;
                const int64_t spr = (nu_max + c - 1) / c;
                const int64_t cpart = cl ? rbpc * rps * M * kRows : 0;
                if (cpart > kMaxClusterPartFloats) continue;
                const int64_t fixed = tc_smem_bytes(M, packed, W, tiles, 0, nu_max, cpart);
                int stages = static_cast<int>(
                    (dev.max_smem_optin - fixed) /
                    (static_cast<int64_t>(tiles) * kRows * kUnitBytes + 16));
                stages = std::min(stages, kMaxStages);
                if (stages < 2) continue;
                const double split_bytes =
                    (S > 1) ? 8.0 * M * S / (kBlockBytes * static_cast<double>(K) / kBlockElems)
                            : 0.0;
                const double short_rows =
                    0.3 * std::max(0.0, 1.0 - nu_max * static_cast<double>(kUnitBytes) / 2048.0);
                const double cost = static_cast<double>(rbpc * spr * tiles) / warp_efficiency(W) *
                                    (1.0 + split_bytes + 0.01 * (S - 1) + short_rows) *
                                    (stages < 3 ? 1.1 : 1.0) *
                                    ((W > rps && rbpc > 1) ? 1.0 + 0.05 * rbpc : 1.0);
                if (cost < best) {
                    best = cost;
                    TcPlan& q = *out;
                    q.wq = nullptr;
                    q.N = static_cast<int>(N);
                    q.K = K;
                    q.U = U;
                    q.RG = static_cast<int>(RG);
                    q.S = S;
                    q.rps = rps;
                    q.c = c;
                    q.hs = hs;
                    q.rbpc = static_cast<int>(rbpc);
                    q.nu_max = nu_max;
                    q.stages = stages;
                    q.cl = cl ? 1 : 0;
                    q.part = (S > 1 && !cl) ? ws->part : nullptr;
                    q.ctr = (S > 1 && !cl) ? ws->ctr : nullptr;
                    *grid = static_cast<int>(g_used * S);
                    *smem = static_cast<int>(tc_smem_bytes(M, packed, W, tiles, stages, nu_max, cpart));
                }
            }
        }
    }
    return best;
}

// The launch plan: whole-unit tiles for the MMA consumer, half-unit warps
// for the packed one (measured on GB300: half units lose with the MMA
// consumer, and give the packed one twice the warps on the same stages).
bool plan_tc(int M, bool packed, int64_t N, int64_t K, const DeviceInfo& dev, const Workspace* ws,
             const int* fit, TcPlan* out, int* grid, int* smem, bool q8 = false) {
    return plan_tc_hs(M, packed, q8, packed ? 2 : 1, N, K, dev, ws, fit, out, grid, smem) < 1e300;
}

template <int M, bool kPk, bool kQ8 = false>
cudaError_t ensure_tc_smem_attr(const DeviceInfo& dev, int bytes) {
    static int configured[64] = {0};
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    if (bytes > dev.max_smem_optin) return cudaErrorInvalidValue;
    if (__atomic_load_n(&configured[dev.device], __ATOMIC_ACQUIRE)) return cudaSuccess;
    cudaError_t err = cudaFuncSetAttribute(gemv_q4_0_tc<M, kPk, kQ8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           dev.max_smem_optin);
    if (err != cudaSuccess) return err;
    __atomic_store_n(&configured[dev.device], 1, __ATOMIC_RELEASE);
    return cudaSuccess;
}

// Resident clusters of 2, 4 and 8 CTAs of one kernel (one CTA per SM: the
// count depends on how the SMs group, not on the launch's shared memory),
// queried once per device.
template <int M, bool kPk, bool kQ8 = false>
cudaError_t cluster_fits(const DeviceInfo& dev, int fit[3]) {
    static int cached[64][3] = {};  // 0: not queried; else 1 + the count
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    for (int i = 0; i < 3; ++i) {
        int f = __atomic_load_n(&cached[dev.device][i], __ATOMIC_ACQUIRE);
        if (f == 0) {
            f = 1 + max_active_clusters(gemv_q4_0_tc<M, kPk, kQ8>, dim3(max_threads(kPk, M, kQ8)),
                                        static_cast<size_t>(dev.max_smem_optin), 2u << i);
            __atomic_store_n(&cached[dev.device][i], f, __ATOMIC_RELEASE);
        }
        fit[i] = f - 1;
    }
    return cudaSuccess;
}

template <int M, bool kPk, bool kQ8 = false>
cudaError_t launch_tc(const float* A, const uint8_t* wq, float* C, int64_t N, int64_t K,
                      cudaStream_t stream, const DeviceInfo& dev, const Workspace* ws,
                      bool clear_counters, bool* launched) {
    *launched = false;
    cudaError_t err = ensure_tc_smem_attr<M, kPk, kQ8>(dev, dev.max_smem_optin);
    if (err != cudaSuccess) return err;
    int fit[3] = {0, 0, 0};
    if (!ws) {
        err = cluster_fits<M, kPk, kQ8>(dev, fit);
        if (err != cudaSuccess) return err;
    }
    TcPlan p;
    int grid = 0, smem = 0;
    if (!plan_tc(M, kPk, N, K, dev, ws, ws ? nullptr : fit, &p, &grid, &smem, kQ8)) return cudaSuccess;
    p.wq = wq;
    if (clear_counters && p.S > 1 && !p.cl) {
        err = cudaMemsetAsync(p.ctr, 0, static_cast<size_t>(p.RG) * sizeof(unsigned), stream);
        if (err != cudaSuccess) return err;
    }
    // Weights as bytes [N rows][U units][144 B]; boxes of (group rows) rps rows x 1 unit.
    const int64_t dims[3] = {kUnitBytes, p.U, N};
    const int64_t strides[2] = {kUnitBytes, static_cast<int64_t>(p.U) * kUnitBytes};
    const int box[3] = {kUnitBytes, 1, p.rps * group_rows(kPk)};
    CUtensorMap wmap, amap;
    err = encode_tiled(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, 3, dims, strides, box);
    if (err != cudaSuccess) return err;
    // Activations as f32 [M][K]; boxes of M rows x 256 k.
    const int64_t adims[2] = {K, M};
    const int64_t astrides[1] = {K * 4};
    const int abox[2] = {kUnitElems, M};
    err = encode_tiled(&amap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, A, 2, adims, astrides, abox);
    if (err != cudaSuccess) return err;
    const dim3 block((p.rps * p.c * p.hs + 1) * 32);
    if (p.cl) {
        err = launch_pdl_cluster(gemv_q4_0_tc<M, kPk, kQ8>, dim3(grid), block, smem, stream,
                                 static_cast<unsigned>(p.S), wmap, amap, A, C, p);
    } else {
        err = launch_pdl(gemv_q4_0_tc<M, kPk, kQ8>, dim3(grid), block, smem, stream, wmap, amap, A, C, p);
    }
    if (err != cudaSuccess) return err;
    note_launch();
    *launched = true;
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemv_q4_0_tc(const float* A, const uint8_t* wq, float* C, int M, int64_t N,
                                int64_t K, cudaStream_t stream, const DeviceInfo& dev,
                                const Workspace* ws, bool packed, bool clear_counters,
                                bool* launched) {
    if (packed) {
        switch (M) {
            case 1: return launch_tc<1, true>(A, wq, C, N, K, stream, dev, ws, clear_counters, launched);
            case 2: return launch_tc<2, true>(A, wq, C, N, K, stream, dev, ws, clear_counters, launched);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (M) {
        case 1: return launch_tc<1, false>(A, wq, C, N, K, stream, dev, ws, clear_counters, launched);
        case 2: return launch_tc<2, false>(A, wq, C, N, K, stream, dev, ws, clear_counters, launched);
        case 3: return launch_tc<3, false>(A, wq, C, N, K, stream, dev, ws, clear_counters, launched);
        case 4: return launch_tc<4, false>(A, wq, C, N, K, stream, dev, ws, clear_counters, launched);
        case 5: return launch_tc<5, false>(A, wq, C, N, K, stream, dev, ws, clear_counters, launched);
        case 6: return launch_tc<6, false>(A, wq, C, N, K, stream, dev, ws, clear_counters, launched);
        case 7: return launch_tc<7, false>(A, wq, C, N, K, stream, dev, ws, clear_counters, launched);
        case 8: return launch_tc<8, false>(A, wq, C, N, K, stream, dev, ws, clear_counters, launched);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gemv_q4_0_q8act_tc(const float* A, const uint8_t* wq, float* C, int M, int64_t N,
                                      int64_t K, cudaStream_t stream, const DeviceInfo& dev, bool* launched) {
    switch (M) {
        case 1: return launch_tc<1, true, true>(A, wq, C, N, K, stream, dev, nullptr, false, launched);
        case 2: return launch_tc<2, true, true>(A, wq, C, N, K, stream, dev, nullptr, false, launched);
        case 3: return launch_tc<3, true, true>(A, wq, C, N, K, stream, dev, nullptr, false, launched);
        case 4: return launch_tc<4, true, true>(A, wq, C, N, K, stream, dev, nullptr, false, launched);
        case 5: return launch_tc<5, true, true>(A, wq, C, N, K, stream, dev, nullptr, false, launched);
        case 6: return launch_tc<6, true, true>(A, wq, C, N, K, stream, dev, nullptr, false, launched);
        case 7: return launch_tc<7, true, true>(A, wq, C, N, K, stream, dev, nullptr, false, launched);
        case 8: return launch_tc<8, true, true>(A, wq, C, N, K, stream, dev, nullptr, false, launched);
        default: return cudaErrorInvalidValue;
    }
}

bool gemv_tc_plan_query(int M, bool packed, int64_t N, int64_t K, int sm_count, int smem_optin,
                        const int* fit, int64_t part_floats, int64_t ctr_count, int64_t out[13]) {
    DeviceInfo dev;
    dev.device = 0;
    dev.sm_count = sm_count;
    dev.max_smem_optin = smem_optin;
    Workspace ws;
    ws.part_floats = static_cast<size_t>(part_floats);
    ws.ctr_count = static_cast<int>(std::min<int64_t>(ctr_count, 0x7FFFFFFF));
    TcPlan p;
    int grid = 0, smem = 0;
    if (!plan_tc(M, packed, N, K, dev, fit ? nullptr : &ws, fit, &p, &grid, &smem)) return false;
    const int64_t v[13] = {p.RG, p.U, p.S, p.rps, p.c, p.hs, p.rbpc, p.nu_max, p.stages, grid, smem,
                           static_cast<int64_t>(p.rps) * p.c * p.hs, p.cl};
    for (int i = 0; i < 13; ++i) out[i] = v[i];
    return true;
}

cudaError_t gemv_tc_read_device_error(unsigned int* bits, bool clear) {
    unsigned int v = 0;
    cudaError_t err = cudaMemcpyFromSymbol(&v, g_gemv_tc_error, sizeof(v));
    if (err != cudaSuccess) return err;
    *bits |= v;
    if (clear && v != 0) {
        const unsigned int zero = 0;
        err = cudaMemcpyToSymbol(g_gemv_tc_error, &zero, sizeof(zero));
    }
    return err;
}

}  // namespace qm

// Decode-regime GEMV over a list of problems in one persistent launch:
// C_p = A_p x dequant(W_p)^T for p = 0 .. count-1, one activation row (M = 1)
// against each Q4_0 weight stream (sections "qmatvec_q4_0" and
// "matmul_q4_0_tiled" of "fuel-vulkan-kernels — quantized (GGML) kernel
// contracts": element j < 16 of a block is the low nibble of quant byte j,
// element j + 16 its high nibble, value (nibble - 8) * d; the GEMV's cost is
// streaming the weight blocks once).
//
// Why one launch: a decode step is a chain of GEMVs of a few to a few tens of
// megabytes each.  Launched one by one, every GEMV pays a fixed price (waiting
// for the previous grid, loading its activations, filling its first stage)
// that is as long as streaming several megabytes.  Here one CTA per SM walks
// all problems in order and streams every weight byte through one ring of
// shared-memory stages, so the weights of the next problem are in flight
// while the current one finishes.  A problem may have to wait for earlier
// ones (its activations are their outputs): each CTA counts its finished
// problems into a global counter, and a problem's activations are loaded only
// once every CTA has finished every problem up to the one it waits for.  The
// weight stream does not wait: the ring keeps filling meanwhile.
//
// Work.  A tile is 16 weight rows over the whole K.  The tiles of problem p
// are dealt round robin over the G CTAs, starting at a rotating offset
// (the tiles of all earlier problems), so every CTA streams about the same
// bytes over the list.  A CTA's tiles of a problem form a sequence of units
// (a unit is 16 rows x 256 k: 8 blocks, 144 bytes of each row); a stage holds
// 16 consecutive units of that sequence (stages never span problems), one
// per consumer warp.  The producer copies a stage as one or two TMA boxes of
// 16 rows x c units (c = 16, or 8 when K/256 is not a multiple of 16), each
// box one copy operation: the copy engine's cost grows with the number of
// copies, and one box per 16 units streams far faster than a copy per row.
// The box spans c + 1 units of a 4-D view of the weights ([N rows][K/256c
// groups][c units][144 B]); the extra unit lies outside its group and lands
// as zeros, which spaces the rows (c + 1) * 144 bytes apart in shared memory:
// an odd number of 16-byte steps, which puts the 32 lanes' 4-byte loads on
// distinct banks.  Rows past N land as zeros too.
//
// Arithmetic (per unit, per warp): mma.sync m16n8k16, bf16 in, f32 out.
//   * A operand: 16 weight rows x 16 k of (q - 8), exact in bf16 (the nibble
//     under the exponent of 128 reads as 128 + q; subtracting 136 is exact).
//     Lane (g, t) owns rows g and g + 8 and one block of each "quad" of four
//     blocks (blocks t*2 + Q, Q = 0, 1: all four blocks of a quad have the
//     same parity, so they sit at the same alignment).
//   * B operand: activation pieces a = hi + lo + r, hi = bf16(a),
//     lo = bf16(a - hi), |r| <= 2^-17 |a|.  Column 2t' holds the hi pieces
//     and column 2t' + 1 the lo pieces of block t' of the quad, non-zero only
//     in the k rows of that block.  So the MMA result D[row][2t'] + D[row][2t'
//     + 1] is row's dot product with block t' alone: eight MMAs cover a quad
//     (32 elements of each of its 4 blocks), and each lane scales its own
//     block's result by that block's d in f32.  Every bf16 product is exact in
//     f32; one product misses a * W by the residual r alone.
//   * A row whose total comes out infinite or NaN is recomputed element by
//     element, as the definition does it (a non-finite d times q = 8 is NaN).
//
// Reduction.  A warp adds its units of a tile in registers, then its four
// lanes of a row group; its 16 row sums go to a shared-memory slot, and the
// last of the tile's warps to finish adds the slots in a fixed warp order and
// writes C.  No atomics touch any sum, so results do not depend on timing.
// A warp hands its stage back to the producer as soon as the unit's bytes are
// in registers, before any of this, so the reduction never holds up a copy.
//
// Launch and waits.  Programmatic dependent launch: before griddepcontrol.wait
// a CTA only initialises barriers and asks L2 for its first stage (a hint that
// cannot return stale data).  Every wait is bounded; a wait that gives up sets
// the device error word and the CTA stops issuing work, waits (bounded) for
// its copies in flight, and returns.
#include <algorithm>
#include <vector>

#include "qm_device.cuh"
#include "qm_internal.h"

namespace qm {

__device__ unsigned int g_gemv_list_error = 0;

namespace {

constexpr int kUnitB = 144;                      // bytes of one row's unit (8 blocks)
// A box of 16 rows x (c + 1) units (c = 16 or 8).
__host__ __device__ constexpr int box_bytes(int c) { return 16 * (c + 1) * kUnitB; }
constexpr int kLFragB = kListMaxK * 4;           // activations (f32 as loaded; M = 1)

constexpr int kLW = 16;                          // consumer warps
constexpr int kLThreads = (kLW + 2) * 32;        // + producer warp + activation-loader warp
// A stage holds 16 units (one per consumer warp) as 16 / c boxes.
constexpr int kStageB = 2 * box_bytes(8);        // 41,472 bytes (c = 8); c = 16 needs 39,168
constexpr int kLStages = 4;
constexpr int kTileSlots = 4;                    // tiles whose partial sums may be in flight
constexpr int kSlotFloats = kLW * 16;            // one tile: 16 warps x 16 rows

// Shared memory: ring | activations | partial-sum slots | barriers and
// counters | 1 KB of zeros.  (24 consumer warps, which
// fit in 72 registers each, on 2 stages of 24 units measured slower: 0.435
// against 0.50 of HBM over the 32-layer sweep; 3 stages ran 4% slower than 4.)
constexpr int kOffFrag = kLStages * kStageB;
constexpr int kOffSlots = kOffFrag + kLFragB;
constexpr int kOffBars = kOffSlots + kTileSlots * kSlotFloats * 4;
// full, empty; a_full, a_empty (activations copied in by the loader); one
// barrier per pair of consumer warps (w, w + 8).
constexpr int kNumBars = 2 * kLStages + 2 + 8;
constexpr int kOffInts = kOffBars + kNumBars * 8;
constexpr int kNumInts = 2 * kTileSlots + kListMaxProblems + 1;  // arrivals, done, tiles per problem, abort
// 1 KB of zeros, 64 bytes past a 128-byte boundary: a lane that reads zeros
// and the lane of the same g that reads real fragments (1024-byte aligned)
// then hit different banks.
constexpr int kOffZero = (kOffInts + kNumInts * 4 + 127) / 128 * 128 + 64;
constexpr int kLSmem = kOffZero + 1024;
static_assert(kLSmem <= 232448, "shared memory of one CTA");
static_assert(kOffFrag % 1024 == 0 && kOffSlots % 16 == 0 && kOffBars % 8 == 0, "alignment");

// Polls of a global completion counter (each followed by a short sleep).
constexpr uint32_t kMaxCounterPolls = 1u << 21;

struct ListProblem {
    const float* A;
    const uint8_t* W;
    float* C;
    int N;
    int K;
    int wait_for;  // -1 or an earlier index of this launch (prefix: problems 0..wait_for)
    int arrive;    // 1: CTAs count their completion of this problem in ctr[p]
    int off;       // rotation of the round-robin tile deal
    int c;         // units per box (16 or 8)
};

// The weight tensor maps first (aligned as CUtensorMap requires), then the
// problems.
struct ListParams {
    CUtensorMap map[kListMaxProblems];
    ListProblem p[kListMaxProblems];
    int count;
    int grid;
    unsigned* ctr;
};

__device__ __forceinline__ uint32_t lds32(const uint8_t* p) { return *reinterpret_cast<const uint32_t*>(p); }

__device__ __forceinline__ void mma_bf16(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1, bool first) {
    if (first) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
            "{%8, %9}, {%10, %10, %10, %10};"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.f));
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
            "{%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

// (q - 8) as bf16 pairs from a quant word holding bytes (b0, b1, b2, b3), b0
// lowest: R0 = low nibbles of (b0, b2), R1 = high nibbles of (b0, b2), R2 =
// low nibbles of (b1, b3), R3 = high nibbles of (b1, b3), the first of each
// pair in the low half.
__device__ __forceinline__ void nib_bf16(uint32_t Q, uint32_t R[4]) {
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

// Quant byte indices of word position p (0..3) of a block of parity `odd`,
// in the order the consumer decodes them.  Even blocks: word 0 joins quant
// bytes 0, 1 (behind d) with 14, 15, then words 1..3 are bytes 2..13.  Odd
// blocks (quants 4-byte aligned): word 0 is bytes 12..15, words 1..3 bytes
// 0..11.
__device__ __forceinline__ int quant_byte(int odd, int p, int i) {
    if (odd) return p == 0 ? 12 + i : 4 * (p - 1) + i;
    return p == 0 ? (i < 2 ? i : 12 + i) : 4 * p - 2 + i;
}

// Rewrite one unit of activations (256 f32 as loaded) in place into its B
// fragments: 1 KB, entry (Q, p, g') of 16 bytes at ((Q * 4 + p) * 8 + g') * 16
// holds, for block 2 (g' / 2) + Q and piece g' % 2 (hi, lo), the fragment
// registers (b0, b1) of slabs 2p and 2p + 1.  Slab 2p pairs quant bytes (b0,
// b2) of word p (low nibbles in b0, high nibbles in b1), slab 2p + 1 bytes
// (b1, b3).  Pieces are formed two at a time (packed conversions; lo by one
// packed FMA x - hi, exact).
__device__ __forceinline__ void unit_fragments(uint8_t* unit, int lane) {
    const float* f = reinterpret_cast<const float*>(unit);
    float x[2][8];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int e = lane + 32 * j;
        const int Q = e >> 5, p = (e >> 3) & 3, gp = e & 7;
        const float* blk = f + 32 * (2 * (gp >> 1) + Q);
        const int c0 = quant_byte(Q, p, 0), c1 = quant_byte(Q, p, 1), c2 = quant_byte(Q, p, 2),
                  c3 = quant_byte(Q, p, 3);
        x[j][0] = blk[c0];
        x[j][1] = blk[c2];
        x[j][2] = blk[c0 + 16];
        x[j][3] = blk[c2 + 16];
        x[j][4] = blk[c1];
        x[j][5] = blk[c3];
        x[j][6] = blk[c1 + 16];
        x[j][7] = blk[c3 + 16];
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        const int e = lane + 32 * j;
        const bool lo_piece = (e & 1) != 0;
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const float2 v = make_float2(x[j][2 * h], x[j][2 * h + 1]);
            const __nv_bfloat162 hb = __floats2bfloat162_rn(v.x, v.y);
            uint32_t hw = *reinterpret_cast<const uint32_t*>(&hb);
            if (lo_piece) {
                const float2 rest = __ffma2_rn(make_float2(__uint_as_float(hw << 16), __uint_as_float(hw & 0xFFFF0000u)),
                                               make_float2(-1.0f, -1.0f), v);
                const __nv_bfloat162 lb = __floats2bfloat162_rn(rest.x, rest.y);
                hw = *reinterpret_cast<const uint32_t*>(&lb);
            }
            w[h] = hw;
        }
        reinterpret_cast<uint4*>(unit)[e] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// One unit of 16 rows: rows g and g + 8 of the stage (ra, rb point at this
// unit in those rows), the unit's fragments F; adds this lane's block sums to
// acc[0] (row g) and acc[1] (row g + 8).
// F is this lane's fragment base: the unit's fragments for the lanes that
// carry a non-zero B fragment ((g >> 1) == t), a kilobyte of zeros for the
// others, so that every lane loads the same way.
__device__ __forceinline__ void unit_mma(const uint8_t* ra, const uint8_t* rb, const uint8_t* F, int g, int t,
                                         float acc[2]) {
    uint32_t wa[2][4], wb[2][4];
    float da[2], db[2];
#pragma unroll
    for (int Q = 0; Q < 2; ++Q) {
        const uint8_t* a = ra + 36 * t + 16 * Q;
        const uint8_t* b = rb + 36 * t + 16 * Q;
        const uint32_t A0 = lds32(a), A1 = lds32(a + 4), A2 = lds32(a + 8), A3 = lds32(a + 12), A4 = lds32(a + 16);
        const uint32_t B0 = lds32(b), B1 = lds32(b + 4), B2 = lds32(b + 8), B3 = lds32(b + 12), B4 = lds32(b + 16);
        if (Q == 0) {  // even block at its start: d, then quant bytes 0, 1 | 2..13 | 14, 15
            wa[Q][0] = __byte_perm(A0, A4, 0x5432u);
            wb[Q][0] = __byte_perm(B0, B4, 0x5432u);
            da[Q] = f16_bits_to_float(A0 & 0xFFFFu);
            db[Q] = f16_bits_to_float(B0 & 0xFFFFu);
        } else {       // odd block, two bytes before its start: d in the high half, then 16 quant bytes
            wa[Q][0] = A4;
            wb[Q][0] = B4;
            da[Q] = f16_bits_to_float(A0 >> 16);
            db[Q] = f16_bits_to_float(B0 >> 16);
        }
        wa[Q][1] = A1; wa[Q][2] = A2; wa[Q][3] = A3;
        wb[Q][1] = B1; wb[Q][2] = B2; wb[Q][3] = B3;
    }
    // Four independent MMA chains (quad Q, words p = 0, 1 or 2, 3), so that
    // no chain is longer than four MMAs.
    float D[2][2][4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
#pragma unroll
        for (int Q = 0; Q < 2; ++Q) {
            uint32_t Ra[4], Rb[4];
            nib_bf16(wa[Q][p], Ra);
            nib_bf16(wb[Q][p], Rb);
            const uint4 Bf = *reinterpret_cast<const uint4*>(F + ((Q * 4 + p) * 8 + g) * 16);
            float* d = D[Q][p >> 1];
            mma_bf16(d, Ra[0], Rb[0], Ra[1], Rb[1], Bf.x, Bf.y, (p & 1) == 0);
            mma_bf16(d, Ra[2], Rb[2], Ra[3], Rb[3], Bf.z, Bf.w, false);
        }
    }
#pragma unroll
    for (int Q = 0; Q < 2; ++Q) {
        acc[0] = fmaf(da[Q], (D[Q][0][0] + D[Q][0][1]) + (D[Q][1][0] + D[Q][1][1]), acc[0]);
        acc[1] = fmaf(db[Q], (D[Q][0][2] + D[Q][0][3]) + (D[Q][1][2] + D[Q][1][3]), acc[1]);
    }
}

// ---- Integer consumer (the list of act-quant GEMVs: activations quantized to
// Q8_0 on chip; see gemv_tc.cu for the exact block factoring).  Lane l takes
// row l % 16 of the 16-row unit and half l / 16 of it (4 blocks, 72 bytes:
// four 16-byte loads and one 8-byte load; rows (c + 1) * 144 bytes apart put
// the 8 lanes of a quarter warp on distinct bank quads), and adds its blocks'
// exact integer dots, scaled once per block, into two sums.
__device__ __forceinline__ void half_unit_q8(const uint8_t* row, int h, const uint8_t* au, float acc[2]) {
    uint32_t w[18];
    if (h == 0) {  // bytes 0 .. 71
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
    } else {  // bytes 72 .. 143
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
    const float* dq = reinterpret_cast<const float*>(au + 256);
    const int* sq = reinterpret_cast<const int*>(au + 256 + 32);
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const uint32_t* Wp = w + 9 * (b >> 1);
        uint32_t q[4];
        float dw;
        if ((b & 1) == 0) {  // even block: d in the low half of word 0, quants at bytes 2..17
            q[0] = __byte_perm(Wp[0], Wp[1], 0x5432u);
            q[1] = __byte_perm(Wp[1], Wp[2], 0x5432u);
            q[2] = __byte_perm(Wp[2], Wp[3], 0x5432u);
            q[3] = __byte_perm(Wp[3], Wp[4], 0x5432u);
            dw = f16_bits_to_float(Wp[0] & 0xFFFFu);
        } else {             // odd block: d in the high half of word 4, quants in words 5..8
            q[0] = Wp[5];
            q[1] = Wp[6];
            q[2] = Wp[7];
            q[3] = Wp[8];
            dw = f16_bits_to_float(Wp[4] >> 16);
        }
        const int bi = 4 * h + b;
        const int4* qa = reinterpret_cast<const int4*>(au + bi * 32);
        const int4 a0 = qa[0], a1 = qa[1];
        int sdot = __dp4a(static_cast<int>(q[0] & 0x0F0F0F0Fu), a0.x, 0);
        sdot = __dp4a(static_cast<int>(q[1] & 0x0F0F0F0Fu), a0.y, sdot);
        sdot = __dp4a(static_cast<int>(q[2] & 0x0F0F0F0Fu), a0.z, sdot);
        sdot = __dp4a(static_cast<int>(q[3] & 0x0F0F0F0Fu), a0.w, sdot);
        sdot = __dp4a(static_cast<int>((q[0] >> 4) & 0x0F0F0F0Fu), a1.x, sdot);
        sdot = __dp4a(static_cast<int>((q[1] >> 4) & 0x0F0F0F0Fu), a1.y, sdot);
        sdot = __dp4a(static_cast<int>((q[2] >> 4) & 0x0F0F0F0Fu), a1.z, sdot);
        sdot = __dp4a(static_cast<int>((q[3] >> 4) & 0x0F0F0F0Fu), a1.w, sdot);
        acc[b & 1] = fmaf(dw * dq[bi], static_cast<float>(sdot - sq[bi]), acc[b & 1]);
    }
}

// Exact row sum of the act-quant product for a non-finite total: each
// activation block quantized again from A (read through L2) exactly as on
// chip, then A'_k = qs_k d_a times (q - 8) d_w element by element.
__device__ __noinline__ float list_row_exact_q8(const uint8_t* row, int nblocks, const float* a) {
    float s = 0.f;
    for (int b = 0; b < nblocks; ++b) {
        const float* x = a + kBlockElems * b;
        float amax = 0.f;
        for (int j = 0; j < kBlockElems; ++j) amax = fmaxf(amax, fabsf(__ldcg(x + j)));
        const float d = __fdiv_rn(amax, 127.f);
        const float da = f16_bits_to_float(f16_bits_rn(d));
        const uint8_t* blk = row + kBlockBytes * b;
        const float dw = f16_bits_to_float(static_cast<uint32_t>(blk[0]) | (static_cast<uint32_t>(blk[1]) << 8));
        for (int j = 0; j < kBlockElems; ++j) {
            const uint32_t byte = blk[2 + (j & 15)];
            const uint32_t nib = (j < 16) ? (byte & 0xFu) : (byte >> 4);
            s = fmaf(static_cast<float>(q8_quant(__ldcg(x + j), d)) * da, magic_minus8(nib | kMagicBits) * dw, s);
        }
    }
    return s;
}

// Exact row sum for a non-finite total (activations read through L2: they may
// have been written by other CTAs during this launch).
__device__ __noinline__ float list_row_exact(const uint8_t* row, int nblocks, const float* a) {
    float s = 0.f;
    for (int b = 0; b < nblocks; ++b) {
        const uint8_t* blk = row + kBlockBytes * b;
        const float d = f16_bits_to_float(static_cast<uint32_t>(blk[0]) | (static_cast<uint32_t>(blk[1]) << 8));
        for (int j = 0; j < kBlockElems; ++j) {
            const uint32_t byte = blk[2 + (j & 15)];
            const uint32_t nib = (j < 16) ? (byte & 0xFu) : (byte >> 4);
            s = fmaf(__ldcg(a + kBlockElems * b + j), magic_minus8(nib | kMagicBits) * d, s);
        }
    }
    return s;
}

// The CTA's share of problem q: tiles first, first + G, ...; returns their count.
__device__ __forceinline__ int cta_tiles(const ListProblem& q, int c, int G, int* first) {
    const int RG = (q.N + 15) >> 4;
    const int f = c >= q.off ? c - q.off : c - q.off + G;
    *first = f;
    return f < RG ? (RG - f + G - 1) / G : 0;
}

// Whether problem q needs its activations loaded (the same decision on every
// warp): another A or K than the loaded one, or a wait beyond the one the
// loaded copy was taken after.
struct AKey {
    const float* A = nullptr;
    int K = 0;
    int waited = -1;
    __device__ bool advance(const ListProblem& q) {
        const bool reload = q.A != A || q.K != K || q.wait_for > waited;
        if (reload) {
            A = q.A;
            K = q.K;
            waited = max(waited, q.wait_for);
        }
        return reload;
    }
};

__device__ __forceinline__ bool aborted(volatile int* flag) { return *flag != 0; }

__device__ __forceinline__ void set_abort(volatile int* flag) {
    atomicOr(&g_gemv_list_error, kErrWaitTimeout);
    *flag = 1;
}

__device__ __forceinline__ bool wait_stage(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    for (uint32_t i = 0; i < kMaxWaitPolls; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 63) == 63 && aborted(abort_flag)) return false;
    }
    set_abort(abort_flag);
    return false;
}

// The same wait for a thread that has nothing else to do meanwhile (the
// producer and the activation loader, which wait most of the time): it
// sleeps between polls so that it does not take issue slots from the
// consumer warps that share its scheduler.
__device__ __forceinline__ bool wait_idle(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    for (uint32_t i = 0; i < kMaxWaitPolls; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if (aborted(abort_flag)) return false;
        __nanosleep(128);
    }
    set_abort(abort_flag);
    return false;
}

template <bool kQ8>
__global__ void __launch_bounds__(kLThreads, 1)
    gemv_q4_0_list(const __grid_constant__ ListParams P) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* ring = smem;
    uint8_t* frag = smem + kOffFrag;
    float* slots = reinterpret_cast<float*>(smem + kOffSlots);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBars);
    uint64_t* empty = full + kLStages;
    uint64_t* a_full = empty + kLStages;
    uint64_t* a_empty = a_full + 1;
    uint64_t* pair_bar = a_empty + 1;  // [8]
    int* arr = reinterpret_cast<int*>(smem + kOffInts);  // [kTileSlots] arrivals per tile slot
    volatile int* done = arr + kTileSlots;               // [kTileSlots] last tile reduced per slot
    int* red = arr + 2 * kTileSlots;                     // [count] tiles of a problem reduced here
    volatile int* abort_flag = red + kListMaxProblems;
    const uint8_t* zeros = smem + kOffZero;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int c = static_cast<int>(blockIdx.x);
    const int G = P.grid;

    grid_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < kLStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kLW);
        }
        mbar_init(a_full, 1);
        mbar_init(a_empty, kLW);
        for (int i = 0; i < 8; ++i) mbar_init(&pair_bar[i], 2);
        for (int i = 0; i < kTileSlots; ++i) {
            arr[i] = 0;
            done[i] = i - kTileSlots;
        }
        for (int i = 0; i < kListMaxProblems; ++i) red[i] = 0;
        for (int i = 0; i < 256; ++i) reinterpret_cast<uint32_t*>(smem + kOffZero)[i] = 0u;
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == kLW) {
        // ------------------------------------------------------- producer
        // Stage s of a problem holds units 16 s .. 16 s + 15 of the CTA's
        // unit sequence of that problem (tile k = i / U, unit u = i % U), as
        // boxes of c units; c divides U, so a box never spans two tiles.
        if (lane != 0) {
            grid_dependency_wait();
            return;
        }
        int st = 0, issued = 0;
        uint32_t ph = 0;
        bool warmed = false;
        const float* a_prev = nullptr;
        for (int qi = 0; qi < P.count; ++qi) {
            const ListProblem& q = P.p[qi];
            int first;
            const int n = cta_tiles(q, c, G, &first);
            if (n == 0) continue;
            const int U = q.K >> 8;
            const int total = n * U;
            const int cu = q.c;
            const CUtensorMap* map = &P.map[qi];
            if (qi + 1 < P.count) prefetch_tensormap(&P.map[qi + 1]);
            if (!warmed) {
                // Ask L2 for the first stage before waiting on earlier kernels.
                warmed = true;
                for (int i = 0; i < min(kLW, total); i += cu)
                    tma_prefetch_l2_4d(map, 0, 0, (i % U) / cu, 16 * (first + (i / U) * G));
                grid_dependency_wait();
            }
            if (q.A != a_prev && q.wait_for < 0) {
                // New activations that nothing in this launch writes: on
                // their way to L2 as this problem's first weights are, a few
                // stages before the consumers read them.
                const uint32_t nb = static_cast<uint32_t>(q.K) * 4u;
                for (uint32_t o = 0; o < nb; o += 16384u)
                    bulk_prefetch_l2(reinterpret_cast<const uint8_t*>(q.A) + o, min(16384u, nb - o));
            }
            a_prev = q.A;
            for (int s0 = 0; s0 < total; s0 += kLW) {
                if (issued >= kLStages && !wait_idle(&empty[st], ph ^ 1u, abort_flag)) break;
                if (aborted(abort_flag)) break;
                const int boxes = (min(kLW, total - s0) + cu - 1) / cu;
                mbar_arrive_expect_tx(&full[st], static_cast<uint32_t>(boxes * box_bytes(cu)));
                uint8_t* stage = ring + st * kStageB;
                for (int j = 0; j < boxes; ++j) {
                    const int i = s0 + j * cu;
                    tma_load_4d(stage + j * box_bytes(cu), map, 0, 0, (i % U) / cu,
                                16 * (first + (i / U) * G), &full[st]);
                }
                ++issued;
                if (++st == kLStages) {
                    st = 0;
                    ph ^= 1u;
                }
            }
            if (aborted(abort_flag)) break;
        }
        if (!warmed) grid_dependency_wait();
        // Before leaving, let the copies still in flight land (bounded): the
        // last kLStages stages issued are the only ones that can be pending.
        for (int j = 0; j < min(issued, kLStages); ++j) {
            if (--st < 0) {
                st = kLStages - 1;
                ph ^= 1u;
            }
            mbar_wait_bounded(&full[st], ph, &g_gemv_list_error);
        }
        return;
    }

    if (warp == kLW + 1) {
        // -------------------------------------------- activation loader
        // New activations of a problem that waits for nothing (wait_for <
        // 0) are read by the consumers straight from global memory; the
        // loader copies in only those that wait for earlier problems, once
        // every consumer is done with the buffer and the problems waited for
        // are finished on every CTA.
        grid_dependency_wait();
        if (lane != 0) return;
        AKey key;
        int rounds = 0, direct = 0, handbacks = 0, verified = -1;
        for (int qi = 0; qi < P.count && !aborted(abort_flag); ++qi) {
            const ListProblem& q = P.p[qi];
            int first;
            if (cta_tiles(q, c, G, &first) == 0) {
                // Nothing of this problem here: count it as finished at once.
                if (q.arrive) {
                    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(P.ctr + qi) : "memory");
                }
                continue;
            }
            if (!key.advance(q)) continue;
            if (q.wait_for < 0) {
                ++rounds;
                continue;
            }
            // The consumers hand the buffer back before every copy after the
            // first round.
            if (rounds > 0) {
                if (!wait_idle(a_empty, handbacks & 1, abort_flag)) break;
                ++handbacks;
            }
            // Activations that are earlier problems' outputs: wait until every
            // CTA has finished every problem up to q.wait_for.
            bool ok = true;
            for (int j = verified + 1; j <= q.wait_for && ok; ++j) {
                uint32_t polls = 0;
                for (;;) {
                    uint32_t v;
                    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(P.ctr + j) : "memory");
                    if (v >= static_cast<uint32_t>(G)) break;
                    if (++polls >= kMaxCounterPolls || aborted(abort_flag)) {
                        ok = false;
                        break;
                    }
                    __nanosleep(64);
                }
            }
            if (!ok) {
                set_abort(abort_flag);
                break;
            }
            verified = max(verified, q.wait_for);
            // Generic-proxy writes of other CTAs, acquired above, before the
            // async-proxy (bulk copy) reads.
            asm volatile("fence.proxy.async.global;" ::: "memory");
            const uint32_t bytes = static_cast<uint32_t>(q.K) * 4u;
            mbar_arrive_expect_tx(a_full, bytes);
            for (uint32_t o = 0; o < bytes; o += 16384u)
                bulk_load_1d(frag + o, reinterpret_cast<const uint8_t*>(q.A) + o, min(16384u, bytes - o), a_full);
            ++direct;
            ++rounds;
        }
        // Let the copy still in flight land (bounded).
        if (direct > 0) mbar_wait_bounded(a_full, (direct - 1) & 1, &g_gemv_list_error);
        return;
    }

    // ----------------------------------------------------------- consumers
    grid_dependency_wait();
    const int g = lane >> 2;
    const int t = lane & 3;
    AKey key;
    int rounds = 0, direct = 0, pair_ph = 0, st = 0, tl = 0;
    bool prev_own = true;  // the fragments in place are read only by the warps that wrote them
    uint32_t ph = 0;
    bool ok = true;
    // A warp pair (w, w + 8) meets at its barrier; bounded, so that a warp
    // that gave up never leaves its partner blocked.
    auto pair_meet = [&]() {
        __syncwarp();
        if (lane == 0) mbar_arrive(&pair_bar[warp & 7]);
        const bool r = wait_stage(&pair_bar[warp & 7], pair_ph & 1, abort_flag);
        ++pair_ph;
        return __all_sync(0xFFFFFFFFu, r);
    };
    for (int qi = 0; qi < P.count && ok; ++qi) {
        const ListProblem& q = P.p[qi];
        int first;
        const int n = cta_tiles(q, c, G, &first);
        if (n == 0) continue;
        if (key.advance(q)) {
            // New activations.  Warp w takes unit u of every tile exactly
            // when u = w (mod 8) (a stage is 16 consecutive units of the
            // CTA's sequence and K / 256 is a multiple of 8), so the
            // fragments of unit u are read by warps u % 8 and u % 8 + 8
            // alone: warp w writes units w, w + 16, w + 32, ..., and only its
            // partner ever has to wait for them.  When K / 256 is a multiple
            // of 16 a warp reads exactly the units it writes ("own").
            const int U = q.K >> 8;
            const bool own = (U % kLW) == 0;
            if (q.wait_for < 0) {
                // Straight from global memory (nothing in this launch writes
                // these activations).  The partner must be done with the
                // units about to be rewritten, unless the warp read them alone.
                if (rounds > 0 && !prev_own) ok = pair_meet();
                if (!ok) break;
                // All of this warp's units in flight at once, then converted.
                const uint8_t* a_g = reinterpret_cast<const uint8_t*>(q.A);
                for (int u = warp; u < U; u += kLW) {
                    cp_async16(frag + u * 1024 + lane * 16, a_g + u * 1024 + lane * 16);
                    cp_async16(frag + u * 1024 + 512 + lane * 16, a_g + u * 1024 + 512 + lane * 16);
                }
                cp_async_wait_all();
                __syncwarp();
                for (int u = warp; u < U; u += kLW) {
                    if constexpr (kQ8) quantize_unit_q8<1>(frag + u * 1024, lane);
                    else unit_fragments(frag + u * 1024, lane);
                }
            } else {
                // Copied in by the loader once every consumer is done with
                // the buffer, then converted in place.
                if (rounds > 0) {
                    // Order this warp's accesses to the buffer before the
                    // loader's next bulk copy.
                    fence_proxy_async_shared();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(a_empty);
                }
                ok = wait_stage(a_full, direct & 1, abort_flag);
                ok = __all_sync(0xFFFFFFFFu, ok);
                if (!ok) break;
                for (int u = warp; u < U; u += kLW) {
                    if constexpr (kQ8) quantize_unit_q8<1>(frag + u * 1024, lane);
                    else unit_fragments(frag + u * 1024, lane);
                }
                ++direct;
            }
            __syncwarp();
            // The partner's units are this warp's too unless it is "own".
            if (!own) ok = pair_meet();
            prev_own = own;
            ++rounds;
            if (!ok) break;
        }
        const int U = q.K >> 8;
        const int total = n * U;
        // This warp's slot of every stage of the problem: box warp / c, unit
        // warp % c of it (c is 16 or 8); its rows g and g + 8 are row_b apart.
        const int cu = q.c;
        const int row_b = (cu + 1) * kUnitB;
        const int slot_off = (cu == 16 ? 0 : (warp >> 3) * box_bytes(8)) + (warp & (cu - 1)) * kUnitB +
                             (kQ8 ? (lane & 15) : g) * row_b;
        const uint8_t* fbase = (g >> 1) == t ? frag : zeros;
        const int fstep = (g >> 1) == t ? 1024 : 0;
        // Position warp, then warp + 16, ... of the CTA's unit sequence:
        // tile k, unit u, advanced without dividing.
        int k = warp / U, u = warp - (warp / U) * U;
        float acc[2] = {0.f, 0.f};
        for (int s0 = 0; s0 < total; s0 += kLW, u += kLW) {
            while (u >= U) {
                u -= U;
                ++k;
            }
            ok = wait_stage(&full[st], ph, abort_flag);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            if (s0 + warp < total) {
                if (u < kLW) acc[0] = acc[1] = 0.f;
                const uint8_t* ra = ring + st * kStageB + slot_off;
                if constexpr (kQ8) half_unit_q8(ra, lane >> 4, frag + u * 1024, acc);
                else unit_mma(ra, ra + 8 * row_b, fbase + u * fstep, g, t, acc);
                // The stage's bytes are in registers: hand it back to the
                // producer before adding anything up.
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
                if (u + kLW >= U) {
                    // This warp's last unit of tile k: its row sums to the slot
                    // (MMA consumer: rows g and g + 8 from the lanes t = 0;
                    // integer consumer: row l from lanes l < 16).
                    float s0v = acc[0], s1v = acc[1];
                    if constexpr (kQ8) {
                        s0v += s1v;
                        s0v += __shfl_xor_sync(0xFFFFFFFFu, s0v, 16);
                    } else {
                        s0v += __shfl_xor_sync(0xFFFFFFFFu, s0v, 1);
                        s1v += __shfl_xor_sync(0xFFFFFFFFu, s1v, 1);
                        s0v += __shfl_xor_sync(0xFFFFFFFFu, s0v, 2);
                        s1v += __shfl_xor_sync(0xFFFFFFFFu, s1v, 2);
                    }
                    const int tile_l = tl + k;
                    const int sl = tile_l % kTileSlots;
                    // The slot's previous tile must have been added up.
                    bool free_ok = true;
                    for (uint32_t polls = 0; done[sl] != tile_l - kTileSlots; ++polls) {
                        if (polls >= kMaxWaitPolls || aborted(abort_flag)) {
                            free_ok = false;
                            break;
                        }
                    }
                    if (!free_ok) {
                        set_abort(abort_flag);
                        ok = false;
                    }
                    ok = __all_sync(0xFFFFFFFFu, ok);
                    if (!ok) break;
                    float* my = slots + (sl * kLW + warp) * 16;
                    if constexpr (kQ8) {
                        if (lane < 16) my[lane] = s0v;
                    } else if (t == 0) {
                        my[g] = s0v;
                        my[g + 8] = s1v;
                    }
                    __threadfence_block();
                    __syncwarp();
                    const int n_part = min(kLW, U);
                    int old = 0;
                    if (lane == 0) old = atomicAdd(&arr[sl], 1);
                    old = __shfl_sync(0xFFFFFFFFu, old, 0);
                    if (old == n_part - 1) {
                        // Last warp of the tile: add the slots in unit order.
                        __threadfence_block();
                        const int tile = first + k * G;
                        float v = 0.f;
                        if (lane < 16) {
                            for (int j = 0; j < n_part; ++j)
                                v += slots[(sl * kLW + ((k * U + j) & (kLW - 1))) * 16 + lane];
                        }
                        const int row = 16 * tile + lane;
                        if (lane < 16 && row < q.N) {
                            if (!isfinite(v)) {
                                const uint8_t* wrow = q.W + static_cast<int64_t>(row) * U * kUnitB;
                                v = kQ8 ? list_row_exact_q8(wrow, U * 8, q.A) : list_row_exact(wrow, U * 8, q.A);
                            }
                            q.C[row] = v;
                        }
                        // Only a problem that others wait on needs its stores
                        // made visible before the CTA counts it finished.
                        if (q.arrive) __threadfence();
                        __syncwarp();
                        if (lane == 0) {
                            arr[sl] = 0;
                            done[sl] = tile_l;
                            if (q.arrive && atomicAdd(&red[qi], 1) == n - 1) {
                                __threadfence();
                                asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(P.ctr + qi)
                                             : "memory");
                            }
                        }
                    }
                }
            }
            if (s0 + warp >= total) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
            }
            if (++st == kLStages) {
                st = 0;
                ph ^= 1u;
            }
        }
        tl += n;
    }
}

}  // namespace

cudaError_t launch_gemv_q4_0_list(const GemvListItem* items, int count, unsigned* counters,
                                  cudaStream_t stream, const DeviceInfo& dev, bool q8) {
    if (count <= 0) return cudaSuccess;
    if (count > kListMaxProblems) return cudaErrorInvalidValue;
    static int configured[2][64] = {};
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    if (kLSmem > dev.max_smem_optin) return cudaErrorInvalidValue;
    void (*const kernel)(ListParams) = q8 ? gemv_q4_0_list<true> : gemv_q4_0_list<false>;
    if (!__atomic_load_n(&configured[q8][dev.device], __ATOMIC_ACQUIRE)) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kLSmem);
        if (e != cudaSuccess) return e;
        __atomic_store_n(&configured[q8][dev.device], 1, __ATOMIC_RELEASE);
    }
    ListParams P;
    P.count = count;
    P.grid = dev.sm_count;
    P.ctr = counters;
    int max_wait = -1;
    for (int i = 0; i < count; ++i) max_wait = std::max(max_wait, items[i].wait_for);
    if (max_wait >= 0 && !counters) return cudaErrorInvalidValue;
    // A launch without waits runs independent problems, whose order does not
    // matter: group those with the same activations (stably, in order of
    // first appearance), so that each CTA loads every activation vector once
    // instead of at every change.
    int order[kListMaxProblems];
    int first_use[kListMaxProblems];
    for (int i = 0; i < count; ++i) {
        order[i] = i;
        first_use[i] = i;
        for (int j = 0; j < i; ++j) {
            if (items[j].A == items[i].A && items[j].K == items[i].K) {
                first_use[i] = first_use[j];
                break;
            }
        }
    }
    if (max_wait < 0)
        std::stable_sort(order, order + count, [&](int a, int b) { return first_use[a] < first_use[b]; });
    int64_t rg_sum = 0;
    for (int o = 0; o < count; ++o) {
        const int i = order[o];
        ListProblem& q = P.p[o];
        q.A = items[i].A;
        q.W = items[i].W;
        q.C = items[i].C;
        q.N = static_cast<int>(items[i].N);
        q.K = static_cast<int>(items[i].K);
        q.wait_for = items[i].wait_for;
        q.arrive = i <= max_wait ? 1 : 0;
        q.off = static_cast<int>(rg_sum % P.grid);
        const int U = q.K / 256;
        if (U % 8 != 0) return cudaErrorInvalidValue;
        q.c = (U % 16 == 0) ? 16 : 8;
        rg_sum += (items[i].N + 15) / 16;
        // Weights as bytes [N rows][U / c groups][c units][144 B]; boxes of
        // 16 rows x 1 group x (c + 1) units x 144 B (the last unit outside
        // the group reads as zeros and pads the shared-memory rows).
        const int64_t dims[4] = {kUnitB, q.c, U / q.c, items[i].N};
        const int64_t strides[3] = {kUnitB, int64_t(kUnitB) * q.c, int64_t(kUnitB) * U};
        const int box[4] = {kUnitB, q.c + 1, 1, 16};
        cudaError_t e = encode_tiled(&P.map[o], CU_TENSOR_MAP_DATA_TYPE_UINT8, items[i].W, 4, dims, strides, box);
        if (e != cudaSuccess) return e;
    }
    if (max_wait >= 0) {
        cudaError_t e = cudaMemsetAsync(counters, 0, static_cast<size_t>(max_wait + 1) * sizeof(unsigned), stream);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = launch_pdl(kernel, dim3(P.grid), dim3(kLThreads), kLSmem, stream, P);
    if (e != cudaSuccess) return e;
    note_launch();
    return cudaSuccess;
}

cudaError_t gemv_list_read_device_error(unsigned int* bits, bool clear) {
    unsigned int v = 0;
    cudaError_t err = cudaMemcpyFromSymbol(&v, g_gemv_list_error, sizeof(v));
    if (err != cudaSuccess) return err;
    *bits |= v;
    if (clear && v != 0) {
        const unsigned int zero = 0;
        err = cudaMemcpyToSymbol(g_gemv_list_error, &zero, sizeof(zero));
    }
    return err;
}

}  // namespace qm

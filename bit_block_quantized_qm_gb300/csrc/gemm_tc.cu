// Prefill GEMM on 5th-generation tensor cores (tcgen05, sm_103a):
// C[M][N] = A[M][K] x dequant(W)^T, W a Q4_0 block stream (section
// "matmul_q4_0_tiled" of "fuel-vulkan-kernels — quantized (GGML) kernel
// contracts": tiles of the weight are decoded once and reused over many
// activation rows).
//
// Exactness of the split-precision products:
//   * a weight (q - 8) * d has at most 4 + 11 significant bits, so it is
//     exactly W_hi + W_lo with W_hi = bf16(W), W_lo = bf16(W - W_hi);
//   * an activation a is a_hi + a_lo + r with a_hi = bf16(a),
//     a_lo = bf16(a - a_hi), |r| <= 2^-17 |a|;
//   * all four products a_hi W_hi, a_hi W_lo, a_lo W_hi, a_lo W_lo are taken
//     (bf16 x bf16 products are exact in the f32 accumulator), so one product
//     misses a W by the activation residual r W alone, at most 2^-17 |a W|;
//   * the large products a_hi W_hi accumulate in one TMEM accumulator and the
//     three small ones (at most 2^-8 of the large one each) in a second one,
//     added once in the epilogue: the rounding of the small terms then
//     happens at their own magnitude, not at the running total's.
//
// Structure (one 128-row output tile of BN = 128 or 256 columns per work
// item, K in 64-wide steps; BN = 128 also runs 112-column tiles, where those
// fill more SMs):
//   * warp 0 (one thread) streams, with TMA, the f32 activation tile of each
//     k-step (128 rows x 64 k) and the weight's raw Q4_0 bytes (BN rows x the
//     48-byte, 16-byte aligned span that holds the step's 36-byte block pair);
//   * warps 2..17 decode each BN x 64 weight tile into W_hi / W_lo, and turn
//     the activation tile, in place, into its a_hi / a_lo tiles (every
//     thread reads its 16 floats, the 16 warps meet at a named barrier, then
//     each writes its pieces), all in the 128-byte swizzled K-major layout
//     the MMA reads; then they run the epilogue;
//   * warp 1 owns the two TMEM accumulators (128 lanes x BN f32 columns
//     each: a_hi W_hi, then the three small products) and one thread issues
//     16 tcgen05.mma (4 products x 4 k-steps of 16, each 128 x N x 16) per
//     k-step, committing completion to the stages' "empty" barriers;
//   * the epilogue reads both accumulators with tcgen05.ld (32 x 32 blocks),
//     adds them, stages a block in shared memory (the freed weight stages)
//     and writes C row by row, 16-byte stores when C's rows allow.
// The 256-wide tile reads each activation tile once per 256 output columns
// and keeps the operand reads of one MMA at 12 KB per 2^20 flops, which the
// shared-memory bandwidth sustains together with the decode's stores.
// Work items (a 1-D grid, one per CTA): whole tiles fill as many full waves
// of SMs as they can; the tiles of a last, partial wave become 128-column
// halves of 256-column tiles, or are split into s_rem = 2, 4 or 8 K ranges of
// whole 256-wide units when the split tiles' clusters of s_rem CTAs all fit
// on the GPU at once.  The partial tiles of a K split meet through the
// thread-block cluster: each CTA keeps its partial tile in shared memory and,
// after a bounded mbarrier handshake, sums a slice of rows of all of them in
// rank order over distributed shared memory, so the result does not depend
// on timing and nothing but C is written to global memory.  An entry that
// comes out infinite or NaN is recomputed element by element from A and the
// Q4_0 stream, so non-finite scales keep the per-element semantics.
// The kernel is launched with programmatic stream serialization: it lets the
// next kernel start its prologue early and waits (griddepcontrol.wait) before
// touching global memory.
// Every wait is bounded; a wait that gives up sets the device error word.
#include <algorithm>

#include "qm_device.cuh"
#include "qm_internal.h"

namespace qm {

__device__ unsigned int g_gemm_error = 0;

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int kDecodeWarps = 16;
constexpr int kThreads = (2 + kDecodeWarps) * 32;
constexpr int kTileA = BM * BK * 2;   // one bf16 activation tile: 16 KB
constexpr int kRawRow = 48;           // raw bytes of one row per k-step (3 x 16 B)

// Tiles of BN = 128 (run 128 or 112 columns wide) or 256 output columns.
template <int BN>
struct Tile {
    static constexpr int kAStages = BN == 128 ? 3 : 2;
    static constexpr int kWStages = 2;
    static constexpr int kRawStages = 2;  // raw Q4_0 bytes of one k-step per stage
    static constexpr int kTileW = BN * BK * 2;  // one bf16 weight tile
    static constexpr int kRawBytes = BN * kRawRow;
    static constexpr int kTmemCols = 2 * BN;    // two f32 accumulators of BN columns
    // Barriers (full and empty per stage, converted per activation stage,
    // acc_full, two cluster-reduction barriers), then the TMEM address,
    // rounded up to 16 bytes.
    static constexpr int kBarBytes = ((2 * (kAStages + kWStages + kRawStages) + kAStages + 3) * 8 + 8 + 15) / 16 * 16;
    static constexpr int kSmemBytes = kAStages * 2 * kTileA + kWStages * 2 * kTileW +
                                      kRawStages * kRawBytes + kBarBytes + 1024;  // + alignment slack
    // Instruction descriptor, kind::f16: D f32, A and B bf16, both K-major,
    // N = BN, M = BM.
    static constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                       (static_cast<uint32_t>(BN >> 3) << 17) |
                                       (static_cast<uint32_t>(BM >> 4) << 24);
    static_assert(kSmemBytes <= 232448, "shared memory of one CTA");
};

// Shared-memory matrix descriptor: K-major, 128-byte swizzle (rows of 128 B,
// 8-row atoms 1024 B apart), start address in 16-byte units.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1) << 16;            // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;    // stride byte offset: one 8-row atom
    d |= static_cast<uint64_t>(1) << 46;            // descriptor version
    d |= static_cast<uint64_t>(2) << 61;            // 128-byte swizzle
    return d;
}

__device__ __forceinline__ void mma_f16(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc,
                                        uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(tmem_d), "l"(da), "l"(db), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive f32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t r[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// 32 consecutive columns of this thread's TMEM lane in the large-product
// accumulator plus the same columns of the small-product one, `small_off`
// columns further on (16 columns of each at a time, to keep registers low).
__device__ __forceinline__ void tmem_ld_acc(uint32_t taddr, uint32_t small_off, float v[32]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint32_t a[16], b[16];
        tmem_ld16(taddr + 16 * h, a);
        tmem_ld16(taddr + small_off + 16 * h, b);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
        for (int i = 0; i < 16; ++i) v[16 * h + i] = __uint_as_float(a[i]) + __uint_as_float(b[i]);
    }
}

// Decode half of one Q4_0 block (18 bytes at `blk`, 2-byte aligned, shared
// memory): quant bytes 8p .. 8p+7, i.e. elements 8p .. 8p+7 (low nibbles) and
// 16+8p .. 16+8p+7 (high nibbles).  A byte permute puts each nibble q in bits
// 16..19 under the byte 0x43, which reads as the float 128 + q; one packed FMA
// per pair, x d - 136 d, gives w = (q - 8) d exactly (136 d and (q - 8) d have
// at most 19 significant bits).  w is then split into bf16 hi = bf16(w) and
// lo = bf16(w - hi), an exact two-piece sum (w - hi has at most 7 significant
// bits); both are stored as row n of 128-byte-swizzled K-major tiles at
// k = 32 * half + j.  Non-finite scales need no care here: they make the
// output entry non-finite and the epilogue recomputes it element by element.
__device__ __forceinline__ void decode_half_block(const uint8_t* blk, int p, int n, int half,
                                                  uint8_t* tile_hi, uint8_t* tile_lo) {
    constexpr uint32_t kHigh = 0x43000000u;
    const uint16_t* h = reinterpret_cast<const uint16_t*>(blk);
    const float d = f16_bits_to_float(h[0]);
    const float2 d2 = make_float2(d, d);
    const float2 b2 = make_float2(-136.0f * d, -136.0f * d);
    const float2 neg1 = make_float2(-1.0f, -1.0f);
    const uint32_t w0 = static_cast<uint32_t>(h[1 + 4 * p]) | (static_cast<uint32_t>(h[2 + 4 * p]) << 16);
    const uint32_t w1 = static_cast<uint32_t>(h[3 + 4 * p]) | (static_cast<uint32_t>(h[4 + 4 * p]) << 16);
#pragma unroll
    for (int side = 0; side < 2; ++side) {  // 0: low nibbles, 1: high nibbles
        const uint32_t v0 = (side ? (w0 >> 4) : w0) & 0x0F0F0F0Fu;
        const uint32_t v1 = (side ? (w1 >> 4) : w1) & 0x0F0F0F0Fu;
        const uint32_t src[4] = {v0, v0, v1, v1};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            // Elements 2e and 2e + 1 of the eight: bytes (2e) % 4 and (2e) % 4 + 1.
            const uint32_t sel0 = 0x7044u | (static_cast<uint32_t>((2 * e) & 3) << 8);
            const uint32_t sel1 = 0x7044u | (static_cast<uint32_t>((2 * e + 1) & 3) << 8);
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(__byte_perm(src[e], kHigh, sel0)),
                                                    __uint_as_float(__byte_perm(src[e], kHigh, sel1))),
                                        d2, b2);
            const __nv_bfloat162 hb = __floats2bfloat162_rn(x.x, x.y);
            const uint32_t hw = *reinterpret_cast<const uint32_t*>(&hb);
            const float2 r = __ffma2_rn(make_float2(__uint_as_float(hw << 16), __uint_as_float(hw & 0xFFFF0000u)),
                                        neg1, x);
            const __nv_bfloat162 lb = __floats2bfloat162_rn(r.x, r.y);
            hi[e] = hw;
            lo[e] = *reinterpret_cast<const uint32_t*>(&lb);
        }
        // Element 8p + e (side 0) or 16 + 8p + e (side 1) of the block sits in
        // 16-byte chunk 4 * half + p + 2 * side of the 128-byte tile row.
        const int chunk = 4 * half + p + 2 * side;
        const int off = n * 128 + ((chunk ^ (n & 7)) << 4);
        *reinterpret_cast<uint4*>(tile_hi + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(tile_lo + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// The activation pieces of four consecutive f32 values x (k = 4f .. 4f + 3 of
// row r of a 128 x 64 tile): hi = bf16(a), lo = bf16(a - hi) (packed
// conversions, lo = a - hi by one packed FMA, exact), stored as 8 bytes of row
// r of the 128-byte swizzled K-major hi and lo tiles.  A non-finite piece
// makes the entries that use it non-finite, and the epilogue recomputes those
// element by element.
__device__ __forceinline__ void split_store4(float4 x, int r, int f, uint8_t* tile_hi, uint8_t* tile_lo) {
    const float2 v[2] = {make_float2(x.x, x.y), make_float2(x.z, x.w)};
    uint32_t hw[2], lw[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const __nv_bfloat162 hb = __floats2bfloat162_rn(v[e].x, v[e].y);
        hw[e] = *reinterpret_cast<const uint32_t*>(&hb);
        const float2 rest = __ffma2_rn(make_float2(__uint_as_float(hw[e] << 16), __uint_as_float(hw[e] & 0xFFFF0000u)),
                                       make_float2(-1.0f, -1.0f), v[e]);
        const __nv_bfloat162 lb = __floats2bfloat162_rn(rest.x, rest.y);
        lw[e] = *reinterpret_cast<const uint32_t*>(&lb);
    }
    const int off = r * 128 + ((((f >> 1) ^ (r & 7))) << 4) + (f & 1) * 8;
    *reinterpret_cast<uint2*>(tile_hi + off) = make_uint2(hw[0], hw[1]);
    *reinterpret_cast<uint2*>(tile_lo + off) = make_uint2(lw[0], lw[1]);
}

// Named barrier over `threads` threads that also ANDs their `v`.
__device__ __forceinline__ bool named_barrier_and(int id, int threads, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(threads)
        : "memory");
    return r != 0;
}

// Exact C[m][n] for an entry whose tensor-core sum is not finite:
// sum_k A[m][k] * ((q - 8) * d) element by element.
__device__ __noinline__ float entry_exact(const float* __restrict__ A, const uint8_t* __restrict__ wq,
                                          int64_t K, int64_t m, int64_t n) {
    const int64_t nb = K / kBlockElems;
    const uint8_t* row = wq + n * nb * kBlockBytes;
    const float* a = A + m * K;
    float s = 0.f;
    for (int64_t b = 0; b < nb; ++b) {
        const uint8_t* blk = row + b * kBlockBytes;
        const float d = f16_bits_to_float(static_cast<uint32_t>(blk[0]) |
                                          (static_cast<uint32_t>(blk[1]) << 8));
        for (int j = 0; j < 32; ++j) {
            const uint32_t byte = blk[2 + (j & 15)];
            const uint32_t nib = (j < 16) ? (byte & 0xFu) : (byte >> 4);
            s = fmaf(a[b * 32 + j], magic_minus8(nib | kMagicBits) * d, s);
        }
    }
    return s;
}

template <int BN>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_q4_0_tc(const __grid_constant__ CUtensorMap map_a,
                 const __grid_constant__ CUtensorMap map_w,
                 const __grid_constant__ CUtensorMap map_w2, const float* __restrict__ A,
                 const uint8_t* __restrict__ wq, float* __restrict__ C, int M, int N, int K,
                 int c_vec, int tw, int nt, int n_full, int s_rem, int hw) {
    using T = Tile<BN>;
    constexpr int kAStages = T::kAStages;
    constexpr int kWStages = T::kWStages;
    constexpr int kRawStages = T::kRawStages;
    constexpr int kTileW = T::kTileW;
    constexpr int kRawBytes = T::kRawBytes;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte alignment for the swizzled tiles, by indexing the shared array
    // itself so the compiler keeps every access below in the shared space.
    uint8_t* base = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint8_t* a_st = base;                                // [kAStages][f32 tile | hi, lo][32 KB]
    uint8_t* w_st = a_st + kAStages * 2 * kTileA;        // [kWStages][hi, lo][BN rows][128 B]
    uint8_t* raw = w_st + kWStages * 2 * kTileW;         // [kRawStages][BN rows][48 B]
    uint64_t* bars = reinterpret_cast<uint64_t*>(raw + kRawStages * kRawBytes);
    uint64_t* a_full = bars;
    uint64_t* a_empty = bars + kAStages;
    uint64_t* w_full = bars + 2 * kAStages;
    uint64_t* w_empty = w_full + kWStages;
    uint64_t* raw_full = w_empty + kWStages;
    uint64_t* raw_empty = raw_full + kRawStages;
    uint64_t* a_conv = raw_empty + kRawStages;  // [kAStages] activation pieces written
    uint64_t* acc_full = a_conv + kAStages;
    uint64_t* red_bar = acc_full + 1;  // [2]: partial tiles written, partial tiles read
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(red_bar + 2);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Work item: CTAs below n_full take whole tiles of tw columns (tw = BN,
    // or 112 with BN = 128 when 112-column tiles fill the SMs better).  Each
    // later tile is either split into s_rem K ranges, one per CTA, or (hw,
    // BN = 256 only) into two 128-column halves, one per CTA.  Tiles are
    // numbered m-tile major.
    const int b = static_cast<int>(blockIdx.x);
    const bool half_item = (BN == 256) && hw != 0 && b >= n_full;
    const int tile = (b < n_full) ? b : n_full + (b - n_full) / (hw ? 2 : s_rem);
    const int split = (b < n_full || hw) ? 0 : (b - n_full) % s_rem;
    const int S = (b < n_full || hw) ? 1 : s_rem;
    const int wn = half_item ? BN / 2 : tw;  // columns of this item
    const int m0 = (tile / nt) * BM;
    const int n0 = (tile % nt) * tw + (half_item ? ((b - n_full) & 1) * (BN / 2) : 0);
    const int KT = K / BK / S;  // k-steps of this CTA's K range
    const int kt0 = split * KT;
    const int cl = S > 1;       // a K split adds up through the cluster

    grid_launch_dependents();
    if (threadIdx.x == 0) {
        for (int s = 0; s < kAStages; ++s) {
            mbar_init(&a_full[s], 1);
            mbar_init(&a_empty[s], 1);
            mbar_init(&a_conv[s], kDecodeWarps);
        }
        for (int s = 0; s < kWStages; ++s) {
            mbar_init(&w_full[s], kDecodeWarps);
            mbar_init(&w_empty[s], 1);
        }
        for (int s = 0; s < kRawStages; ++s) {
            mbar_init(&raw_full[s], 1);
            mbar_init(&raw_empty[s], kDecodeWarps);
        }
        mbar_init(acc_full, 1);
        mbar_init(&red_bar[0], S);  // one arrival per CTA of the cluster
        mbar_init(&red_bar[1], S);
        fence_barrier_init();
    }
    if (warp == 1) {
        asm volatile(
            "tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                smem_addr(tmem_slot)),
            "r"(T::kTmemCols)
            : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // Cluster launches: every CTA's barriers are initialised before any CTA
    // can arrive on them remotely.
    if (cl) cluster_sync_all();
    const uint32_t tmem = *tmem_slot;
    grid_dependency_wait();  // A and C may belong to the kernel before this one

    if (warp == 0) {
        if (lane == 0) {
            // Producer: the raw weight bytes and the activation tiles of each
            // k-step.  The step's block pair is bytes 36 j .. 36 j + 35 of each
            // row (j = k-step); the 48-byte box starts at the 16-byte boundary
            // below it, which TMA requires, and still covers the pair.
            prefetch_tensormap(&map_a);
            const CUtensorMap* mw = half_item ? &map_w2 : &map_w;
            prefetch_tensormap(mw);
            for (int kt = 0; kt < KT; ++kt) {
                const int rs = kt % kRawStages;
                if (kt >= kRawStages &&
                    !mbar_wait_bounded(&raw_empty[rs], ((kt / kRawStages) - 1) & 1, &g_gemm_error))
                    break;
                // The box is BN rows (BN / 2 for a half item), whatever wn is.
                mbar_arrive_expect_tx(&raw_full[rs], static_cast<uint32_t>((half_item ? BN / 2 : BN) * kRawRow));
                tma_load_2d(raw + rs * kRawBytes, mw, (36 * (kt0 + kt)) & ~15, n0, &raw_full[rs]);
                const int as = kt % kAStages;
                if (kt >= kAStages &&
                    !mbar_wait_bounded(&a_empty[as], ((kt / kAStages) - 1) & 1, &g_gemm_error))
                    break;
                // The f32 tile (128 rows x 256 B) fills the stage's hi and lo space.
                mbar_arrive_expect_tx(&a_full[as], 2 * kTileA);
                tma_load_2d(a_st + (2 * as) * kTileA, &map_a, (kt0 + kt) * BK, m0, &a_full[as]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // MMA issuer: 4 products x 4 k-steps of 16 per 64-wide k-step, N =
            // wn; the large product into columns 0.., the small ones into
            // columns BN.. of the TMEM allocation.
            const uint32_t idesc =
                (T::kIdesc & ~(0x3Fu << 17)) | (static_cast<uint32_t>(wn >> 3) << 17);
            bool ok = true;
            for (int kt = 0; kt < KT && ok; ++kt) {
                const int as = kt % kAStages;
                const int ws = kt % kWStages;
                ok = mbar_wait_bounded(&a_conv[as], (kt / kAStages) & 1, &g_gemm_error) &&
                     mbar_wait_bounded(&w_full[ws], (kt / kWStages) & 1, &g_gemm_error);
                if (!ok) break;
                tc_fence_after();
                const uint32_t ahi = smem_addr(a_st + (2 * as) * kTileA);
                const uint32_t alo = ahi + kTileA;
                const uint32_t whi = smem_addr(w_st + (2 * ws) * kTileW);
                const uint32_t wlo = whi + kTileW;
                // Descriptors once per stage; a k-step of 16 bf16 (32 bytes) is +2
                // in the start-address field (16-byte units, below 2^14 here).
                const uint64_t dah = sw128_desc(ahi), dal = sw128_desc(alo);
                const uint64_t dwh = sw128_desc(whi), dwl = sw128_desc(wlo);
#pragma unroll
                for (int kk = 0; kk < BK / 16; ++kk) {
                    const uint64_t o = static_cast<uint64_t>(2 * kk);
                    const uint32_t acc_on = (kt | kk) != 0;
                    mma_f16(tmem, dah + o, dwh + o, idesc, acc_on);
                    mma_f16(tmem + BN, dah + o, dwl + o, idesc, acc_on);
                    mma_f16(tmem + BN, dal + o, dwh + o, idesc, 1u);
                    mma_f16(tmem + BN, dal + o, dwl + o, idesc, 1u);
                }
                mma_commit(&a_empty[as]);
                mma_commit(&w_empty[ws]);
            }
            mma_commit(acc_full);
        }
    } else {
        // Decode warps: tpr threads per weight row.  With 2 (256 columns)
        // thread t of 512 owns row t / 2 and block t % 2 of the 64-wide k-step,
        // both halves of its quant bytes; with 4 (128 columns) it owns row
        // t / 4, block (t / 2) % 2 and quant bytes 8 (t % 2) .. 8 (t % 2) + 7.
        const int tpr = wn > 128 ? 2 : 4;
        const int dt = threadIdx.x - 64;
        const int a_rows = min(BM, M - m0);  // activation rows of this tile
        const int n = dt / tpr;
        const int half = (tpr == 2) ? (dt & 1) : ((dt >> 1) & 1);
        for (int kt = 0; kt < KT; ++kt) {
            const int rs = kt % kRawStages;
            const int ws = kt % kWStages;
            const int as = kt % kAStages;
            bool ok = mbar_wait_bounded(&raw_full[rs], (kt / kRawStages) & 1, &g_gemm_error);
            if (ok && kt >= kWStages)
                ok = mbar_wait_bounded(&w_empty[ws], ((kt / kWStages) - 1) & 1, &g_gemm_error);
            if (ok) {
                // The weight tile first: the activation tile's copy, issued
                // when its stage came free, lands meanwhile.
                const uint8_t* blk =
                    raw + rs * kRawBytes + n * kRawRow + ((36 * (kt0 + kt)) & 15) + half * kBlockBytes;
                uint8_t* thi = w_st + (2 * ws) * kTileW;
                if (tpr == 2) {
                    decode_half_block(blk, 0, n, half, thi, thi + kTileW);
                    decode_half_block(blk, 1, n, half, thi, thi + kTileW);
                } else if (n < wn) {  // rows past a 112-column tile are not decoded
                    decode_half_block(blk, dt & 1, n, half, thi, thi + kTileW);
                }
            }
            if (ok) ok = mbar_wait_bounded(&a_full[as], (kt / kAStages) & 1, &g_gemm_error);
            uint8_t* ast = a_st + (2 * as) * kTileA;
            float4 x[4];
            if (ok) {
                // This thread's 16 floats of the f32 activation tile: float4
                // j * 512 + dt, i.e. row 32 j + dt / 16, k = 4 (dt % 16) .. + 3
                // (each quarter warp reads 128 contiguous bytes).  Rows past
                // M are not split: whatever their pieces hold reaches only
                // the MMA rows of outputs past M, which are never stored.
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (32 * j < a_rows) x[j] = *reinterpret_cast<const float4*>(ast + (j * 512 + dt) * 16);
            }
            // Every thread has read its floats before any piece overwrites
            // them; a failed wait anywhere stops all decode warps together.
            if (!named_barrier_and(2, kDecodeWarps * 32, ok)) break;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                if (32 * j < a_rows) split_store4(x[j], 32 * j + (dt >> 4), dt & 15, ast, ast + kTileA);
            fence_proxy_async_shared();  // make the tiles visible to the tensor cores
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&w_full[ws]);
                mbar_arrive(&raw_empty[rs]);
                mbar_arrive(&a_conv[as]);
            }
        }
        // Epilogue: TMEM lane quarter q = warp % 4; warp (q, cq) owns rows
        // 32 q .. 32 q + 31 and columns wn/4 cq .. wn/4 cq + wn/4 - 1, as
        // blocks of 32 x 32 (the last one narrower when wn/4 = 28).  Lane i holds row i of a block; the block
        // goes through shared memory (rows 36 floats apart: conflict-free
        // 16-byte writes and reads) so that C is written a row at a time.  All
        // MMAs have completed when acc_full fires, and it fires only after
        // every decode warp has left its loop, so the activation and weight
        // stages are free.
        // (Warp-uniform decision: tcgen05.ld below is a warp-wide instruction.)
        const bool acc_ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(acc_full, 0, &g_gemm_error));
        static_assert(kDecodeWarps * 32 * 36 * 4 <= kAStages * 2 * kTileA + kWStages * 2 * kTileW,
                      "staging space");
        const int q = warp & 3;
        const int cq = (warp - 2) >> 2;
        const int mrow = m0 + 32 * q;
        float* stg = reinterpret_cast<float*>(a_st) + (warp - 2) * (32 * 36);
        const int cw = wn / 4;              // columns of this warp (28, 32, 64)
        const int ncb = (cw + 31) / 32;     // 32-column blocks of this warp
        if (cl) {
            // Split K through the cluster (the S CTAs of this tile, ranks in
            // range order): each CTA leaves its partial tile in its own shared
            // memory, [128 rows][wn + 4] f32, then adds rows r 128/S ..
            // (r + 1) 128/S - 1 of all S tiles in rank order, reading the
            // others' through distributed shared memory, and writes C.  The
            // arrivals come on every path, whatever the waits returned.
            const int ld = wn + 4;  // row stride: 16-byte stores of 8 lanes hit distinct banks
            float* ptile = reinterpret_cast<float*>(a_st);
            for (int jb = 0; jb < ncb; ++jb) {
                const int col = cw * cq + 32 * jb;
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) v[i] = 0.f;
                if (acc_ok) {
                    tc_fence_after();
                    tmem_ld_acc(tmem + (static_cast<uint32_t>(32 * q) << 16) + col, BN, v);
                }
                float* dst = ptile + (32 * q + lane) * ld + col;
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    *reinterpret_cast<float4*>(dst + 4 * j) =
                        make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            }
            asm volatile("fence.acq_rel.cluster;" ::: "memory");
            named_barrier_sync(1, kDecodeWarps * 32);
            const uint32_t rank = cluster_ctarank();
            if (threadIdx.x == 64) {
                for (int r = 0; r < S; ++r)
                    mbar_arrive_cluster(mapa_shared(smem_addr(&red_bar[0]), static_cast<uint32_t>(r)));
            }
            if (mbar_wait_cluster_bounded(&red_bar[0], 0, &g_gemm_error)) {
                const int rows = BM / S;
                const int c4n = wn / 4;
                const uint32_t tbase = smem_addr(ptile);
                for (int it = threadIdx.x - 64; it < rows * c4n; it += kDecodeWarps * 32) {
                    const int rl = static_cast<int>(rank) * rows + it / c4n;  // row in the tile
                    const int c4 = it % c4n;
                    const uint32_t off = static_cast<uint32_t>((rl * ld + 4 * c4) * 4);
                    float4 acc4 = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int r = 0; r < S; ++r) {
                        const float4 x = ld_dsmem_f4(mapa_shared(tbase + off, static_cast<uint32_t>(r)));
                        acc4.x += x.x;
                        acc4.y += x.y;
                        acc4.z += x.z;
                        acc4.w += x.w;
                    }
                    const int m = m0 + rl;
                    const int n = n0 + 4 * c4;
                    if (m >= M || n >= N) continue;
                    float o[4] = {acc4.x, acc4.y, acc4.z, acc4.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        if (n + e < N && !isfinite(o[e])) o[e] = entry_exact(A, wq, K, m, n + e);
                    }
                    float* crow = C + static_cast<int64_t>(m) * N;
                    if (c_vec) {
                        *reinterpret_cast<float4*>(crow + n) = make_float4(o[0], o[1], o[2], o[3]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            if (n + e < N) crow[n + e] = o[e];
                    }
                }
            }
            // No CTA leaves while another may still read its partial tile.
            named_barrier_sync(1, kDecodeWarps * 32);
            if (threadIdx.x == 64) {
                for (int r = 0; r < S; ++r)
                    mbar_arrive_cluster(mapa_shared(smem_addr(&red_bar[1]), static_cast<uint32_t>(r)));
            }
            mbar_wait_cluster_bounded(&red_bar[1], 0, &g_gemm_error);
        } else {
        for (int jb = 0; jb < ncb; ++jb) {
            const int col = cw * cq + 32 * jb;
            const int valid = min(32, cw - 32 * jb);  // columns of this block inside the tile
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
            if (acc_ok) {
                tc_fence_after();
                tmem_ld_acc(tmem + (static_cast<uint32_t>(32 * q) << 16) + col, BN, v);
            }
            __syncwarp();  // the previous block's reads of the staging rows are done
            // v[i]: row mrow + lane, column n0 + col + i.  Staged so that lane i
            // then holds column i of every row.
#pragma unroll
            for (int j = 0; j < 8; ++j)
                *reinterpret_cast<float4*>(stg + lane * 36 + 4 * j) =
                    make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
            __syncwarp();
            const int nn = n0 + col + lane;  // this lane's column in the row-wise passes
            {
                if (!acc_ok) continue;
                // Entries that came out non-finite: recompute element by element.
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    if (i < valid && !isfinite(v[i]) && mrow + lane < M && n0 + col + i < N)
                        stg[lane * 36 + i] = entry_exact(A, wq, K, mrow + lane, n0 + col + i);
                }
                __syncwarp();
                if (c_vec) {
                    // 8 lanes per row, 16 bytes each: 4 rows per store instruction.
                    const int c4 = lane & 7;
                    const int n4 = n0 + col + 4 * c4;
#pragma unroll
                    for (int r4 = 0; r4 < 8; ++r4) {
                        const int row = 4 * r4 + (lane >> 3);
                        const float4 x = *reinterpret_cast<const float4*>(stg + row * 36 + 4 * c4);
                        if (mrow + row < M && n4 < N && 4 * c4 < valid)
                            *reinterpret_cast<float4*>(C + static_cast<int64_t>(mrow + row) * N + n4) = x;
                    }
                } else {
                    for (int row = 0; row < 32; ++row) {
                        if (mrow + row < M && nn < N && lane < valid)
                            C[static_cast<int64_t>(mrow + row) * N + nn] = stg[row * 36 + lane];
                    }
                }
            }
        }
        }  // whole tiles
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "r"(T::kTmemCols)
                     : "memory");
    }
}

}  // namespace

bool gemm_tc_supported(const float* A, const uint8_t* wq, int64_t M, int64_t N, int64_t K) {
    // (Work items are numbered in one int: at most 2^26 tiles of 128 x 128.)
    return M >= 1 && N >= 1 && (K % 256) == 0 && K > 0 && K <= (int64_t(1) << 24) &&
           M <= (int64_t(1) << 30) && N <= (int64_t(1) << 30) &&
           ((M + BM - 1) / BM) * ((N + 127) / 128) <= (int64_t(1) << 26) &&
           (reinterpret_cast<uintptr_t>(wq) & 15u) == 0 && (reinterpret_cast<uintptr_t>(A) & 15u) == 0;
}

namespace {

// Tile width: 256 columns when M is at least 256 and N at least 2048 (or K is
// long), 128 columns otherwise.  With the activation split inside the kernel a
// 256-column tile splits each activation tile for twice the columns, and
// that decides most shapes (CUDA-graph replay on GB300): 256 x 4096 x 4096
// runs in 36.7 against 49.2 us, 512 x 4096 x 4096 in 61.7 (K split in two
// through clusters) against 83.1 us with 112-column tiles; 512 x 1024 x 4096
// stays faster with 128 columns (29.5 against 37.3 us), and so does M = 32
// (29.0 against 29.3, 36.8 us with N-wide tiles at any M).
int choose_bn(int64_t M, int64_t N, int64_t K, const DeviceInfo& /*dev*/) {
    return (M >= 256 && (N >= 2048 || K >= 8192)) ? 256 : 128;
}

// Work items for one CTA per SM.  Whole tiles fill as many full waves as they
// can; the tiles of the last, partial wave (all tiles when there are fewer
// than SMs) are split so that the last wave is not left mostly idle:
// 256-column tiles after a full wave into two 128-column halves when those fit
// the SMs (no partial sums to add), otherwise into s_rem = 2, 4 or 8 K ranges
// of whole 256-wide units, the most that fit the SMs, where the split tiles'
// clusters of s_rem CTAs can all be resident at once (fit[0..2] clusters of
// 2, 4 and 8) and the whole tiles before them come in whole clusters (a
// split adds up through its cluster); else the last wave stays whole.
struct GemmItems {
    int64_t nt, tiles, rem, n_full, items;
    int s_rem, hw;
};

GemmItems plan_gemm_items(int bn, int64_t M, int64_t N, int64_t K, int64_t P, const int fit[3]) {
    GemmItems g;
    g.nt = (N + bn - 1) / bn;
    g.tiles = g.nt * ((M + BM - 1) / BM);
    g.rem = g.tiles % P;
    g.hw = (bn == 256 && g.tiles >= P && g.rem > 0 && 2 * g.rem <= P) ? 1 : 0;
    g.s_rem = 1;
    for (int i = 0; i < 3 && !g.hw && g.rem > 0; ++i) {
        const int c = 2 << i;
        if ((K / 256) % c == 0 && g.rem * c <= P && (g.tiles - g.rem) % c == 0 && fit[i] >= g.rem)
            g.s_rem = c;
    }
    g.n_full = (g.s_rem > 1 || g.hw) ? g.tiles - g.rem : g.tiles;
    g.items = g.n_full + (g.tiles - g.n_full) * (g.hw ? 2 : g.s_rem);
    return g;
}

// 112-column tiles (with the 128-column kernel) where 128-column tiles leave
// SMs idle, need no K split, and 112-column ones fill more SMs, still without
// a split: 512 x 4096 makes 148 tiles of 112 against 128 tiles of 128 on 152
// SMs, each with 12.5% less work.
bool narrow_tiles(int64_t M, int64_t N, int64_t K, int64_t P, const int fit[3]) {
    const GemmItems g128 = plan_gemm_items(128, M, N, K, P, fit);
    const GemmItems g112 = plan_gemm_items(112, M, N, K, P, fit);
    return g128.tiles < P && g128.s_rem == 1 && g112.s_rem == 1 && g112.tiles <= P &&
           g112.tiles > g128.tiles;
}

// Resident clusters of 2, 4 and 8 CTAs of the BN kernel, queried once per
// device.
template <int BN>
cudaError_t gemm_cluster_fits(const DeviceInfo& dev, int fit[3]) {
    static int cached[64][3] = {};  // 0: not queried; else 1 + the count
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    for (int i = 0; i < 3; ++i) {
        int f = __atomic_load_n(&cached[dev.device][i], __ATOMIC_ACQUIRE);
        if (f == 0) {
            f = 1 + max_active_clusters(gemm_q4_0_tc<BN>, dim3(kThreads), Tile<BN>::kSmemBytes, 2u << i);
            __atomic_store_n(&cached[dev.device][i], f, __ATOMIC_RELEASE);
        }
        fit[i] = f - 1;
    }
    return cudaSuccess;
}

// Shared-memory attribute of the BN kernel, set once per device.
template <int BN>
cudaError_t ensure_gemm_smem_attr(const DeviceInfo& dev) {
    static int configured[64] = {0};
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    if (!__atomic_load_n(&configured[dev.device], __ATOMIC_ACQUIRE)) {
        cudaError_t e = cudaFuncSetAttribute(gemm_q4_0_tc<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Tile<BN>::kSmemBytes);
        if (e != cudaSuccess) return e;
        __atomic_store_n(&configured[dev.device], 1, __ATOMIC_RELEASE);
    }
    return cudaSuccess;
}

template <int BN>
cudaError_t launch_bn(const float* A, const uint8_t* wq, float* C, int64_t M, int64_t N, int64_t K,
                      cudaStream_t stream, const DeviceInfo& dev, int tw, const int fit[3]) {
    const GemmItems g = plan_gemm_items(tw, M, N, K, dev.sm_count, fit);
    const int64_t nt = g.nt, n_full = g.n_full, items = g.items;
    const int s_rem = g.s_rem, hw = g.hw;

    CUtensorMap map_a, map_w, map_w2;
    // Activations as f32 [M][K]; boxes of 128 rows x 64 k (256-byte rows).
    const int64_t adims[2] = {K, M};
    const int64_t astrides[1] = {K * 4};
    const int abox[2] = {BK, BM};
    cudaError_t err = encode_tiled(&map_a, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, A, 2, adims, astrides, abox);
    if (err != cudaSuccess) return err;
    // Weights as bytes [N rows][K/32 * 18 B] (a row is a multiple of 144 B,
    // so of 16 B); boxes of BN rows x 48 B, bytes past a row's end read as 0.
    const int64_t row_bytes = K / kBlockElems * kBlockBytes;
    const int64_t wdims[2] = {row_bytes, N};
    const int64_t wstrides[1] = {row_bytes};
    const int wbox[2] = {kRawRow, BN};
    err = encode_tiled(&map_w, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, 2, wdims, wstrides, wbox);
    if (err != cudaSuccess) return err;
    const int wbox2[2] = {kRawRow, BN / 2};  // half-width items
    err = encode_tiled(&map_w2, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, 2, wdims, wstrides, wbox2);
    if (err != cudaSuccess) return err;

    const int c_vec = ((reinterpret_cast<uintptr_t>(C) & 15u) == 0 && (N % 4) == 0) ? 1 : 0;
    if (s_rem > 1) {
        err = launch_pdl_cluster(gemm_q4_0_tc<BN>, dim3(static_cast<unsigned>(items)), dim3(kThreads),
                                 Tile<BN>::kSmemBytes, stream, static_cast<unsigned>(s_rem), map_a, map_w,
                                 map_w2, A, wq, C, static_cast<int>(M), static_cast<int>(N),
                                 static_cast<int>(K), c_vec, tw, static_cast<int>(nt),
                                 static_cast<int>(n_full), s_rem, hw);
    } else {
        err = launch_pdl(gemm_q4_0_tc<BN>, dim3(static_cast<unsigned>(items)), dim3(kThreads),
                         Tile<BN>::kSmemBytes, stream, map_a, map_w, map_w2, A, wq, C, static_cast<int>(M),
                         static_cast<int>(N), static_cast<int>(K), c_vec, tw, static_cast<int>(nt),
                         static_cast<int>(n_full), s_rem, hw);
    }
    if (err != cudaSuccess) return err;
    note_launch();
    return cudaSuccess;
}

}  // namespace

cudaError_t launch_gemm_q4_0_tc(const float* A, const uint8_t* wq, float* C, int64_t M, int64_t N,
                                int64_t K, cudaStream_t stream, const DeviceInfo& dev) {
    int fit[3] = {0, 0, 0};
    if (choose_bn(M, N, K, dev) == 256) {
        cudaError_t err = ensure_gemm_smem_attr<256>(dev);
        if (err == cudaSuccess) err = gemm_cluster_fits<256>(dev, fit);
        if (err != cudaSuccess) return err;
        return launch_bn<256>(A, wq, C, M, N, K, stream, dev, 256, fit);
    }
    cudaError_t err = ensure_gemm_smem_attr<128>(dev);
    if (err == cudaSuccess) err = gemm_cluster_fits<128>(dev, fit);
    if (err != cudaSuccess) return err;
    return launch_bn<128>(A, wq, C, M, N, K, stream, dev, narrow_tiles(M, N, K, dev.sm_count, fit) ? 112 : 128,
                          fit);
}

void gemm_tc_plan_query(int64_t M, int64_t N, int64_t K, int sm_count, const int fit[3], int64_t out[8]) {
    const DeviceInfo dev{0, sm_count, 0};
    int bn = choose_bn(M, N, K, dev);
    if (bn == 128 && narrow_tiles(M, N, K, sm_count, fit)) bn = 112;
    const GemmItems g = plan_gemm_items(bn, M, N, K, sm_count, fit);
    const int64_t v[8] = {bn, g.nt, g.tiles, g.n_full, g.s_rem, g.hw, g.items, g.s_rem > 1 ? 1 : 0};
    for (int i = 0; i < 8; ++i) out[i] = v[i];
}

cudaError_t gemm_tc_read_device_error(unsigned int* bits, bool clear) {
    unsigned int v = 0;
    cudaError_t err = cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(v));
    if (err != cudaSuccess) return err;
    *bits |= v;
    if (clear && v != 0) {
        const unsigned int zero = 0;
        err = cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(zero));
    }
    return err;
}

}  // namespace qm

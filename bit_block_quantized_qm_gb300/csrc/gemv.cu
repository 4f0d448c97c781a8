// Decode-regime GEMV: C[m][n] = sum_k A[m][k] * W[n][k] for M = 1..8 rows of
// f32 activations against a Q4_0 weight stream (sections "qmatvec_q4_0" and
// "matmul_q4_0_tiled" of "fuel-vulkan-kernels — quantized (GGML) kernel
// contracts"; element j < 16 of a block is the low nibble of quant byte j,
// element j + 16 its high nibble, value (nibble - 8) * d).
//
// This file holds the FP32 FMA kernels; the tensor-core GEMV is in gemv_tc.cu.
//
// Persistent kernel (K % 256 == 0, 16-byte aligned wq and A):
//   * A "unit" is 8 consecutive blocks of one weight row: 144 bytes = 9
//     aligned 16-byte words covering 256 k.  A "row group" is 32 rows.  The
//     work is the grid of (row group, unit) tiles; the launch splits it into
//     G row-group ranges x S unit ranges, one CTA (one per SM) for each,
//     sized so every CTA gets nearly the same number of tiles.
//   * In each CTA a producer warp streams the CTA's 32-row x 144-byte tiles
//     into a ring of shared-memory stages with 2-D TMA loads (and the CTA's
//     activation slice with 1-D bulk copies), so HBM latency overlaps the
//     decode of earlier tiles.  Eight consumer warps take tiles in turn.
//   * Lane l of a consumer warp owns row l of the tile.  It reads its row's
//     unit with nine 16-byte shared loads (the 144-byte row stride sends the
//     8 lanes of each quarter-warp to 8 distinct 4-bank groups) and decodes
//     the 8 blocks with fixed byte permutes; the activations are broadcast
//     16-byte shared loads.  Nibbles are masked in place, moved under the
//     exponent of 2^23 with one byte permute and turned into (q - 8) by one
//     subtraction, all exact; 32 products are summed per block and scaled
//     once by d (element by element when d is not finite).
//   * Partial sums of a row group meet in shared memory (fixed warp order).
//     When K is split (S > 1: only with scratch memory, which the regular
//     entry point does not give this kernel) each CTA writes its row groups'
//     partials to the scratch and the last of the S CTAs to arrive at a row
//     group adds them in split order and writes C, so results do not depend
//     on timing.
// Generic kernel (any K % 32 == 0, 2-byte aligned wq, 4-byte aligned A): one
// warp per row, lanes striding over blocks, shuffle reduction.
#include <algorithm>
#include <mutex>

#include "qm_device.cuh"
#include "qm_internal.h"

namespace qm {

__device__ unsigned int g_gemv_error = 0;

namespace {

constexpr int kUnitBytes = 144;  // 8 blocks
constexpr int kUnitElems = 256;
constexpr int kRowsPerTile = 32;  // one row per lane
constexpr int kTileBytes = kUnitBytes * kRowsPerTile;
// Consumer warps per CTA: as many as the registers of one CTA per SM allow.
template <int M>
__host__ __device__ constexpr int consumer_warps() { return M <= 4 ? 16 : 8; }
template <int M>
__host__ __device__ constexpr int cta_threads() {
    return (consumer_warps<M>() + 1) * 32;  // + producer warp
}
constexpr int kMaxSplits = 16;  // at most 16 K ranges
constexpr int kMaxRowGroupsPerCta = 16;

// Where block_dot reads activations from.
enum class ASrc { kGlobalVec, kGlobalScalar, kShared };

template <ASrc kSrc>
__device__ __forceinline__ float4 load_a4(const float* p) {
    if constexpr (kSrc == ASrc::kGlobalVec) {
        return __ldg(reinterpret_cast<const float4*>(p));
    } else if constexpr (kSrc == ASrc::kShared) {
        return *reinterpret_cast<const float4*>(p);
    } else {
        return make_float4(__ldg(p), __ldg(p + 1), __ldg(p + 2), __ldg(p + 3));
    }
}

// t[m] = sum over the 32 elements of one block of A[m][k0 + j] * (q_j - 8),
// with row m of the activations at A + m * lda.  q[w] holds quant bytes
// 4w..4w+3 (byte 4w in the low 8 bits).
template <int M, ASrc kSrc>
__device__ __forceinline__ void block_dot(const float* __restrict__ A, int64_t lda, int64_t k0,
                                          const uint32_t q[4], float t[M]) {
    // Independent FMA chains per activation row (more when M is small) so a
    // warp keeps several multiply-adds in flight.
    constexpr int kChains = (M == 1) ? 4 : (M <= 3 ? 2 : 1);
    float c[M][kChains];
#pragma unroll
    for (int m = 0; m < M; ++m)
#pragma unroll
        for (int h = 0; h < kChains; ++h) c[m][h] = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint32_t lo = q[w] & 0x0F0F0F0Fu;         // elements 4w .. 4w+3
        const uint32_t hi = (q[w] >> 4) & 0x0F0F0F0Fu;  // elements 16+4w .. 16+4w+3
        float v[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            v[e] = magic_minus8(__byte_perm(lo, kMagicBits, 0x7540u + e));
            v[4 + e] = magic_minus8(__byte_perm(hi, kMagicBits, 0x7540u + e));
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const float* am = A + m * lda + k0 + 4 * w;
            const float4 al = load_a4<kSrc>(am);
            const float4 ah = load_a4<kSrc>(am + 16);
            const float a[8] = {al.x, al.y, al.z, al.w, ah.x, ah.y, ah.z, ah.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) c[m][e % kChains] = fmaf(a[e], v[e], c[m][e % kChains]);
        }
    }
#pragma unroll
    for (int m = 0; m < M; ++m) {
        float x = c[m][0];
#pragma unroll
        for (int h = 1; h < kChains; ++h) x += c[m][h];
        t[m] = x;
    }
}

// The block's contribution taken element by element, sum_j A[m][k0+j] *
// ((q_j - 8) * d).  Used only when d is infinite or NaN: there the factored
// form d * sum_j A_j (q_j - 8) can lose the NaN that a zero weight (q = 8)
// times an infinite d, or infinities of both signs, put into the sum.
template <int M, ASrc kSrc>
__device__ __noinline__ void block_exact(const float* __restrict__ A, int64_t lda, int64_t k0,
                                         const uint32_t q[4], float d, float t[M]) {
#pragma unroll
    for (int m = 0; m < M; ++m) t[m] = 0.f;
    for (int j = 0; j < 32; ++j) {
        const int byte = j & 15;
        const uint32_t b = (q[byte >> 2] >> (8 * (byte & 3))) & 0xFFu;
        const uint32_t nib = (j < 16) ? (b & 0xFu) : (b >> 4);
        const float w = magic_minus8(nib | kMagicBits) * d;
#pragma unroll
        for (int m = 0; m < M; ++m) {
            float a;
            if constexpr (kSrc == ASrc::kShared) {
                a = A[m * lda + k0 + j];
            } else {
                a = __ldg(A + m * lda + k0 + j);
            }
            t[m] = fmaf(a, w, t[m]);
        }
    }
}

// acc[m] += d * t[m], or the exact per-element sum when d is not finite.
template <int M, ASrc kSrc>
__device__ __forceinline__ void scale_block(const float* __restrict__ A, int64_t lda, int64_t k0,
                                            const uint32_t q[4], float d, const float t[M],
                                            float acc[M]) {
    if (isfinite(d)) {
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m] = fmaf(d, t[m], acc[m]);
    } else {
        float e[M];
        block_exact<M, kSrc>(A, lda, k0, q, d, e);
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m] += e[m];
    }
}

// One 144-byte unit (8 blocks) of one row, 16-byte aligned in shared memory.
// Blocks come in pairs of 36 bytes = 9 words: the even block's d is the low
// half of word 0 and its quants are bytes 2..17 (realigned with byte
// permutes); the odd block's d is the high half of word 4 and its quants are
// words 5..8.
template <int M>
__device__ __forceinline__ void unit_dot(const uint8_t* tile_row, const float* __restrict__ A,
                                         int64_t lda, int64_t kbase, float acc[M]) {
    uint32_t w[36];
    const uint4* src = reinterpret_cast<const uint4*>(tile_row);
#pragma unroll
    for (int i = 0; i < 9; ++i) {
        const uint4 v = src[i];
        w[4 * i + 0] = v.x;
        w[4 * i + 1] = v.y;
        w[4 * i + 2] = v.z;
        w[4 * i + 3] = v.w;
    }
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        const uint32_t* W = w + 9 * p;
        float t[M];
        const uint32_t qa[4] = {__byte_perm(W[0], W[1], 0x5432u), __byte_perm(W[1], W[2], 0x5432u),
                                __byte_perm(W[2], W[3], 0x5432u), __byte_perm(W[3], W[4], 0x5432u)};
        block_dot<M, ASrc::kShared>(A, lda, kbase + 64 * p, qa, t);
        const float da = f16_bits_to_float(W[0] & 0xFFFFu);
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m] = fmaf(da, t[m], acc[m]);
        const uint32_t qb[4] = {W[5], W[6], W[7], W[8]};
        block_dot<M, ASrc::kShared>(A, lda, kbase + 64 * p + 32, qb, t);
        const float db = f16_bits_to_float(W[4] >> 16);
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m] = fmaf(db, t[m], acc[m]);
    }
}

// Work decomposition of one persistent launch.
struct GemvGrid {
    const uint8_t* wq;  // the weight stream (read directly only by the exact fix-up)
    int N;
    int64_t K;
    int U;          // units per row, K / 256
    int RG;         // row groups, ceil(N / 32)
    int S;          // unit ranges (K splits); U is a multiple of S
    int nu;         // units per range, U / S
    int uc;         // units per stage (a divisor of nu): a stage is 32 rows x uc units
    int box0;       // units in the first TMA box of a stage (the second has uc - box0)
    int rpg;        // row groups per range of rows
    int stages;     // ring depth in row-group stages
    float* part;    // [RG][S][M][32] split partial sums (S > 1)
    unsigned* ctr;  // [RG] arrival counters (S > 1), zero between launches
};

template <int M>
__global__ void __launch_bounds__(cta_threads<M>(), 1)
    gemv_q4_0_persistent(const __grid_constant__ CUtensorMap map0,
                         const __grid_constant__ CUtensorMap map1, const float* __restrict__ A,
                         float* __restrict__ C, const GemvGrid g) {
    constexpr int W = consumer_warps<M>();
    extern __shared__ __align__(128) uint8_t smem[];
    // ring [stages][32 rows x nu units x 144 B] (first box0 units of every row,
    // then the rest) | activations f32 [M][nu * 256] | partial sums
    // [rpg][slots][M][32] | full[stages] | empty[stages] | a_bar | seq[stages]
    const int stage_bytes = kTileBytes * g.uc;
    uint8_t* ring = smem;
    float* a_s = reinterpret_cast<float*>(smem + g.stages * stage_bytes);
    const int lda = g.nu * kUnitElems;
    // Row group r's tiles go to warps (r * nu + j) % W, j < nu: min(nu, W)
    // distinct warps, each with its own partial-sum slot.
    const int slots = min(g.nu, W);
    float* partial = a_s + M * lda;
    uint64_t* full = reinterpret_cast<uint64_t*>(partial + g.rpg * slots * M * 32);
    uint64_t* empty = full + g.stages;
    uint64_t* a_bar = empty + g.stages;
    // seq[st]: the chunk the producer last issued into stage st.  A warp waits
    // for its chunk's number before the parity wait on full[st], so it can
    // never mistake an older phase of the stage for its own.
    volatile int* seq = reinterpret_cast<volatile int*>(a_bar + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int split = static_cast<int>(blockIdx.x) % g.S;
    const int rg0 = (static_cast<int>(blockIdx.x) / g.S) * g.rpg;
    const int nrg = max(0, min(g.rpg, g.RG - rg0));
    const int u0 = split * g.nu;
    const int nu = g.nu;
    const int uc = g.uc;
    const int chunks = nu / uc;  // stages per row group
    const int box1 = uc - g.box0;
    const int items = nrg * nu;

    for (int i = threadIdx.x; i < g.rpg * slots * M * 32; i += blockDim.x) partial[i] = 0.f;
    if (threadIdx.x == 0) {
        for (int s = 0; s < g.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], uc);  // one arrival per consumed tile
            seq[s] = -1;
        }
        mbar_init(a_bar, 1);
        fence_barrier_init();
    }
    __syncthreads();

    if (warp == W) {
        // Producer: the activation slice, then one row group per stage.
        if (lane == 0 && items > 0) {
            prefetch_tensormap(&map0);
            if (box1 > 0) prefetch_tensormap(&map1);
            const uint32_t a_bytes = static_cast<uint32_t>(nu) * kUnitElems * 4;
            mbar_arrive_expect_tx(a_bar, a_bytes * M);
            for (int m = 0; m < M; ++m)
                bulk_load_1d(a_s + m * lda, A + m * g.K + static_cast<int64_t>(u0) * kUnitElems,
                             a_bytes, a_bar);
            // Chunk c = (row group c / chunks, units [(c % chunks) * uc, +uc)).
            for (int c = 0; c < nrg * chunks; ++c) {
                const int st = c % g.stages;
                if (c >= g.stages &&
                    !mbar_wait_bounded(&empty[st], ((c / g.stages) - 1) & 1, &g_gemv_error))
                    break;
                uint8_t* dst = ring + st * stage_bytes;
                const int row = (rg0 + c / chunks) * kRowsPerTile;
                const int ub = u0 + (c % chunks) * uc;
                seq[st] = c;
                mbar_arrive_expect_tx(&full[st], stage_bytes);
                tma_load_3d(dst, &map0, 0, ub, row, &full[st]);
                if (box1 > 0)
                    tma_load_3d(dst + kTileBytes * g.box0, &map1, 0, ub + g.box0, row, &full[st]);
            }
        }
    } else if (items > 0 && mbar_wait_bounded(a_bar, 0, &g_gemv_error)) {
        // Consumers: tile i (row group i / nu, unit i % nu) goes to warp i % W.
        float acc[M];
        int cur = -1;
        auto flush = [&](int r) {
            const int slot = (g.nu >= W) ? warp : ((warp - (r * g.nu) % W) + W) % W;
            float* pw = partial + (r * slots + slot) * M * 32;
#pragma unroll
            for (int m = 0; m < M; ++m) pw[m * 32 + lane] += acc[m];
        };
        for (int i = warp; i < items; i += W) {
            const int r = i / nu;
            const int j = i - r * nu;
            if (r != cur) {
                if (cur >= 0) flush(cur);
#pragma unroll
                for (int q = 0; q < M; ++q) acc[q] = 0.f;
                cur = r;
            }
            const int c = i / uc;  // chunk (items of a chunk are consecutive)
            const int jc = i - c * uc;
            const int st = c % g.stages;
            bool issued = false;
            for (uint32_t poll = 0; poll < kMaxWaitPolls; ++poll) {
                if (seq[st] == c) {
                    issued = true;
                    break;
                }
                __nanosleep(32);
            }
            if (!issued) atomicOr(&g_gemv_error, kErrWaitTimeout);
            if (issued && mbar_wait_bounded(&full[st], (c / g.stages) & 1, &g_gemv_error)) {
                const uint8_t* base = ring + st * stage_bytes;
                // Start of the tile's unit (jc of this stage) in tile row `row`.
                auto row_unit = [&](int row) -> const uint8_t* {
                    return (jc < g.box0)
                               ? base + (row * g.box0 + jc) * kUnitBytes
                               : base + kTileBytes * g.box0 + (row * box1 + (jc - g.box0)) * kUnitBytes;
                };
                unit_dot<M>(row_unit(lane), a_s, lda, j * kUnitElems, acc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[st]);
        }
        if (cur >= 0) flush(cur);
    }
    __syncthreads();

    // Row-group totals in fixed slot order; split partials meet in the workspace.
    if (warp < W) {
        for (int r = warp; r < nrg; r += W) {
            const int row = (rg0 + r) * kRowsPerTile + lane;
            float tot[M];
#pragma unroll
            for (int m = 0; m < M; ++m) {
                float v = 0.f;
                for (int q = 0; q < slots; ++q) v += partial[((r * slots + q) * M + m) * 32 + lane];
                tot[m] = v;
            }
            if (row < g.N) {
                const uint8_t* row_blocks =
                    g.wq + (static_cast<int64_t>(row) * g.U + u0) * kUnitBytes;
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    if (!isfinite(tot[m]))
                        tot[m] = row_range_exact(row_blocks, nu * 8,
                                                 A + m * g.K + static_cast<int64_t>(u0) * kUnitElems);
                }
            }
            if (g.S == 1) {
                if (row < g.N) {
#pragma unroll
                    for (int m = 0; m < M; ++m) C[static_cast<int64_t>(m) * g.N + row] = tot[m];
                }
                continue;
            }
            const int64_t rg = rg0 + r;
            float* slot = g.part + (rg * g.S + split) * (M * 32);
#pragma unroll
            for (int m = 0; m < M; ++m) slot[m * 32 + lane] = tot[m];
            __threadfence();
            __syncwarp();
            unsigned old = 0;
            if (lane == 0) old = atomicAdd(&g.ctr[rg], 1u);
            old = __shfl_sync(0xFFFFFFFFu, old, 0);
            if (old == static_cast<unsigned>(g.S - 1)) {
                __threadfence();
#pragma unroll
                for (int m = 0; m < M; ++m) {
                    float v = 0.f;
                    for (int q = 0; q < g.S; ++q)
                        v += __ldcg(g.part + (rg * g.S + q) * (M * 32) + m * 32 + lane);
                    if (row < g.N) C[static_cast<int64_t>(m) * g.N + row] = v;
                }
                if (lane == 0) atomicExch(&g.ctr[rg], 0u);
            }
        }
    }
}

template <int M>
__global__ void __launch_bounds__(256)
    gemv_q4_0_generic(const float* __restrict__ A, const uint8_t* __restrict__ wq,
                      float* __restrict__ C, int64_t N, int64_t K) {
    const int lane = threadIdx.x & 31;
    const int64_t warps_total = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
    const int64_t nb = K / kBlockElems;
    for (int64_t n = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
         n < N; n += warps_total) {
        float acc[M];
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m] = 0.f;
        for (int64_t b = lane; b < nb; b += 32) {
            const uint16_t* h = reinterpret_cast<const uint16_t*>(wq + (n * nb + b) * kBlockBytes);
            uint32_t q[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                q[w] = static_cast<uint32_t>(h[1 + 2 * w]) |
                       (static_cast<uint32_t>(h[2 + 2 * w]) << 16);
            }
            float t[M];
            block_dot<M, ASrc::kGlobalScalar>(A, K, b * kBlockElems, q, t);
            const float d = f16_bits_to_float(h[0]);
            scale_block<M, ASrc::kGlobalScalar>(A, K, b * kBlockElems, q, d, t, acc);
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1)
                acc[m] += __shfl_xor_sync(0xFFFFFFFFu, acc[m], off);
        }
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < M; ++m) C[m * N + n] = acc[m];
        }
    }
}

// Per-device one-time opt-in to large dynamic shared memory.
template <int M>
cudaError_t ensure_smem_attr(const DeviceInfo& dev, int bytes) {
    static int configured[64] = {0};
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    if (bytes > dev.max_smem_optin) return cudaErrorInvalidValue;
    if (__atomic_load_n(&configured[dev.device], __ATOMIC_ACQUIRE)) return cudaSuccess;
    cudaError_t err = cudaFuncSetAttribute(gemv_q4_0_persistent<M>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           dev.max_smem_optin);
    if (err != cudaSuccess) return err;
    __atomic_store_n(&configured[dev.device], 1, __ATOMIC_RELEASE);
    return cudaSuccess;
}

int64_t smem_bytes(int M, int W, int stages, int uc, int nu, int rpg) {
    return static_cast<int64_t>(stages) * kTileBytes * uc +
           static_cast<int64_t>(M) * nu * kUnitElems * 4 +
           static_cast<int64_t>(rpg) * std::min(nu, W) * M * 32 * 4 + (2 * stages + 1) * 8 +
           stages * 4;
}

// Split a stage's nu units into at most two TMA boxes whose widths keep the
// 144-byte row stride from piling the lanes of a quarter-warp onto one bank
// group: an odd width is conflict-free, 2 mod 4 is two-way.
int first_box(int nu) {
    if (nu % 4 != 0) return nu;
    return nu / 2 - 1;  // nu / 2 is even, so both halves become odd
}

// Choose (G row-group ranges) x (S unit ranges) for one CTA per SM.  The
// largest share (rpg * nu tiles, times the number of waves) decides; among
// shapes whose stages are at least kMinStageBytes (small TMA copies stream
// poorly), the cheapest wins, fewer splits breaking ties.
constexpr int64_t kMinStageBytes = 16 * 1024;

bool plan_grid(int M, int W, int64_t N, int64_t K, const DeviceInfo& dev,
               const Workspace& ws, GemvGrid* g, int* grid, int* smem) {
    const int U = static_cast<int>(K / kUnitElems);
    const int64_t RG = (N + kRowsPerTile - 1) / kRowsPerTile;
    const int P = dev.sm_count;
    int64_t best[2] = {INT64_MAX, INT64_MAX};  // [small stages, big stages]
    GemvGrid cand[2];
    int cgrid[2] = {0, 0}, csmem[2] = {0, 0};
    for (int S = 1; S <= kMaxSplits && S <= U; ++S) {
        if (U % S != 0) continue;
        const int nu = U / S;
        if (nu > 2 * 255) continue;
        const int G = std::max(1, P / S);
        const int64_t rpg = std::min<int64_t>((RG + G - 1) / G, kMaxRowGroupsPerCta);
        const int64_t g_used = (RG + rpg - 1) / rpg;
        // Stage = 32 rows x uc units.  Halve uc while the stage stays at least
        // kMinStageBytes and the ring would hold fewer than four stages, so
        // more copies stay in flight and refills start sooner.
        int uc = nu;
        auto fit = [&](int u) {
            int st = 8;
            while (st > 1 && smem_bytes(M, W, st, u, nu, static_cast<int>(rpg)) > dev.max_smem_optin)
                --st;
            return smem_bytes(M, W, st, u, nu, static_cast<int>(rpg)) <= dev.max_smem_optin ? st : 0;
        };
        int stages = fit(uc);
        while (uc % 2 == 0 && static_cast<int64_t>(kTileBytes) * (uc / 2) >= kMinStageBytes &&
               stages < 4 && fit(uc / 2) > stages) {
            uc /= 2;
            stages = fit(uc);
        }
        if (stages == 0) continue;
        if (stages < 2 && rpg * (nu / uc) > 1) continue;
        if (S > 1 && (RG * S * M * 32 > static_cast<int64_t>(ws.part_floats) ||
                      RG > static_cast<int64_t>(ws.ctr_count)))
            continue;
        const int64_t waves = (g_used * S + P - 1) / P;
        const int64_t cost = rpg * nu * waves;
        const int big = (static_cast<int64_t>(kTileBytes) * uc >= kMinStageBytes) ? 1 : 0;
        if (cost < best[big]) {
            best[big] = cost;
            GemvGrid& c = cand[big];
            c.wq = nullptr;
            c.N = static_cast<int>(N);
            c.K = K;
            c.U = U;
            c.RG = static_cast<int>(RG);
            c.S = S;
            c.nu = nu;
            c.uc = uc;
            c.box0 = first_box(uc);
            c.rpg = static_cast<int>(rpg);
            c.stages = stages;
            c.part = ws.part;
            c.ctr = ws.ctr;
            cgrid[big] = static_cast<int>(g_used * S);
            csmem[big] = static_cast<int>(smem_bytes(M, W, stages, uc, nu, static_cast<int>(rpg)));
        }
    }
    const int pick = (best[1] != INT64_MAX) ? 1 : 0;
    if (best[pick] == INT64_MAX) return false;
    *g = cand[pick];
    *grid = cgrid[pick];
    *smem = csmem[pick];
    return g->box0 <= 255 && g->uc - g->box0 <= 255;
}

// Whether the persistent kernel can take this operand layout at all.
bool persistent_ok(const float* A, const uint8_t* wq, int64_t N, int64_t K) {
    const int64_t units = K / kUnitElems;
    return (K % kUnitElems) == 0 && units > 0 && (reinterpret_cast<uintptr_t>(wq) & 15u) == 0 &&
           (reinterpret_cast<uintptr_t>(A) & 15u) == 0 && N <= (int64_t(1) << 30) &&
           units <= (int64_t(1) << 20);
}

// Plan and launch the persistent kernel with split-K scratch `ws`.  Sets
// *launched = false (and launches nothing) when no plan fits.  With
// clear_counters the row-group counters are zeroed on the stream first.
template <int M>
cudaError_t launch_persistent(const float* A, const uint8_t* wq, float* C, int64_t N, int64_t K,
                              cudaStream_t stream, const DeviceInfo& dev, const Workspace& ws,
                              bool clear_counters, bool* launched) {
    *launched = false;
    GemvGrid g;
    int grid = 0, smem = 0;
    if (!plan_grid(M, consumer_warps<M>(), N, K, dev, ws, &g, &grid, &smem))
        return cudaSuccess;
    g.wq = wq;
    cudaError_t err = ensure_smem_attr<M>(dev, smem);
    if (err != cudaSuccess) return err;
    if (clear_counters && g.S > 1) {
        err = cudaMemsetAsync(g.ctr, 0, static_cast<size_t>(g.RG) * sizeof(unsigned), stream);
        if (err != cudaSuccess) return err;
    }
    // The weight stream as bytes [N rows][U units][144 B]; boxes of
    // 32 rows x box units x 144 B.
    const int64_t units = K / kUnitElems;
    const int64_t dims[3] = {kUnitBytes, units, N};
    const int64_t strides[2] = {kUnitBytes, units * kUnitBytes};
    CUtensorMap map0, map1;
    const int box_a[3] = {kUnitBytes, g.box0, kRowsPerTile};
    err = encode_tiled(&map0, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, 3, dims, strides, box_a);
    if (err != cudaSuccess) return err;
    map1 = map0;
    if (g.uc > g.box0) {
        const int box_b[3] = {kUnitBytes, g.uc - g.box0, kRowsPerTile};
        err = encode_tiled(&map1, CU_TENSOR_MAP_DATA_TYPE_UINT8, wq, 3, dims, strides, box_b);
        if (err != cudaSuccess) return err;
    }
    gemv_q4_0_persistent<M><<<grid, cta_threads<M>(), smem, stream>>>(map0, map1, A, C, g);
    note_launch();
    *launched = true;
    return cudaGetLastError();
}

template <int M>
cudaError_t launch_generic(const float* A, const uint8_t* wq, float* C, int64_t N, int64_t K,
                           cudaStream_t stream, const DeviceInfo& dev) {
    const int64_t ctas = (N + 7) / 8;
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * 16;
    const unsigned grid = static_cast<unsigned>(ctas < cap ? ctas : cap);
    gemv_q4_0_generic<M><<<grid, 256, 0, stream>>>(A, wq, C, N, K);
    note_launch();
    return cudaGetLastError();
}

template <int M>
cudaError_t launch_m(const float* A, const uint8_t* wq, float* C, int64_t N, int64_t K,
                     cudaStream_t stream, const DeviceInfo& dev, GemvKind kind) {
    if (persistent_ok(A, wq, N, K)) {
        // No scratch: the FP32 FMA kernel then takes whole K ranges, and the
        // staged GEMV adds a split K up through thread-block clusters.
        const Workspace none;
        bool launched = false;
        cudaError_t err = kind == GemvKind::kSimt
                              ? launch_persistent<M>(A, wq, C, N, K, stream, dev, none, false, &launched)
                              : launch_gemv_q4_0_tc(A, wq, C, M, N, K, stream, dev, nullptr,
                                                    kind == GemvKind::kPacked, false, &launched);
        if (err != cudaSuccess || launched) return err;
    }
    return launch_generic<M>(A, wq, C, N, K, stream, dev);
}

}  // namespace

cudaError_t launch_gemv_q4_0(const float* A, const uint8_t* wq, float* C, int M, int64_t N,
                             int64_t K, cudaStream_t stream, const DeviceInfo& dev, GemvKind kind) {
    switch (M) {
        case 1: return launch_m<1>(A, wq, C, N, K, stream, dev, kind);
        case 2: return launch_m<2>(A, wq, C, N, K, stream, dev, kind);
        case 3: return launch_m<3>(A, wq, C, N, K, stream, dev, kind);
        case 4: return launch_m<4>(A, wq, C, N, K, stream, dev, kind);
        case 5: return launch_m<5>(A, wq, C, N, K, stream, dev, kind);
        case 6: return launch_m<6>(A, wq, C, N, K, stream, dev, kind);
        case 7: return launch_m<7>(A, wq, C, N, K, stream, dev, kind);
        case 8: return launch_m<8>(A, wq, C, N, K, stream, dev, kind);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t gemv_read_device_error(unsigned int* bits, bool clear) {
    unsigned int v = 0;
    cudaError_t err = cudaMemcpyFromSymbol(&v, g_gemv_error, sizeof(v));
    if (err != cudaSuccess) return err;
    *bits |= v;
    if (clear && v != 0) {
        const unsigned int zero = 0;
        err = cudaMemcpyToSymbol(g_gemv_error, &zero, sizeof(zero));
    }
    return err;
}

// ---------------------------------------------------------------------------
// Allocation-free variant (qm_matmul_q4_0_noalloc).  Some callers cannot call
// cudaMalloc: code that runs where the CUDA allocator is off limits (inside a
// custom allocator or memory-pool callback, under a process-wide memory cap,
// or in a runtime that owns all device memory and forbids stray allocations).
// For them the split-K GEMV takes its scratch from this fixed array.  (The
// regular entry point allocates nothing either: it adds split K ranges up
// through thread-block clusters.  This entry point keeps its own split, which
// needs no cluster launch.)  Every GPU that loads the library holds the array
// until the process exits; all calls share it.
static __device__ __align__(256) float g_noalloc_scratch[kNoallocPartFloats + kNoallocCounters];

namespace {

// Device address of g_noalloc_scratch, found once per device with that device
// current.  (In host code the array's name is only a host-side stand-in.)  The
// address belongs to the device's context: after cudaDeviceReset the next call
// gets a new context, with the module loaded anew, so the address is looked
// up again when the current context is not the one it was found in.
void* g_noalloc_addr[64] = {nullptr};
CUcontext g_noalloc_ctx[64] = {nullptr};
std::mutex g_noalloc_mutex;

using CtxGetCurrent = CUresult (*)(CUcontext*);

CUcontext current_context() {
    static CtxGetCurrent fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return static_cast<CtxGetCurrent>(nullptr);
        return reinterpret_cast<CtxGetCurrent>(f);
    }();
    CUcontext ctx = nullptr;
    if (fn) fn(&ctx);
    return ctx;
}

cudaError_t noalloc_workspace(const DeviceInfo& dev, Workspace* out) {
    if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    const CUcontext ctx = current_context();
    if (!g_noalloc_addr[dev.device] || g_noalloc_ctx[dev.device] != ctx) {
        void* p = nullptr;
        cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (err != cudaSuccess) return err;
        g_noalloc_addr[dev.device] = p;
        g_noalloc_ctx[dev.device] = ctx;
    }
    float* base = static_cast<float*>(g_noalloc_addr[dev.device]);
    out->part = base;
    out->part_floats = kNoallocPartFloats;
    out->ctr = reinterpret_cast<unsigned*>(base + kNoallocPartFloats);
    out->ctr_count = kNoallocCounters;
    return cudaSuccess;
}

template <int M>
cudaError_t launch_m_noalloc(const float* A, const uint8_t* wq, float* C, int64_t N, int64_t K,
                             cudaStream_t stream, const DeviceInfo& dev) {
    if (persistent_ok(A, wq, N, K)) {
        Workspace ws;
        cudaError_t err = noalloc_workspace(dev, &ws);
        if (err != cudaSuccess) return err;
        // The arrival counters must start at zero; the array keeps whatever
        // the previous call (or an abandoned one) left, so clear them first.
        bool launched = false;
        err = launch_gemv_q4_0_tc(A, wq, C, M, N, K, stream, dev, &ws,
                                  gemv_auto_kind(M, N, K) == GemvKind::kPacked, true, &launched);
        if (err != cudaSuccess || launched) return err;
    }
    return launch_generic<M>(A, wq, C, N, K, stream, dev);
}

}  // namespace

cudaError_t launch_gemv_q4_0_noalloc(const float* A, const uint8_t* wq, float* C, int M, int64_t N,
                                     int64_t K, cudaStream_t stream, const DeviceInfo& dev) {
    switch (M) {
        case 1: return launch_m_noalloc<1>(A, wq, C, N, K, stream, dev);
        case 2: return launch_m_noalloc<2>(A, wq, C, N, K, stream, dev);
        case 3: return launch_m_noalloc<3>(A, wq, C, N, K, stream, dev);
        case 4: return launch_m_noalloc<4>(A, wq, C, N, K, stream, dev);
        case 5: return launch_m_noalloc<5>(A, wq, C, N, K, stream, dev);
        case 6: return launch_m_noalloc<6>(A, wq, C, N, K, stream, dev);
        case 7: return launch_m_noalloc<7>(A, wq, C, N, K, stream, dev);
        case 8: return launch_m_noalloc<8>(A, wq, C, N, K, stream, dev);
        default: return cudaErrorInvalidValue;
    }
}

// ---------------------------------------------------------------------------
// Failure-path self-test (qm_selftest_wait_timeout): one thread waits, with a
// short bound, on an mbarrier whose phase nothing completes.  The wait gives
// up, sets the device error word the other kernels use, and the kernel
// returns: the host then sees QM_ERR_TIMEOUT and the context stays usable.
// No asynchronous copy is in flight, so returning early leaves nothing behind.
constexpr uint32_t kSelftestPolls = 1u << 16;

__global__ void wait_timeout_selftest(uint32_t polls) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_barrier_init();
    for (uint32_t i = 0; i < polls; ++i) {
        if (mbar_try_wait(&bar, 0)) return;
    }
    atomicOr(&g_gemv_error, kErrWaitTimeout);
}

cudaError_t launch_wait_timeout_selftest(cudaStream_t stream) {
    wait_timeout_selftest<<<1, 32, 0, stream>>>(kSelftestPolls);
    note_launch();
    return cudaGetLastError();
}

}  // namespace qm

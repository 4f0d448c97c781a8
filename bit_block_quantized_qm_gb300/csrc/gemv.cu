// Decode-regime GEMV: C[m][n] = sum_k A[m][k] * W[n][k] for M = 1..8 rows of
// f32 activations against a Q4_0 weight stream (sections "qmatvec_q4_0" and
// "matmul_q4_0_tiled" of "fuel-vulkan-kernels — quantized (GGML) kernel
// contracts"; element j < 16 of a block is the low nibble of quant byte j,
// element j + 16 its high nibble, value (nibble - 8) * d).
//
// Fast kernel (K % 256 == 0, 16-byte aligned wq and A):
//   * A "unit" is 8 consecutive blocks of one weight row: 144 bytes = 9
//     aligned 16-byte words covering 256 k.  A CTA owns 32 rows and a range of
//     units; each unit's 32 x 144-byte tile is brought into shared memory by
//     one 2-D TMA load, so HBM sees whole-line reads and the SM spends no load
//     instructions on the weight stream.
//   * Lane l of every warp owns row l.  It reads its row's unit with nine
//     16-byte shared loads (a 144-byte row stride maps the 8 lanes of each
//     quarter-warp to 8 distinct 4-bank groups: conflict-free) and decodes
//     the 8 blocks with fixed byte permutes.  All lanes of a warp use the same
//     activations, so A is read with broadcast 16-byte loads.
//   * Decode: nibbles are masked in place, moved under the exponent of 2^23
//     with one byte-permute each and turned into (q - 8) by one subtraction,
//     all exact; 32 products are summed per block and scaled once by d.
//   * K is split over the CTAs of a thread-block cluster when there are too
//     few row groups to fill the GPU; partial sums are combined in a fixed
//     order through distributed shared memory, so results are deterministic.
// Generic kernel (any K % 32 == 0, 2-byte aligned wq, 4-byte aligned A): one
// warp per row, lanes striding over blocks, shuffle reduction.
#include <cooperative_groups.h>

#include "qm_device.cuh"
#include "qm_internal.h"

namespace cg = cooperative_groups;

namespace qm {

__device__ unsigned int g_gemv_error = 0;

namespace {

constexpr int kUnitBytes = 144;  // 8 blocks
constexpr int kUnitElems = 256;
constexpr int kRowsPerCta = 32;  // one row per lane
constexpr int kTileBytes = kUnitBytes * kRowsPerCta;
constexpr int kMaxUnitsPerCta = 40;  // 184 KB of tiles
constexpr int kMaxCluster = 8;

template <bool kVecA>
__device__ __forceinline__ float4 load_a4(const float* p) {
    if constexpr (kVecA) {
        return __ldg(reinterpret_cast<const float4*>(p));
    } else {
        return make_float4(__ldg(p), __ldg(p + 1), __ldg(p + 2), __ldg(p + 3));
    }
}

// t[m] = sum over the 32 elements of one block of A[m][k0 + j] * (q_j - 8).
// q[w] holds quant bytes 4w..4w+3 (byte 4w in the low 8 bits).
template <int M, bool kVecA>
__device__ __forceinline__ void block_dot(const float* __restrict__ A, int64_t K, int64_t k0,
                                          const uint32_t q[4], float t[M]) {
#pragma unroll
    for (int m = 0; m < M; ++m) t[m] = 0.f;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint32_t lo = q[w] & 0x0F0F0F0Fu;         // elements 4w .. 4w+3
        const uint32_t hi = (q[w] >> 4) & 0x0F0F0F0Fu;  // elements 16+4w .. 16+4w+3
        float vl[4], vh[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            vl[c] = magic_minus8(__byte_perm(lo, kMagicBits, 0x7540u + c));
            vh[c] = magic_minus8(__byte_perm(hi, kMagicBits, 0x7540u + c));
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
            const float* am = A + m * K + k0 + 4 * w;
            const float4 al = load_a4<kVecA>(am);
            const float4 ah = load_a4<kVecA>(am + 16);
            float s = t[m];
            s = fmaf(al.x, vl[0], s);
            s = fmaf(al.y, vl[1], s);
            s = fmaf(al.z, vl[2], s);
            s = fmaf(al.w, vl[3], s);
            s = fmaf(ah.x, vh[0], s);
            s = fmaf(ah.y, vh[1], s);
            s = fmaf(ah.z, vh[2], s);
            s = fmaf(ah.w, vh[3], s);
            t[m] = s;
        }
    }
}

// One 144-byte unit (8 blocks) of one row, 16-byte aligned in shared memory.
// Blocks come in pairs of 36 bytes = 9 words: the even block's d is the low
// half of word 0 and its quants are bytes 2..17 (realigned with byte
// permutes); the odd block's d is the high half of word 4 and its quants are
// words 5..8.
template <int M>
__device__ __forceinline__ void unit_dot(const uint8_t* tile_row, const float* __restrict__ A,
                                         int64_t K, int64_t kbase, float acc[M]) {
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
        block_dot<M, true>(A, K, kbase + 64 * p, qa, t);
        const float da = f16_bits_to_float(W[0] & 0xFFFFu);
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m] = fmaf(da, t[m], acc[m]);
        const uint32_t qb[4] = {W[5], W[6], W[7], W[8]};
        block_dot<M, true>(A, K, kbase + 64 * p + 32, qb, t);
        const float db = f16_bits_to_float(W[4] >> 16);
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m] = fmaf(db, t[m], acc[m]);
    }
}

template <int M>
__global__ void __launch_bounds__(256)
    gemv_q4_0_tma(const __grid_constant__ CUtensorMap wmap, const float* __restrict__ A,
                  float* __restrict__ C, int N, int64_t K, int units_total, int units_per_cta,
                  int cluster) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* tiles = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + units_per_cta * kTileBytes);
    float* partial = reinterpret_cast<float*>(bars + units_per_cta);  // [nwarps][M][32]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int rank = static_cast<int>(blockIdx.x) % cluster;
    const int row0 = (static_cast<int>(blockIdx.x) / cluster) * kRowsPerCta;
    const int u0 = rank * units_per_cta;
    int nunits = units_total - u0;
    nunits = nunits < 0 ? 0 : (nunits > units_per_cta ? units_per_cta : nunits);

    if (threadIdx.x == 0) {
        prefetch_tensormap(&wmap);
        for (int j = 0; j < nunits; ++j) mbar_init(&bars[j], 1);
        fence_barrier_init();
        for (int j = 0; j < nunits; ++j) {
            mbar_arrive_expect_tx(&bars[j], kTileBytes);
            tma_load_2d(tiles + j * kTileBytes, &wmap, (u0 + j) * kUnitBytes, row0, &bars[j]);
        }
    }
    __syncthreads();

    float acc[M];
#pragma unroll
    for (int m = 0; m < M; ++m) acc[m] = 0.f;
    for (int j = warp; j < nunits; j += nwarps) {
        if (!mbar_wait_bounded(&bars[j], 0, &g_gemv_error)) continue;
        unit_dot<M>(tiles + j * kTileBytes + lane * kUnitBytes, A, K,
                    static_cast<int64_t>(u0 + j) * kUnitElems, acc);
    }
#pragma unroll
    for (int m = 0; m < M; ++m) partial[(warp * M + m) * 32 + lane] = acc[m];
    __syncthreads();

    const int row = row0 + lane;
    if (cluster == 1) {
        if (warp == 0 && row < N) {
#pragma unroll
            for (int m = 0; m < M; ++m) {
                float s = 0.f;
                for (int w = 0; w < nwarps; ++w) s += partial[(w * M + m) * 32 + lane];
                C[static_cast<int64_t>(m) * N + row] = s;
            }
        }
    } else {
        cg::cluster_group cl = cg::this_cluster();
        cl.sync();
        if (rank == 0 && warp == 0 && row < N) {
#pragma unroll
            for (int m = 0; m < M; ++m) {
                float s = 0.f;
                for (int q = 0; q < cluster; ++q) {
                    const float* rp = cl.map_shared_rank(partial, q);
                    for (int w = 0; w < nwarps; ++w) s += rp[(w * M + m) * 32 + lane];
                }
                C[static_cast<int64_t>(m) * N + row] = s;
            }
        }
        cl.sync();  // peers keep their shared memory alive until rank 0 has read it
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
            block_dot<M, false>(A, K, b * kBlockElems, q, t);
            const float d = f16_bits_to_float(h[0]);
#pragma unroll
            for (int m = 0; m < M; ++m) acc[m] = fmaf(d, t[m], acc[m]);
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
    if (__atomic_load_n(&configured[dev.device], __ATOMIC_ACQUIRE) >= bytes) return cudaSuccess;
    const int want = dev.max_smem_optin;
    cudaError_t err =
        cudaFuncSetAttribute(gemv_q4_0_tma<M>, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
    if (err != cudaSuccess) return err;
    __atomic_store_n(&configured[dev.device], want, __ATOMIC_RELEASE);
    return bytes <= want ? cudaSuccess : cudaErrorInvalidValue;
}

template <int M>
cudaError_t launch_m(const float* A, const uint8_t* wq, float* C, int64_t N, int64_t K,
                     cudaStream_t stream, const DeviceInfo& dev) {
    const int64_t units = K / kUnitElems;
    const int64_t row_bytes = units * kUnitBytes;
    const bool fast = (K % kUnitElems) == 0 && units > 0 &&
                      (reinterpret_cast<uintptr_t>(wq) & 15u) == 0 &&
                      (reinterpret_cast<uintptr_t>(A) & 15u) == 0 && N <= (int64_t(1) << 30) &&
                      row_bytes < (int64_t(1) << 32);
    if (fast) {
        const int64_t row_groups = (N + kRowsPerCta - 1) / kRowsPerCta;
        const int64_t target = static_cast<int64_t>(dev.sm_count) * 6;
        int cluster = 1;
        while (cluster < kMaxCluster && row_groups * cluster < target && cluster * 2 <= units)
            cluster *= 2;
        int64_t upc = (units + cluster - 1) / cluster;
        while (upc > kMaxUnitsPerCta && cluster < kMaxCluster) {
            cluster *= 2;
            upc = (units + cluster - 1) / cluster;
        }
        if (upc <= kMaxUnitsPerCta) {
            int nwarps = upc < 8 ? static_cast<int>(upc) : 8;
            for (int d = 8; d >= 4; --d) {
                if (upc % d == 0) {
                    nwarps = d;
                    break;
                }
            }
            const int smem = static_cast<int>(upc * kTileBytes + upc * 8 + nwarps * M * 32 * 4);
            cudaError_t err = ensure_smem_attr<M>(dev, smem);
            if (err != cudaSuccess) return err;
            CUtensorMap map;
            err = encode_weight_map_2d(&map, wq, row_bytes, N, kUnitBytes, kRowsPerCta);
            if (err != cudaSuccess) return err;

            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(row_groups * cluster));
            cfg.blockDim = dim3(nwarps * 32);
            cfg.dynamicSmemBytes = smem;
            cfg.stream = stream;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = cluster;
            attr[0].val.clusterDim.y = 1;
            attr[0].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            err = cudaLaunchKernelEx(&cfg, gemv_q4_0_tma<M>, map, A, C, static_cast<int>(N), K,
                                     static_cast<int>(units), static_cast<int>(upc), cluster);
            if (err != cudaSuccess) return err;
            note_launch();
            return cudaGetLastError();
        }
    }
    const int64_t warps_needed = N;
    const int64_t ctas = (warps_needed + 7) / 8;
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * 16;
    const unsigned grid = static_cast<unsigned>(ctas < cap ? ctas : cap);
    gemv_q4_0_generic<M><<<grid, 256, 0, stream>>>(A, wq, C, N, K);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv_q4_0(const float* A, const uint8_t* wq, float* C, int M, int64_t N,
                             int64_t K, cudaStream_t stream, const DeviceInfo& dev) {
    switch (M) {
        case 1: return launch_m<1>(A, wq, C, N, K, stream, dev);
        case 2: return launch_m<2>(A, wq, C, N, K, stream, dev);
        case 3: return launch_m<3>(A, wq, C, N, K, stream, dev);
        case 4: return launch_m<4>(A, wq, C, N, K, stream, dev);
        case 5: return launch_m<5>(A, wq, C, N, K, stream, dev);
        case 6: return launch_m<6>(A, wq, C, N, K, stream, dev);
        case 7: return launch_m<7>(A, wq, C, N, K, stream, dev);
        case 8: return launch_m<8>(A, wq, C, N, K, stream, dev);
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

}  // namespace qm

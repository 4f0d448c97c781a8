// Prefill GEMM on FP32 FMA: C[M][N] = A[M][K] x dequant(W)^T for any M >= 1
// (section "matmul_q4_0_tiled" of "fuel-vulkan-kernels — quantized (GGML)
// kernel contracts": shared-memory tiles, each weight block decoded once per
// tile and reused over the tile's rows).
//
// A CTA computes a BM x BN tile of C.  Each k-step covers one Q4_0 block per
// weight row (32 k): the CTA stages the A slab [BM x 32] (k-major) and the
// decoded weights [32 x BN] in shared memory, each thread decoding its share
// of the BN blocks exactly once as (q - 8) * d.  Every thread then runs a
// TM x TN register tile of FFMAs over the 32 k.  The next slab is fetched
// into registers while the current one is multiplied.  Only 2-byte alignment
// of wq and 4-byte alignment of A are assumed (16-byte A takes vector loads).
#include "qm_device.cuh"
#include "qm_internal.h"

namespace qm {
namespace {

constexpr int kThreads = 256;

template <int BM, int BN, int TM, int TN>
struct Tile {
    static constexpr int kParts = kThreads / BN;          // threads decoding one weight row
    static constexpr int kBytesPerPart = 16 / kParts;     // quant bytes each of them decodes
    static constexpr int kHalfWords = kBytesPerPart / 2;  // 2-byte loads per thread
    static constexpr int kAVec = BM * 32 / kThreads / 4;  // float4 of A per thread
    static constexpr int kColThreads = BN / TN;
    static_assert(kThreads % BN == 0 && kParts >= 1 && kParts <= 8, "BN");
    static_assert((BM / TM) * (BN / TN) == kThreads, "thread tile");
    static_assert(kAVec >= 1, "BM");
    static_assert(TM == 4 || TM == 8, "TM");
    static_assert(TN == 2 || TN == 4 || TN == 8, "TN");

    // Row offset (within the tile) of the thread's x-th row / column.
    __device__ static __forceinline__ int row(int tm, int x) {
        return (TM == 8) ? ((x < 4) ? 4 * tm + x : BM / 2 + 4 * tm + x - 4) : 4 * tm + x;
    }
    __device__ static __forceinline__ int col(int tn, int x) {
        if constexpr (TN == 8) return (x < 4) ? 4 * tn + x : BN / 2 + 4 * tn + x - 4;
        if constexpr (TN == 4) return 4 * tn + x;
        return 2 * tn + x;
    }
};

template <int BM, int BN, int TM, int TN>
__global__ void __launch_bounds__(kThreads)
    gemm_q4_0_simt(const float* __restrict__ A, const uint8_t* __restrict__ wq,
                   float* __restrict__ C, int64_t M, int64_t N, int64_t K, int a_vec) {
    using T = Tile<BM, BN, TM, TN>;
    __shared__ __align__(16) float As[32][BM];
    __shared__ __align__(16) float Ws[32][BN];

    const int t = threadIdx.x;
    const int64_t m0 = static_cast<int64_t>(blockIdx.y) * BM;
    const int64_t n0 = static_cast<int64_t>(blockIdx.x) * BN;
    const int64_t nb = K / kBlockElems;

    // A staging: thread t loads float4 c = t / BM + (kThreads / BM) * i of row t % BM.
    const int a_row = t % BM;
    const int a_c0 = t / BM;
    const bool a_ok = (m0 + a_row) < M;
    const float* a_src = A + (m0 + a_row) * K;
    // W staging: thread t decodes quant bytes [p * kBytesPerPart, ...) of row t % BN.
    const int w_row = t % BN;
    const int w_part = t / BN;
    const bool w_ok = (n0 + w_row) < N;
    const uint8_t* w_src = wq + (n0 + w_row) * nb * kBlockBytes;

    float4 a_reg[T::kAVec];
    uint32_t w_d = 0;
    uint32_t w_h[T::kHalfWords];

    auto fetch = [&](int64_t kb) {
#pragma unroll
        for (int i = 0; i < T::kAVec; ++i) {
            const int c = a_c0 + (kThreads / BM) * i;
            if (a_ok) {
                const float* p = a_src + kb * kBlockElems + 4 * c;
                a_reg[i] = a_vec ? __ldg(reinterpret_cast<const float4*>(p))
                                 : make_float4(__ldg(p), __ldg(p + 1), __ldg(p + 2), __ldg(p + 3));
            } else {
                a_reg[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        if (w_ok) {
            const uint16_t* h = reinterpret_cast<const uint16_t*>(w_src + kb * kBlockBytes);
            w_d = h[0];
#pragma unroll
            for (int i = 0; i < T::kHalfWords; ++i) w_h[i] = h[1 + w_part * T::kHalfWords + i];
        } else {
            w_d = 0;
#pragma unroll
            for (int i = 0; i < T::kHalfWords; ++i) w_h[i] = 0x8888u;
        }
    };
    auto stage = [&]() {
#pragma unroll
        for (int i = 0; i < T::kAVec; ++i) {
            const int c = a_c0 + (kThreads / BM) * i;
            As[4 * c + 0][a_row] = a_reg[i].x;
            As[4 * c + 1][a_row] = a_reg[i].y;
            As[4 * c + 2][a_row] = a_reg[i].z;
            As[4 * c + 3][a_row] = a_reg[i].w;
        }
        const float d = f16_bits_to_float(w_d);
#pragma unroll
        for (int i = 0; i < T::kHalfWords; ++i) {
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const uint32_t byte = (w_h[i] >> (8 * b)) & 0xFFu;
                const int j = w_part * T::kBytesPerPart + 2 * i + b;  // quant byte index
                Ws[j][w_row] = magic_minus8((byte & 0xFu) | kMagicBits) * d;
                Ws[j + 16][w_row] = magic_minus8((byte >> 4) | kMagicBits) * d;
            }
        }
    };

    const int tn = t % T::kColThreads;
    const int tm = t / T::kColThreads;
    float acc[TM][TN];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;

    if (nb > 0) fetch(0);
    for (int64_t kb = 0; kb < nb; ++kb) {
        __syncthreads();  // previous slab fully consumed
        stage();
        __syncthreads();
        if (kb + 1 < nb) fetch(kb + 1);
#pragma unroll 4
        for (int k = 0; k < 32; ++k) {
            float a[TM], w[TN];
#pragma unroll
            for (int x = 0; x < TM; x += 4) {
                const float4 v = *reinterpret_cast<const float4*>(&As[k][T::row(tm, x)]);
                a[x] = v.x;
                a[x + 1] = v.y;
                a[x + 2] = v.z;
                a[x + 3] = v.w;
            }
            if constexpr (TN == 2) {
                const float2 v = *reinterpret_cast<const float2*>(&Ws[k][T::col(tn, 0)]);
                w[0] = v.x;
                w[1] = v.y;
            } else {
#pragma unroll
                for (int x = 0; x < TN; x += 4) {
                    const float4 v = *reinterpret_cast<const float4*>(&Ws[k][T::col(tn, x)]);
                    w[x] = v.x;
                    w[x + 1] = v.y;
                    w[x + 2] = v.z;
                    w[x + 3] = v.w;
                }
            }
#pragma unroll
            for (int i = 0; i < TM; ++i)
#pragma unroll
                for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], w[j], acc[i][j]);
        }
    }

#pragma unroll
    for (int i = 0; i < TM; ++i) {
        const int64_t m = m0 + T::row(tm, i);
        if (m >= M) continue;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            const int64_t n = n0 + T::col(tn, j);
            if (n < N) C[m * N + n] = acc[i][j];
        }
    }
}

template <int BM, int BN, int TM, int TN>
cudaError_t launch_tile(const float* A, const uint8_t* wq, float* C, int64_t M, int64_t N,
                        int64_t K, cudaStream_t stream) {
    const int64_t gx = (N + BN - 1) / BN;
    const int64_t gy = (M + BM - 1) / BM;
    if (gx > 0x7FFFFFFF || gy > 65535) return cudaErrorInvalidConfiguration;
    const int a_vec = ((reinterpret_cast<uintptr_t>(A) & 15u) == 0) ? 1 : 0;
    gemm_q4_0_simt<BM, BN, TM, TN><<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)),
                                     kThreads, 0, stream>>>(A, wq, C, M, N, K, a_vec);
    note_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_q4_0_simt(const float* A, const uint8_t* wq, float* C, int64_t M,
                                  int64_t N, int64_t K, cudaStream_t stream,
                                  const DeviceInfo& dev) {
    (void)dev;
    if (M >= 128) return launch_tile<128, 128, 8, 8>(A, wq, C, M, N, K, stream);
    return launch_tile<32, 64, 4, 2>(A, wq, C, M, N, K, stream);
}

}  // namespace qm

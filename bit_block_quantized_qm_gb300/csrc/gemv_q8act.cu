// The decode-regime product with the activations quantized to Q8_0 first:
// C = A' x dequant(W)^T, A' = dequant_q8_0(quantize_q8_0(A)) row by row, for
// M = 1..8 — the GEMV fused with a preceding activation quantization ("act-
// quant fusion" in "vulkan: shader and sequencing efficiency backlog";
// quantization and dequantization as in sections "quantize_q8_0" and
// "dequant_q8_0", the product as in "qmatvec_q4_0" of "fuel-vulkan-kernels —
// quantized (GGML) kernel contracts").  A is read once as f32 and never
// written back quantized: each kernel quantizes the blocks it needs on chip.
//
// K % 256 == 0 with 16-byte aligned A and wq runs the staged GEMV's integer
// consumer (gemv_tc.cu).  Other shapes run the generic kernel here: one warp
// per output row, lanes striding over the row's blocks; a lane quantizes the
// activation block of each of its blocks itself (max, scale, quants, exactly
// as the staged kernel does), takes sum_j (q_j - 8) qs_j in integers and adds
// d_w d_a times it; the lanes' sums meet by shuffles.  A row whose total is
// not finite is recomputed element by element by lane 0.
#include "qm_device.cuh"
#include "qm_internal.h"

namespace qm {
namespace {

constexpr int kWarpsPerCta = 8;

// Quantize one 32-element activation block (4-byte aligned): its quants and
// the binary16 scale as f32.
__device__ __forceinline__ float quantize_block(const float* x, int8_t qs[32]) {
    float amax = 0.f;
    for (int j = 0; j < kBlockElems; ++j) amax = fmaxf(amax, fabsf(x[j]));
    const float d = __fdiv_rn(amax, 127.f);
    for (int j = 0; j < kBlockElems; ++j) qs[j] = static_cast<int8_t>(q8_quant(x[j], d));
    return f16_bits_to_float(f16_bits_rn(d));
}

__device__ __forceinline__ float weight_scale(const uint8_t* blk) {
    return f16_bits_to_float(static_cast<uint32_t>(blk[0]) | (static_cast<uint32_t>(blk[1]) << 8));
}

template <int M>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    gemv_q4_0_q8act_generic(const float* __restrict__ A, const uint8_t* __restrict__ wq, float* __restrict__ C,
                            int64_t N, int64_t K) {
    const int lane = threadIdx.x & 31;
    const int64_t nb = K / kBlockElems;
    grid_launch_dependents();
    grid_dependency_wait();
    for (int64_t n = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5); n < N;
         n += static_cast<int64_t>(gridDim.x) * kWarpsPerCta) {
        const uint8_t* row = wq + n * nb * kBlockBytes;
        float acc[M];
#pragma unroll
        for (int m = 0; m < M; ++m) acc[m] = 0.f;
        for (int64_t b = lane; b < nb; b += 32) {
            const uint8_t* blk = row + b * kBlockBytes;
            const float dw = weight_scale(blk);
            int qw[32];
            for (int j = 0; j < 16; ++j) {
                qw[j] = static_cast<int>(blk[2 + j] & 0xFu) - 8;
                qw[j + 16] = static_cast<int>(blk[2 + j] >> 4) - 8;
            }
#pragma unroll
            for (int m = 0; m < M; ++m) {
                int8_t qs[32];
                const float da = quantize_block(A + m * K + b * kBlockElems, qs);
                int s = 0;
                for (int j = 0; j < kBlockElems; ++j) s += qw[j] * static_cast<int>(qs[j]);
                acc[m] = fmaf(dw * da, static_cast<float>(s), acc[m]);
            }
        }
#pragma unroll
        for (int m = 0; m < M; ++m) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[m] += __shfl_xor_sync(0xFFFFFFFFu, acc[m], o);
        }
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < M; ++m) {
                float v = acc[m];
                if (!isfinite(v)) {
                    // Element by element: A'_k = qs_k d_a (exact), times (q - 8) d_w.
                    v = 0.f;
                    for (int64_t b = 0; b < nb; ++b) {
                        const uint8_t* blk = row + b * kBlockBytes;
                        const float dw = weight_scale(blk);
                        int8_t qs[32];
                        const float da = quantize_block(A + m * K + b * kBlockElems, qs);
                        for (int j = 0; j < kBlockElems; ++j) {
                            const uint32_t byte = blk[2 + (j & 15)];
                            const uint32_t nib = (j < 16) ? (byte & 0xFu) : (byte >> 4);
                            v = fmaf(static_cast<float>(qs[j]) * da, magic_minus8(nib | kMagicBits) * dw, v);
                        }
                    }
                }
                C[m * N + n] = v;
            }
        }
    }
}

template <int M>
cudaError_t launch_generic(const float* A, const uint8_t* wq, float* C, int64_t N, int64_t K,
                           cudaStream_t stream, const DeviceInfo& dev) {
    const int64_t ctas = (N + kWarpsPerCta - 1) / kWarpsPerCta;
    const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
    const unsigned grid = static_cast<unsigned>(ctas < cap ? ctas : cap);
    cudaError_t err = launch_pdl(gemv_q4_0_q8act_generic<M>, dim3(grid), dim3(kWarpsPerCta * 32), 0, stream,
                                 A, wq, C, N, K);
    if (err == cudaSuccess) note_launch();
    return err;
}

}  // namespace

cudaError_t launch_matmul_q4_0_q8act(const float* A, const uint8_t* wq, float* C, int M, int64_t N, int64_t K,
                                     cudaStream_t stream, const DeviceInfo& dev) {
    if (K % 256 == 0 && (reinterpret_cast<uintptr_t>(A) & 15u) == 0 && (reinterpret_cast<uintptr_t>(wq) & 15u) == 0 &&
        N <= (int64_t(1) << 30) && K / 256 <= (int64_t(1) << 20)) {
        bool launched = false;
        cudaError_t err = launch_gemv_q4_0_q8act_tc(A, wq, C, M, N, K, stream, dev, &launched);
        if (err != cudaSuccess || launched) return err;
    }
    switch (M) {
        case 1: return launch_generic<1>(A, wq, C, N, K, stream, dev);
        case 2: return launch_generic<2>(A, wq, C, N, K, stream, dev);
        case 3: return launch_generic<3>(A, wq, C, N, K, stream, dev);
        case 4: return launch_generic<4>(A, wq, C, N, K, stream, dev);
        case 5: return launch_generic<5>(A, wq, C, N, K, stream, dev);
        case 6: return launch_generic<6>(A, wq, C, N, K, stream, dev);
        case 7: return launch_generic<7>(A, wq, C, N, K, stream, dev);
        case 8: return launch_generic<8>(A, wq, C, N, K, stream, dev);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace qm

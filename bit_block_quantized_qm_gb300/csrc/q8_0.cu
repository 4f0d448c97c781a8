// GGML Q8_0: dequant (block stream -> f32) and quantize (f32 -> block stream).
//
// Follows "fuel-vulkan-kernels — quantized (GGML) kernel contracts":
//   * section "dequant_q8_0": a 34-byte block holds an f16 scale d (bytes
//     0-1, little-endian) and 32 signed 8-bit quants; element j = qs_j * d.
//     An 8-bit integer times a binary16 value is exact in f32, so the output
//     is bit-identical to the definition (signed zeros, infinities and NaN
//     included);
//   * section "quantize_q8_0": per 32-element block d = max|x| / 127; the
//     block stores d narrowed to binary16 and qs = round(x / d).  Where the
//     section is silent this library reads: f32 arithmetic with correctly
//     rounded divisions; NaN elements do not raise the max; the narrowing
//     rounds to nearest even (overflow to infinity); round() takes halfway
//     cases away from zero; qs is clamped to [-127, 127] (which binds only
//     when d is an f32 subnormal); qs = 0 where d = 0 or x / d is NaN.
//
// Both directions are HBM-bound: dequant reads 34 and writes 128 bytes per
// block, quantize reads 128 and writes 34.  The fast kernels move 32 blocks
// per warp step with coalesced 16-byte loads and stores through a staging
// buffer in shared memory (32 blocks of 34 bytes are 68 aligned 16-byte
// words); generic kernels take misaligned pointers and the last partial
// group.  The fast kernels are launched with programmatic stream
// serialization and touch global memory only after griddepcontrol.wait.
#include "qm_device.cuh"
#include "qm_internal.h"

namespace qm {
namespace {

constexpr int kQ8Bytes = 34;
constexpr int kGroupBlocks = 32;
constexpr int kGroupBytes = kGroupBlocks * kQ8Bytes;  // 1088 = 68 * 16
constexpr int kWarps = 8;

// A signed byte b as an exact float: (b ^ 0x80) is b + 128 in 0..255; under the
// exponent of 2^23 it reads 2^23 + b + 128, and subtracting 2^23 + 128 leaves b.
constexpr float kMagicPlus128 = 8388736.0f;  // 2^23 + 128

// Four consecutive outputs of a block from its 4 quant bytes q (q0 lowest).
__device__ __forceinline__ float4 q8_decode4(uint32_t q, float d) {
    const uint32_t u = q ^ 0x80808080u;
    float4 v;
    v.x = (__uint_as_float(__byte_perm(u, kMagicBits, 0x7650u)) - kMagicPlus128) * d;
    v.y = (__uint_as_float(__byte_perm(u, kMagicBits, 0x7651u)) - kMagicPlus128) * d;
    v.z = (__uint_as_float(__byte_perm(u, kMagicBits, 0x7652u)) - kMagicPlus128) * d;
    v.w = (__uint_as_float(__byte_perm(u, kMagicBits, 0x7653u)) - kMagicPlus128) * d;
    return v;
}

__global__ void __launch_bounds__(kWarps * 32)
    dequant_q8_0_fast(const uint8_t* __restrict__ wq, int64_t n_groups, float* __restrict__ out) {
    __shared__ __align__(16) uint8_t stage[kWarps][kGroupBytes];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint8_t* buf = stage[warp];
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps;
    int64_t g = static_cast<int64_t>(blockIdx.x) * kWarps + warp;

    grid_launch_dependents();
    grid_dependency_wait();

    // 68 words per group: lanes take words lane, lane + 32, and (lanes < 4) lane + 64.
    uint4 r0 = make_uint4(0, 0, 0, 0), r1 = r0, r2 = r0;
    auto fetch = [&](int64_t grp) {
        const uint8_t* src = wq + grp * kGroupBytes;
        r0 = ldg_nc_v4(src + lane * 16);
        r1 = ldg_nc_v4(src + 512 + lane * 16);
        if (lane < 4) r2 = ldg_nc_v4(src + 1024 + lane * 16);
    };
    if (g < n_groups) fetch(g);
    for (; g < n_groups; g += stride) {
        *reinterpret_cast<uint4*>(buf + lane * 16) = r0;
        *reinterpret_cast<uint4*>(buf + 512 + lane * 16) = r1;
        if (lane < 4) *reinterpret_cast<uint4*>(buf + 1024 + lane * 16) = r2;
        __syncwarp();
        if (g + stride < n_groups) fetch(g + stride);
        float* og = out + g * (kGroupBlocks * kBlockElems);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int f = lane + 32 * i;  // float4 index within the group's output
            const int b = f >> 3;
            const int c = f & 7;          // elements 4c .. 4c + 3
            const uint8_t* blk = buf + b * kQ8Bytes;
            const float d = f16_bits_to_float(*reinterpret_cast<const uint16_t*>(blk));
            const uint32_t lo = *reinterpret_cast<const uint16_t*>(blk + 2 + 4 * c);
            const uint32_t hi = *reinterpret_cast<const uint16_t*>(blk + 4 + 4 * c);
            const float4 v = q8_decode4(lo | (hi << 16), d);
            st_global_cs_v4(og + 4 * f, v.x, v.y, v.z, v.w);
        }
        __syncwarp();
    }
}

// One thread per (block, 4-element chunk): byte loads, any alignment of wq;
// out needs 4-byte alignment (16-byte when out16).
__global__ void __launch_bounds__(256)
    dequant_q8_0_generic(const uint8_t* __restrict__ wq, int64_t b_begin, int64_t n_blocks,
                         float* __restrict__ out, int out16) {
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t b = b_begin + (t >> 3);
    const int c = static_cast<int>(t & 7);
    if (b >= n_blocks) return;
    const uint8_t* blk = wq + b * kQ8Bytes;
    const float d = f16_bits_to_float(static_cast<uint32_t>(blk[0]) | (static_cast<uint32_t>(blk[1]) << 8));
    const uint8_t* q = blk + 2 + 4 * c;
    const uint32_t word = static_cast<uint32_t>(q[0]) | (static_cast<uint32_t>(q[1]) << 8) |
                          (static_cast<uint32_t>(q[2]) << 16) | (static_cast<uint32_t>(q[3]) << 24);
    const float4 v = q8_decode4(word, d);
    float* o = out + b * kBlockElems + 4 * c;
    if (out16) {
        *reinterpret_cast<float4*>(o) = v;
    } else {
        o[0] = v.x;
        o[1] = v.y;
        o[2] = v.z;
        o[3] = v.w;
    }
}

__device__ __forceinline__ uint32_t pack_q4(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    return a | (b << 8) | (c << 16) | (d << 24);
}

// 32 blocks per warp step: lane l loads float4 (32 i + l), i < 8, which holds
// elements 4 (l % 8) .. +3 of block 4 i + l / 8; the 8 lanes of a block share
// its max by shuffles, each quantizes its 4 elements (q8_quant_byte), and the
// 34-byte blocks are assembled in shared memory and written as 68 16-byte
// words.
__global__ void __launch_bounds__(kWarps * 32)
    quantize_q8_0_fast(const float* __restrict__ x, int64_t n_groups, uint8_t* __restrict__ out) {
    __shared__ __align__(16) uint8_t stage[kWarps][kGroupBytes];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint8_t* buf = stage[warp];
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps;
    const int sub = lane & 7;

    grid_launch_dependents();
    grid_dependency_wait();

    for (int64_t g = static_cast<int64_t>(blockIdx.x) * kWarps + warp; g < n_groups; g += stride) {
        const float4* src = reinterpret_cast<const float4*>(x + g * (kGroupBlocks * kBlockElems));
        float4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __ldcs(src + 32 * i + lane);
        // The max of block 4 i + l / 8 over its 8 lanes, then gathered so that
        // lane l holds block l's: one division and one reciprocal per block.
        float mine = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float m = fmaxf(fmaxf(fabsf(v[i].x), fabsf(v[i].y)), fmaxf(fabsf(v[i].z), fabsf(v[i].w)));
            m = fmaxf(m, 0.f);
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
            m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
            const float mb = __shfl_sync(0xFFFFFFFFu, m, 8 * (lane & 3));  // block 4 i + (lane & 3)
            if ((lane >> 2) == i) mine = mb;
        }
        const float d_mine = __fdiv_rn(mine, 127.f);
        const float r_mine = __frcp_rn(d_mine);
        *reinterpret_cast<uint16_t*>(buf + lane * kQ8Bytes) = static_cast<uint16_t>(f16_bits_rn(d_mine));
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int b = 4 * i + (lane >> 3);
            const float d = __shfl_sync(0xFFFFFFFFu, d_mine, b);
            const float r = __shfl_sync(0xFFFFFFFFu, r_mine, b);
            uint8_t* blk = buf + b * kQ8Bytes;
            const uint32_t w = pack_q4(q8_quant_byte(v[i].x, d, r), q8_quant_byte(v[i].y, d, r),
                                       q8_quant_byte(v[i].z, d, r), q8_quant_byte(v[i].w, d, r));
            // Quant bytes 4 sub .. 4 sub + 3 at block offset 2 + 4 sub (2-byte aligned).
            *reinterpret_cast<uint16_t*>(blk + 2 + 4 * sub) = static_cast<uint16_t>(w & 0xFFFFu);
            *reinterpret_cast<uint16_t*>(blk + 4 + 4 * sub) = static_cast<uint16_t>(w >> 16);
        }
        __syncwarp();
        uint8_t* dst = out + g * kGroupBytes;
        *reinterpret_cast<uint4*>(dst + lane * 16) = *reinterpret_cast<const uint4*>(buf + lane * 16);
        *reinterpret_cast<uint4*>(dst + 512 + lane * 16) =
            *reinterpret_cast<const uint4*>(buf + 512 + lane * 16);
        if (lane < 4)
            *reinterpret_cast<uint4*>(dst + 1024 + lane * 16) =
                *reinterpret_cast<const uint4*>(buf + 1024 + lane * 16);
        __syncwarp();
    }
}

// One thread per block: 4-byte loads of x, byte stores (any alignment of out).
// The block's 34 bytes are assembled as 9 little-endian words (the last one
// half used) and written byte by byte.
__global__ void __launch_bounds__(256)
    quantize_q8_0_generic(const float* __restrict__ x, int64_t b_begin, int64_t n_blocks,
                          uint8_t* __restrict__ out) {
    const int64_t b = b_begin + static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (b >= n_blocks) return;
    const float* xb = x + b * kBlockElems;
    float m = 0.f;
    for (int j = 0; j < kBlockElems; ++j) m = fmaxf(m, fabsf(xb[j]));
    const float d = __fdiv_rn(m, 127.f);
    uint32_t w[9];
    // word 0: scale (bytes 0-1), quants 0-1; word i (1..7): quants 4i-2 .. 4i+1;
    // word 8: quants 30-31
    int q[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) q[j] = q8_quant(xb[j], d) & 0xFF;
    w[0] = f16_bits_rn(d) | (static_cast<uint32_t>(q[0]) << 16) | (static_cast<uint32_t>(q[1]) << 24);
#pragma unroll
    for (int i = 1; i < 8; ++i)
        w[i] = static_cast<uint32_t>(q[4 * i - 2]) | (static_cast<uint32_t>(q[4 * i - 1]) << 8) |
               (static_cast<uint32_t>(q[4 * i]) << 16) | (static_cast<uint32_t>(q[4 * i + 1]) << 24);
    w[8] = static_cast<uint32_t>(q[30]) | (static_cast<uint32_t>(q[31]) << 8);
    uint8_t* blk = out + b * kQ8Bytes;
#pragma unroll
    for (int i = 0; i < kQ8Bytes; ++i) blk[i] = static_cast<uint8_t>(w[i >> 2] >> (8 * (i & 3)));
}

}  // namespace

cudaError_t launch_dequant_q8_0(const uint8_t* wq, int64_t n_blocks, float* out,
                                cudaStream_t stream, const DeviceInfo& dev) {
    const bool in16 = (reinterpret_cast<uintptr_t>(wq) & 15u) == 0;
    const bool out16 = (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
    const int64_t n_groups = (in16 && out16) ? n_blocks / kGroupBlocks : 0;
    if (n_groups > 0) {
        const int64_t ctas = (n_groups + kWarps - 1) / kWarps;
        const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
        cudaError_t err = launch_pdl(dequant_q8_0_fast, dim3(static_cast<unsigned>(ctas < cap ? ctas : cap)),
                                     dim3(kWarps * 32), 0, stream, wq, n_groups, out);
        if (err != cudaSuccess) return err;
        note_launch();
    }
    const int64_t b_begin = n_groups * kGroupBlocks;
    const int64_t rest = n_blocks - b_begin;
    if (rest > 0) {
        const int64_t grid = (rest * 8 + 255) / 256;
        dequant_q8_0_generic<<<static_cast<unsigned>(grid), 256, 0, stream>>>(wq, b_begin, n_blocks, out,
                                                                              out16 ? 1 : 0);
        note_launch();
        return cudaGetLastError();
    }
    return cudaSuccess;
}

cudaError_t launch_quantize_q8_0(const float* x, int64_t n_blocks, uint8_t* out,
                                 cudaStream_t stream, const DeviceInfo& dev) {
    const bool in16 = (reinterpret_cast<uintptr_t>(x) & 15u) == 0;
    const bool out16 = (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
    const int64_t n_groups = (in16 && out16) ? n_blocks / kGroupBlocks : 0;
    if (n_groups > 0) {
        const int64_t ctas = (n_groups + kWarps - 1) / kWarps;
        const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
        cudaError_t err = launch_pdl(quantize_q8_0_fast, dim3(static_cast<unsigned>(ctas < cap ? ctas : cap)),
                                     dim3(kWarps * 32), 0, stream, x, n_groups, out);
        if (err != cudaSuccess) return err;
        note_launch();
    }
    const int64_t b_begin = n_groups * kGroupBlocks;
    const int64_t rest = n_blocks - b_begin;
    if (rest > 0) {
        const int64_t grid = (rest + 255) / 256;
        quantize_q8_0_generic<<<static_cast<unsigned>(grid), 256, 0, stream>>>(x, b_begin, n_blocks, out);
        note_launch();
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace qm

// dequant_q4_0: GGML Q4_0 block stream -> dense f32.
//
// Follows "fuel-vulkan-kernels — quantized (GGML) kernel contracts", section
// "dequant_q4_0": out[32*b + j] = (nibble_j - 8) * d, with element j < 16 in
// the low nibble of quant byte j and element j + 16 in its high nibble.  The
// product of an integer in [-8, 7] and a binary16 value is exact in f32, so
// the output is bit-identical to the definition, signed zeros included.
//
// HBM-bound: 18 bytes read and 128 bytes written per block; the f32 write is
// 88% of the traffic.  The fast kernel gives each warp 32 consecutive blocks
// per step (576 input bytes = 36 aligned 16-byte words, read with coalesced
// 16-byte loads and staged in shared memory) and writes their 4 KB of output
// as 256 coalesced 16-byte streaming stores, prefetching the next step's
// input while it writes.  A generic kernel (2-byte loads, 4- or 16-byte
// stores) covers misaligned pointers and the last partial group.
//
// The fast kernel is launched with programmatic stream serialization: it lets
// the next kernel start its prologue at once and, before waiting for the
// kernels it depends on, only asks L2 for its first group (a hint that cannot
// return stale data); every load and store comes after griddepcontrol.wait.
#include "qm_device.cuh"
#include "qm_internal.h"

namespace qm {
namespace {

constexpr int kGroupBlocks = 32;
constexpr int kGroupInBytes = kGroupBlocks * kBlockBytes;  // 576 = 36 * 16
constexpr int kWarpsPerCta = 8;

// Four consecutive output floats of one block: chunk c (0..7) covers elements
// 4*(c&3) .. +3 (low nibbles, c < 4) or 16 + 4*(c&3) .. +3 (high nibbles).
__device__ __forceinline__ float4 decode_chunk(uint32_t dbits, uint32_t qword, int c) {
    const float d = f16_bits_to_float(dbits);
    const uint32_t w = (c >= 4) ? (qword >> 4) : qword;
    float4 v;
    v.x = magic_minus8((w & 0xFu) | kMagicBits) * d;
    v.y = magic_minus8(((w >> 8) & 0xFu) | kMagicBits) * d;
    v.z = magic_minus8(((w >> 16) & 0xFu) | kMagicBits) * d;
    v.w = magic_minus8(((w >> 24) & 0xFu) | kMagicBits) * d;
    return v;
}

__global__ void __launch_bounds__(kWarpsPerCta * 32)
    dequant_q4_0_fast(const uint8_t* __restrict__ wq, int64_t n_groups, float* __restrict__ out) {
    __shared__ __align__(16) uint8_t stage[kWarpsPerCta][kGroupInBytes];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    uint8_t* buf = stage[warp];
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarpsPerCta;
    int64_t g = static_cast<int64_t>(blockIdx.x) * kWarpsPerCta + warp;

    grid_launch_dependents();
    if (g < n_groups && lane < 5)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(wq + g * kGroupInBytes + lane * 128));
    grid_dependency_wait();

    uint4 r0 = make_uint4(0, 0, 0, 0), r1 = make_uint4(0, 0, 0, 0);
    if (g < n_groups) {
        const uint8_t* src = wq + g * kGroupInBytes;
        r0 = ldg_nc_v4(src + lane * 16);
        if (lane < 4) r1 = ldg_nc_v4(src + 512 + lane * 16);
    }
    for (; g < n_groups; g += stride) {
        *reinterpret_cast<uint4*>(buf + lane * 16) = r0;
        if (lane < 4) *reinterpret_cast<uint4*>(buf + 512 + lane * 16) = r1;
        __syncwarp();
        const int64_t gn = g + stride;
        if (gn < n_groups) {
            const uint8_t* src = wq + gn * kGroupInBytes;
            r0 = ldg_nc_v4(src + lane * 16);
            if (lane < 4) r1 = ldg_nc_v4(src + 512 + lane * 16);
        }
        float* og = out + g * (kGroupBlocks * kBlockElems);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int f = lane + 32 * i;  // float4 index within the group's output
            const int b = f >> 3;
            const int c = f & 7;
            const uint8_t* blk = buf + b * kBlockBytes;
            const uint32_t dbits = *reinterpret_cast<const uint16_t*>(blk);
            const int off = 2 + 4 * (c & 3);
            const uint32_t lo = *reinterpret_cast<const uint16_t*>(blk + off);
            const uint32_t hi = *reinterpret_cast<const uint16_t*>(blk + off + 2);
            const float4 v = decode_chunk(dbits, lo | (hi << 16), c);
            st_global_cs_v4(og + 4 * f, v.x, v.y, v.z, v.w);
        }
        __syncwarp();
    }
}

// One thread per (block, chunk): 2-byte loads, so any 2-byte-aligned stream
// works; out needs 4-byte alignment (16-byte when out16).
__global__ void __launch_bounds__(256)
    dequant_q4_0_generic(const uint8_t* __restrict__ wq, int64_t b_begin, int64_t n_blocks,
                         float* __restrict__ out, int out16) {
    const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t b = b_begin + (t >> 3);
    const int c = static_cast<int>(t & 7);
    if (b >= n_blocks) return;
    const uint8_t* blk = wq + b * kBlockBytes;
    const uint32_t dbits = *reinterpret_cast<const uint16_t*>(blk);
    const int off = 2 + 4 * (c & 3);
    const uint32_t lo = *reinterpret_cast<const uint16_t*>(blk + off);
    const uint32_t hi = *reinterpret_cast<const uint16_t*>(blk + off + 2);
    const float4 v = decode_chunk(dbits, lo | (hi << 16), c);
    float* o = out + b * kBlockElems + 4 * (c & 3) + ((c >= 4) ? 16 : 0);
    if (out16) {
        *reinterpret_cast<float4*>(o) = v;
    } else {
        o[0] = v.x;
        o[1] = v.y;
        o[2] = v.z;
        o[3] = v.w;
    }
}

}  // namespace

cudaError_t launch_dequant_q4_0(const uint8_t* wq, int64_t n_blocks, float* out,
                                cudaStream_t stream, const DeviceInfo& dev) {
    const bool in16 = (reinterpret_cast<uintptr_t>(wq) & 15u) == 0;
    const bool out16 = (reinterpret_cast<uintptr_t>(out) & 15u) == 0;
    int64_t n_groups = (in16 && out16) ? n_blocks / kGroupBlocks : 0;
    if (n_groups > 0) {
        const int64_t ctas_needed = (n_groups + kWarpsPerCta - 1) / kWarpsPerCta;
        const int64_t cap = static_cast<int64_t>(dev.sm_count) * 8;
        const int grid = static_cast<int>(ctas_needed < cap ? ctas_needed : cap);
        cudaError_t err = launch_pdl(dequant_q4_0_fast, dim3(grid), dim3(kWarpsPerCta * 32), 0,
                                     stream, wq, n_groups, out);
        if (err != cudaSuccess) return err;
        note_launch();
    }
    const int64_t b_begin = n_groups * kGroupBlocks;
    const int64_t rest = n_blocks - b_begin;
    if (rest > 0) {
        const int64_t threads = rest * 8;
        const int64_t grid = (threads + 255) / 256;
        dequant_q4_0_generic<<<static_cast<unsigned>(grid), 256, 0, stream>>>(
            wq, b_begin, n_blocks, out, out16 ? 1 : 0);
        note_launch();
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace qm

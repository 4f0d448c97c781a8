// Device-side helpers shared by the libqm kernels (sm_103a): Q4_0 block
// decoding primitives, mbarrier and TMA wrappers with bounded waits.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace qm {

constexpr int kBlockBytes = 18;  // Q4_0 block: f16 d + 16 quant bytes
constexpr int kBlockElems = 32;

// Bits of the float 2^23: OR-ing a value v < 2^23 into its mantissa gives the
// float 2^23 + v exactly; subtracting 2^23 + 8 then leaves (v - 8) exactly.
constexpr uint32_t kMagicBits = 0x4B000000u;
constexpr float kMagicPlus8 = 8388616.0f;  // 2^23 + 8

// Device error bits (one word per translation unit that waits on copies).
constexpr unsigned int kErrWaitTimeout = 1u;

// Polls of an mbarrier before a wait gives up.  try_wait blocks for a
// hardware-defined slice per poll, so this bounds a wait to well under a
// second while never firing on a healthy copy.
constexpr uint32_t kMaxWaitPolls = 1u << 22;

// The f16 scale d -> f32 (exact).
__device__ __forceinline__ float f16_bits_to_float(uint32_t bits16) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(bits16)));
}

// (nibble - 8) as f32, exactly, for a value v in 0..15 already placed in the
// low bits of a word whose other bits match kMagicBits.
__device__ __forceinline__ float magic_minus8(uint32_t word_with_magic) {
    return __uint_as_float(word_with_magic) - kMagicPlus8;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_shared() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for phase `parity` of `bar`.  Returns false (and sets bit
// kErrWaitTimeout in *err) if the phase did not complete within the limit.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  unsigned int* err) {
    for (uint32_t i = 0; i < kMaxWaitPolls; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
    }
    atomicOr(err, kErrWaitTimeout);
    return false;
}

// 2-D TMA tile load (global -> this CTA's shared memory), completing on `bar`.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// src, dst 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_load_1d(void* dst, const void* src, uint32_t bytes,
                                             uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// 3-D TMA tile load (global -> this CTA's shared memory), completing on `bar`.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

// 4-D TMA tile load (global -> this CTA's shared memory), completing on `bar`.
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_addr(bar))
        : "memory");
}

// Hint: bring a 4-D TMA box into L2 (see tma_prefetch_l2_3d).
__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap* map, int x, int y, int z, int w) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// 16 bytes global -> shared memory, asynchronously, cached at L2 only (so no
// line cached in L1 before this launch can be returned); the thread waits
// for its own copies with cp_async_wait_all.  Both addresses 16-byte aligned.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)),
                 "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// Hint: bring `bytes` (a multiple of 16) at a 16-byte aligned global address
// into L2 (see tma_prefetch_l2_3d on why this can never return stale data).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Hint: bring a 3-D TMA box into L2 without copying it anywhere.  L2 is the
// device's point of coherence, so a line fetched early is still updated by
// any later write; only a load into shared memory or registers must wait.
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map, int x, int y, int z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

// Programmatic dependent launch.  launch_dependents lets the next kernel on
// the stream (when launched with programmatic serialization) start its
// prologue while this one runs; wait blocks until every kernel this one
// depends on has finished and its writes are visible.  Both are no-ops for
// a kernel launched the ordinary way.
__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Named barrier over the first `threads` threads of the CTA (a multiple of 32).
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---- thread-block clusters -------------------------------------------------

// All threads of every CTA of the cluster meet here.  Used only where no
// thread can have left the kernel (right after barrier initialisation), so
// the wait always ends.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" :::
                     "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// The shared::cluster address of the object at shared address `saddr` in the
// CTA of rank `rank` of this cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}

__device__ __forceinline__ float4 ld_dsmem_f4(uint32_t caddr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(caddr)
                 : "memory");
    return v;
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t caddr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(caddr) : "memory");
    return v;
}

// Arrive on the mbarrier at shared::cluster address `caddr` (possibly another
// CTA's), releasing this thread's earlier shared-memory writes to the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t caddr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(caddr) : "memory");
}

// Bounded wait on this CTA's mbarrier `bar`, acquiring the writes that other
// CTAs of the cluster released with their arrivals.
__device__ __forceinline__ bool mbar_wait_cluster_bounded(uint64_t* bar, uint32_t parity,
                                                          unsigned int* err) {
    for (uint32_t i = 0; i < kMaxWaitPolls; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    atomicOr(err, kErrWaitTimeout);
    return false;
}

// ---- Q8_0 quantization (section "quantize_q8_0": d = max|x| / 127, the
// block keeps d narrowed to binary16 and qs = round(x / d)), with the readings
// the library takes where the section is silent: f32 arithmetic with
// correctly rounded divisions, NaN elements do not raise the max, the
// narrowing rounds to nearest even, round() takes halfway cases away from
// zero, qs is clamped to [-127, 127], qs = 0 where d = 0 or x / d is NaN.

// d narrowed to binary16 (round to nearest even), as its 16 bits in the low
// half of a word: the packed conversion of (0, d), kept in 32-bit registers.
__device__ __forceinline__ uint32_t f16_bits_rn(float d) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(0.f), "f"(d));
    return r & 0xFFFFu;
}

// The quant of x for the block scale d (see the readings above).
__device__ __forceinline__ int q8_quant(float x, float d) {
    if (d == 0.f) return 0;
    const float t = __fdiv_rn(x, d);
    if (isnan(t)) return 0;
    return static_cast<int>(fminf(fmaxf(roundf(t), -127.f), 127.f));
}

// The quant byte of x, as q8_quant gives it, without a division in the
// common case.  With r = 1/d correctly rounded and t' = x * r rounded,
// t' = (x/d)(1 + e1)(1 + e2) and fl(x/d) = (x/d)(1 + e3), |e_i| <= 2^-24, so
// |t' - fl(x/d)| <= 127.5 * (3 * 2^-24 + 2^-48) < 2.3e-5 when |t'| < 127.4.
// Rounding t' to the nearest integer (adding 1.5 * 2^23 leaves it in the low
// mantissa bits, two's complement for negatives) then gives the same integer
// as rounding fl(x/d), half away from zero, unless t' is within 1e-4 of a
// half-integer; those, and every t' out of range or not finite (d = 0, a
// subnormal d whose reciprocal overflows, NaN or infinite x), take q8_quant.
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23
__device__ __forceinline__ uint32_t q8_quant_byte(float x, float d, float r) {
    const float t = __fmul_rn(x, r);
    const float m = __fadd_rn(t, kRoundMagic);
    const float ri = __fsub_rn(m, kRoundMagic);  // t rounded to an integer, exactly
    if (fabsf(t) < 127.4f && fabsf(__fsub_rn(t, ri)) < 0.4999f) return __float_as_uint(m) & 0xFFu;
    return static_cast<uint32_t>(q8_quant(x, d)) & 0xFFu;
}

// Quantize one unit of staged activations, f32 [M][256] as the TMA box lands,
// in place into [M][256] signed quants, then [M][8] f32 scales (the narrowed
// binary16 d, as f32), then [M][8] int32 values 8 * sum qs.  Lane l takes
// elements 8 (l % 4) .. + 7 of block l / 4 of every row; a block's max and
// quant sum meet over its four lanes by shuffles.  All rows are read before
// anything is written (the outputs overlap the inputs).
template <int M>
__device__ __forceinline__ void quantize_unit_q8(uint8_t* unit, int lane) {
    const int bl = lane >> 2;
    const int part = lane & 3;
    uint32_t qw[M][2];
    float dv[M];
    int bs[M];
#pragma unroll
    for (int m = 0; m < M; ++m) {
        const float4* src = reinterpret_cast<const float4*>(unit + (m * 256 + bl * 32 + 8 * part) * 4);
        const float4 x0 = src[0], x1 = src[1];
        const float x[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
        float amax = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
        const float d = __fdiv_rn(amax, 127.f);
        const float r = __frcp_rn(d);
        uint32_t qb[8];
        int sum = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            qb[e] = q8_quant_byte(x[e], d, r);
            sum += static_cast<int>(static_cast<int8_t>(qb[e]));
        }
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
        sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
        qw[m][0] = qb[0] | (qb[1] << 8) | (qb[2] << 16) | (qb[3] << 24);
        qw[m][1] = qb[4] | (qb[5] << 8) | (qb[6] << 16) | (qb[7] << 24);
        dv[m] = f16_bits_to_float(f16_bits_rn(d));
        bs[m] = 8 * sum;
    }
    __syncwarp();
    float* dq = reinterpret_cast<float*>(unit + M * 256);
    int* sq = reinterpret_cast<int*>(unit + M * 256 + M * 32);
#pragma unroll
    for (int m = 0; m < M; ++m) {
        *reinterpret_cast<uint2*>(unit + m * 256 + bl * 32 + 8 * part) = make_uint2(qw[m][0], qw[m][1]);
        if (part == 0) {
            dq[m * 8 + bl] = dv[m];
            sq[m * 8 + bl] = bs[m];
        }
    }
}

// 16-byte streaming store (output written once, not re-read by this kernel).
__device__ __forceinline__ void st_global_cs_v4(float* p, float a, float b, float c, float d) {
    asm volatile("st.global.cs.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(a), "f"(b), "f"(c),
                 "f"(d)
                 : "memory");
}

// 16-byte read-only load through the non-coherent path.
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Exact sum over `nblocks` consecutive Q4_0 blocks of one weight row against
// one activation row a_m: sum_k a_m[k] * ((q_k - 8) * d), element by element.
// Taken for a row whose block-scaled sum came out infinite or NaN: there a
// non-finite d times a zero weight (q = 8), or infinities of both signs, must
// give NaN exactly as the definition does.
static __device__ __noinline__ float row_range_exact(const uint8_t* row_blocks, int nblocks,
                                                     const float* a_m) {
    float s = 0.f;
    for (int b = 0; b < nblocks; ++b) {
        const uint8_t* blk = row_blocks + kBlockBytes * b;
        const float d = f16_bits_to_float(static_cast<uint32_t>(blk[0]) |
                                          (static_cast<uint32_t>(blk[1]) << 8));
        for (int j = 0; j < kBlockElems; ++j) {
            const uint32_t byte = blk[2 + (j & 15)];
            const uint32_t nib = (j < 16) ? (byte & 0xFu) : (byte >> 4);
            s = fmaf(__ldg(a_m + kBlockElems * b + j), magic_minus8(nib | kMagicBits) * d, s);
        }
    }
    return s;
}

}  // namespace qm

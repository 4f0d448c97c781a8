// Host-side interface between the C ABI (qm_api.cu) and the kernel files.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace qm {

struct DeviceInfo {
    int device = 0;
    int sm_count = 0;
    int max_smem_optin = 0;  // bytes of dynamic shared memory a CTA may opt into
};

// Scratch memory of a split-K GEMV that meets its partial sums in global
// memory: partial sums and per-row-group arrival counters.  Only the
// allocation-free entry point has one (a fixed array inside the library, of
// kNoallocPartFloats floats and kNoallocCounters counters); the regular path
// adds its K ranges up through thread-block clusters and needs none.
struct Workspace {
    float* part = nullptr;
    unsigned* ctr = nullptr;
    size_t part_floats = 0;
    int ctr_count = 0;
};
constexpr size_t kNoallocPartFloats = size_t(256) * 1024;  // 1 MB of split partial sums
constexpr int kNoallocCounters = 4096;                      // row groups with a split K

// Cached properties of the current device (queried once per device).
cudaError_t current_device_info(DeviceInfo* out);

// Tiled TMA descriptor: `rank` dimensions of `dtype` elements (innermost
// first), the byte strides of dimensions 1..rank-1 (multiples of 16), a box
// of box[d] elements, zero fill outside the tensor.
cudaError_t encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                         const int64_t* dims, const int64_t* strides, const int* box,
                         CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE);

cudaError_t launch_dequant_q4_0(const uint8_t* wq, int64_t n_blocks, float* out,
                                cudaStream_t stream, const DeviceInfo& dev);

// Q8_0 block stream <-> f32 (q8_0.cu).
cudaError_t launch_dequant_q8_0(const uint8_t* wq, int64_t n_blocks, float* out,
                                cudaStream_t stream, const DeviceInfo& dev);
cudaError_t launch_quantize_q8_0(const float* x, int64_t n_blocks, uint8_t* out,
                                 cudaStream_t stream, const DeviceInfo& dev);

// Consumers of the decode-regime GEMV.
enum class GemvKind { kSimt, kMma, kPacked };

// The automatic choice between the GEMV consumers.  Measured on GB300
// (back-to-back launches, both consumers in the same run): the packed FP32
// consumer is faster for M = 1..2 at N = 1024 (M = 1: 5.2 against 6.0 us;
// M = 2: 5.9 against 6.7 us at K = 4096); from N = 2048 up the tensor-core
// consumer is as fast or faster (M = 1, 2048 x 4096: 6.1 against 6.7 us;
// 4096 x 4096: 6.6 against 6.4 us; 14336 x 4096: 11.7 against 12.0 us), and
// for M = 3..8 it is the only consumer.
inline GemvKind gemv_auto_kind(int64_t M, int64_t N, int64_t /*K*/) {
    return (M <= 2 && N <= 1024) ? GemvKind::kPacked : GemvKind::kMma;
}

// Decode-regime GEMV, M = 1..8.  When wq and A are 16-byte aligned and
// K % 256 == 0: the staged GEMV (gemv_tc.cu) on tensor cores (kMma) or on
// packed FP32 FMAs (kPacked, M <= 2), else the persistent FP32 FMA kernel
// (kSimt); otherwise the generic kernel.
cudaError_t launch_gemv_q4_0(const float* A, const uint8_t* wq, float* C, int M, int64_t N,
                             int64_t K, cudaStream_t stream, const DeviceInfo& dev, GemvKind kind);

// The staged GEMV for K % 256 == 0 and 16-byte aligned A and wq: on tensor
// cores (mma.sync on bf16 pieces) for M = 1..8, or with packed FP32 FMAs
// (fma.rn.f32x2, one row per lane) for M = 1..2 when `packed`.  With ws null
// a split K adds up through thread-block clusters; otherwise through the
// scratch *ws (its counters zeroed on the stream first when clear_counters).
// Sets *launched = false and enqueues nothing when no launch plan fits.
cudaError_t launch_gemv_q4_0_tc(const float* A, const uint8_t* wq, float* C, int M, int64_t N,
                                int64_t K, cudaStream_t stream, const DeviceInfo& dev,
                                const Workspace* ws, bool packed, bool clear_counters,
                                bool* launched);
cudaError_t gemv_tc_read_device_error(unsigned int* bits, bool clear);

// The staged GEMV's integer consumer for the product with the activations
// quantized to Q8_0 first (K % 256 == 0, 16-byte aligned A and wq, M = 1..8);
// a split K adds up through thread-block clusters.  Sets *launched = false and
// enqueues nothing when no launch plan fits.
cudaError_t launch_gemv_q4_0_q8act_tc(const float* A, const uint8_t* wq, float* C, int M, int64_t N,
                                      int64_t K, cudaStream_t stream, const DeviceInfo& dev, bool* launched);

// C = dequant_q8_0(quantize_q8_0(A)) x dequant(W)^T for M = 1..8, K % 32 == 0
// (gemv_q8act.cu): the staged kernel where it applies, else a generic one.
cudaError_t launch_matmul_q4_0_q8act(const float* A, const uint8_t* wq, float* C, int M, int64_t N, int64_t K,
                                     cudaStream_t stream, const DeviceInfo& dev);

// The staged GEMV's launch plan for a device with sm_count SMs and smem_optin
// bytes of opt-in shared memory, without touching a device: with fit (the
// resident clusters of 2, 4 and 8 CTAs) the regular path's, else that of a
// split-K scratch of the given size: {RG, U, S, rps, c, hs, rbpc, nu_max,
// stages, grid, smem, W, cluster split}.  False when no plan fits.
bool gemv_tc_plan_query(int M, bool packed, int64_t N, int64_t K, int sm_count, int smem_optin,
                        const int* fit, int64_t part_floats, int64_t ctr_count, int64_t out[13]);

// The prefill GEMM's work items for a device with sm_count SMs on which fit[i]
// clusters of 2, 4, 8 CTAs can be resident at once: {BN, n-tiles, tiles,
// whole-tile items, s_rem, half-width split, items, cluster split}.
void gemm_tc_plan_query(int64_t M, int64_t N, int64_t K, int sm_count, const int fit[3], int64_t out[8]);

// The same GEMV with its split-K scratch in a fixed device array instead of
// a workspace (no allocation).  The first call on a device looks up the
// array's address.
cudaError_t launch_gemv_q4_0_noalloc(const float* A, const uint8_t* wq, float* C, int M, int64_t N,
                                     int64_t K, cudaStream_t stream, const DeviceInfo& dev);

// One problem of the persistent list GEMV (gemv_list.cu): M = 1, K % 2048 == 0,
// K <= kListMaxK, A and W 16-byte aligned; wait_for is -1 or an earlier index
// of the same launch (A is read once problems 0..wait_for are complete).
constexpr int kListMaxK = 14336;
constexpr int kListMaxProblems = 128;
struct GemvListItem {
    const float* A;
    const uint8_t* W;
    float* C;
    int64_t N;
    int64_t K;
    int wait_for;
};

// The list GEMV: one persistent launch over `count` (<= kListMaxProblems)
// problems.  `counters` (count unsigned, device memory) is required when some
// wait_for >= 0; it is cleared on the stream first.  With q8 every problem is
// the act-quant product (activations quantized to Q8_0 on chip, integer
// consumer).
cudaError_t launch_gemv_q4_0_list(const GemvListItem* items, int count, unsigned* counters,
                                  cudaStream_t stream, const DeviceInfo& dev, bool q8 = false);
cudaError_t gemv_list_read_device_error(unsigned int* bits, bool clear);


// Prefill GEMM on tcgen05 tensor cores: K % 256 == 0, 16-byte aligned A and wq.
bool gemm_tc_supported(const float* A, const uint8_t* wq, int64_t M, int64_t N, int64_t K);
cudaError_t launch_gemm_q4_0_tc(const float* A, const uint8_t* wq, float* C, int64_t M, int64_t N,
                                int64_t K, cudaStream_t stream, const DeviceInfo& dev);
cudaError_t gemm_tc_read_device_error(unsigned int* bits, bool clear);

// Prefill GEMM on FP32 FMA, any M >= 1.
cudaError_t launch_gemm_q4_0_simt(const float* A, const uint8_t* wq, float* C, int64_t M,
                                  int64_t N, int64_t K, cudaStream_t stream,
                                  const DeviceInfo& dev);

// Count one kernel enqueued by the library.
void note_launch();

// Launch `kernel` with programmatic stream serialization: it may start while
// the previous kernel on the stream is still running, as far as that kernel
// allows (griddepcontrol.launch_dependents), and must itself execute
// griddepcontrol.wait before touching memory that earlier work writes or reads.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same with thread-block clusters of `cluster_x` CTAs along x
// (gridDim.x a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t stream, unsigned cluster_x, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster_x;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// How many clusters of `cluster_x` CTAs of `kernel` can be resident at once
// (0 when the query fails).
template <typename... KArgs>
int max_active_clusters(void (*kernel)(KArgs...), dim3 block, size_t smem, unsigned cluster_x) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster_x);
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster_x;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}

// Read (and optionally clear) the device error words of the kernel files
// that wait on asynchronous copies; ORs them into *bits.
cudaError_t gemv_read_device_error(unsigned int* bits, bool clear);

// One-thread kernel whose bounded wait on an mbarrier nothing completes runs
// out and sets the device error word (qm_selftest_wait_timeout).
cudaError_t launch_wait_timeout_selftest(cudaStream_t stream);

}  // namespace qm

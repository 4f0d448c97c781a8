// The C ABI of libqm (declared in include/qm.h): argument checks, algorithm
// choice and launches on the caller's stream.  No call allocates device or
// host-pinned memory and none synchronizes with the device, except
// qm_device_status, which waits for the stream it is given; there is no host
// fallback.  What a call keeps between calls is host-side only: the device
// properties and the kernels' shared-memory attributes, set once per device.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

#include "qm.h"
#include "qm_internal.h"
#ifdef QM_TEST_HOOKS
#include <atomic>

#include "qm_test.h"
#endif

namespace qm {

namespace {

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
int g_dev_ready[kMaxDevices] = {0};
std::mutex g_dev_mutex;

PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;
uint64_t g_launches = 0;
std::once_flag g_encode_once;

}  // namespace

#ifdef QM_TEST_HOOKS
namespace {
std::atomic<int> g_injected_errors{0};
}  // namespace

bool take_injected_error() {
    int n = g_injected_errors.load();
    while (n > 0 && !g_injected_errors.compare_exchange_weak(n, n - 1)) {
    }
    return n > 0;
}
#endif

void note_launch() { __atomic_fetch_add(&g_launches, 1, __ATOMIC_RELAXED); }

uint64_t launch_count() { return __atomic_load_n(&g_launches, __ATOMIC_RELAXED); }

cudaError_t current_device_info(DeviceInfo* out) {
#ifdef QM_TEST_HOOKS
    // An injected failure (qm_test_inject_error): the calling entry point
    // returns QM_ERR_CUDA before anything is enqueued.
    if (take_injected_error()) return cudaErrorUnknown;
#endif
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (__atomic_load_n(&g_dev_ready[dev], __ATOMIC_ACQUIRE)) {
        *out = g_dev[dev];
        return cudaSuccess;
    }
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (!g_dev_ready[dev]) {
        DeviceInfo info;
        info.device = dev;
        err = cudaDeviceGetAttribute(&info.sm_count, cudaDevAttrMultiProcessorCount, dev);
        if (err != cudaSuccess) return err;
        err = cudaDeviceGetAttribute(&info.max_smem_optin,
                                     cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (err != cudaSuccess) return err;
        g_dev[dev] = info;
        __atomic_store_n(&g_dev_ready[dev], 1, __ATOMIC_RELEASE);
    }
    *out = g_dev[dev];
    return cudaSuccess;
}

// Tiled TMA descriptor: `rank` dimensions of `dtype` elements (innermost
// first), the byte strides of dimensions 1..rank-1 (multiples of 16), a box
// of box[d] elements, zero fill outside the tensor.
cudaError_t encode_tiled(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                         const int64_t* dims, const int64_t* strides, const int* box,
                         CUtensorMapSwizzle swizzle) {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    });
    if (!g_encode_tiled) return cudaErrorNotSupported;
    if (rank < 1 || rank > 5) return cudaErrorInvalidValue;
    cuuint64_t d[5], st[4];
    cuuint32_t b[5], es[5];
    for (int i = 0; i < rank; ++i) {
        d[i] = static_cast<cuuint64_t>(dims[i]);
        b[i] = static_cast<cuuint32_t>(box[i]);
        es[i] = 1;
        if (i > 0) st[i - 1] = static_cast<cuuint64_t>(strides[i - 1]);
    }
    CUresult r = g_encode_tiled(map, dtype, rank, const_cast<void*>(base), d,
                                st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace qm

namespace {

constexpr int kVersion = 100;  // 0.1.0

bool mul_ok(int64_t a, int64_t b, int64_t* out) {
    if (a < 0 || b < 0) return false;
    if (a != 0 && b > INT64_MAX / a) return false;
    *out = a * b;
    return true;
}

bool overlaps(const void* a, int64_t a_bytes, const void* b, int64_t b_bytes) {
    if (a_bytes <= 0 || b_bytes <= 0) return false;
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + static_cast<uintptr_t>(b_bytes) && b0 < a0 + static_cast<uintptr_t>(a_bytes);
}

// The pointer must be device-accessible memory of `device`: device or managed
// memory, or host memory registered/mapped with a device address.
int check_pointer(const void* p, int device) {
    cudaPointerAttributes attr;
    cudaError_t err = cudaPointerGetAttributes(&attr, p);
    if (err != cudaSuccess) {
        cudaGetLastError();
        return QM_ERR_POINTER;
    }
    switch (attr.type) {
        case cudaMemoryTypeDevice:
            return attr.device == device ? QM_OK : QM_ERR_POINTER;
        case cudaMemoryTypeManaged:
            return QM_OK;
        case cudaMemoryTypeHost:
            return attr.devicePointer == p ? QM_OK : QM_ERR_POINTER;
        default:
            return QM_ERR_POINTER;
    }
}

int from_cuda(cudaError_t err) { return err == cudaSuccess ? QM_OK : QM_ERR_CUDA; }

int run_matmul(const float* A, const void* wq, float* C, int64_t M, int64_t N, int64_t K, int algo,
               cudaStream_t s, const qm::DeviceInfo& dev);

// Host checks of one product's operands (the qm_matmul_q4_0 rules); on
// success the byte counts of A, wq and C.
int check_matmul(const float* A, const void* wq, const float* C, int64_t M, int64_t N, int64_t K,
                 int64_t* a_bytes, int64_t* w_bytes, int64_t* c_bytes) {
    if (M < 0 || N < 0 || K < 0 || (K % 32) != 0) return QM_ERR_SHAPE;
    int64_t a_elems, c_elems, w_elems;
    if (!mul_ok(M, K, &a_elems) || !mul_ok(a_elems, 4, a_bytes) || !mul_ok(M, N, &c_elems) ||
        !mul_ok(c_elems, 4, c_bytes) || !mul_ok(N, K / 32, &w_elems) || !mul_ok(w_elems, 18, w_bytes))
        return QM_ERR_SHAPE;
    if (M == 0 || N == 0) return QM_OK;
    if (!C) return QM_ERR_NULL;
    if (K > 0 && (!A || !wq)) return QM_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(C) & 3u) != 0) return QM_ERR_ALIGN;
    if (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 3u) != 0 || (reinterpret_cast<uintptr_t>(wq) & 1u) != 0))
        return QM_ERR_ALIGN;
    if (overlaps(C, *c_bytes, A, *a_bytes) || overlaps(C, *c_bytes, wq, *w_bytes)) return QM_ERR_ALIAS;
    if (M > 0x7FFFFFFF || N > 0x7FFFFFFF) return QM_ERR_SHAPE;
    return QM_OK;
}

int matmul_impl(const float* A, const void* wq, float* C, int64_t M, int64_t N, int64_t K,
                int algo, void* stream) {
    if (algo < QM_ALGO_AUTO || algo > QM_ALGO_GEMV_PK) return QM_ERR_SHAPE;
    int64_t a_bytes = 0, w_bytes = 0, c_bytes = 0;
    int rc = check_matmul(A, wq, C, M, N, K, &a_bytes, &w_bytes, &c_bytes);
    if (rc != QM_OK) return rc;
    if ((algo == QM_ALGO_GEMV || algo == QM_ALGO_GEMV_SIMT) && M > 8) return QM_ERR_UNSUPPORTED;
    if (algo == QM_ALGO_GEMV_PK && M > 2) return QM_ERR_UNSUPPORTED;
    if (M == 0 || N == 0) return QM_OK;

    qm::DeviceInfo dev;
    if (qm::current_device_info(&dev) != cudaSuccess) return QM_ERR_CUDA;
    rc = check_pointer(C, dev.device);
    if (rc == QM_OK && K > 0) rc = check_pointer(A, dev.device);
    if (rc == QM_OK && K > 0) rc = check_pointer(wq, dev.device);
    if (rc != QM_OK) return rc;

    return run_matmul(A, wq, C, M, N, K, algo, static_cast<cudaStream_t>(stream), dev);
}

// The launch part of qm_matmul_q4_0 for arguments already checked.
int run_matmul(const float* A, const void* wq, float* C, int64_t M, int64_t N, int64_t K, int algo,
               cudaStream_t s, const qm::DeviceInfo& dev) {
    if (K == 0) return from_cuda(cudaMemsetAsync(C, 0, static_cast<size_t>(M * N * 4), s));
    const uint8_t* w = static_cast<const uint8_t*>(wq);
    const bool tc_ok = qm::gemm_tc_supported(A, w, M, N, K);
    if (algo == QM_ALGO_AUTO) {
        if (M <= 8)
            algo = qm::gemv_auto_kind(M, N, K) == qm::GemvKind::kPacked ? QM_ALGO_GEMV_PK : QM_ALGO_GEMV;
        else algo = tc_ok ? QM_ALGO_GEMM_TC : QM_ALGO_GEMM_SIMT;
    }
    if (algo == QM_ALGO_GEMV || algo == QM_ALGO_GEMV_SIMT || algo == QM_ALGO_GEMV_PK) {
        const qm::GemvKind kind = algo == QM_ALGO_GEMV      ? qm::GemvKind::kMma
                                  : algo == QM_ALGO_GEMV_PK ? qm::GemvKind::kPacked
                                                            : qm::GemvKind::kSimt;
        return from_cuda(qm::launch_gemv_q4_0(A, w, C, static_cast<int>(M), N, K, s, dev, kind));
    }
    if (algo == QM_ALGO_GEMM_TC) {
        if (!tc_ok) return QM_ERR_UNSUPPORTED;
        return from_cuda(qm::launch_gemm_q4_0_tc(A, w, C, M, N, K, s, dev));
    }
    return from_cuda(qm::launch_gemm_q4_0_simt(A, w, C, M, N, K, s, dev));
}

}  // namespace

extern "C" {

int qm_version(void) { return kVersion; }

const char* qm_status_string(int status) {
    switch (status) {
        case QM_OK: return "ok";
        case QM_ERR_NULL: return "a required pointer is NULL";
        case QM_ERR_SHAPE: return "invalid size (negative, K not a multiple of 32, or overflow)";
        case QM_ERR_ALIGN: return "misaligned pointer (wq needs 2 bytes, A/C/out 4 bytes)";
        case QM_ERR_ALIAS: return "an output overlaps an input";
        case QM_ERR_CUDA: return "a CUDA call or kernel launch failed";
        case QM_ERR_TIMEOUT: return "a kernel gave up a bounded wait (an asynchronous copy or a peer that did not arrive)";
        case QM_ERR_UNSUPPORTED: return "the forced algorithm cannot run this shape";
        case QM_ERR_POINTER: return "a pointer is not device memory of the current device";
        case QM_ERR_TOO_LARGE: return "beyond the fixed scratch of qm_matmul_q4_0_noalloc (M > 8)";
        default: return "unknown status";
    }
}

int qm_dequant_q4_0(const void* wq, int64_t n_blocks, float* out, void* stream) {
    if (n_blocks < 0) return QM_ERR_SHAPE;
    int64_t in_bytes, out_bytes;
    if (!mul_ok(n_blocks, 18, &in_bytes) || !mul_ok(n_blocks, 128, &out_bytes)) return QM_ERR_SHAPE;
    if (n_blocks == 0) return QM_OK;
    if (!wq || !out) return QM_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(wq) & 1u) != 0 || (reinterpret_cast<uintptr_t>(out) & 3u) != 0)
        return QM_ERR_ALIGN;
    if (overlaps(out, out_bytes, wq, in_bytes)) return QM_ERR_ALIAS;
    qm::DeviceInfo dev;
    if (qm::current_device_info(&dev) != cudaSuccess) return QM_ERR_CUDA;
    int rc = check_pointer(wq, dev.device);
    if (rc == QM_OK) rc = check_pointer(out, dev.device);
    if (rc != QM_OK) return rc;
    return from_cuda(qm::launch_dequant_q4_0(static_cast<const uint8_t*>(wq), n_blocks, out,
                                             static_cast<cudaStream_t>(stream), dev));
}

int qm_dequant_q8_0(const void* wq, int64_t n_blocks, float* out, void* stream) {
    if (n_blocks < 0) return QM_ERR_SHAPE;
    int64_t in_bytes, out_bytes;
    if (!mul_ok(n_blocks, 34, &in_bytes) || !mul_ok(n_blocks, 128, &out_bytes)) return QM_ERR_SHAPE;
    if (n_blocks == 0) return QM_OK;
    if (!wq || !out) return QM_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(out) & 3u) != 0) return QM_ERR_ALIGN;
    if (overlaps(out, out_bytes, wq, in_bytes)) return QM_ERR_ALIAS;
    qm::DeviceInfo dev;
    if (qm::current_device_info(&dev) != cudaSuccess) return QM_ERR_CUDA;
    int rc = check_pointer(wq, dev.device);
    if (rc == QM_OK) rc = check_pointer(out, dev.device);
    if (rc != QM_OK) return rc;
    return from_cuda(qm::launch_dequant_q8_0(static_cast<const uint8_t*>(wq), n_blocks, out,
                                             static_cast<cudaStream_t>(stream), dev));
}

int qm_quantize_q8_0(const float* x, int64_t n_elements, void* out, void* stream) {
    if (n_elements < 0 || (n_elements % 32) != 0) return QM_ERR_SHAPE;
    const int64_t n_blocks = n_elements / 32;
    int64_t in_bytes, out_bytes;
    if (!mul_ok(n_elements, 4, &in_bytes) || !mul_ok(n_blocks, 34, &out_bytes)) return QM_ERR_SHAPE;
    if (n_blocks == 0) return QM_OK;
    if (!x || !out) return QM_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(x) & 3u) != 0) return QM_ERR_ALIGN;
    if (overlaps(out, out_bytes, x, in_bytes)) return QM_ERR_ALIAS;
    qm::DeviceInfo dev;
    if (qm::current_device_info(&dev) != cudaSuccess) return QM_ERR_CUDA;
    int rc = check_pointer(x, dev.device);
    if (rc == QM_OK) rc = check_pointer(out, dev.device);
    if (rc != QM_OK) return rc;
    return from_cuda(qm::launch_quantize_q8_0(x, n_blocks, static_cast<uint8_t*>(out),
                                              static_cast<cudaStream_t>(stream), dev));
}

int qm_matmul_q4_0(const float* A, const void* wq, float* C, int64_t M, int64_t N, int64_t K,
                   void* stream) {
    return matmul_impl(A, wq, C, M, N, K, QM_ALGO_AUTO, stream);
}

int qm_matmul_q4_0_algo(const float* A, const void* wq, float* C, int64_t M, int64_t N, int64_t K,
                        int algo, void* stream) {
    return matmul_impl(A, wq, C, M, N, K, algo, stream);
}

// Allocation-free GEMV: the same checks as qm_matmul_q4_0, scratch from a
// fixed device array (see include/qm.h).
int qm_matmul_q4_0_noalloc(const float* A, const void* wq, float* C, int64_t M, int64_t N,
                           int64_t K, void* stream) {
    if (M < 0 || N < 0 || K < 0 || (K % 32) != 0) return QM_ERR_SHAPE;
    int64_t a_elems, c_elems, w_elems, a_bytes, c_bytes, w_bytes;
    if (!mul_ok(M, K, &a_elems) || !mul_ok(a_elems, 4, &a_bytes) || !mul_ok(M, N, &c_elems) ||
        !mul_ok(c_elems, 4, &c_bytes) || !mul_ok(N, K / 32, &w_elems) ||
        !mul_ok(w_elems, 18, &w_bytes))
        return QM_ERR_SHAPE;
    if (M > 8) return QM_ERR_TOO_LARGE;
    if (M == 0 || N == 0) return QM_OK;
    if (!C) return QM_ERR_NULL;
    if (K > 0 && (!A || !wq)) return QM_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(C) & 3u) != 0) return QM_ERR_ALIGN;
    if (K > 0 && ((reinterpret_cast<uintptr_t>(A) & 3u) != 0 ||
                  (reinterpret_cast<uintptr_t>(wq) & 1u) != 0))
        return QM_ERR_ALIGN;
    if (overlaps(C, c_bytes, A, a_bytes) || overlaps(C, c_bytes, wq, w_bytes)) return QM_ERR_ALIAS;
    if (N > 0x7FFFFFFF) return QM_ERR_SHAPE;
    qm::DeviceInfo dev;
    if (qm::current_device_info(&dev) != cudaSuccess) return QM_ERR_CUDA;
    int rc = check_pointer(C, dev.device);
    if (rc == QM_OK && K > 0) rc = check_pointer(A, dev.device);
    if (rc == QM_OK && K > 0) rc = check_pointer(wq, dev.device);
    if (rc != QM_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) return from_cuda(cudaMemsetAsync(C, 0, static_cast<size_t>(c_bytes), s));
    return from_cuda(qm::launch_gemv_q4_0_noalloc(A, static_cast<const uint8_t*>(wq), C,
                                                  static_cast<int>(M), N, K, s, dev));
}

// The product with the activations quantized to Q8_0 first: the checks of
// qm_matmul_q4_0, M <= 8.
int qm_matmul_q4_0_q8act(const float* A, const void* wq, float* C, int64_t M, int64_t N, int64_t K,
                         void* stream) {
    int64_t a_bytes = 0, w_bytes = 0, c_bytes = 0;
    int rc = check_matmul(A, wq, C, M, N, K, &a_bytes, &w_bytes, &c_bytes);
    if (rc != QM_OK) return rc;
    if (M > 8) return QM_ERR_TOO_LARGE;
    if (M == 0 || N == 0) return QM_OK;
    qm::DeviceInfo dev;
    if (qm::current_device_info(&dev) != cudaSuccess) return QM_ERR_CUDA;
    rc = check_pointer(C, dev.device);
    if (rc == QM_OK && K > 0) rc = check_pointer(A, dev.device);
    if (rc == QM_OK && K > 0) rc = check_pointer(wq, dev.device);
    if (rc != QM_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (K == 0) return from_cuda(cudaMemsetAsync(C, 0, static_cast<size_t>(c_bytes), s));
    return from_cuda(qm::launch_matmul_q4_0_q8act(A, static_cast<const uint8_t*>(wq), C, static_cast<int>(M), N,
                                                  K, s, dev));
}

// The list GEMV: checks every problem as qm_matmul_q4_0 does, then the
// ordering rules between problems, then runs maximal runs of problems the
// persistent kernel takes (M = 1, K % 2048 == 0, K <= 14336, 16-byte aligned
// A and wq) as launches of up to 128 problems; any other problem runs alone
// through qm_matmul_q4_0's path, in list order on the same stream.
}  // extern "C"

namespace {

// qm_gemv_q4_0_list and qm_gemv_q4_0_q8act_list: the same checks and
// grouping; q8 selects the act-quant product.
int gemv_list_impl(const qm_gemv_problem* problems, int64_t count, int64_t M, uint32_t* counters,
                   void* stream, bool q8) {
    if (count < 0 || M < 0) return QM_ERR_SHAPE;
    if (count == 0 || M == 0) return QM_OK;
    if (!problems) return QM_ERR_NULL;
    if (count > (int64_t(1) << 24)) return QM_ERR_SHAPE;
    if (q8 && M > 8) return QM_ERR_TOO_LARGE;
    if (counters && (reinterpret_cast<uintptr_t>(counters) & 3u) != 0) return QM_ERR_ALIGN;
    std::vector<int64_t> ab(count), wb(count), cb(count);
    for (int64_t i = 0; i < count; ++i) {
        const qm_gemv_problem& p = problems[i];
        if (p.reserved != 0 || p.wait_for < -1 || p.wait_for >= i) return QM_ERR_SHAPE;
        const int rc = check_matmul(p.A, p.wq, p.C, M, p.N, p.K, &ab[i], &wb[i], &cb[i]);
        if (rc != QM_OK) return rc;
        if (p.N == 0) ab[i] = wb[i] = cb[i] = 0;
        if (p.K == 0) ab[i] = wb[i] = 0;
    }
    // Ordering between problems: no output overlaps any weight stream; an
    // output of problem i that overlaps an operand of a later problem j (or j's
    // output overlaps i's activations) needs j to wait for i; the counters
    // overlap nothing.
    const int64_t ctr_bytes = counters ? count * 4 : 0;
    for (int64_t i = 0; i < count; ++i) {
        const qm_gemv_problem& p = problems[i];
        if (overlaps(counters, ctr_bytes, p.A, ab[i]) || overlaps(counters, ctr_bytes, p.wq, wb[i]) ||
            overlaps(counters, ctr_bytes, p.C, cb[i]))
            return QM_ERR_ALIAS;
        for (int64_t j = 0; j < count; ++j) {
            if (j != i && overlaps(p.C, cb[i], problems[j].wq, wb[j])) return QM_ERR_ALIAS;
        }
        for (int64_t j = i + 1; j < count; ++j) {
            const qm_gemv_problem& q = problems[j];
            const bool touch = overlaps(p.C, cb[i], q.A, ab[j]) || overlaps(p.C, cb[i], q.C, cb[j]) ||
                               overlaps(q.C, cb[j], p.A, ab[i]);
            if (touch && q.wait_for < i) return QM_ERR_ALIAS;
        }
    }
    qm::DeviceInfo dev;
    if (qm::current_device_info(&dev) != cudaSuccess) return QM_ERR_CUDA;
    for (int64_t i = 0; i < count; ++i) {
        const qm_gemv_problem& p = problems[i];
        if (p.N == 0) continue;
        int rc = check_pointer(p.C, dev.device);
        if (rc == QM_OK && p.K > 0) rc = check_pointer(p.A, dev.device);
        if (rc == QM_OK && p.K > 0) rc = check_pointer(p.wq, dev.device);
        if (rc != QM_OK) return rc;
    }
    if (counters && check_pointer(counters, dev.device) != QM_OK) return QM_ERR_POINTER;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto list_ok = [&](const qm_gemv_problem& p) {
        return M == 1 && p.N > 0 && p.K > 0 && (p.K % 2048) == 0 && p.K <= qm::kListMaxK &&
               (reinterpret_cast<uintptr_t>(p.A) & 15u) == 0 && (reinterpret_cast<uintptr_t>(p.wq) & 15u) == 0;
    };
    std::vector<qm::GemvListItem> items;
    int64_t i = 0;
    while (i < count) {
        const qm_gemv_problem& p = problems[i];
        if (p.N == 0) {
            ++i;
            continue;
        }
        if (!list_ok(p)) {
            int rc;
            if (!q8) {
                rc = run_matmul(p.A, p.wq, p.C, M, p.N, p.K, QM_ALGO_AUTO, s, dev);
            } else if (p.K == 0) {
                rc = from_cuda(cudaMemsetAsync(p.C, 0, static_cast<size_t>(M * p.N * 4), s));
            } else {
                rc = from_cuda(qm::launch_matmul_q4_0_q8act(p.A, static_cast<const uint8_t*>(p.wq), p.C,
                                                            static_cast<int>(M), p.N, p.K, s, dev));
            }
            if (rc != QM_OK) return rc;
            ++i;
            continue;
        }
        // A run of list problems from i: at most kListMaxProblems; without
        // counters it ends before a problem that waits on one inside it
        // (the launch boundary then orders them).
        items.clear();
        const int64_t start = i;
        while (i < count && static_cast<int>(items.size()) < qm::kListMaxProblems && list_ok(problems[i])) {
            const qm_gemv_problem& q = problems[i];
            const int w = q.wait_for >= start ? static_cast<int>(q.wait_for - start) : -1;
            if (w >= 0 && !counters) break;
            items.push_back({q.A, static_cast<const uint8_t*>(q.wq), q.C, q.N, q.K, w});
            ++i;
        }
        const int rc = from_cuda(qm::launch_gemv_q4_0_list(items.data(), static_cast<int>(items.size()),
                                                           counters ? counters + start : nullptr, s, dev, q8));
        if (rc != QM_OK) return rc;
    }
    return QM_OK;
}

}  // namespace

extern "C" {

int qm_gemv_q4_0_list(const qm_gemv_problem* problems, int64_t count, int64_t M, uint32_t* counters,
                      void* stream) {
    return gemv_list_impl(problems, count, M, counters, stream, false);
}

int qm_gemv_q4_0_q8act_list(const qm_gemv_problem* problems, int64_t count, int64_t M, uint32_t* counters,
                            void* stream) {
    return gemv_list_impl(problems, count, M, counters, stream, true);
}

uint64_t qm_launch_count(void) { return qm::launch_count(); }

int qm_gemm_plan(int64_t M, int64_t N, int64_t K, int sm_count, int fit2, int fit4, int fit8,
                 int64_t* out) {
    if (!out) return QM_ERR_NULL;
    if (M < 1 || N < 1 || K < 256 || (K % 256) != 0 || sm_count < 1 ||
        !qm::gemm_tc_supported(reinterpret_cast<const float*>(16), reinterpret_cast<const uint8_t*>(16),
                               M, N, K))
        return QM_ERR_SHAPE;
    const int fit[3] = {fit2, fit4, fit8};
    qm::gemm_tc_plan_query(M, N, K, sm_count, fit, out);
    return QM_OK;
}

int qm_gemv_plan(int64_t M, int64_t N, int64_t K, int packed, int sm_count, int smem_optin, int fit2,
                 int fit4, int fit8, int noalloc, int64_t* out) {
    if (!out) return QM_ERR_NULL;
    if (M < 1 || M > (packed ? 2 : 8) || N < 1 || N > 0x7FFFFFFF || K < 256 || (K % 256) != 0 ||
        K > (int64_t(1) << 30) || sm_count < 1 || smem_optin < 1 || fit2 < 0 || fit4 < 0 || fit8 < 0)
        return QM_ERR_SHAPE;
    const int fit[3] = {fit2, fit4, fit8};
    return qm::gemv_tc_plan_query(static_cast<int>(M), packed != 0, N, K, sm_count, smem_optin,
                                  noalloc ? nullptr : fit, static_cast<int64_t>(qm::kNoallocPartFloats),
                                  qm::kNoallocCounters, out)
               ? QM_OK
               : QM_ERR_UNSUPPORTED;
}

int qm_selftest_wait_timeout(void* stream) {
    qm::DeviceInfo dev;
    if (qm::current_device_info(&dev) != cudaSuccess) return QM_ERR_CUDA;
    return from_cuda(qm::launch_wait_timeout_selftest(static_cast<cudaStream_t>(stream)));
}

int qm_device_status(void* stream, int clear) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return QM_ERR_CUDA;
    unsigned int bits = 0;
    if (qm::gemv_read_device_error(&bits, clear != 0) != cudaSuccess) return QM_ERR_CUDA;
    if (qm::gemm_tc_read_device_error(&bits, clear != 0) != cudaSuccess) return QM_ERR_CUDA;
    if (qm::gemv_tc_read_device_error(&bits, clear != 0) != cudaSuccess) return QM_ERR_CUDA;
    if (qm::gemv_list_read_device_error(&bits, clear != 0) != cudaSuccess) return QM_ERR_CUDA;
    return bits ? QM_ERR_TIMEOUT : QM_OK;
}

#ifdef QM_TEST_HOOKS
int qm_test_inject_error(int calls) {
    if (calls < 0) return QM_ERR_SHAPE;
    qm::g_injected_errors.store(calls);
    return QM_OK;
}
#endif

}  // extern "C"

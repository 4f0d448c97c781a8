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

// Cached properties of the current device (queried once per device).
cudaError_t current_device_info(DeviceInfo* out);

// 2-D TMA descriptor over a weight stream seen as a byte matrix
// [rows][row_bytes] (row_bytes a multiple of 16), box box_rows x box_bytes,
// zero fill outside the matrix.
cudaError_t encode_weight_map_2d(CUtensorMap* map, const void* base, int64_t row_bytes,
                                 int64_t rows, int box_bytes, int box_rows);

cudaError_t launch_dequant_q4_0(const uint8_t* wq, int64_t n_blocks, float* out,
                                cudaStream_t stream, const DeviceInfo& dev);

// Decode-regime GEMV, M = 1..8.  Picks the TMA-staged kernel when wq and A
// are 16-byte aligned and K % 256 == 0, else the generic kernel.
cudaError_t launch_gemv_q4_0(const float* A, const uint8_t* wq, float* C, int M, int64_t N,
                             int64_t K, cudaStream_t stream, const DeviceInfo& dev);

// Prefill GEMM on FP32 FMA, any M >= 1.
cudaError_t launch_gemm_q4_0_simt(const float* A, const uint8_t* wq, float* C, int64_t M,
                                  int64_t N, int64_t K, cudaStream_t stream,
                                  const DeviceInfo& dev);

// Count one kernel enqueued by the library.
void note_launch();

// Read (and optionally clear) the device error words of the kernel files
// that wait on asynchronous copies; ORs them into *bits.
cudaError_t gemv_read_device_error(unsigned int* bits, bool clear);

}  // namespace qm

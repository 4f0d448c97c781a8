/*
 * qm_test.h — test-only hooks of libqm.  They exist only in the copy of the
 * library built with -DQM_TEST_HOOKS (bit_block_quantized_qm_gb300/build.py,
 * build_test_hooks(), into _build/test/libqm.so); the product library does
 * not export them.
 */
#ifndef QM_TEST_H
#define QM_TEST_H

#include "qm.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * qm_test_inject_error — the next `calls` calls of entry points that would
 * enqueue work on a device (every qm_dequant_*, qm_quantize_q8_0,
 * qm_matmul_*, qm_gemv_q4_0_list and qm_selftest_wait_timeout call that passes
 * its host-side argument checks) fail with QM_ERR_CUDA and enqueue nothing, as
 * a failed CUDA call in them would.  Host-only queries (plans, strings,
 * qm_device_status) are not counted.  calls = 0 clears a pending injection.
 * Returns QM_OK, or QM_ERR_SHAPE for calls < 0.  Thread-safe; the count is
 * process-wide.
 */
QM_API int qm_test_inject_error(int calls);

#ifdef __cplusplus
}
#endif

#endif /* QM_TEST_H */

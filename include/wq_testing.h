/*
 * wq_testing.h -- a hook of libwq for its own failure-path tests; not part of
 * the matmul ABI of wq.h.
 *
 * Every barrier wait in the library's kernels is bounded: one that runs out
 * records a flag in the device status word (read and cleared by
 * wq_check_device, WQ_ERR_TIMEOUT), raises its thread block's abort flag so
 * that the block's other waits end at once, waits (bounded) for its own
 * copies in flight, and the kernel returns.  The pages have no counterpart:
 * the barrier_acquire of Marlin's cross-block reduction (aphrodite-engine
 * marlin_cuda_kernel.cu) spins without a limit.  This hook makes that path
 * run without any fault.
 */
#ifndef WQ_TESTING_H
#define WQ_TESTING_H

#include "wq.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * wq_testing_decode_timeout -- wq_matmul on the few-token kernel (M <= 64,
 * WQ_ERR_SHAPE otherwise) with every barrier wait limited to
 * wait_limit_cycles SM clock cycles (1e4 .. 8e9) and the producer of every
 * thread block withholding ring stage withhold_stage (>= 0): it never arms
 * that stage's barrier nor copies into it, so the consumers' wait for it runs
 * out.  The call returns WQ_OK once the kernel is enqueued; wq_check_device
 * then reports WQ_ERR_TIMEOUT if a wait ran out (a block with fewer stages
 * than withhold_stage + 1 finishes normally).  `out` holds no meaningful
 * result afterwards; the device stays usable.  Other arguments as wq_matmul.
 */
WQ_API wq_status wq_testing_decode_timeout(const void *x, wq_dtype x_dtype, const void *packed_w,
                                           const void *scales, wq_dtype s_dtype, const int32_t *zeros,
                                           int M, int N, int K, int w_bit, int group_size, float *out,
                                           void *workspace, size_t workspace_bytes,
                                           long long wait_limit_cycles, int withhold_stage, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* WQ_TESTING_H */

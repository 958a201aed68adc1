/*
 * fastweight_selftest.h -- self-test of the tensor-core building blocks that
 * the bf16 forward of fastweight.h is made of.  Not part of the layer's
 * arithmetic: it exists so a test can pin, on the GPU, the operand layouts,
 * matrix and instruction descriptors, the tensor-memory accumulator layout and
 * the completion barriers against a plain matrix product.
 */
#ifndef FASTWEIGHT_SELFTEST_H
#define FASTWEIGHT_SELFTEST_H

#include "fastweight.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * fw_selftest_umma -- D = A * B^T on one CTA with tcgen05.mma (bf16 operands,
 * fp32 accumulation in tensor memory), M = 128.
 *
 *   A : [128, K] fp32 device buffer whose values are exactly representable in
 *       bf16 (they are converted on the device without loss);
 *   B : [N, K] fp32 device buffer, same condition;
 *   D : [128, N] fp32 device output.
 *   N in {16, 32, 64, 128, 256};  K in {16, 32, 64, 128}.
 *   a_mn / b_mn : 0 stages that operand K-major, 1 stages it MN-major, both
 *                 with the 128-byte swizzle, exactly as the forward does.
 *   swap_mn     : 0 (the layout the forward uses) or 1 (leading and stride
 *                 byte offsets of MN-major descriptors exchanged; a check
 *                 that the test can tell the two conventions apart).
 * Returns FW_OK, FW_ERR_INVALID_ARG, FW_ERR_CUDA.  Asynchronous on `stream`;
 * a bounded wait that gives up is reported by fw_device_status().
 */
FW_API int fw_selftest_umma(const float *A, const float *B, float *D, int N, int K, int a_mn,
                            int b_mn, int swap_mn, void *stream);

/*
 * fw_selftest_wait_timeout -- exercises the failure path of the library's
 * bounded waits without hanging or faulting the GPU: one CTA waits on an
 * mbarrier that nothing ever arrives at, gives up after limit_us
 * microseconds (1 .. 100000), records FW_ERR_TIMEOUT in the device status
 * word and exits normally.  The next fw_device_status() returns
 * FW_ERR_TIMEOUT and clears it; the CUDA context stays usable.
 */
FW_API int fw_selftest_wait_timeout(int limit_us, void *stream);

/*
 * fw_selftest_flag_timeout -- the same for the ready-flag waits of the
 * single-launch forward (a CTA spinning, with sleeps, on a flag in global
 * memory that another CTA sets): one CTA waits on a flag that nothing ever
 * sets, gives up after limit_us microseconds (1 .. 100000), records
 * FW_ERR_TIMEOUT in the device status word and exits normally.
 */
FW_API int fw_selftest_flag_timeout(int limit_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FASTWEIGHT_SELFTEST_H */

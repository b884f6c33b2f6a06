/*
 * lrkv_testing.h -- test-only controls of liblrkv. Not for production use.
 *
 * The paper has no counterpart: these entry points exist so that tests can
 * drive the library's failure paths without faulting or hanging the GPU.
 */
#ifndef LRKV_TESTING_H_
#define LRKV_TESTING_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * lrkv_testing_set_decode_stall -- enable != 0: every following
 * lrkv_attn_decode call that runs the G-mode decode kernel (any rank but the
 * rank-64 rebuild mode) makes its W-issuing warp wait, once, on an mbarrier
 * that nothing arrives at. The wait gives up after about 2^20 cycles, stores
 * LRKV_ERR_TIMEOUT in dev_status and raises the CTA's abort flag; every other
 * role leaves its loop, the MMAs and copies already issued are waited for, and
 * the kernel returns (its output is not valid). enable = 0 restores normal
 * calls. Process-wide; not synchronised with calls already enqueued.
 */
void lrkv_testing_set_decode_stall(int32_t enable);

#ifdef __cplusplus
}
#endif

#endif /* LRKV_TESTING_H_ */

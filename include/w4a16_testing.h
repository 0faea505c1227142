/*
 * w4a16_testing.h - test hooks of the W4A16 library (not for production use).
 *
 * They exist so that a test can drive the failure path of the device-side
 * bounded waits (a wait that expires reports W4_ERR_TIMEOUT through
 * w4a16_device_status and the kernel returns) without faulting or hanging a
 * GPU.  Status codes are those of w4a16.h.
 */
#ifndef W4A16_TESTING_H
#define W4A16_TESTING_H

#include "w4a16.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * w4a16_testing_set_seq_wait - settings of the completion-counter waits of
 * w4_gemv_seq launches issued after this call (process-wide).
 *   wait_ns      limit of each counter wait in nanoseconds, at most 2 s;
 *                0 restores the default of 2 s.
 *   target_bump  added to every counter target.  0 is normal operation; any
 *                other value makes every counter wait unmeetable (no CTA can
 *                pass the first one, so the count never grows), so each waits
 *                out its limit, records the expiry (w4a16_device_status then
 *                returns W4_ERR_TIMEOUT) and the launch finishes without valid
 *                results.  Call with (0, 0) to restore normal operation.
 * Returns W4A16_OK, or W4_ERR_SHAPE if wait_ns exceeds 2 s.  Not synchronised
 * with w4_gemv_seq calls on other host threads.
 */
W4A16_API int w4a16_testing_set_seq_wait(unsigned long long wait_ns, unsigned target_bump);

#ifdef __cplusplus
}
#endif

#endif /* W4A16_TESTING_H */

/*
 * st24_selftest.h -- self-test entry point of the st24 library (not part of
 * the product path; declared apart from st24.h).
 */
#ifndef ST24_SELFTEST_H
#define ST24_SELFTEST_H

#include "st24.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Enqueues on `stream` one CTA that waits, with the same bounded wait the
 * kernels use on their mbarriers, on a barrier nothing arrives at.  After
 * the wait's limit (about one second) the kernel records a timeout in the
 * device status word and returns; the next st24_device_status() on the
 * stream returns ST24_ERR_TIMEOUT and clears it.  It exercises the failure
 * detection of the library without faulting or hanging the GPU.  Returns
 * ST24_ERR_CUDA if the launch fails.
 */
ST24_API st24_status st24_selftest_wait_timeout(void* stream);

#ifdef __cplusplus
}
#endif

#endif

/*
 * fp8g — hooks for testing the library's failure handling.  Not needed to use
 * the library; the entry points of fp8g.h do not depend on them.
 */
#ifndef FP8G_TESTING_H
#define FP8G_TESTING_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Bound, in nanoseconds, of every pipeline wait inside the GEMM and bmm_fp8
 * kernels that the CALLING THREAD launches from now on (0 restores the default
 * of 2 s).  A wait that runs past it gives up: the launch stops, drains the
 * copies and tensor-core operations it has in flight, frees its tensor memory
 * and raises FP8G_DEVICE_TIMEOUT in the device status word, which
 * fp8g_get_device_status() then reports as FP8G_ERR_TIMEOUT.  Outputs of a
 * launch that gave up are unspecified.  A limit far below a launch's running
 * time makes that launch give up: the timeout path can so be exercised
 * without breaking the pipeline itself.  Never fails.
 */
void fp8g_testing_set_wait_limit_ns(uint64_t ns);

/*
 * Tile shape of the calling thread's last fp8_gemm_nt_groupwise or bmm_fp8
 * launch: 1 if it ran on CTA pairs (256 x 256 tiles, tcgen05 cta_group::2), 0
 * if on one CTA per 128 x 256 tile, -1 if the thread has launched none.  The
 * shape never changes results; this tells a test which one was chosen.
 */
int fp8g_testing_last_gemm_cta_pair(void);

#ifdef __cplusplus
}
#endif

#endif /* FP8G_TESTING_H */

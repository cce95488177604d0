/*
 * ibp_testing.h -- testing hooks of the GB300 IBP codec library (libibp_gb300.so).
 *
 * Not part of the codec: the paper has no counterpart. They exist so that the
 * failure path of the gather's bounded waits can be exercised on a GPU without
 * faulting, trapping or hanging it.
 *
 * The warp-specialised decompress-gather kernel (slots in device memory, rows of
 * more than 1 KiB) hands work from planner warps to decoder warps through
 * shared-memory barriers. Every wait on them is bounded: by default it gives up after
 * 2 s of GPU global time, records IBP_ERR_TIMEOUT in *d_status, raises a flag that
 * ends the other warps' loops, waits for the warp's own copies in flight and returns.
 */
#ifndef IBP_TESTING_H
#define IBP_TESTING_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Set the limit, in ns of GPU global time, of every bounded wait of the gather
 * kernels launched from now on, in this process and on every device; ns = 0 restores
 * the default (2 s). Returns the previous setting (0 = the default). A limit of a
 * few ns makes a wait run out almost surely; the call's output is then incomplete and
 * *d_status reads IBP_ERR_TIMEOUT. Host-side only: no CUDA call, never fails. Not
 * meant for normal use; a test that lowers the limit restores it. */
uint64_t ibp_testing_set_wait_limit_ns(uint64_t ns);

/* on != 0: the planner warps of warp-specialised gathers launched from now on (in
 * this process, on every device) plan their units but never hand them to the
 * decoders, so the decoders' first wait cannot complete and runs out after the wait
 * limit: the call then records IBP_ERR_TIMEOUT in *d_status and its output is
 * incomplete; every warp still ends within the limit. on = 0 restores normal
 * operation. Returns the previous setting. Host-side only: no CUDA call, never fails.
 * Gathers served by the other kernels are unaffected. Not meant for normal use; a
 * test that sets it clears it. */
int ibp_testing_withhold_plans(int on);

#ifdef __cplusplus
}
#endif
#endif

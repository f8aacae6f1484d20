/* mhc_boundary_test.h -- test hooks of the mHC boundary library (not for
 * production use).
 *
 * Failure detection without a GPU fault: every wait in the library's
 * kernels is bounded.  A wait that gives up sets a bit of the handle's error
 * word, the kernel leaves its outputs invalid and exits, and the next
 * mhc_boundary_check_errors (or run) returns MHC_ERR_TIMEOUT; the CUDA
 * context stays usable.  This hook makes that happen on purpose.
 */
#ifndef MHC_BOUNDARY_TEST_H
#define MHC_BOUNDARY_TEST_H

#include "mhc_boundary.h"

#ifdef __cplusplus
extern "C" {
#endif

/* With on != 0, the tensor-core stage kernels and the one-kernel path for a
 * few tokens launched from now on, on the current device, issue no input
 * copies: their waits for those copies run out (after about a second) and
 * they report MHC_ERR_TIMEOUT.  on == 0
 * restores normal operation.  Affects every handle on the device; call it
 * only while no boundary call is in flight.  Returns MHC_ERR_CUDA if the
 * device flag cannot be set. */
mhc_status_t mhc_test_stall_stage_copies(int32_t on);

#ifdef __cplusplus
}
#endif

#endif /* MHC_BOUNDARY_TEST_H */

/*
 * tfqmm_debug.h -- entry points of the bounds-checking debug build only
 * (libtfqmm_debug.so, compiled from the same sources with TF_DEBUG_BOUNDS).
 * That library exports everything tfqmm.h declares, with the same results;
 * its kernels additionally check every shared- and global-memory index
 * against its buffer before the access, skip an access that would fall
 * outside, and record it in the device status word, which tf_device_status
 * then reports as TF_EBOUNDS.  No check traps or faults.
 */
#ifndef TFQMM_DEBUG_H
#define TFQMM_DEBUG_H

#include "tfqmm.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Test hook of the checker itself: the next product launch treats its y as
 * `rows` rows shorter than the call's arguments say (0..16), so its stores to
 * the last rows fail the bounds check: they are skipped and reported, and the
 * caller's memory there stays untouched.  One shot; TF_OK or TF_EINVAL_ROWS.
 */
int tf_debug_shrink_y(int rows);

#ifdef __cplusplus
}
#endif
#endif

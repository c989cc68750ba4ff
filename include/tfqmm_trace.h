/*
 * tfqmm_trace.h -- the phase-trace build of libtfqmm (libtfqmm_trace.so, built
 * from the same sources with TF_TRACE by mlx_affine_bit_gb300.build.build_trace).
 *
 * Every entry point of tfqmm.h behaves as in the product library; in addition
 * every CTA of every row-kernel launch writes one record of 9 uint64 words:
 *   [0] the launch's number (0, 1, ... since the last tf_trace_reset, in launch
 *       order on the host), [1] (SM id << 32) | block index, then %globaltimer
 *   (ns) at [2] kernel entry, [3] the producer's first stage issued, [4] that
 *   stage landed (0 in early-x launches of one or two rows, whose producer does
 *   not wait for it), [5] consumer thread 0 past the dependency wait (programmatic
 *   dependent launch; a launch without it passes at once), [6] the first x
 *   slice placed and summed, [7] the first stage's group products done, [8]
 *   consumer thread 0's last store issued.  A phase the CTA did not reach is 0.
 * Records go to a per-device buffer of 65536 records allocated at the first
 * traced launch (a failed allocation leaves launches untraced); records past
 * 65536 are dropped.  The trace costs a few global stores per CTA; its times are
 * for reading phases, not for the bench.
 */
#ifndef TFQMM_TRACE_H
#define TFQMM_TRACE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Waits for the device, clears every record and the launch numbering.  0 or a
 * negative TF_E* status. */
int tf_trace_reset(void);

/* Waits for the device and copies up to max_records records (9 words each, the
 * layout above) into the host array buf; returns how many, or a negative
 * TF_E* status. */
int tf_trace_read(uint64_t *buf, int max_records);

#ifdef __cplusplus
}
#endif

#endif

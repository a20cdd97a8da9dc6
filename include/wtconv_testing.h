/*
 * wtconv_testing.h -- test hook of libwtconv (not part of the layer; the paper has no
 * counterpart).
 *
 * The kernels bound every wait on an mbarrier (1 s by default), so that a copy that never
 * lands ends the kernel with a recorded status instead of a hang. This hook shortens that
 * limit so that a test can make waits run out on purpose and check that the status is
 * reported (wtconv_workspace_status) and that the next ordinary call is unaffected.
 */
#ifndef WTCONV_TESTING_H_
#define WTCONV_TESTING_H_

#include "wtconv.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Sets the limit of every bounded wait of the kernels launched afterwards by any host
 * thread, in nanoseconds; 0 restores the default (1 s). Process-wide; meant for tests only.
 * A limit below the default is counted in SM clock cycles (the device's nanosecond timer
 * advances in steps of up to a microsecond, too coarse for a short limit), which at SM
 * clocks of 1 GHz or more last no longer than the nanoseconds asked for, and is checked
 * before each probe of the barrier: with a limit of 1, every wait runs out at once, whether
 * or not its copy has landed, so the first wait of every CTA reports a timeout.
 * The bounded wait for in-flight copies that a CTA performs before it leaves after a
 * timeout always keeps the default limit. Returns WT_OK.
 */
wt_status wtconv_testing_set_wait_limit_ns(unsigned long long ns);

#ifdef __cplusplus
}
#endif

#endif /* WTCONV_TESTING_H_ */

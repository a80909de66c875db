/*
 * mamba_scan_testing.h -- test-only entry points of libmamba_scan.so.
 *
 * Not part of the operation's ABI (include/mamba_scan.h): nothing here
 * computes anything the pages define.  These calls let tests exercise the
 * library's failure reporting without faulting or hanging a GPU.
 */
#ifndef MAMBA_SCAN_TESTING_H
#define MAMBA_SCAN_TESTING_H

#include "mamba_scan.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Launch, on `stream`, one thread that waits on a shared-memory mbarrier that
 * nothing ever arrives on, giving up after `polls` polls (mbarrier try_wait;
 * each may suspend the thread briefly), and records the give-up in the device
 * error word exactly as the scans' bounded copy waits do.  The next
 * mamba_device_status(stream) then returns MAMBA_ERR_TIMEOUT and clears the
 * word; the CUDA context stays usable.
 *
 * polls must be in [1, 1048576] (else MAMBA_ERR_SIZE, nothing launched).
 * Returns MAMBA_OK, or MAMBA_ERR_LAUNCH if the launch failed.
 */
int mamba_test_bounded_wait(int polls, mamba_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA_SCAN_TESTING_H */

/*
 * pkv_selftest.h - a diagnostic call of the paged-KV-cache library.
 *
 * Every pipeline wait inside the library's kernels is bounded in time: if a
 * wait does not complete within its limit, the waiting warp ORs
 * PKV_FLAG_TIMEOUT (pkv.h) into the caller's err_flag and returns instead of
 * spinning forever, so a pipeline bug reports an error and the CUDA context
 * stays usable.  The pages describe no such mechanism (it belongs to this
 * implementation), so this call exists only to let a test exercise it on a
 * GPU without faulting or hanging anything.
 */
#ifndef PKV_SELFTEST_H_
#define PKV_SELFTEST_H_

#include <stdint.h>

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * pkv_selftest_bounded_wait - run the library's bounded mbarrier wait once.
 *
 * Launches one warp that initialises a shared-memory mbarrier with an
 * arrival count of 1 and waits on its first phase with the same helper the
 * decode and prefill kernels use, giving up after limit_ns nanoseconds of
 * %globaltimer.  With arrive == 0 nothing arrives and no copy targets the
 * barrier, so the wait runs out: the warp ORs PKV_FLAG_TIMEOUT into *err_flag
 * and returns.  With arrive != 0 one lane arrives first, the wait completes at
 * once and err_flag is left alone.  If waited_ns is not NULL the warp stores
 * there how long the wait took.
 *
 *   limit_ns   1 .. 100000000 (at most 0.1 s), else PKV_ERR_INVALID_ARG
 *   err_flag   device int32 (required), OR-ed with PKV_FLAG_TIMEOUT on timeout
 *   waited_ns  device uint64 or NULL
 *   stream     cudaStream_t (NULL = the legacy default stream)
 *
 * Only enqueues the kernel; the caller synchronises and reads the words back.
 */
pkv_status pkv_selftest_bounded_wait(uint64_t limit_ns, int arrive, int32_t *err_flag,
                                     uint64_t *waited_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_SELFTEST_H_ */

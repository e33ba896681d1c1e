/*
 * gdn_debug.h -- self-tests of the library's failure reporting.  Not needed to
 * compute anything; the tests call them to check, on the GPU and without
 * faulting it, that a device-side wait which never completes gives up and is
 * reported through the workspace status word.
 */
#ifndef GDN_DEBUG_H
#define GDN_DEBUG_H

#include <stddef.h>
#include <stdint.h>

#include "gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * gdn_debug_wait_timeout -- launch one CTA whose two warps each wait on an
 * mbarrier that nothing completes, through the same bounded wait the
 * tensor-core kernels use: the first to pass its limit (2 s of wall time)
 * records GDN_ERR_TIMEOUT (seq = 7, head = 3) and raises the CTA's abort flag,
 * and the other leaves on seeing the flag.  Asynchronous on `stream`; read the
 * result with gdn_check(workspace, stream), which returns GDN_ERR_TIMEOUT.
 *
 *   workspace   device, at least 256 bytes, status word zeroed (gdn_workspace_init)
 *
 * Returns GDN_OK once enqueued, GDN_ERR_WORKSPACE for a missing or small
 * workspace, GDN_ERR_INVALID_ARG for a misaligned one, GDN_ERR_CUDA if the
 * launch fails.
 */
gdn_status gdn_debug_wait_timeout(void *workspace, size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_DEBUG_H */

/* Debug build of the masked attention library: libmattn_debug.so.
 *
 * The same sources as libmattn.so compiled with -DMATTN_DEBUG. Every index
 * that a kernel computes for a global load or store outside the tensor-map
 * copies (which the hardware bounds itself) is checked against the size of
 * its buffer first; an index out of range is recorded and the access is
 * skipped (a load reads 0, a store does not happen). Nothing traps, so the
 * CUDA context stays usable and the host reads the record afterwards. The
 * library exports everything mattn.h declares plus the calls below; the
 * release library exports none of these. The kernels run slower than in the
 * release build: the debug build is for tests, not for timing.
 */
#ifndef MATTN_DEBUG_H_
#define MATTN_DEBUG_H_

#include "mattn.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct attn_debug_info {
  unsigned long long count; /* failed checks since the last clear, over all kernels */
  int site;                 /* access site of the first one (attn_debug_site_name), 0 if none */
  int pad;
  long long index;          /* its index */
  long long bound;          /* and the size it broke */
} attn_debug_info;

/* Reads the failed-check records of every kernel into *out (the first
 * failure found and the total count). With clear != 0 the records are reset
 * afterwards. Synchronises the device. ATTN_ERR_INVALID_ARG for out = NULL,
 * ATTN_ERR_CUDA if a copy fails. */
attn_status attn_debug_record(attn_debug_info* out, int clear);

/* Name of an access site reported in attn_debug_info::site ("unknown" for
 * other values). */
const char* attn_debug_site_name(int site);

/* Checks the checking itself: launches a 16-thread kernel on `stream` over a
 * 16-element buffer that the call allocates, in which thread 0's index is
 * planted 3 past the end and threads 1..15 add 1 to their own element. The
 * check must refuse thread 0's access (no access happens) and record exactly
 * that index; the other threads' updates must land. Returns ATTN_OK when both
 * hold (and clears the record it made), ATTN_ERR_UNSUPPORTED when not,
 * ATTN_ERR_CUDA on a CUDA error. Synchronises `stream`. */
attn_status attn_debug_selftest(struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* MATTN_DEBUG_H_ */

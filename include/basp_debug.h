/*
 * basp_debug.h -- the extra entry point of the bounds-checking debug build,
 * libbasp_debug.so (the same sources compiled with -DBASP_CHECK_BOUNDS=1).
 * The release library, libbasp.so, does not export it.
 *
 * In the debug build every load and store of the re-layout kernels is checked
 * against the extent of the buffer it belongs to.  An access outside it is
 * not made; it is counted in a device-side counter instead.  This stands in
 * for an out-of-bounds sanitizer; the paper has no counterpart.
 */
#ifndef BASP_DEBUG_H
#define BASP_DEBUG_H

#include "basp.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Synchronise the current device, store into *count the number of
 * out-of-bounds accesses the kernels have skipped on it since the last call,
 * and reset that number to zero.  BASP_ERR_INVALID_ARG for a NULL count,
 * BASP_ERR_CUDA if the synchronisation or the copies fail.
 */
basp_status basp_debug_bounds_violations(unsigned long long *count);

#ifdef __cplusplus
}
#endif

#endif /* BASP_DEBUG_H */

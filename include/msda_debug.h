/*
 * msda_debug.h -- the one extra entry point of the debug build of libmsda
 * (libmsda_debug.so, compiled with -DMSDA_DEBUG; libmsda.so does not export it).
 *
 * In that build every value gather, grad_output load and grad_value (or
 * fixed-point) reduction of the kernels is checked against the extent of its
 * tensor, and 16-byte vector accesses against their alignment.  A bad access
 * is not made: a load reads the tensor's first elements instead, a reduction is
 * dropped, and the access is counted.  The kernels never trap, so a wrong index
 * shows up as a count and as wrong results, with the context intact.
 */
#ifndef MSDA_DEBUG_H_
#define MSDA_DEBUG_H_

#if defined(__GNUC__)
#define MSDA_DEBUG_API __attribute__((visibility("default")))
#else
#define MSDA_DEBUG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Accesses skipped since the library was loaded (or since the last reset) on
 * the current device, over every kernel; waits for the device first.
 * reset != 0: zero the counts after reading them. */
MSDA_DEBUG_API unsigned long long msda_debug_violations(int reset);

#ifdef __cplusplus
}
#endif

#endif /* MSDA_DEBUG_H_ */

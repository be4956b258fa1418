/*
 * msda_probes.h -- measurement kernels shipped beside libmsda (in
 * libmsda_probes.so, not in libmsda.so): the rates at which this GPU's SMs
 * move random 128-byte lines, which bound the MSDeformAttn kernels (a bilinear
 * sample gathers four value rows of head_dim channels, 128 bytes at
 * head_dim = 32 in fp32, from random places; the backward adds into as many
 * rows of grad_value).  Nothing of the method is computed here.
 *
 * Every probe runs msda_probe_accesses(lines) >= `lines` line operations (each
 * thread runs whole rounds of eight) over a device buffer of `n_lines`
 * 128-byte lines (16-byte aligned, 1 <= n_lines < 2^31): each quarter-warp
 * draws its lines from its own 32-bit linear congruential stream (seeded from
 * `seed` and its index), reduced uniformly into [0, n_lines), so every access
 * stays inside the buffer.  A warp instruction covers four lines (eight lanes
 * x 16 bytes each), as the kernels' gathers and reductions do, and a thread
 * keeps eight accesses in flight.
 * `hot_lines` > 0 restricts the lines to the first hot_lines of the buffer
 * (a set that stays in L1).  Launches are asynchronous on `stream`; the
 * caller times them with events.  Return value: 0, or a cudaError_t.
 *
 *   msda_probe_gather   ld.global.nc.v4 of each line (the sum lands in sink,
 *                       which needs 16 bytes per launched thread:
 *                       msda_probe_sink_bytes())
 *   msda_probe_reduce   red.global.add.v4.f32 of 1.0 into each line (the
 *                       buffer must hold floats; its contents change)
 *   msda_probe_bulk_reduce  the same reductions through the TMA unit: each
 *                       quarter-warp stages its line's 128 bytes of 1.0 in
 *                       shared memory and issues one cp.reduce.async.bulk
 *                       .add.f32 of them into the line (the buffer must hold
 *                       floats; its contents change)
 *   msda_probe_mixed    per eight gathers, `reds_per_8` (0..8) reductions into
 *                       other lines (from a second stream): the backward's mix;
 *                       msda_probe_accesses(lines) gathers, that times
 *                       reds_per_8 / 8 reductions
 */
#ifndef MSDA_PROBES_H_
#define MSDA_PROBES_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

size_t msda_probe_sink_bytes(void);
int64_t msda_probe_accesses(int64_t lines);
int msda_probe_gather(const void *buf, int64_t n_lines, int64_t hot_lines, int64_t lines, void *sink, uint32_t seed,
                      void *stream);
int msda_probe_reduce(void *buf, int64_t n_lines, int64_t hot_lines, int64_t lines, uint32_t seed, void *stream);
int msda_probe_bulk_reduce(void *buf, int64_t n_lines, int64_t lines, uint32_t seed, void *stream);
int msda_probe_mixed(void *buf, int64_t n_lines, int64_t lines, int reds_per_8, void *sink, uint32_t seed,
                     void *stream);

#ifdef __cplusplus
}
#endif

#endif /* MSDA_PROBES_H_ */

/*
 * gma_profile.h -- instrumentation entry points of libgma.so (not part of the GMA method).
 *
 * They let a benchmark count the library's kernel launches and time each kernel with CUDA
 * events recorded on the stream the kernel is launched on.  The method itself is described
 * in gma.h; nothing here changes what the forward pass computes.
 */
#ifndef GMA_PROFILE_H_
#define GMA_PROFILE_H_

#include <stddef.h>

#include "gma.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Number of kernels libgma.so has launched in this process (all devices, all streams). */
GMA_API unsigned long long gma_launch_count(void);

/*
 * on != 0: start recording a CUDA event pair around every kernel the library launches (the
 * previous records are dropped); on == 0: stop recording (records are kept for reading).
 * Recording adds two event records per launch on the launch stream.  Returns GMA_ERR_CUDA if
 * an event could not be created.
 */
GMA_API gma_status_t gma_profile_enable(int on);

/*
 * Waits for every recorded event, then writes one line per kernel kind into `buf`:
 *   "<kernel name> <launches> <total milliseconds>\n"
 * NUL-terminated, truncated to `len` bytes.  Returns the number of lines, or -1 on a CUDA error.
 */
GMA_API int gma_profile_read(char *buf, size_t len);

/*
 * Measures the throughput of the GPU's base-2 exponential instruction (ex2.approx.f32, the one the
 * softmax over mixture components uses) with a short all-SM microbenchmark on `stream`, and writes
 * exponentials per second to *exps_per_second.  Synchronous; allocates nothing on the device.
 */
GMA_API gma_status_t gma_probe_ex2_rate(void *stream, double *exps_per_second);

/*
 * Test hook for the bounded device waits.  The next gma_forward_bidir call with dtype GMA_BF16
 * launches its write kernel with the first key-tile load withheld: the waits on that tile run out
 * after their limit (about one second), the kernel records the timeout in the workspace error word
 * and every CTA exits normally, releasing its tensor memory.  gma_check_device_error() on that
 * workspace then returns GMA_ERR_TIMEOUT.  Nothing traps or faults; the context stays usable.
 * Setting the environment variable GMA_FAULT_INJECT (to anything but "" or "0") before the first
 * bf16 bidirectional call of the process has the same effect on that call.
 */
GMA_API void gma_debug_withhold_first_load(void);

/*
 * Bounds-check debug build (libgma_checked.so, compiled with -DGMA_BOUNDS_CHECK).  In that build every
 * computed global-memory index of the forward kernels (both paths: workspace sections, outputs, the
 * float32 path's input rows) is compared with the extent the host planned for its buffer; a failed
 * check skips the access and is recorded, nothing traps.  gma_debug_bounds_read() copies the record to
 * out[4]: the first failing site (0: none), its index, its extent, and the number of failed checks
 * since the last gma_debug_bounds_clear(); read it after the kernels have completed (for instance
 * after cudaDeviceSynchronize()).  gma_debug_bounds_selftest()
 * enqueues one kernel that fails one check on purpose (site 999, index 3, extent 3) without touching
 * memory.  In the normal build all three return GMA_ERR_UNSUPPORTED.
 */
GMA_API gma_status_t gma_debug_bounds_read(unsigned long long *out);
GMA_API gma_status_t gma_debug_bounds_clear(void);
GMA_API gma_status_t gma_debug_bounds_selftest(void *stream);

#ifdef __cplusplus
}
#endif

#endif /* GMA_PROFILE_H_ */

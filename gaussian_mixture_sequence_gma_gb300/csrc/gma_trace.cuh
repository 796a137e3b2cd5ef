// gma_trace.cuh -- optional cycle trace of one CTA (development builds only).
//
// Compiled to nothing unless the library is built with -DGMA_TRACE.  A trace build records, for the CTA
// at grid position (0, 0), clock64() at numbered points of each role's tile loop into a device array
// of kTraceIds x kTraceTiles slots (point id, tile index), read back with gma_debug_trace_read().
#pragma once

#ifdef GMA_TRACE
namespace gma {
constexpr int kTraceIds = 64, kTraceTiles = 64;
static __device__ unsigned long long g_trace[kTraceIds * kTraceTiles];  // one per translation unit
}  // namespace gma
#ifdef GMA_TRACE_SPANS_ONLY
// span points only: the tile-loop points compile to nothing, so the loops run as in a release build
#define GMA_TRACE_AT(id, t) \
  do {                      \
  } while (0)
#else
#define GMA_TRACE_AT(id, t)                                                                        \
  do {                                                                                             \
    if (blockIdx.x == 0 && blockIdx.y == 0 && (threadIdx.x & 31) == 0 && (t) < ::gma::kTraceTiles) \
      ::gma::g_trace[(id) * ::gma::kTraceTiles + (t)] = clock64();                                 \
  } while (0)
#endif
// Span points: %globaltimer (ns) of every CTA (linear index below kSpanCtas) at point `slot`, taken by
// the calling thread, shifted left by 8 with the CTA's SM index in the low 8 bits.
namespace gma {
constexpr int kSpanSlots = 10, kSpanCtas = 2048;
static __device__ unsigned long long g_span[kSpanSlots * kSpanCtas];
}  // namespace gma
#define GMA_SPAN_AT(slot)                                                                  \
  do {                                                                                     \
    const unsigned cta_ = blockIdx.y * gridDim.x + blockIdx.x;                             \
    if (cta_ < (unsigned)::gma::kSpanCtas) {                                               \
      unsigned long long g_;                                                               \
      unsigned sm_;                                                                        \
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(g_));                               \
      asm volatile("mov.u32 %0, %%smid;" : "=r"(sm_));                                     \
      ::gma::g_span[(slot) * ::gma::kSpanCtas + cta_] = (g_ << 8) | (sm_ & 0xffu);         \
    }                                                                                      \
  } while (0)
#else
#define GMA_SPAN_AT(slot) \
  do {                    \
  } while (0)
#define GMA_TRACE_AT(id, t) \
  do {                      \
  } while (0)
#endif

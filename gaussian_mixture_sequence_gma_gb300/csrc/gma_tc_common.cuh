// gma_tc_common.cuh -- sm_103a device primitives for the tensor-core path: mbarriers with bounded
// waits, TMA (tensor and bulk) loads, tcgen05 TMEM allocation / MMA / loads and stores, and the
// shared-memory and instruction descriptors of the 128-byte-swizzled operand layouts.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gma_internal.h"

#ifndef GMA_WAIT_SPIN
#define GMA_WAIT_SPIN 4
#endif
#ifndef GMA_WAIT_SLEEP_NS
#define GMA_WAIT_SLEEP_NS 64
#endif

// ---------------------------------------------------------------------------------------------- bounds checks
// Debug build (-DGMA_BOUNDS_CHECK): GMA_INB(i, n, site) is false when the element index i is not below n,
// the extent the host planned for the buffer it indexes, and the caller then skips the access.  The first
// failing site, its index and extent, and the number of failures go to this translation unit's record
// (g_bounds), which gma_debug_bounds_read() collects; nothing traps.  In the normal build it is true.
#ifdef GMA_BOUNDS_CHECK
namespace gma {
namespace {
__device__ unsigned long long g_bounds[4];  // first site, its index, its extent; failures

__device__ __noinline__ bool bounds_fail(unsigned long long i, unsigned long long n, unsigned site) {
  if (atomicCAS(&g_bounds[0], 0ull, (unsigned long long)site) == 0ull) {
    g_bounds[1] = i;
    g_bounds[2] = n;
  }
  atomicAdd(&g_bounds[3], 1ull);
  return false;
}

// Host side: copies this translation unit's record to h[4] (clear: then zeroes it).
inline gma_status_t bounds_record_io(unsigned long long* h, bool clear) {
  if (h && cudaMemcpyFromSymbol(h, g_bounds, sizeof g_bounds) != cudaSuccess) return GMA_ERR_CUDA;
  static const unsigned long long zero[4] = {0, 0, 0, 0};
  if (clear && cudaMemcpyToSymbol(g_bounds, zero, sizeof zero) != cudaSuccess) return GMA_ERR_CUDA;
  return GMA_OK;
}
}  // namespace
}  // namespace gma
#define GMA_INB(i, n, site)                                        \
  ((unsigned long long)(i) < (unsigned long long)(n) ||            \
   ::gma::bounds_fail((unsigned long long)(i), (unsigned long long)(n), (site)))
#else
#define GMA_INB(i, n, site) true
#endif

namespace gma {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------------------------- launch order
// Waits until the previous kernel on the stream has completed and its writes are visible (a no-op for a
// kernel launched without programmatic dependent launch).
__device__ __forceinline__ void dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel on the stream (launched as dependent) start once every CTA of this one has
// executed this or exited.
__device__ __forceinline__ void dep_launch_next() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// ---------------------------------------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// Shared abort state of one CTA: the first wait that runs out of time records the site in the
// workspace error word and raises `abort`; every other wait then gives up at once, so all roles
// leave their loops and reach the common exit (where TMEM is released).
struct Abort {
  volatile uint32_t flag;
};

// Bounded wait on phase `parity` of `bar`.  Returns false on timeout or abort.  try_wait itself
// suspends the thread for a while; the clock and the abort flag are checked every 16 tries.
__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity, Abort* ab, Ctrl* ctrl, uint32_t site,
                                             uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = 0;
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15) == 0) {
      if (ab->flag) return false;
      const uint64_t now = global_timer_ns();
      if (t0 == 0) t0 = now;
      if (now - t0 > limit_ns) {
        ab->flag = 1;
        if (atomicCAS(&ctrl->err, kErrNone, kErrTimeout) == kErrNone) ctrl->err_site = site;
        return false;
      }
    }
  }
}

// wait_bounded for a single control thread (producer, MMA issuer): after a few unsuccessful tries it
// sleeps between tries, so that waiting threads take few issue slots and shared-memory cycles from the
// row warps.
__device__ __forceinline__ bool wait_bounded_bo(uint64_t* bar, uint32_t parity, Abort* ab, Ctrl* ctrl, uint32_t site,
                                                uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  uint64_t t0 = 0;
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if (i >= GMA_WAIT_SPIN) __nanosleep(GMA_WAIT_SLEEP_NS);
    if ((i & 15) == 0) {
      if (ab->flag) return false;
      const uint64_t now = global_timer_ns();
      if (t0 == 0) t0 = now;
      if (now - t0 > limit_ns) {
        ab->flag = 1;
        if (atomicCAS(&ctrl->err, kErrNone, kErrTimeout) == kErrNone) ctrl->err_site = site;
        return false;
      }
    }
  }
}

// wait_bounded taken by a whole warp with one outcome for every lane (row-warp control flow stays
// uniform, which the warp-level arrivals and tcgen05 .sync.aligned operations rely on).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, Abort* ab, Ctrl* ctrl, uint32_t site,
                                          uint64_t limit_ns) {
  return __all_sync(0xffffffffu, wait_bounded(bar, parity, ab, ctrl, site, limit_ns));
}

// One arrival per warp on `bar` (barriers counted in warps): the warp's lanes synchronise first, which
// orders their earlier shared-memory and tensor-memory accesses before lane 0's release-arrive.
__device__ __forceinline__ void warp_arrive(uint64_t* bar) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// ---------------------------------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          smem_u32(dst)),
      "l"((uint64_t)map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}
// Plain bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"((uint64_t)src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
// Plain bulk copy shared -> global (16-byte aligned addresses, size a multiple of 16), bulk-group completion.
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"((uint64_t)dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
}
// Bulk float32 add shared -> global (each element of the global range += the shared one, performed at
// L2; 16-byte aligned addresses, size a multiple of 16), bulk-group completion.
__device__ __forceinline__ void bulk_reduce_add_f32(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"((uint64_t)dst),
               "r"(src), "r"(bytes)
               : "memory");
}
// Tiled store shared -> global (rows past the tensor's extent are not written), bulk-group completion.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"((uint64_t)map),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the committed stores have finished reading shared memory / have completed
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---------------------------------------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc]^T
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]^T
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
          d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// The same with the descriptors given as a base plus an offset (in 16-byte units) added right before the
// instruction, so unrolled issue loops keep only their base descriptors live.
__device__ __forceinline__ void mma_ss_off(uint32_t d, uint64_t a, uint32_t a_off, uint64_t b, uint32_t b_off,
                                           uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 ad, bd, ao, bo;\n setp.ne.b32 p, %6, 0;\n cvt.u64.u32 ao, %2;\n"
      " cvt.u64.u32 bo, %4;\n add.s64 ad, %1, ao;\n add.s64 bd, %3, bo;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], ad, bd, %5, p;\n}\n" ::"r"(d),
      "l"(a), "r"(a_off), "l"(b), "r"(b_off), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_ts_off(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t b_off, uint32_t idesc,
                                           uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n .reg .b64 bd, bo;\n setp.ne.b32 p, %5, 0;\n cvt.u64.u32 bo, %3;\n add.s64 bd, %2, bo;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p;\n}\n" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(b_off), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%"
      "21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait_tied8(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]),"+r"(r[1]),"+r"(r[2]),"+r"(r[3]),"+r"(r[4]),"+r"(r[5]),"+r"(r[6]),"+r"(r[7]) : : "memory");
}
__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];\n" : "=r"(r) : "r"(taddr));
  return r;
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld_wait_tied1(uint32_t& r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r) : : "memory");
}
__device__ __forceinline__ void tmem_ld_wait_tied16(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]),"+r"(r[1]),"+r"(r[2]),"+r"(r[3]),"+r"(r[4]),"+r"(r[5]),"+r"(r[6]),"+r"(r[7]),"+r"(r[8]),"+r"(r[9]),"+r"(r[10]),"+r"(r[11]),"+r"(r[12]),"+r"(r[13]),"+r"(r[14]),"+r"(r[15]) : : "memory");
}
// Wait for outstanding TMEM loads with 32 destination registers tied to the wait, so no use of them
// can be scheduled before it while later loads are still in flight.
__device__ __forceinline__ void tmem_ld_wait_tied32(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;" : "+r"(r[0]),"+r"(r[1]),"+r"(r[2]),"+r"(r[3]),"+r"(r[4]),"+r"(r[5]),"+r"(r[6]),"+r"(r[7]),"+r"(r[8]),"+r"(r[9]),"+r"(r[10]),"+r"(r[11]),"+r"(r[12]),"+r"(r[13]),"+r"(r[14]),"+r"(r[15]),"+r"(r[16]),"+r"(r[17]),"+r"(r[18]),"+r"(r[19]),"+r"(r[20]),"+r"(r[21]),"+r"(r[22]),"+r"(r[23]),"+r"(r[24]),"+r"(r[25]),"+r"(r[26]),"+r"(r[27]),"+r"(r[28]),"+r"(r[29]),"+r"(r[30]),"+r"(r[31]) : : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Warpgroup-wide register re-allocation (all four warps of a warpgroup execute the same one).
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------------------------- shared memory
// Accesses through 32-bit shared-window addresses, so address arithmetic stays 32-bit (an XOR with a
// 16-byte chunk index is one logic op) and every access is a shared-memory instruction.
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ float lds32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts32(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}
__device__ __forceinline__ void sts16(uint32_t a, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(a), "h"(v) : "memory");
}

// ---------------------------------------------------------------------------------------------- descriptors
// Instruction descriptor, kind::f16 with float32 accumulation.  a_type/b_type: 0 = f16, 1 = bf16;
// a_mn/b_mn: 0 = K-major, 1 = MN-major.  N in bits 17-22 (N >> 3), M in bits 24-28 (M >> 4).
__host__ __device__ constexpr uint32_t make_idesc(int M, int N, int a_type, int b_type, int a_mn, int b_mn) {
  return (1u << 4) | ((uint32_t)a_type << 7) | ((uint32_t)b_type << 10) | ((uint32_t)a_mn << 15) |
         ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor for the 128-byte swizzle: start address, leading-dimension byte
// offset (MN-major: stride between 64-element swizzle atoms along M/N), stride byte offset (stride
// between groups of 8 rows), version 1, swizzle mode 2 (128B).
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo & 0x3FFFF) >> 4) << 16;
  d |= (uint64_t)((sbo & 0x3FFFF) >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// The same for the 32-byte swizzle (swizzle mode 6): atoms of 8 rows x 32 bytes (16 bf16 along MN for
// an MN-major operand), lbo = stride between 16-element atoms along MN, sbo = stride between 8-row groups.
__device__ __forceinline__ uint64_t make_sdesc32(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo & 0x3FFFF) >> 4) << 16;
  d |= (uint64_t)((sbo & 0x3FFFF) >> 4) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)6 << 61;
  return d;
}

// Byte offset of 16-byte chunk `c` (0 or 1) of row r in a 32B-swizzled atom of 32-byte rows
// (chunk index XOR bit 2 of the row, the TMA / MMA 32B swizzle).
__host__ __device__ __forceinline__ uint32_t sw32_chunk(int r, int c) {
  return (uint32_t)r * 32u + ((uint32_t)(c ^ ((r >> 2) & 1)) << 4);
}

// Byte offset of 16-bit element (row r, column k) of a 128B-swizzled tile whose rows hold 64
// elements per block and whose column blocks lie `block_stride` bytes apart.  Used both for
// K-major operands (rows = M or N, columns = contraction) and for MN-major operands (rows =
// contraction, columns = M or N): the physical image is the same.
__host__ __device__ __forceinline__ uint32_t sw128_off(int r, int k, uint32_t block_stride) {
  const int kb = k >> 6, kk = k & 63;
  return kb * block_stride + (r >> 3) * 1024 + (r & 7) * 128 + ((((kk >> 3) ^ (r & 7)) & 7) << 4) + (kk & 7) * 2;
}
// ---------------------------------------------------------------------------------------------- numerics
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// 1/x from the approximate reciprocal instruction (relative error within a few float32 ulps; every
// use here rounds the result to bf16 or scales a float32 output).
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// (a, b) += (c, d) with one packed float32x2 add.
__device__ __forceinline__ void add_f32x2(float& a, float& b, float c, float d) {
  asm("{\n .reg .b64 x, y;\n mov.b64 x, {%0, %1};\n mov.b64 y, {%2, %3};\n add.rn.f32x2 x, x, y;\n"
      " mov.b64 {%0, %1}, x;\n}\n"
      : "+f"(a), "+f"(b)
      : "f"(c), "f"(d));
}
// Three-input maximum.
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

}  // namespace tc
}  // namespace gma

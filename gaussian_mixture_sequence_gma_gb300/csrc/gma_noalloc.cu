// gma_noalloc.cu -- bidirectional forward for callers that cannot allocate device memory.
//
// Some callers have no way to obtain a device workspace at all: plugins whose execute hook runs in
// a host framework that forbids allocation on that path, pre-planned inference runtimes where every
// byte is budgeted before the first request, or plain C programs that link this library without a
// device allocator of their own.  gma_forward_bidir_static_ws() serves them from a scratch array
// that lives in the library itself: a file-scope __device__ array, so each GPU that loads the library
// holds kStaticWsBytes of it until the process exits.
//
// Host code may not pass the array's name to a kernel -- on the host that name is only a stand-in,
// not a device address.  The address is obtained with cudaGetSymbolAddress (with the device current)
// and cached per device together with the identity of the CUDA context it was looked up in; a call
// made in another context (for instance after cudaDeviceReset recreated the primary context, which
// loads the module again and may place the array elsewhere) looks it up afresh.  The first call on a
// device (or in a new context) does this set-up, so that first call should be made before any stream
// capture begins.  Every call shares the one array and it keeps the last call's contents; the
// bidirectional path clears the parts that must start at zero (the error word and the write-phase
// accumulator) at the start of every call.  Calls whose work overlaps on the GPU (two streams, or two
// host threads) race on the array: serialise them.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "gma_internal.h"

namespace gma {
namespace {

constexpr size_t kStaticWsBytes = (size_t)16 << 20;  // 16 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct CachedAddr {
  unsigned long long ctx_id;  // context the address belongs to (0: none cached)
  void* addr;
};

std::mutex g_mu;
CachedAddr g_cache[kMaxDevices] = {};

// Identity of the calling thread's current CUDA context, or 0 if it cannot be read.  The driver
// entry points come from the runtime (no link-time dependency on the driver library).
unsigned long long current_ctx_id() {
  static std::once_flag once;
  static CtxGetCurrentFn get_cur = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_cur || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_cur(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_static_ws in the current device's context.  Looked up once per device and
// context; without a readable context identity it is looked up on every call (cudaGetSymbolAddress
// allocates nothing).
gma_status_t static_ws_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GMA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GMA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  unsigned long long id = current_ctx_id();
  if (id != 0 && g_cache[dev].ctx_id == id) {
    *out = g_cache[dev].addr;
    return GMA_OK;
  }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_ws);  // also makes the primary context current
  if (e != cudaSuccess || p == nullptr) return cuda_fail("cudaGetSymbolAddress(static workspace)", e);
  if (id == 0) id = current_ctx_id();
  g_cache[dev] = {id, id != 0 ? p : nullptr};
  *out = p;
  return GMA_OK;
}

}  // namespace
}  // namespace gma

extern "C" {

size_t gma_static_ws_capacity(void) { return gma::kStaticWsBytes; }

gma_status_t gma_forward_bidir_static_ws(const gma_problem_t* p, const void* Q, const void* K, const void* V,
                                         const float* mu, const float* sigma2, const float* log_pi, void* O,
                                         void* stream) {
  const size_t need = gma_workspace_bytes(p, GMA_OP_BIDIR);
  if (need == 0) {
    // invalid problem: let the regular entry point report the precise status without launching
    return gma_forward_bidir(p, Q, K, V, mu, sigma2, log_pi, O, nullptr, 0, stream);
  }
  if (need > gma::kStaticWsBytes) return GMA_ERR_WORKSPACE;
  void* ws = nullptr;
  gma_status_t s = gma::static_ws_address(&ws);
  if (s != GMA_OK) return s;
  return gma_forward_bidir(p, Q, K, V, mu, sigma2, log_pi, O, ws, gma::kStaticWsBytes, stream);
}

gma_status_t gma_static_ws_check_error(void* stream) {
  void* ws = nullptr;
  gma_status_t s = gma::static_ws_address(&ws);
  if (s != GMA_OK) return s;
  // reads the control block at the start of the array into host memory (no allocation)
  return gma_check_device_error(ws, stream);
}

}  // extern "C"

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
// not a device address.  The address is obtained once per device with cudaGetSymbolAddress (with that
// device current) and cached; the first call on a device does this set-up, so that first call should
// be made before any stream capture begins.  Every call shares the one array and it keeps the last
// call's contents; the bidirectional path clears the parts that must start at zero (the error word and
// the write-phase accumulator) at the start of every call.  Calls whose work overlaps on the GPU (two
// streams, or two host threads) race on the array: serialise them.
#include <cuda_runtime.h>

#include <mutex>

#include "gma_internal.h"

namespace gma {
namespace {

constexpr size_t kStaticWsBytes = (size_t)16 << 20;  // 16 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_static_ws on the current device (set up once per device).
gma_status_t static_ws_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GMA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GMA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || p == nullptr) return GMA_ERR_CUDA;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
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

}  // extern "C"

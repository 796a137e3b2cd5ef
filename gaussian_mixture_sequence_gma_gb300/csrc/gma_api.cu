// gma_api.cu -- the extern "C" boundary of libgma.so: argument validation, workspace sizing,
// dispatch to the float32 CUDA-core path or the bf16 tensor-core path, and status mapping.
#include <cuda_runtime.h>

#include <cstdio>
#include <atomic>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "gma_internal.h"

namespace gma {

namespace {
thread_local char g_detail[256] = "";
}

void set_error_detail(const char* msg) { snprintf(g_detail, sizeof g_detail, "%s", msg); }

gma_status_t cuda_fail(const char* step, cudaError_t err, const void* func) {
  const cudaError_t e = err != cudaSuccess ? err : cudaGetLastError();
  int n = snprintf(g_detail, sizeof g_detail, "%s: %s", step, e == cudaSuccess ? "failed" : cudaGetErrorString(e));
  cudaFuncAttributes fa;
  if (func && n > 0 && n < (int)sizeof g_detail && cudaFuncGetAttributes(&fa, func) == cudaSuccess)
    snprintf(g_detail + n, sizeof g_detail - n, " (kernel: %d registers, max %d threads, %zu B static smem, %d B max dynamic)",
             fa.numRegs, fa.maxThreadsPerBlock, fa.sharedSizeBytes, fa.maxDynamicSharedSizeBytes);
  return GMA_ERR_CUDA;
}

gma_status_t check_launch(const char* step, const void* func) {
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? GMA_OK : cuda_fail(step, e, func);
}

gma_status_t set_smem_optin(const void* func, int bytes, int /*slot*/) {
  // the default limit on dynamic shared memory is 48 KB minus the kernel's static shared memory
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, func) != cudaSuccess) return cuda_fail("cudaFuncGetAttributes", cudaSuccess, func);
  if ((size_t)bytes + fa.sharedSizeBytes <= 48 * 1024) return GMA_OK;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GMA_ERR_CUDA;
  struct Entry { const void* f; int dev; int bytes; };
  static std::mutex mu;
  static std::vector<Entry> done;
  std::lock_guard<std::mutex> lock(mu);
  for (auto& e : done)
    if (e.f == func && e.dev == dev && e.bytes >= bytes) return GMA_OK;
  if (cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return cuda_fail("cudaFuncSetAttribute(max dynamic shared memory)");
  done.push_back({func, dev, bytes});
  return GMA_OK;
}

namespace {
constexpr uint64_t kDefaultWaitNs = 1000000000ull;  // 1 s
constexpr uint64_t kMinWaitNs = 1000000ull;         // 1 ms
constexpr uint64_t kMaxWaitNs = 600000000000ull;    // 10 min
std::atomic<uint64_t> g_wait_ns{0};                 // 0: not set through the API

uint64_t env_wait_ns() {
  static const uint64_t v = [] {
    const char* e = std::getenv("GMA_WAIT_LIMIT_MS");
    if (!e || !*e) return (uint64_t)0;
    char* end = nullptr;
    const double ms = std::strtod(e, &end);
    if (end == e || !(ms > 0)) return (uint64_t)0;
    const double ns = ms * 1e6;
    return ns < (double)kMinWaitNs ? kMinWaitNs : (ns > (double)kMaxWaitNs ? kMaxWaitNs : (uint64_t)ns);
  }();
  return v;
}
}  // namespace

uint64_t wait_limit_ns() {
  const uint64_t v = g_wait_ns.load(std::memory_order_relaxed);
  if (v) return v;
  const uint64_t e = env_wait_ns();
  return e ? e : kDefaultWaitNs;
}

namespace {
std::atomic<int> g_det{-1};  // -1: not set through the API

bool env_det() {
  static const bool v = [] {
    const char* e = std::getenv("GMA_DETERMINISTIC");
    return e && *e && !(e[0] == '0' && e[1] == 0);
  }();
  return v;
}
}  // namespace

bool deterministic() {
  const int v = g_det.load(std::memory_order_relaxed);
  return v < 0 ? env_det() : v != 0;
}

gma_status_t set_carveout_max(const void* func) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GMA_ERR_CUDA;
  struct Entry { const void* f; int dev; };
  static std::mutex mu;
  static std::vector<Entry> done;
  std::lock_guard<std::mutex> lock(mu);
  for (auto& e : done)
    if (e.f == func && e.dev == dev) return GMA_OK;
  if (cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
      cudaSuccess)
    return cuda_fail("cudaFuncSetAttribute(shared memory carveout)");
  done.push_back({func, dev});
  return GMA_OK;
}

namespace {

bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

gma_status_t validate_problem(const gma_problem_t* p) {
  if (!p) return GMA_ERR_INVALID_ARG;
  if (p->B < 1 || p->H < 1 || p->N < 0 || p->K < 1 || p->d < 1 || p->dv < 1) return GMA_ERR_INVALID_ARG;
  if (!(p->eps >= 0.0f) || p->eps == INFINITY) return GMA_ERR_INVALID_ARG;
  if (p->dtype != GMA_F32 && p->dtype != GMA_BF16) return GMA_ERR_UNSUPPORTED;
  if (p->d != kD || p->dv != kDv || p->K > kMaxK) return GMA_ERR_UNSUPPORTED;
  if ((long long)p->B * p->H * (long long)p->N >= (1LL << 31)) return GMA_ERR_UNSUPPORTED;
  return GMA_OK;
}

// Projected forward: [the forward's own workspace | GEMM workspace | Y float32 [B*N][3*H*64] | Q | K | V].
struct ProjLayout {
  size_t base, lt, y, q, k, v, total;
};
ProjLayout proj_layout(const gma_problem_t& p, bool causal, bool det);

// det: the deterministic reduction mode (taken once per call, so that the size checked is the one used).
size_t required_bytes(const gma_problem_t& p, gma_op_t op, bool det) {
  if (op == GMA_OP_PROJECTED_BIDIR || op == GMA_OP_PROJECTED_CAUSAL)
    return proj_layout(p, op == GMA_OP_PROJECTED_CAUSAL, det).total;
  if (op == GMA_OP_CROSS) op = GMA_OP_BIDIR;  // the same workspace: it does not depend on N
  if (op == GMA_OP_CAUSAL_DECODE) return simt_decode_bytes(p);
  if (op == GMA_OP_BACKWARD_BIDIR || op == GMA_OP_BACKWARD_CAUSAL)
    return simt_backward_bytes(p, op == GMA_OP_BACKWARD_CAUSAL, det);
  if (p.dtype == GMA_BF16) return tc_plan(p, op, det).total;
  return simt_plan(p, op, det).total;
}

ProjLayout proj_layout(const gma_problem_t& p, bool causal, bool det) {
  ProjLayout L{};
  const size_t es = p.dtype == GMA_BF16 ? 2 : 4;
  const size_t qkv = align_up((size_t)p.B * p.H * p.N * kD * es);
  L.base = align_up(required_bytes(p, causal ? GMA_OP_CAUSAL : GMA_OP_BIDIR, det));
  L.lt = L.base;
  const bool lib_gemm = p.dtype != GMA_BF16;  // float32 I/O: library GEMM workspace and a float32 Y
  L.y = L.lt + (lib_gemm ? align_up(proj_lt_workspace_bytes()) : 0);
  L.q = L.y + (lib_gemm ? align_up((size_t)p.B * p.N * 3 * p.H * kD * sizeof(float)) : 0);
  L.k = L.q + qkv;
  L.v = L.k + qkv;
  L.total = L.v + qkv;
  return L;
}

// Nk: keys / values per (b, h); N (= p->N) except for cross-attention.
gma_status_t run(const gma_problem_t* p, gma_op_t op, int Nk, const void* Q, const void* K, const void* V,
                 const float* mu, const float* sigma2, const float* log_pi, void* out, void* ws, size_t ws_bytes,
                 void* stream, bool clear_err = true, int det_mode = -1) {
  static const char* const kNames[] = {"gma_responsibilities", "gma_forward_bidir", "gma_forward_causal",
                                       "gma_forward_cross", "gma_causal_state"};
  const int oi = (int)op;
  NvtxScope range(oi >= 0 && oi < 5 ? kNames[oi] : "gma_call");
  gma_status_t s = validate_problem(p);
  if (s != GMA_OK) return s;
  if (Nk < 0) return GMA_ERR_INVALID_ARG;
  if ((long long)p->B * p->H * (long long)Nk >= (1LL << 31)) return GMA_ERR_UNSUPPORTED;
  if (!mu || !sigma2 || !log_pi || !ws) return GMA_ERR_INVALID_ARG;
  if (p->N > 0) {  // with N == 0 nothing is read or written, so empty tensors may be null
    if (!Q || !out) return GMA_ERR_INVALID_ARG;
    if (op != GMA_OP_RESPONSIBILITIES && Nk > 0 && (!K || !V)) return GMA_ERR_INVALID_ARG;
    if (op != GMA_OP_RESPONSIBILITIES && (out == Q || (K && out == K) || (V && out == V))) return GMA_ERR_INVALID_ARG;
  }
  const void* ptrs[] = {Q, K, V, mu, sigma2, log_pi, out};
  for (const void* q : ptrs)
    if (q && !aligned(q, 16)) return GMA_ERR_INVALID_ARG;
  if (!aligned(ws, kAlign)) return GMA_ERR_INVALID_ARG;
  const bool det = det_mode < 0 ? deterministic() : det_mode != 0;
  if (ws_bytes < required_bytes(*p, op, det)) return GMA_ERR_WORKSPACE;
  if (p->N == 0) return GMA_OK;
  cudaStream_t st = (cudaStream_t)stream;
  cudaGetLastError();  // a stale error from earlier caller work is not ours to report
  if (op == GMA_OP_CROSS) op = GMA_OP_BIDIR;  // the bidirectional kernels, with the key length Nk
  if (p->dtype == GMA_BF16) return tc_run(*p, op, Nk, Q, K, V, mu, sigma2, log_pi, out, ws, st, clear_err, det);
  return simt_run(*p, op, Nk, Q, K, V, mu, sigma2, log_pi, out, ws, st, det);
}

gma_status_t run_backward(const gma_problem_t* p, bool causal, const void* Q, const void* K, const void* V, const float* mu,
                                const float* sigma2, const float* log_pi, const void* dO, void* dQ, void* dK, void* dV,
                                float* dmu, float* dsigma2, float* dlog_pi, void* ws, size_t ws_bytes, void* stream) {
  gma_status_t s = validate_problem(p);
  if (s != GMA_OK) return s;
  if (!mu || !sigma2 || !log_pi || !ws || !dmu || !dsigma2 || !dlog_pi) return GMA_ERR_INVALID_ARG;
  const void* ins[] = {Q, K, V, mu, sigma2, log_pi, dO};
  const void* outs[] = {dQ, dK, dV, dmu, dsigma2, dlog_pi};
  if (p->N > 0)
    for (const void* q : ins)
      if (!q) return GMA_ERR_INVALID_ARG;
  if (p->N > 0 && (!dQ || !dK || !dV)) return GMA_ERR_INVALID_ARG;
  for (const void* q : ins)
    if (q && !aligned(q, 16)) return GMA_ERR_INVALID_ARG;
  for (const void* q : outs) {
    if (q && !aligned(q, 16)) return GMA_ERR_INVALID_ARG;
    for (const void* r : ins)
      if (q && q == r) return GMA_ERR_INVALID_ARG;
  }
  for (int i = 0; i < 6; ++i)
    for (int j = i + 1; j < 6; ++j)
      if (outs[i] && outs[i] == outs[j]) return GMA_ERR_INVALID_ARG;
  if (!aligned(ws, kAlign)) return GMA_ERR_INVALID_ARG;
  const bool det = deterministic();
  if (ws_bytes < required_bytes(*p, causal ? GMA_OP_BACKWARD_CAUSAL : GMA_OP_BACKWARD_BIDIR, det))
    return GMA_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  cudaGetLastError();
  return simt_backward(*p, causal, Q, K, V, mu, sigma2, log_pi, dO, dQ, dK, dV, dmu, dsigma2, dlog_pi, ws, st, det);
}

}  // namespace
}  // namespace gma

using namespace gma;

extern "C" {

gma_status_t gma_set_wait_limit_ns(uint64_t ns) {
  if (ns != 0 && (ns < gma::kMinWaitNs || ns > gma::kMaxWaitNs)) return GMA_ERR_INVALID_ARG;
  gma::g_wait_ns.store(ns, std::memory_order_relaxed);
  return GMA_OK;
}

uint64_t gma_get_wait_limit_ns(void) { return gma::wait_limit_ns(); }

gma_status_t gma_set_deterministic(int mode) {
  if (mode < -1 || mode > 1) return GMA_ERR_INVALID_ARG;
  gma::g_det.store(mode, std::memory_order_relaxed);
  return GMA_OK;
}

int gma_get_deterministic(void) { return gma::deterministic() ? 1 : 0; }

size_t gma_workspace_bytes(const gma_problem_t* p, gma_op_t op) {
  if (validate_problem(p) != GMA_OK) return 0;
  if (op < GMA_OP_RESPONSIBILITIES || op > GMA_OP_PROJECTED_CAUSAL) return 0;
  return required_bytes(*p, op, deterministic());
}

gma_status_t gma_forward_projected(const gma_problem_t* p, int causal, int dm, const void* X, const void* Wqkv,
                                   const float* bqkv, const float* mu, const float* sigma2, const float* log_pi,
                                   void* O, void* ws, size_t ws_bytes, void* stream) {
  gma_status_t s = validate_problem(p);
  if (s != GMA_OK) return s;
  if (causal != 0 && causal != 1) return GMA_ERR_INVALID_ARG;
  if (dm < 8 || dm % 8 != 0 || dm > (1 << 16)) return GMA_ERR_UNSUPPORTED;
  if (!mu || !sigma2 || !log_pi || !ws || !Wqkv || !bqkv) return GMA_ERR_INVALID_ARG;
  if (p->N > 0 && (!X || !O)) return GMA_ERR_INVALID_ARG;
  if (O && (O == X || O == Wqkv || O == (const void*)bqkv)) return GMA_ERR_INVALID_ARG;
  const void* ptrs[] = {X, Wqkv, bqkv, mu, sigma2, log_pi, O};
  for (const void* q : ptrs)
    if (q && !aligned(q, 16)) return GMA_ERR_INVALID_ARG;
  if (!aligned(ws, kAlign)) return GMA_ERR_INVALID_ARG;
  const gma_op_t op = causal ? GMA_OP_PROJECTED_CAUSAL : GMA_OP_PROJECTED_BIDIR;
  const bool det = deterministic();
  if (ws_bytes < required_bytes(*p, op, det)) return GMA_ERR_WORKSPACE;
  if (p->N == 0) return GMA_OK;
  cudaStream_t st = (cudaStream_t)stream;
  cudaGetLastError();
  const ProjLayout L = proj_layout(*p, causal != 0, det);
  char* w = (char*)ws;
  s = proj_run(*p, dm, X, Wqkv, bqkv, (float*)(w + L.y), w + L.q, w + L.k, w + L.v, w + L.lt, (Ctrl*)ws, st, det);
  if (s != GMA_OK) return s;
  // bf16: the projection kernel cleared the error word and reports its bounded waits there
  return run(p, causal ? GMA_OP_CAUSAL : GMA_OP_BIDIR, p->N, w + L.q, w + L.k, w + L.v, mu, sigma2, log_pi, O, ws,
             L.base, stream, p->dtype != GMA_BF16, det ? 1 : 0);
}

gma_status_t gma_responsibilities(const gma_problem_t* p, const void* X, const float* mu, const float* sigma2,
                                  const float* log_pi, float* gamma_out, void* ws, size_t ws_bytes, void* stream) {
  return run(p, GMA_OP_RESPONSIBILITIES, p ? p->N : 0, X, nullptr, nullptr, mu, sigma2, log_pi, gamma_out, ws, ws_bytes, stream);
}

gma_status_t gma_forward_bidir(const gma_problem_t* p, const void* Q, const void* K, const void* V, const float* mu,
                               const float* sigma2, const float* log_pi, void* O, void* ws, size_t ws_bytes,
                               void* stream) {
  return run(p, GMA_OP_BIDIR, p ? p->N : 0, Q, K, V, mu, sigma2, log_pi, O, ws, ws_bytes, stream);
}

gma_status_t gma_forward_causal(const gma_problem_t* p, const void* Q, const void* K, const void* V, const float* mu,
                                const float* sigma2, const float* log_pi, void* O, void* ws, size_t ws_bytes,
                                void* stream) {
  return run(p, GMA_OP_CAUSAL, p ? p->N : 0, Q, K, V, mu, sigma2, log_pi, O, ws, ws_bytes, stream);
}

gma_status_t gma_forward_cross(const gma_problem_t* p, int Nk, const void* Q, const void* K, const void* V,
                               const float* mu, const float* sigma2, const float* log_pi, void* O, void* ws,
                               size_t ws_bytes, void* stream) {
  return run(p, GMA_OP_CROSS, Nk, Q, K, V, mu, sigma2, log_pi, O, ws, ws_bytes, stream);
}

size_t gma_state_bytes(const gma_problem_t* p) {
  if (validate_problem(p) != GMA_OK) return 0;
  return (size_t)p->B * p->H * p->K * (p->dv + 1) * sizeof(float);
}

gma_status_t gma_causal_state(const gma_problem_t* p, const void* K, const void* V, const float* mu,
                              const float* sigma2, const float* log_pi, float* state, void* ws, size_t ws_bytes,
                              void* stream) {
  gma_status_t s = validate_problem(p);
  if (s != GMA_OK) return s;
  if (!mu || !sigma2 || !log_pi || !ws || !state) return GMA_ERR_INVALID_ARG;
  if (p->N > 0 && (!K || !V)) return GMA_ERR_INVALID_ARG;
  const void* ptrs[] = {K, V, mu, sigma2, log_pi, state};
  for (const void* q : ptrs)
    if (q && !aligned(q, 16)) return GMA_ERR_INVALID_ARG;
  if (!aligned(ws, kAlign)) return GMA_ERR_INVALID_ARG;
  const bool det = deterministic();
  if (ws_bytes < required_bytes(*p, GMA_OP_CAUSAL_STATE, det)) return GMA_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  cudaGetLastError();
  if (p->dtype == GMA_BF16)
    return tc_run(*p, GMA_OP_CAUSAL_STATE, p->N, nullptr, K, V, mu, sigma2, log_pi, state, ws, st, true, det);
  return simt_run(*p, GMA_OP_CAUSAL_STATE, p->N, nullptr, K, V, mu, sigma2, log_pi, state, ws, st, det);
}

gma_status_t gma_causal_decode(const gma_problem_t* p, const void* Q, const void* K, const void* V, const float* mu,
                               const float* sigma2, const float* log_pi, float* state, void* O, void* ws,
                               size_t ws_bytes, void* stream) {
  gma_status_t s = validate_problem(p);
  if (s != GMA_OK) return s;
  if (!mu || !sigma2 || !log_pi || !ws || !state) return GMA_ERR_INVALID_ARG;
  if (p->N > 0) {
    if (!Q || !K || !V || !O) return GMA_ERR_INVALID_ARG;
    if (O == Q || O == K || O == V || O == (const void*)state) return GMA_ERR_INVALID_ARG;
  }
  const void* ptrs[] = {Q, K, V, mu, sigma2, log_pi, state, O};
  for (const void* q : ptrs)
    if (q && !aligned(q, 16)) return GMA_ERR_INVALID_ARG;
  if (!aligned(ws, kAlign)) return GMA_ERR_INVALID_ARG;
  if (ws_bytes < required_bytes(*p, GMA_OP_CAUSAL_DECODE, false)) return GMA_ERR_WORKSPACE;
  if (p->N == 0) return GMA_OK;
  cudaStream_t st = (cudaStream_t)stream;
  cudaGetLastError();
  return simt_decode(*p, Q, K, V, mu, sigma2, log_pi, state, O, ws, st);
}

gma_status_t gma_decode_prepare(const gma_problem_t* p, const float* mu, const float* sigma2, const float* log_pi,
                                void* ws, size_t ws_bytes, void* stream) {
  gma_status_t s = validate_problem(p);
  if (s != GMA_OK) return s;
  if (!mu || !sigma2 || !log_pi || !ws) return GMA_ERR_INVALID_ARG;
  const void* ptrs[] = {mu, sigma2, log_pi};
  for (const void* q : ptrs)
    if (!aligned(q, 16)) return GMA_ERR_INVALID_ARG;
  if (!aligned(ws, kAlign)) return GMA_ERR_INVALID_ARG;
  if (ws_bytes < required_bytes(*p, GMA_OP_CAUSAL_DECODE, false)) return GMA_ERR_WORKSPACE;
  cudaGetLastError();
  return simt_decode_fold(*p, mu, sigma2, log_pi, ws, (cudaStream_t)stream);
}

gma_status_t gma_causal_decode_prepared(const gma_problem_t* p, const void* Q, const void* K, const void* V,
                                        float* state, void* O, void* ws, size_t ws_bytes, void* stream) {
  gma_status_t s = validate_problem(p);
  if (s != GMA_OK) return s;
  if (!ws || !state) return GMA_ERR_INVALID_ARG;
  if (p->N > 0) {
    if (!Q || !K || !V || !O) return GMA_ERR_INVALID_ARG;
    if (O == Q || O == K || O == V || O == (const void*)state) return GMA_ERR_INVALID_ARG;
  }
  const void* ptrs[] = {Q, K, V, state, O};
  for (const void* q : ptrs)
    if (q && !aligned(q, 16)) return GMA_ERR_INVALID_ARG;
  if (!aligned(ws, kAlign)) return GMA_ERR_INVALID_ARG;
  if (ws_bytes < required_bytes(*p, GMA_OP_CAUSAL_DECODE, false)) return GMA_ERR_WORKSPACE;
  if (p->N == 0) return GMA_OK;
  cudaGetLastError();
  return simt_decode_run(*p, Q, K, V, state, O, ws, false, (cudaStream_t)stream);
}


gma_status_t gma_backward_bidir(const gma_problem_t* p, const void* Q, const void* K, const void* V, const float* mu,
                                const float* sigma2, const float* log_pi, const void* dO, void* dQ, void* dK, void* dV,
                                float* dmu, float* dsigma2, float* dlog_pi, void* ws, size_t ws_bytes, void* stream) {
  return gma::run_backward(p, false, Q, K, V, mu, sigma2, log_pi, dO, dQ, dK, dV, dmu, dsigma2, dlog_pi, ws, ws_bytes,
                           stream);
}

gma_status_t gma_backward_causal(const gma_problem_t* p, const void* Q, const void* K, const void* V, const float* mu,
                                 const float* sigma2, const float* log_pi, const void* dO, void* dQ, void* dK, void* dV,
                                 float* dmu, float* dsigma2, float* dlog_pi, void* ws, size_t ws_bytes, void* stream) {
  return gma::run_backward(p, true, Q, K, V, mu, sigma2, log_pi, dO, dQ, dK, dV, dmu, dsigma2, dlog_pi, ws, ws_bytes,
                           stream);
}

gma_status_t gma_check_device_error(void* ws, void* stream) {
  if (!ws || !aligned(ws, kAlign)) return GMA_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)stream;
  Ctrl c;
  if (cudaMemcpyAsync(&c, ws, sizeof(Ctrl), cudaMemcpyDeviceToHost, st) != cudaSuccess) return GMA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return GMA_ERR_CUDA;
  return c.err == kErrNone ? GMA_OK : (c.err == kErrRange ? GMA_ERR_RANGE : GMA_ERR_TIMEOUT);
}

const char* gma_status_string(gma_status_t s) {
  switch (s) {
    case GMA_OK: return "ok";
    case GMA_ERR_INVALID_ARG: return "invalid argument";
    case GMA_ERR_UNSUPPORTED: return "unsupported problem (d, dv, K or dtype)";
    case GMA_ERR_WORKSPACE: return "workspace too small";
    case GMA_ERR_CUDA: return "CUDA runtime error";
    case GMA_ERR_TIMEOUT: return "a bounded device wait timed out";
    case GMA_ERR_RANGE: return "a parameter is outside the range of the fp16 log-density operands";
  }
  return "unknown status";
}

int gma_version(void) { return (0 << 16) | 1; }

const char* gma_last_error(void) { return g_detail; }

}  // extern "C"

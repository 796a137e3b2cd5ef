// gma_internal.h -- host-side plumbing shared by the translation units of libgma.so.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "gma.h"

namespace gma {

constexpr int kD = 64;          // routing width d supported by this build
constexpr int kDv = 64;         // value width dv supported by this build
constexpr int kMaxK = 256;      // largest mixture size
constexpr int kStateCols = 65;  // CUDA-core path: [Vt | Z] row width (dv + 1)
constexpr size_t kAlign = 256;  // alignment of every workspace section
constexpr int kTargetUnits = 304;  // work units the split heuristics aim for (2 per SM on 152 SMs)

// Control block at the start of every workspace.
struct Ctrl {
  uint32_t err;       // non-zero: a bounded device wait gave up
  uint32_t err_site;  // which wait (kernel-defined code)
  uint32_t pad[62];
};
static_assert(sizeof(Ctrl) == 256, "control block is one aligned section");

// Device error codes written into Ctrl::err.
enum : uint32_t { kErrNone = 0, kErrTimeout = 1, kErrRange = 2 };

inline size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }
inline int cdiv(long long a, long long b) { return (int)((a + b - 1) / b); }

// ---- CUDA-core (float32) path -------------------------------------------------------------------
constexpr int kSimtTile = 32;  // tokens per tile

struct SimtPlan {
  int tiles;       // ceil(N / tile)
  int splits;      // CTAs per (b,h) for the write phase (bidir) or segments (causal)
  int seg_tiles;   // tiles per segment / split
  bool det;        // deterministic reduction mode: the write's partial states are stored, then summed
  size_t off_params, off_state, off_agg, total;  // off_agg: the partial states (det only)
};
// det: plan for the deterministic reduction mode (the bidirectional, cross and state workspaces then
// hold the write's partial states of at most kTargetUnits + B*H CTAs, whatever the key length).
SimtPlan simt_plan(const gma_problem_t& p, gma_op_t op, bool det = false);
// Nk: keys / values per (b, h) for the write phase (p.N except for cross-attention).
gma_status_t simt_run(const gma_problem_t& p, gma_op_t op, int Nk, const void* Q, const void* K, const void* V,
                      const float* mu, const float* sigma2, const float* log_pi, void* out, void* ws,
                      cudaStream_t stream, bool det = false);

// ---- tensor-core (bf16 I/O) path ----------------------------------------------------------------
struct TcPlan {
  int Kp;          // K rounded up to 64, 128 or 256: the width of the log-density contraction (4 x the components per row thread)
  int tiles;       // ceil(N / 128)
  int splits;      // CTAs per (b,h) in the write phase / segments in the causal path
  int seg_tiles;   // tiles per split or segment
  bool det;        // deterministic reduction mode: the write's per-CTA states are stored, then summed
  size_t off_w, off_c, off_flags, off_state;  // off_flags: per-head range flags of the parameter fold
  size_t off_agg;  // det only: the write's per-CTA states (at most max(152, B*H) CTAs, any key length)
  size_t total;
};
TcPlan tc_plan(const gma_problem_t& p, gma_op_t op, bool det = false);
// clear_err: the parameter fold clears the workspace error word first (false when an earlier kernel of
// the same call, the tcgen05 projection, has already cleared it and may have reported into it).
// ctrl: the control block the kernels report into (null: the one at the start of ws).
gma_status_t tc_run(const gma_problem_t& p, gma_op_t op, int Nk, const void* Q, const void* K, const void* V,
                    const float* mu, const float* sigma2, const float* log_pi, void* out, void* ws,
                    cudaStream_t stream, bool clear_err = true, bool det = false, Ctrl* ctrl = nullptr);
bool tc_available();
// Tensor map over a row-major bf16 matrix [rows][cols]: boxes of box_cols x box_rows, 128-byte swizzle,
// zero fill outside (a 3-D map with a unit outer dimension, read with 3-D tensor loads).
bool make_map_rows(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                   uint32_t box_rows);
// Backward pass of the bidirectional or causal forward (float32 CUDA-core kernels, both I/O dtypes).
// det: every sum across CTAs (the state, its gradient and the parameter sums) is taken from stored
// partials in a fixed order.
size_t simt_backward_bytes(const gma_problem_t& p, bool causal, bool det = false);
gma_status_t simt_backward(const gma_problem_t& p, bool causal, const void* Q, const void* K, const void* V, const float* mu,
                           const float* sigma2, const float* log_pi, const void* dO, void* dQ, void* dK, void* dV,
                           float* dmu, float* dsigma2, float* dlog_pi, void* ws, cudaStream_t stream, bool det = false);
// Decode T = p.N new tokens per (b, h) against `state` (float32 [B*H][K][dv + 1], in place).  Workspace:
// simt_decode_bytes(p) (a control block and every head's folded parameters).
size_t simt_decode_bytes(const gma_problem_t& p);
gma_status_t simt_decode(const gma_problem_t& p, const void* Q, const void* K, const void* V, const float* mu,
                         const float* sigma2, const float* log_pi, float* state, void* out, void* ws,
                         cudaStream_t stream);
// The two halves of simt_decode: the parameter fold into the workspace, and the decode reading it
// (dependent = 1: launched as a dependent of the fold just before it).
gma_status_t simt_decode_fold(const gma_problem_t& p, const float* mu, const float* sigma2, const float* log_pi,
                              void* ws, cudaStream_t st);
gma_status_t simt_decode_run(const gma_problem_t& p, const void* Q, const void* K, const void* V, float* state,
                             void* out, void* ws, bool dependent, cudaStream_t st);
// Q / K / V projection of a Transformer block into Q, K, V ([B][H][N][64], I/O dtype, bias added).  bf16:
// one tcgen05 GEMM with the layout in its epilogue; it clears ctrl's error word and reports its own
// bounded waits there (Y and lt_ws unused).  float32: library GEMM into Y (float32), then a layout
// kernel; lt_ws: proj_lt_workspace_bytes() bytes.  det: the library GEMM is restricted to algorithms
// without a split-K reduction (the tcgen05 GEMM has none).
size_t proj_lt_workspace_bytes();
gma_status_t proj_run(const gma_problem_t& p, int dm, const void* X, const void* W, const float* bias, float* Y,
                      void* Q, void* K, void* V, void* lt_ws, Ctrl* ctrl, cudaStream_t st, bool det = false);
// Test hook: bit 0 makes the next bidirectional write launch skip its first X-tile load, so that a
// bounded device wait runs out and reports GMA_ERR_TIMEOUT.  The environment variable GMA_FAULT_INJECT
// (anything but "" or "0") sets it for the first bidirectional call of the process.
void tc_set_fault_injection(uint32_t mask);

// Bounds-check debug build (-DGMA_BOUNDS_CHECK): the per-translation-unit records of failed checks
// (first site, its index and extent, failures), copied to h[4] and optionally cleared, and a kernel that
// fails one check on purpose without touching memory.  GMA_ERR_UNSUPPORTED in the normal build.
gma_status_t tc_bounds_io(unsigned long long* h, bool clear);
gma_status_t simt_bounds_io(unsigned long long* h, bool clear);
gma_status_t bounds_selftest(cudaStream_t st);

// NVTX range for the lifetime of the object (one per C-ABI call).
struct NvtxScope {
  explicit NvtxScope(const char* name);
  ~NvtxScope();
  NvtxScope(const NvtxScope&) = delete;
  NvtxScope& operator=(const NvtxScope&) = delete;
};

// Limit of every bounded device wait of the tensor-core kernels, in ns: gma_set_wait_limit_ns(), else the
// environment variable GMA_WAIT_LIMIT_MS (read once), else 1 s.
uint64_t wait_limit_ns();

// Deterministic reduction mode: gma_set_deterministic(), else the environment variable GMA_DETERMINISTIC
// (read once; a value other than empty or "0" turns it on), else off.  When on, no sum across CTAs uses
// atomics: each CTA stores its partial, and one thread per element adds the partials up in a fixed
// order, so that repeated calls on the same inputs give bitwise-equal outputs.  The workspaces of the
// affected calls grow by the partials.
bool deterministic();

// Launch bookkeeping: counts every kernel launch, brackets it with an NVTX range named for its phase
// and, while profiling is on, with a CUDA event pair on the launch stream.
void* prof_before(cudaStream_t st, const char* name);
void prof_after(cudaStream_t st, void* token);

#define GMA_LAUNCH(name, kernel, grid, block, smem, stream, ...)    \
  do {                                                              \
    void* gma_prof_token_ = ::gma::prof_before((stream), (name));   \
    kernel<<<(grid), (block), (smem), (stream)>>>(__VA_ARGS__);     \
    ::gma::prof_after((stream), gma_prof_token_);                   \
  } while (0)

// Programmatic dependent launch: the kernel may start while the previous kernel on the stream is
// finishing; it must execute griddepcontrol.wait (dep_wait) in every thread before it reads what that
// kernel wrote, and it may read what kernels before that one wrote only after the wait as well.
template <typename... KArgs, typename... Args>
inline void launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                             Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

#define GMA_LAUNCH_DEPENDENT(name, kernel, grid, block, smem, stream, ...)                  \
  do {                                                                                    \
    void* gma_prof_token_ = ::gma::prof_before((stream), (name));                         \
    ::gma::launch_dependent(kernel, dim3(grid), dim3(block), (smem), (stream), __VA_ARGS__); \
    ::gma::prof_after((stream), gma_prof_token_);                                         \
  } while (0)

// Records a description of the failing step (and the pending CUDA error, if any) for
// gma_last_error(); returns GMA_ERR_CUDA.
gma_status_t cuda_fail(const char* step, cudaError_t err = cudaSuccess, const void* func = nullptr);
// cudaGetLastError() after a launch; on failure records the step, CUDA's message and the kernel's
// attributes.
gma_status_t check_launch(const char* step, const void* func);
void set_error_detail(const char* msg);

// Sets the dynamic shared-memory opt-in of a kernel once per device.
gma_status_t set_smem_optin(const void* func, int bytes, int slot);
// Asks for the largest shared-memory carveout for a small kernel that runs between the large-shared-memory
// kernels, so that the SMs need not change their L1 / shared split around it (once per device).
gma_status_t set_carveout_max(const void* func);

}  // namespace gma

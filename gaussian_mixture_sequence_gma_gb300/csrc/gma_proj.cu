// gma_proj.cu -- the Q / K / V projection of the Transformer-block form of the forward pass
// (Gaussian Mixture Attention pages, gist.science summary "Variants and training": GMA replaces the
// attention of a Transformer block whose queries, keys and values are linear projections of the
// block input; the causal language model of the experiments uses it at d_model = 768, 12 heads).
//
// One plain library GEMM, Y [B*N][3*H*64] = X [B*N][dm] Wqkv [dm][3*H*64], float32 accumulation and
// float32 output (cuBLASLt), then one layout kernel that adds the bias in float32, rounds once to the
// I/O dtype and writes Q, K, V as [B][H][N][64] for the GMA kernels.  Column block 0 of Y holds Q,
// block 1 K, block 2 V; within a block, columns 64h .. 64h+63 are head h.
#include <cublasLt.h>

#include <cstdio>
#include <mutex>

#include "gma_internal.h"

namespace gma {
namespace {

constexpr int kMaxDevices = 64;

struct LtPlan {
  int M = 0, Ncol = 0, dm = 0, dtype = -1;
  cublasLtMatmulAlgo_t algo{};
  bool valid = false;
};

std::mutex g_lt_mu;
cublasLtHandle_t g_lt[kMaxDevices] = {};
LtPlan g_plan[kMaxDevices];

gma_status_t lt_fail(const char* what, cublasStatus_t st) {
  char msg[128];
  snprintf(msg, sizeof msg, "%s returned cublasStatus_t %d", what, (int)st);
  set_error_detail(msg);
  return GMA_ERR_CUDA;
}

// One thread per 8 consecutive dims of one output row: index i = (((w * B + b) * H + h) * N + n) * 8 + j.
template <typename IO>
__global__ void __launch_bounds__(256) proj_layout_kernel(const float* __restrict__ Y, const float* __restrict__ bias,
                                                          int B, int H, int N, IO* __restrict__ Q, IO* __restrict__ K,
                                                          IO* __restrict__ V) {
  const size_t total = (size_t)3 * B * H * N * 8;
  const int ncol = 3 * H * kD;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int j = (int)(i & 7);
    size_t r = i >> 3;
    const int n = (int)(r % N);
    r /= N;
    const int h = (int)(r % H);
    r /= H;
    const int b = (int)(r % B);
    const int w = (int)(r / B);
    const int col = (w * H + h) * kD + 8 * j;
    const float4* src = reinterpret_cast<const float4*>(Y + ((size_t)b * N + n) * ncol + col);
    const float4* bs = reinterpret_cast<const float4*>(bias + col);
    const float4 y0 = __ldg(src), y1 = __ldg(src + 1), b0 = __ldg(bs), b1 = __ldg(bs + 1);
    const float v[8] = {y0.x + b0.x, y0.y + b0.y, y0.z + b0.z, y0.w + b0.w,
                        y1.x + b1.x, y1.y + b1.y, y1.z + b1.z, y1.w + b1.w};
    IO* dst = (w == 0 ? Q : (w == 1 ? K : V)) + (((size_t)b * H + h) * N + n) * kD + 8 * j;
    if constexpr (sizeof(IO) == 2) {
      uint32_t u[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 p2 = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
        u[k] = *reinterpret_cast<const uint32_t*>(&p2);
      }
      *reinterpret_cast<uint4*>(dst) = make_uint4(u[0], u[1], u[2], u[3]);
    } else {
      reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
      reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
}

}  // namespace

size_t proj_lt_workspace_bytes() { return (size_t)32 << 20; }

gma_status_t proj_run(const gma_problem_t& p, int dm, const void* X, const void* W, const float* bias, float* Y,
                      void* Q, void* K, void* V, void* lt_ws, cudaStream_t st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cuda_fail("cudaGetDevice");
  const int M = p.B * p.N, Ncol = 3 * p.H * kD;
  const bool bf16 = p.dtype == GMA_BF16;
  const cudaDataType_t io = bf16 ? CUDA_R_16BF : CUDA_R_32F;
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t la = nullptr, lb = nullptr, lc = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  gma_status_t ret = GMA_OK;
  cublasStatus_t s;
  std::lock_guard<std::mutex> lock(g_lt_mu);
  if (!g_lt[dev] && (s = cublasLtCreate(&g_lt[dev])) != CUBLAS_STATUS_SUCCESS) return lt_fail("cublasLtCreate", s);
  // column-major view: Y^T [Ncol x M] = W^T [Ncol x dm] . X^T [dm x M]; row-major W, X, Y are exactly these
  if ((s = cublasLtMatmulDescCreate(&op, CUBLAS_COMPUTE_32F, CUDA_R_32F)) != CUBLAS_STATUS_SUCCESS ||
      (s = cublasLtMatrixLayoutCreate(&la, io, Ncol, dm, Ncol)) != CUBLAS_STATUS_SUCCESS ||
      (s = cublasLtMatrixLayoutCreate(&lb, io, dm, M, dm)) != CUBLAS_STATUS_SUCCESS ||
      (s = cublasLtMatrixLayoutCreate(&lc, CUDA_R_32F, Ncol, M, Ncol)) != CUBLAS_STATUS_SUCCESS) {
    ret = lt_fail("cublasLt descriptor setup", s);
  }
  LtPlan& plan = g_plan[dev];
  if (ret == GMA_OK && !(plan.valid && plan.M == M && plan.Ncol == Ncol && plan.dm == dm && plan.dtype == (int)p.dtype)) {
    size_t wsb = proj_lt_workspace_bytes();
    cublasLtMatmulHeuristicResult_t res{};
    int found = 0;
    if ((s = cublasLtMatmulPreferenceCreate(&pref)) != CUBLAS_STATUS_SUCCESS ||
        (s = cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &wsb, sizeof wsb)) !=
            CUBLAS_STATUS_SUCCESS ||
        (s = cublasLtMatmulAlgoGetHeuristic(g_lt[dev], op, la, lb, lc, lc, pref, 1, &res, &found)) !=
            CUBLAS_STATUS_SUCCESS) {
      ret = lt_fail("cublasLtMatmulAlgoGetHeuristic", s);
    } else if (found < 1) {
      set_error_detail("cublasLt found no algorithm for the projection GEMM");
      ret = GMA_ERR_UNSUPPORTED;
    } else {
      plan.M = M;
      plan.Ncol = Ncol;
      plan.dm = dm;
      plan.dtype = (int)p.dtype;
      plan.algo = res.algo;
      plan.valid = true;
    }
  }
  if (ret == GMA_OK) {
    const float alpha = 1.f, beta = 0.f;
    if ((s = cublasLtMatmul(g_lt[dev], op, &alpha, W, la, X, lb, &beta, Y, lc, Y, lc, &plan.algo, lt_ws,
                            proj_lt_workspace_bytes(), st)) != CUBLAS_STATUS_SUCCESS)
      ret = lt_fail("cublasLtMatmul", s);
  }
  if (pref) cublasLtMatmulPreferenceDestroy(pref);
  if (lc) cublasLtMatrixLayoutDestroy(lc);
  if (lb) cublasLtMatrixLayoutDestroy(lb);
  if (la) cublasLtMatrixLayoutDestroy(la);
  if (op) cublasLtMatmulDescDestroy(op);
  if (ret != GMA_OK) return ret;
  const size_t total = (size_t)3 * p.B * p.H * p.N * 8;
  const unsigned grid = (unsigned)std::min<size_t>((total + 255) / 256, 152 * 16);
  if (bf16) {
    GMA_LAUNCH("proj_layout", proj_layout_kernel<__nv_bfloat16>, grid, 256, 0, st, Y, bias, p.B, p.H, p.N,
               (__nv_bfloat16*)Q, (__nv_bfloat16*)K, (__nv_bfloat16*)V);
    return check_launch("launch proj_layout", (const void*)proj_layout_kernel<__nv_bfloat16>);
  }
  GMA_LAUNCH("proj_layout", proj_layout_kernel<float>, grid, 256, 0, st, Y, bias, p.B, p.H, p.N, (float*)Q, (float*)K,
             (float*)V);
  return check_launch("launch proj_layout", (const void*)proj_layout_kernel<float>);
}

}  // namespace gma

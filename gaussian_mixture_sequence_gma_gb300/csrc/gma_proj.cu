// gma_proj.cu -- the Q / K / V projection of the Transformer-block form of the forward pass
// (Gaussian Mixture Attention pages, gist.science summary "Variants and training": GMA replaces the
// attention of a Transformer block whose queries, keys and values are linear projections of the
// block input; the causal language model of the experiments uses it at d_model = 768, 12 heads).
//
// bf16 I/O: one hand-written tcgen05 GEMM, Y [B*N][3*H*64] = X [B*N][dm] Wqkv [dm][3*H*64] with float32
// accumulation in TMEM, whose epilogue adds the bias in float32, rounds once to bf16 and writes Q, K, V
// as [B][H][N][64] for the GMA kernels (no float32 Y).  float32 I/O: one plain library GEMM (cuBLASLt,
// float32 output) and one layout kernel doing the same.  Column block 0 of Y holds Q, block 1 K, block 2
// V; within a block, columns 64h .. 64h+63 are head h.
#include <cublasLt.h>

#include <cstdio>
#include <mutex>

#include "gma_internal.h"
#include "gma_tc_common.cuh"

namespace gma {
namespace {

constexpr int kMaxDevices = 64;

struct LtPlan {
  int M = 0, Ncol = 0, dm = 0, dtype = -1, det = -1;
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

// ---- bf16: one hand-written tcgen05 GEMM with the bias, the rounding and the layout in its epilogue ----
// Y [M = B*N][Ncol] = X [M][dm] Wqkv [dm][Ncol] in 256 x 256 tiles, one tile per CTA, one CTA per SM.  The
// tile is two 128-row halves with their own accumulators (all 512 TMEM columns) that share every Wqkv
// stage, so each stage of Wqkv is read from L2 once per 256 rows of X: the operands of this GEMM are
// re-read by every tile, and L2-to-SM traffic, not the tensor pipe, bounds it at smaller tiles.
// A = X rows (K-major, 128-byte swizzle, two 128-row boxes); B = Wqkv read as an MN-major operand: four
// 64-column boxes of 64 rows, 8 KB apart.  The K loop runs over 64-wide blocks of dm in a three-stage
// TMA ring (zero fill past dm, M and Ncol).  Warp 0 loads; one thread of warp 1 (rows 0-127) and one of
// warp 2 (rows 128-255) issue the contractions of their half (a thread issuing tcgen05.mma waits about
// as long as the instruction runs, so one issuer would bound the tile); warp 1 owns the TMEM columns.
// Warps 4-11 each take one lane quarter of one half: 16 columns at a time, + bias in float32, rounded
// once to bf16, stored straight into Q, K or V [B][H][N][64].
constexpr int kPBM = 256, kPBN = 256, kPBK = 64, kPStages = 3, kPThreads = 384;
constexpr uint32_t kPStageA = kPBM * kPBK * 2, kPStageB = kPBN * kPBK * 2, kPStage = kPStageA + kPStageB;
constexpr uint32_t kPSmem = kPStages * kPStage + 1024;  // + 1 KB alignment slack

struct ProjBars {
  uint64_t full[kPStages], empty[kPStages], acc[2];
  uint32_t tmem;
  tc::Abort ab;
};

__global__ void __launch_bounds__(kPThreads, 1)
    proj_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   const float* __restrict__ bias, int M, int Ncol, int dm, int H, int N, __nv_bfloat16* __restrict__ Q,
                   __nv_bfloat16* __restrict__ K, __nv_bfloat16* __restrict__ V, Ctrl* ctrl, uint64_t wait_ns) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
  __shared__ ProjBars B;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m0 = blockIdx.x * kPBM, n0 = blockIdx.y * kPBN;
  const int KB = (dm + kPBK - 1) / kPBK;
  // this call's error word starts clear (the forward that follows leaves it as this kernel left it)
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) {
    ctrl->err = kErrNone;
    ctrl->err_site = 0;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      tc::mbar_init(&B.full[s], 1);
      tc::mbar_init(&B.empty[s], 2);  // both issuers read every stage
    }
    tc::mbar_init(&B.acc[0], 1);
    tc::mbar_init(&B.acc[1], 1);
    B.ab.flag = 0;
    tc::mbar_fence_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(&B.tmem, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = B.tmem;
  const uint32_t sa = tc::smem_u32(smem);
  if (warp == 0) {
    if (lane == 0) {
      int last[kPStages];
      for (int s = 0; s < kPStages; ++s) last[s] = -1;
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % kPStages;
        const uint32_t ph = (uint32_t)(kb / kPStages) & 1u;
        // the slot is free once both halves' contractions of its previous block have read it
        if (kb >= kPStages && !tc::wait_bounded(&B.empty[s], ph ^ 1u, &B.ab, ctrl, 130, wait_ns)) break;
        tc::mbar_expect_tx(&B.full[s], kPStage);
        uint8_t* st = smem + (size_t)s * kPStage;
        tc::tma_load_3d(st, &tmX, kPBK * kb, m0, 0, &B.full[s]);
        tc::tma_load_3d(st + kPStageA / 2, &tmX, kPBK * kb, m0 + kPBM / 2, 0, &B.full[s]);
#pragma unroll
        for (int i = 0; i < kPBN / 64; ++i)
          tc::tma_load_3d(st + kPStageA + 8192 * i, &tmW, n0 + 64 * i, kPBK * kb, 0, &B.full[s]);
        last[s] = (int)ph;
      }
      // never leave with copies in flight
      tc::Abort none{0};
      for (int s = 0; s < kPStages; ++s)
        if (last[s] >= 0) tc::wait_bounded(&B.full[s], (uint32_t)last[s], &none, ctrl, 131, wait_ns);
    }
  } else if (warp == 1 || warp == 2) {
    if (lane == 0) {
      const int hf = warp - 1;  // row half: rows 128 hf .. 128 hf + 127, accumulator columns 256 hf ..
      constexpr uint32_t idesc = tc::make_idesc(128, kPBN, 1, 1, 0, 1);  // bf16 x bf16, A K-major, B MN-major
      for (int kb = 0; kb < KB; ++kb) {
        const int s = kb % kPStages;
        if (!tc::wait_bounded(&B.full[s], (uint32_t)(kb / kPStages) & 1u, &B.ab, ctrl, 132, wait_ns)) break;
        tc::tc_fence_after();
        const uint32_t a = sa + (uint32_t)s * kPStage;
        const uint64_t da = tc::make_sdesc(a + (uint32_t)hf * (kPStageA / 2), 16, 1024);
        const uint64_t db = tc::make_sdesc(a + kPStageA, 8192, 1024);
#pragma unroll
        for (int ks = 0; ks < kPBK / 16; ++ks)
          tc::mma_ss_off(tmem + 256u * (uint32_t)hf, da, (uint32_t)(32 * ks) >> 4, db, (uint32_t)(2048 * ks) >> 4,
                         idesc, (kb > 0 || ks > 0) ? 1u : 0u);
        tc::mma_commit(&B.empty[s]);
      }
      tc::mma_commit(&B.acc[hf]);
      tc::Abort none{0};
      tc::wait_bounded(&B.acc[hf], 0, &none, ctrl, 133, wait_ns);  // contractions done before TMEM is freed
    }
  } else if (warp >= 4) {
    // epilogue: warp w reads TMEM lane quarter w % 4 of half (w - 4) / 4: token row m0 + 128 half + 32 q + lane
    const int q = warp & 3, hf = (warp - 4) >> 2, m = m0 + 128 * hf + 32 * q + lane;
    const bool ok = tc::warp_wait(&B.acc[hf], 0, &B.ab, ctrl, 134, wait_ns);
    if (ok) {
      tc::tc_fence_after();
      const int b = m / N, n = m - (m / N) * N;
      const int hc = H * kD;  // columns of each of Q, K, V
      // four 16-column loads in flight per wait (one round trip per 64 columns, not per 16)
#pragma unroll 1
      for (int c4 = 0; c4 < kPBN / 64; ++c4) {
        uint32_t r[64];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          tc::tmem_ld16(tmem + ((uint32_t)(32 * q) << 16) + 256u * (uint32_t)hf + 64 * c4 + 16 * j, r + 16 * j);
#pragma unroll
        for (int j = 0; j < 4; ++j) tc::tmem_ld_wait_tied16(r + 16 * j);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int col = n0 + 64 * c4 + 16 * j;
          if (col < Ncol && m < M) {
            const float4* bs = reinterpret_cast<const float4*>(bias + col);
            const uint32_t* rj = r + 16 * j;
            uint32_t u[8];
#pragma unroll
            for (int k4 = 0; k4 < 4; ++k4) {
              const float4 bb = __ldg(bs + k4);
              u[2 * k4] = tc::pack_bf16x2(__uint_as_float(rj[4 * k4]) + bb.x, __uint_as_float(rj[4 * k4 + 1]) + bb.y);
              u[2 * k4 + 1] =
                  tc::pack_bf16x2(__uint_as_float(rj[4 * k4 + 2]) + bb.z, __uint_as_float(rj[4 * k4 + 3]) + bb.w);
            }
            const int w = col / hc, hh = (col - w * hc) / kD, d = col - w * hc - hh * kD;
            __nv_bfloat16* dst = (w == 0 ? Q : (w == 1 ? K : V)) + (((size_t)b * H + hh) * N + n) * kD + d;
            reinterpret_cast<uint4*>(dst)[0] = make_uint4(u[0], u[1], u[2], u[3]);
            reinterpret_cast<uint4*>(dst)[1] = make_uint4(u[4], u[5], u[6], u[7]);
          }
        }
      }
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem, 512);
  }
}

}  // namespace

size_t proj_lt_workspace_bytes() { return (size_t)32 << 20; }

gma_status_t proj_run(const gma_problem_t& p, int dm, const void* X, const void* W, const float* bias, float* Y,
                      void* Q, void* K, void* V, void* lt_ws, Ctrl* ctrl, cudaStream_t st, bool det) {
  if (p.dtype == GMA_BF16) {
    const int M = p.B * p.N, Ncol = 3 * p.H * kD;
    CUtensorMap mx, mw;
    if (!make_map_rows(&mx, X, (uint64_t)M, (uint64_t)dm, kPBK, kPBM / 2) ||
        !make_map_rows(&mw, W, (uint64_t)dm, (uint64_t)Ncol, 64, kPBK))
      return GMA_ERR_CUDA;
    if (set_smem_optin((const void*)proj_tc_kernel, (int)kPSmem, 5) != GMA_OK) return GMA_ERR_CUDA;
    GMA_LAUNCH("proj_tc", proj_tc_kernel, dim3(cdiv(M, kPBM), cdiv(Ncol, kPBN)), kPThreads, kPSmem, st, mx, mw, bias, M,
               Ncol, dm, p.H, p.N, (__nv_bfloat16*)Q, (__nv_bfloat16*)K, (__nv_bfloat16*)V, ctrl, wait_limit_ns());
    return check_launch("launch proj_tc", (const void*)proj_tc_kernel);
  }
  (void)ctrl;
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
  if (ret == GMA_OK && !(plan.valid && plan.M == M && plan.Ncol == Ncol && plan.dm == dm && plan.dtype == (int)p.dtype &&
                        plan.det == (int)det)) {
    size_t wsb = proj_lt_workspace_bytes();
    // deterministic reduction mode: no split-K reduction scheme, so each output is one in-order sum
    uint32_t schemes = (uint32_t)CUBLASLT_REDUCTION_SCHEME_NONE;
    cublasLtMatmulHeuristicResult_t res{};
    int found = 0;
    if ((s = cublasLtMatmulPreferenceCreate(&pref)) != CUBLAS_STATUS_SUCCESS ||
        (s = cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &wsb, sizeof wsb)) !=
            CUBLAS_STATUS_SUCCESS ||
        (det && (s = cublasLtMatmulPreferenceSetAttribute(pref, CUBLASLT_MATMUL_PREF_REDUCTION_SCHEME_MASK, &schemes,
                                                          sizeof schemes)) != CUBLAS_STATUS_SUCCESS) ||
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
      plan.det = (int)det;
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

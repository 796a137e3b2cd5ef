// gma_simt.cu -- float32 CUDA-core path of the GMA forward pass (dtype GMA_F32).
//
// This is the precision path: float32 I/O asks for float32-level agreement, which
// the 16-bit tensor-core operands cannot give, and at the small K this dtype is
// used with the work is memory- and launch-bound rather than tensor-bound.
//
// Method (Gaussian Mixture Attention pages, gist.science summaries):
//   "Core mechanism" item 1  gamma_ik = softmax_k( log pi_k + log N(x_i; mu_k, diag sigma2_k) )
//   "Core mechanism" item 2  Vt = Gamma_K^T V, Z = Gamma_K^T 1, O = Gamma_Q Vt / (Gamma_Q Z + eps)
//   "Variants and training" item 3  causal: inclusive prefix sums over key positions.
// The log-density is evaluated in centered form, c_k - 1/2 sum_d (x_d - mu_kd)^2 / sigma2_kd with
// c_k = log pi_k - 1/2 sum_d log sigma2_kd; the -(d/2) log 2pi term is common to all k and
// cancels in the softmax.
#include <cuda_bf16.h>

#include "gma_internal.h"

namespace gma {
namespace {

constexpr int T = kSimtTile;
constexpr int kThreads = 256;

template <typename IO>
__device__ __forceinline__ float ld_io(const IO* p);
template <>
__device__ __forceinline__ float ld_io<float>(const float* p) { return __ldg(p); }
template <>
__device__ __forceinline__ float ld_io<__nv_bfloat16>(const __nv_bfloat16* p) { return __bfloat162float(*p); }

template <typename IO>
__device__ __forceinline__ void st_io(IO* p, float v);
template <>
__device__ __forceinline__ void st_io<float>(float* p, float v) { *p = v; }
template <>
__device__ __forceinline__ void st_io<__nv_bfloat16>(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// Prepared parameters, per head: mu_t[d][K], w_t[d][K] = 1/sigma2 (component index fastest so that a
// warp of consecutive components reads consecutive addresses), c[K].
struct SimtParams {
  float* mu_t;
  float* w_t;
  float* c;
};

__device__ __forceinline__ SimtParams params_at(float* base, int H, int K) {
  SimtParams P;
  P.mu_t = base;
  P.w_t = base + (size_t)H * kD * K;
  P.c = base + (size_t)2 * H * kD * K;
  return P;
}

// Folds (mu, sigma2, log_pi) into the prepared layout, clears the error word and zeroes `zero_n`
// floats at `zero` (the write-phase accumulator).
__global__ void simt_prep_kernel(const float* __restrict__ mu, const float* __restrict__ sigma2,
                                 const float* __restrict__ log_pi, int H, int K, float* params, Ctrl* ctrl,
                                 float* zero, size_t zero_n) {
  SimtParams P = params_at(params, H, K);
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t nth = (size_t)gridDim.x * blockDim.x;
  if (tid == 0) { ctrl->err = kErrNone; ctrl->err_site = 0; }
  const size_t nkd = (size_t)H * K * kD;
  for (size_t i = tid; i < nkd; i += nth) {
    const int j = (int)(i % kD);
    const int k = (int)((i / kD) % K);
    const int h = (int)(i / ((size_t)kD * K));
    const size_t o = ((size_t)h * kD + j) * K + k;
    P.mu_t[o] = mu[i];
    P.w_t[o] = 1.0f / sigma2[i];
  }
  // c_k: one warp per component, two dims per lane, then a warp sum (coalesced, no serial chain)
  const int lane = threadIdx.x & 31;
  const size_t warp_id = tid >> 5, nwarps = nth >> 5;
  for (size_t i = warp_id; i < (size_t)H * K; i += nwarps) {
    float s = logf(sigma2[i * kD + lane]) + logf(sigma2[i * kD + 32 + lane]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) P.c[i] = log_pi[i] - 0.5f * s;
  }
  for (size_t i = tid; i < zero_n; i += nth) zero[i] = 0.f;
}

// Loads `n` valid rows (of 64) starting at row `r0` of a [rows][64] matrix into smem as float32;
// rows past `n` are zero.
template <typename IO>
__device__ __forceinline__ void load_rows(const IO* __restrict__ src, int r0, int n, float* dst) {
  for (int i = threadIdx.x; i < T * kD; i += blockDim.x) {
    const int r = i / kD;
    dst[i] = r < n ? ld_io<IO>(src + (size_t)(r0 + r) * kD + (i % kD)) : 0.f;
  }
}

// Responsibilities of the T rows in xs (first `nvalid` valid) into G[T][K]; invalid rows are zero.
__device__ void gamma_tile(const float* xs, int nvalid, const SimtParams& P, int h, int K, float* G) {
  const float* mu_t = P.mu_t + (size_t)h * kD * K;
  const float* w_t = P.w_t + (size_t)h * kD * K;
  const float* c = P.c + (size_t)h * K;
  for (int p = threadIdx.x; p < K * (T / 8); p += blockDim.x) {
    const int k = p % K, tg = p / K;
    float acc[8];
#pragma unroll
    for (int ii = 0; ii < 8; ++ii) acc[ii] = 0.f;
    for (int j = 0; j < kD; ++j) {
      const float m = __ldg(mu_t + (size_t)j * K + k);
      const float w = __ldg(w_t + (size_t)j * K + k);
#pragma unroll
      for (int ii = 0; ii < 8; ++ii) {
        const float diff = xs[(tg * 8 + ii) * kD + j] - m;
        acc[ii] = fmaf(diff * w, diff, acc[ii]);
      }
    }
    const float ck = __ldg(c + k);
#pragma unroll
    for (int ii = 0; ii < 8; ++ii) G[(tg * 8 + ii) * K + k] = ck - 0.5f * acc[ii];
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  for (int i = warp; i < T; i += nwarps) {
    float* row = G + i * K;
    if (i >= nvalid) {
      for (int k = lane; k < K; k += 32) row[k] = 0.f;
      continue;
    }
    float m = -INFINITY;
    for (int k = lane; k < K; k += 32) m = fmaxf(m, row[k]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = 0.f;
    for (int k = lane; k < K; k += 32) {
      const float e = expf(row[k] - m);
      row[k] = e;
      s += e;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float inv = 1.0f / s;
    for (int k = lane; k < K; k += 32) row[k] *= inv;
  }
  __syncthreads();
}

// sacc[(k, c)] += sum_i G[i][k] * [v_i | 1]_c over one tile; each pair is owned by one thread.
__device__ __forceinline__ void accumulate_state(const float* G, const float* vs, int K, float* sacc) {
  const int npairs = K * kStateCols;
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
    const int k = p / kStateCols, c = p % kStateCols;
    float s = 0.f;
    if (c < kDv) {
      for (int i = 0; i < T; ++i) s = fmaf(G[i * K + k], vs[i * kDv + c], s);
    } else {
      for (int i = 0; i < T; ++i) s += G[i * K + k];
    }
    sacc[p] += s;
  }
}

// ---------------------------------------------------------------------------------------------
// Responsibilities export: grid (tiles, B*H).
template <typename IO>
__global__ void __launch_bounds__(kThreads) simt_resp_kernel(const IO* __restrict__ X, float* params, int H, int N,
                                                             int K, float* __restrict__ gamma) {
  extern __shared__ float sm[];
  float* xs = sm;
  float* G = xs + T * kD;
  const int unit = blockIdx.y, h = unit % H;
  const int t0 = blockIdx.x * T;
  const int nvalid = min(T, N - t0);
  const SimtParams P = params_at(params, H, K);
  load_rows<IO>(X + (size_t)unit * N * kD, t0, nvalid, xs);
  __syncthreads();
  gamma_tile(xs, nvalid, P, h, K, G);
  float* out = gamma + ((size_t)unit * N + t0) * K;
  for (int i = threadIdx.x; i < nvalid * K; i += blockDim.x) out[i] = G[i];
}

// Write phase (bidirectional) or segment aggregate (causal): grid (splits, B*H).  Each CTA covers
// tiles [split * seg_tiles, ...) of its (b,h).  atomic != 0: add into state[unit][K][65];
// atomic == 0: store into state[unit][split][K][65].
template <typename IO>
__global__ void __launch_bounds__(kThreads) simt_write_kernel(const IO* __restrict__ Kx, const IO* __restrict__ V,
                                                              float* params, int H, int N, int K, int seg_tiles,
                                                              int splits, float* state, int atomic) {
  extern __shared__ float sm[];
  float* xs = sm;
  float* vs = xs + T * kD;
  float* G = vs + T * kDv;
  float* sacc = G + T * K;  // [K][65] partial state of this CTA
  const int unit = blockIdx.y, h = unit % H, split = blockIdx.x;
  const SimtParams P = params_at(params, H, K);
  const int npairs = K * kStateCols;
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) sacc[p] = 0.f;
  const int tiles = (N + T - 1) / T;
  const int tb = split * seg_tiles, te = min(tiles, tb + seg_tiles);
  for (int t = tb; t < te; ++t) {
    const int t0 = t * T, nvalid = min(T, N - t0);
    load_rows<IO>(Kx + (size_t)unit * N * kD, t0, nvalid, xs);
    load_rows<IO>(V + (size_t)unit * N * kDv, t0, nvalid, vs);
    __syncthreads();
    gamma_tile(xs, nvalid, P, h, K, G);
    accumulate_state(G, vs, K, sacc);
    __syncthreads();
  }
  float* dst = atomic ? state + (size_t)unit * npairs : state + ((size_t)unit * splits + split) * npairs;
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
    if (atomic) atomicAdd(dst + p, sacc[p]); else dst[p] = sacc[p];
  }
}

// Read phase (bidirectional): grid (tiles, B*H).
template <typename IO>
__global__ void __launch_bounds__(kThreads) simt_read_kernel(const IO* __restrict__ Q, float* params, int H, int N,
                                                             int K, const float* __restrict__ state, float eps,
                                                             IO* __restrict__ O) {
  extern __shared__ float sm[];
  float* xs = sm;
  float* G = xs + T * kD;
  float* num = G + T * K;
  const int unit = blockIdx.y, h = unit % H;
  const int t0 = blockIdx.x * T, nvalid = min(T, N - t0);
  const SimtParams P = params_at(params, H, K);
  load_rows<IO>(Q + (size_t)unit * N * kD, t0, nvalid, xs);
  __syncthreads();
  gamma_tile(xs, nvalid, P, h, K, G);
  const float* S = state + (size_t)unit * K * kStateCols;
  for (int p = threadIdx.x; p < T * kStateCols; p += blockDim.x) {
    const int i = p / kStateCols, c = p % kStateCols;
    float s = 0.f;
    for (int k = 0; k < K; ++k) s = fmaf(G[i * K + k], __ldg(S + k * kStateCols + c), s);
    num[p] = s;
  }
  __syncthreads();
  IO* out = O + ((size_t)unit * N + t0) * kDv;
  for (int p = threadIdx.x; p < nvalid * kDv; p += blockDim.x) {
    const int i = p / kDv, c = p % kDv;
    st_io<IO>(out + p, num[i * kStateCols + c] / (num[i * kStateCols + kDv] + eps));
  }
}

// Exclusive scan over segments: agg[unit][p][e] <- sum_{p' < p} agg[unit][p'][e].  grid (ceil(K*65/256), B*H).
__global__ void simt_scan_kernel(float* agg, int P, int npairs) {
  const int unit = blockIdx.y;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= npairs) return;
  float* base = agg + (size_t)unit * P * npairs + e;
  float run = 0.f;
  for (int p = 0; p < P; ++p) {
    const float t = base[(size_t)p * npairs];
    base[(size_t)p * npairs] = run;
    run += t;
  }
}

// Causal sweep: grid (segments, B*H).  Starts from the exclusive prefix state of its segment and walks
// the segment tile by tile: O_i = [gQ_i . S + sum_{j in tile, j <= i} (gQ_i . gK_j) [v_j|1]] normalised,
// then S += Gamma_K(tile)^T [V|1].
template <typename IO>
__global__ void __launch_bounds__(kThreads) simt_causal_kernel(const IO* __restrict__ Q, const IO* __restrict__ Kx,
                                                               const IO* __restrict__ V, float* params, int H, int N,
                                                               int K, int seg_tiles, int P, const float* agg,
                                                               float eps, IO* __restrict__ O) {
  extern __shared__ float sm[];
  const int npairs = K * kStateCols;
  float* S = sm;                 // [K][65]
  float* xs = S + npairs;        // [T][64]
  float* vs = xs + T * kD;       // [T][64]
  float* GQ = vs + T * kDv;      // [T][K]
  float* GK = GQ + T * K;        // [T][K]
  float* A = GK + T * K;         // [T][T]
  float* num = A + T * T;        // [T][65]
  const int unit = blockIdx.y, h = unit % H, seg = blockIdx.x;
  const SimtParams Pp = params_at(params, H, K);
  const float* S0 = agg + ((size_t)unit * P + seg) * npairs;
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) S[p] = S0[p];
  const int tiles = (N + T - 1) / T;
  const int tb = seg * seg_tiles, te = min(tiles, tb + seg_tiles);
  for (int t = tb; t < te; ++t) {
    const int t0 = t * T, nvalid = min(T, N - t0);
    __syncthreads();
    load_rows<IO>(Q + (size_t)unit * N * kD, t0, nvalid, xs);
    __syncthreads();
    gamma_tile(xs, nvalid, Pp, h, K, GQ);
    load_rows<IO>(Kx + (size_t)unit * N * kD, t0, nvalid, xs);
    load_rows<IO>(V + (size_t)unit * N * kDv, t0, nvalid, vs);
    __syncthreads();
    gamma_tile(xs, nvalid, Pp, h, K, GK);
    // masked intra-tile affinity, j <= i inclusive
    for (int p = threadIdx.x; p < T * T; p += blockDim.x) {
      const int i = p / T, j = p % T;
      float s = 0.f;
      if (j <= i)
        for (int k = 0; k < K; ++k) s = fmaf(GQ[i * K + k], GK[j * K + k], s);
      A[p] = s;
    }
    __syncthreads();
    for (int p = threadIdx.x; p < T * kStateCols; p += blockDim.x) {
      const int i = p / kStateCols, c = p % kStateCols;
      float s = 0.f;
      for (int k = 0; k < K; ++k) s = fmaf(GQ[i * K + k], S[k * kStateCols + c], s);
      if (c < kDv) {
        for (int j = 0; j <= i; ++j) s = fmaf(A[i * T + j], vs[j * kDv + c], s);
      } else {
        for (int j = 0; j <= i; ++j) s += A[i * T + j];
      }
      num[p] = s;
    }
    __syncthreads();
    IO* out = O + ((size_t)unit * N + t0) * kDv;
    for (int p = threadIdx.x; p < nvalid * kDv; p += blockDim.x) {
      const int i = p / kDv, c = p % kDv;
      st_io<IO>(out + p, num[i * kStateCols + c] / (num[i * kStateCols + kDv] + eps));
    }
    for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
      const int k = p / kStateCols, c = p % kStateCols;
      float s = 0.f;
      if (c < kDv) {
        for (int j = 0; j < T; ++j) s = fmaf(GK[j * K + k], vs[j * kDv + c], s);
      } else {
        for (int j = 0; j < T; ++j) s += GK[j * K + k];
      }
      S[p] += s;
    }
  }
}

// ----------------------------------------------------------------------------------------------- backward
// Gradients of the bidirectional forward ("Variants and training" item 3: the mixture is learned end to
// end by backpropagation), float32 on the CUDA cores.  With Vt, Z from the forward write and G = dL/dO:
//   den_i = gamma_Qi . Z + eps, O_i = gamma_Qi . Vt / den_i, dn_i = G_i / den_i, dden_i = -(G_i . O_i) / den_i,
//   dgamma_Qi = [Vt | Z] [dn_i | dden_i],   [dVt | dZ] = sum_i gamma_Qi [dn_i | dden_i]^T,
//   dgamma_Kj = [dVt | dZ] [v_j | 1],       dv_j = dVt^T gamma_Kj,
//   dl = gamma * (dgamma - gamma . dgamma)  (softmax),
//   dx_d = sum_k dl_k (mu_kd - x_d) / sigma2_kd,  and per head, over every query and key row:
//   D1_kd = sum dl_k (x_d - mu_kd), D2_kd = sum dl_k (x_d - mu_kd)^2, b_k = sum dl_k,
//   dmu = D1 / sigma2,  dsigma2 = (D2 / sigma2 - b) / (2 sigma2),  dlog_pi = b.
// The per-row dl of both sides go through the workspace to the parameter-gradient pass.

// dx for the T rows of xs from dl [T][K]: sum_k dl_ik w_kd (mu_kd - x_id) = (dl (w mu))_id - x_id (dl w)_id.
// Thread (column j, row group) walks k reading mu[h][k][j] and sigma2[h][k][j] (consecutive j across a
// warp: coalesced) and updates its T / 4 rows.
template <typename IO>
__device__ void dx_tile(const float* xs, const float* dl, int nvalid, const float* __restrict__ mu,
                        const float* __restrict__ sigma2, int h, int K, IO* dst) {
  constexpr int kRowGroups = kThreads / kD;  // 4
  constexpr int kRows = T / kRowGroups;      // 8 rows per thread
  const int j = threadIdx.x % kD, rg = threadIdx.x / kD;
  const float* muh = mu + (size_t)h * K * kD + j;
  const float* s2h = sigma2 + (size_t)h * K * kD + j;
  float a1[kRows], a2[kRows];
#pragma unroll
  for (int r = 0; r < kRows; ++r) a1[r] = a2[r] = 0.f;
  for (int k = 0; k < K; ++k) {
    const float w = 1.0f / __ldg(s2h + (size_t)k * kD), wm = w * __ldg(muh + (size_t)k * kD);
#pragma unroll
    for (int r = 0; r < kRows; ++r) {
      const float d = dl[(rg * kRows + r) * K + k];
      a1[r] = fmaf(d, wm, a1[r]);
      a2[r] = fmaf(d, w, a2[r]);
    }
  }
#pragma unroll
  for (int r = 0; r < kRows; ++r) {
    const int i = rg * kRows + r;
    if (i < nvalid) st_io<IO>(dst + (size_t)i * kD + j, a1[r] - xs[i * kD + j] * a2[r]);
  }
}

// Softmax backward in place: dG <- G * (dG - G . dG), one warp per row.
__device__ void softmax_backward_tile(const float* G, float* dG, int K) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  for (int i = warp; i < T; i += nwarps) {
    float dot = 0.f;
    for (int k = lane; k < K; k += 32) dot = fmaf(G[i * K + k], dG[i * K + k], dot);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
    for (int k = lane; k < K; k += 32) dG[i * K + k] = G[i * K + k] * (dG[i * K + k] - dot);
  }
  __syncthreads();
}

// Query side: grid (splits, B*H).  Recomputes O, pushes dO back through the read, writes dQ and dl_Q,
// and adds [dVt | dZ] into dstate[unit][K][65].
template <typename IO>
__global__ void __launch_bounds__(kThreads) simt_bwd_query_kernel(const IO* __restrict__ Q, const IO* __restrict__ dO,
                                                                  float* params, const float* __restrict__ mu,
                                                                  const float* __restrict__ sigma2, int H, int N, int K,
                                                                  int seg_tiles,
                                                                  const float* __restrict__ state, float eps,
                                                                  float* dstate, float* dlq, IO* __restrict__ dQ) {
  extern __shared__ float sm[];
  const int npairs = K * kStateCols;
  float* S = sm;                // [K][65]  Vt | Z
  float* sacc = S + npairs;     // [K][65]  dVt | dZ of this CTA
  float* xs = sacc + npairs;    // [T][64]
  float* gs = xs + T * kD;      // [T][64]  dO rows
  float* dn = gs + T * kDv;     // [T][65]  numerators, then dn | dden
  float* G = dn + T * kStateCols;  // [T][K]
  float* dG = G + T * K;        // [T][K]
  const int unit = blockIdx.y, h = unit % H, split = blockIdx.x;
  const SimtParams P = params_at(params, H, K);
  const float* S0 = state + (size_t)unit * npairs;
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
    S[p] = S0[p];
    sacc[p] = 0.f;
  }
  const int tiles = (N + T - 1) / T;
  const int tb = split * seg_tiles, te = min(tiles, tb + seg_tiles);
  for (int t = tb; t < te; ++t) {
    const int t0 = t * T, nvalid = min(T, N - t0);
    __syncthreads();
    load_rows<IO>(Q + (size_t)unit * N * kD, t0, nvalid, xs);
    load_rows<IO>(dO + (size_t)unit * N * kDv, t0, nvalid, gs);
    __syncthreads();
    gamma_tile(xs, nvalid, P, h, K, G);
    for (int p = threadIdx.x; p < T * kStateCols; p += blockDim.x) {  // [num | den - eps]
      const int i = p / kStateCols, c = p % kStateCols;
      float s = 0.f;
      for (int k = 0; k < K; ++k) s = fmaf(G[i * K + k], S[k * kStateCols + c], s);
      dn[p] = s;
    }
    __syncthreads();
    {  // one warp per row: O, G . O, then dn | dden (rows past N have G = 0, so all zero)
      const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
      for (int i = warp; i < T; i += nwarps) {
        if (i >= nvalid) {  // rows past N: no gradient (and no 0 / 0 when eps = 0)
          dn[i * kStateCols + lane] = 0.f;
          dn[i * kStateCols + 32 + lane] = 0.f;
          if (lane == 0) dn[i * kStateCols + kDv] = 0.f;
          continue;
        }
        const float den = dn[i * kStateCols + kDv] + eps;
        const float o0 = dn[i * kStateCols + lane] / den, o1 = dn[i * kStateCols + 32 + lane] / den;
        float go = gs[i * kDv + lane] * o0 + gs[i * kDv + 32 + lane] * o1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) go += __shfl_xor_sync(0xffffffffu, go, o);
        __syncwarp();
        dn[i * kStateCols + lane] = gs[i * kDv + lane] / den;
        dn[i * kStateCols + 32 + lane] = gs[i * kDv + 32 + lane] / den;
        if (lane == 0) dn[i * kStateCols + kDv] = -go / den;
      }
    }
    __syncthreads();
    for (int p = threadIdx.x; p < T * K; p += blockDim.x) {  // dgamma_Q = [Vt | Z] [dn | dden]
      const int i = p / K, k = p % K;
      float s = 0.f;
      for (int c = 0; c < kStateCols; ++c) s = fmaf(dn[i * kStateCols + c], S[k * kStateCols + c], s);
      dG[p] = s;
    }
    for (int p = threadIdx.x; p < npairs; p += blockDim.x) {  // [dVt | dZ] += gamma_Q^T [dn | dden]
      const int k = p / kStateCols, c = p % kStateCols;
      float s = 0.f;
      for (int i = 0; i < T; ++i) s = fmaf(G[i * K + k], dn[i * kStateCols + c], s);
      sacc[p] += s;
    }
    __syncthreads();
    softmax_backward_tile(G, dG, K);
    float* dst = dlq + ((size_t)unit * N + t0) * K;
    for (int p = threadIdx.x; p < nvalid * K; p += blockDim.x) dst[p] = dG[p];
    dx_tile<IO>(xs, dG, nvalid, mu, sigma2, h, K, dQ + ((size_t)unit * N + t0) * kD);
  }
  __syncthreads();
  float* dS = dstate + (size_t)unit * npairs;
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) atomicAdd(dS + p, sacc[p]);
}

// Key side: grid (tiles, B*H).  Pushes [dVt | dZ] back through the write: dV, dK and dl_K.
template <typename IO>
__global__ void __launch_bounds__(kThreads) simt_bwd_key_kernel(const IO* __restrict__ Kx, const IO* __restrict__ V,
                                                                float* params, const float* __restrict__ mu,
                                                                const float* __restrict__ sigma2, int H, int N, int K,
                                                                const float* __restrict__ dstate, float* dlk,
                                                                IO* __restrict__ dK, IO* __restrict__ dV) {
  extern __shared__ float sm[];
  const int npairs = K * kStateCols;
  float* dS = sm;               // [K][65]  dVt | dZ
  float* xs = dS + npairs;      // [T][64]
  float* vs = xs + T * kD;      // [T][64]
  float* G = vs + T * kDv;      // [T][K]
  float* dG = G + T * K;        // [T][K]
  const int unit = blockIdx.y, h = unit % H;
  const int t0 = blockIdx.x * T, nvalid = min(T, N - t0);
  const SimtParams P = params_at(params, H, K);
  const float* dS0 = dstate + (size_t)unit * npairs;
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) dS[p] = dS0[p];
  load_rows<IO>(Kx + (size_t)unit * N * kD, t0, nvalid, xs);
  load_rows<IO>(V + (size_t)unit * N * kDv, t0, nvalid, vs);
  __syncthreads();
  gamma_tile(xs, nvalid, P, h, K, G);
  for (int p = threadIdx.x; p < T * K; p += blockDim.x) {  // dgamma_K = [dVt | dZ] [v | 1]
    const int j = p / K, k = p % K;
    float s = dS[k * kStateCols + kDv];
    for (int c = 0; c < kDv; ++c) s = fmaf(vs[j * kDv + c], dS[k * kStateCols + c], s);
    dG[p] = s;
  }
  IO* dv_out = dV + ((size_t)unit * N + t0) * kDv;
  for (int p = threadIdx.x; p < nvalid * kDv; p += blockDim.x) {  // dv = dVt^T gamma_K
    const int j = p / kDv, c = p % kDv;
    float s = 0.f;
    for (int k = 0; k < K; ++k) s = fmaf(G[j * K + k], dS[k * kStateCols + c], s);
    st_io<IO>(dv_out + p, s);
  }
  __syncthreads();
  softmax_backward_tile(G, dG, K);
  float* dst = dlk + ((size_t)unit * N + t0) * K;
  for (int p = threadIdx.x; p < nvalid * K; p += blockDim.x) dst[p] = dG[p];
  dx_tile<IO>(xs, dG, nvalid, mu, sigma2, h, K, dK + ((size_t)unit * N + t0) * kD);
}

// ---- causal backward.  S_i = sum_{j <= i} gamma_Kj [v_j | 1] (running state), u_i = [G_i / den_i |
// -(G_i . O_i) / den_i], R_j = sum_{i >= j} gamma_Qi u_i^T (suffix sum of the queries' contributions):
//   dgamma_Qi = S_i u_i,   dgamma_Kj = R_j [v_j | 1],   dv_j = R_j[:, :dv]^T gamma_Kj.
// Chunked like the forward: segment aggregates and an exclusive scan give S at each segment start; the
// query pass walks its segment forward (intra-tile terms masked to j <= i) and leaves the segment's
// aggregate of gamma_Q u^T; an exclusive suffix scan gives R after each segment; the key pass walks its
// segment backward.

// Masked tile products for the causal backward: A_ij = gQ_i . gK_j and W_ij = u_i . [v_j | 1] for j <= i.
__device__ void causal_tile_products(const float* GQ, const float* GK, const float* us, const float* vs, int K,
                                     float* A, float* W) {
  for (int p = threadIdx.x; p < T * T; p += blockDim.x) {
    const int i = p / T, j = p % T;
    float a = 0.f, w = 0.f;
    if (j <= i) {
      for (int k = 0; k < K; ++k) a = fmaf(GQ[i * K + k], GK[j * K + k], a);
      w = us[i * kStateCols + kDv];
      for (int c = 0; c < kDv; ++c) w = fmaf(us[i * kStateCols + c], vs[j * kDv + c], w);
    }
    A[p] = a;
    W[p] = w;
  }
}

// Query side: grid (segments, B*H).  S starts at agg[unit][seg] (scanned); writes u, dl_Q, dQ and the
// segment aggregate sum_i gamma_Qi u_i^T into bagg[unit][seg].
template <typename IO>
__global__ void __launch_bounds__(kThreads) simt_bwd_causal_query_kernel(
    const IO* __restrict__ Q, const IO* __restrict__ Kx, const IO* __restrict__ V, const IO* __restrict__ dO,
    float* params, const float* __restrict__ mu, const float* __restrict__ sigma2, int H, int N, int K, int seg_tiles,
    int P, const float* agg, float eps, float* bagg, float* uglob, float* dlq, IO* __restrict__ dQ) {
  extern __shared__ float sm[];
  const int npairs = K * kStateCols;
  float* S = sm;                   // [K][65]
  float* xs = S + npairs;          // [T][64]  queries, then keys
  float* vs = xs + T * kD;         // [T][64]
  float* gs = vs + T * kDv;        // [T][64]  dO rows
  float* us = gs + T * kDv;        // [T][65]  numerators, then u
  float* GQ = us + T * kStateCols;  // [T][K]
  float* GK = GQ + T * K;          // [T][K]
  float* dG = GK + T * K;          // [T][K]
  float* A = dG + T * K;           // [T][T]
  float* W = A + T * T;            // [T][T]
  __shared__ float xq[T * kD];     // the query rows, kept for dQ
  const int unit = blockIdx.y, h = unit % H, seg = blockIdx.x;
  const SimtParams Pp = params_at(params, H, K);
  const float* S0 = agg + ((size_t)unit * P + seg) * npairs;
  float* bout = bagg + ((size_t)unit * P + seg) * npairs;
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) {
    S[p] = S0[p];
    bout[p] = 0.f;
  }
  const int tiles = (N + T - 1) / T;
  const int tb = seg * seg_tiles, te = min(tiles, tb + seg_tiles);
  for (int t = tb; t < te; ++t) {
    const int t0 = t * T, nvalid = min(T, N - t0);
    __syncthreads();
    load_rows<IO>(Q + (size_t)unit * N * kD, t0, nvalid, xq);
    load_rows<IO>(dO + (size_t)unit * N * kDv, t0, nvalid, gs);
    __syncthreads();
    gamma_tile(xq, nvalid, Pp, h, K, GQ);
    load_rows<IO>(Kx + (size_t)unit * N * kD, t0, nvalid, xs);
    load_rows<IO>(V + (size_t)unit * N * kDv, t0, nvalid, vs);
    __syncthreads();
    gamma_tile(xs, nvalid, Pp, h, K, GK);
    // numerators [num | den - eps] of the causal output: gQ_i . S + sum_{j <= i} A_ij [v_j | 1]
    for (int p = threadIdx.x; p < T * T; p += blockDim.x) {
      const int i = p / T, j = p % T;
      float a = 0.f;
      if (j <= i)
        for (int k = 0; k < K; ++k) a = fmaf(GQ[i * K + k], GK[j * K + k], a);
      A[p] = a;
    }
    __syncthreads();
    for (int p = threadIdx.x; p < T * kStateCols; p += blockDim.x) {
      const int i = p / kStateCols, c = p % kStateCols;
      float s = 0.f;
      for (int k = 0; k < K; ++k) s = fmaf(GQ[i * K + k], S[k * kStateCols + c], s);
      if (c < kDv) {
        for (int j = 0; j <= i; ++j) s = fmaf(A[i * T + j], vs[j * kDv + c], s);
      } else {
        for (int j = 0; j <= i; ++j) s += A[i * T + j];
      }
      us[p] = s;
    }
    __syncthreads();
    {  // one warp per row: O, G . O, then u (rows past N: zero)
      const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
      for (int i = warp; i < T; i += nwarps) {
        float* ui = us + i * kStateCols;
        if (i >= nvalid) {
          ui[lane] = 0.f;
          ui[32 + lane] = 0.f;
          if (lane == 0) ui[kDv] = 0.f;
          continue;
        }
        const float den = ui[kDv] + eps;
        const float o0 = ui[lane] / den, o1 = ui[32 + lane] / den;
        float go = gs[i * kDv + lane] * o0 + gs[i * kDv + 32 + lane] * o1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) go += __shfl_xor_sync(0xffffffffu, go, o);
        __syncwarp();
        ui[lane] = gs[i * kDv + lane] / den;
        ui[32 + lane] = gs[i * kDv + 32 + lane] / den;
        if (lane == 0) ui[kDv] = -go / den;
      }
    }
    __syncthreads();
    float* ug = uglob + ((size_t)unit * N + t0) * kStateCols;
    for (int p = threadIdx.x; p < nvalid * kStateCols; p += blockDim.x) ug[p] = us[p];
    causal_tile_products(GQ, GK, us, vs, K, A, W);
    __syncthreads();
    for (int p = threadIdx.x; p < T * K; p += blockDim.x) {  // dgamma_Q = S u + sum_{j <= i} W_ij gK_j
      const int i = p / K, k = p % K;
      float s = 0.f;
      for (int c = 0; c < kStateCols; ++c) s = fmaf(S[k * kStateCols + c], us[i * kStateCols + c], s);
      for (int j = 0; j <= i; ++j) s = fmaf(W[i * T + j], GK[j * K + k], s);
      dG[p] = s;
    }
    __syncthreads();
    for (int p = threadIdx.x; p < npairs; p += blockDim.x) {  // segment aggregate and the running state
      const int k = p / kStateCols, c = p % kStateCols;
      float b = 0.f, a = 0.f;
      for (int i = 0; i < T; ++i) b = fmaf(GQ[i * K + k], us[i * kStateCols + c], b);
      if (c < kDv) {
        for (int j = 0; j < T; ++j) a = fmaf(GK[j * K + k], vs[j * kDv + c], a);
      } else {
        for (int j = 0; j < T; ++j) a += GK[j * K + k];
      }
      bout[p] += b;
      S[p] += a;
    }
    __syncthreads();
    softmax_backward_tile(GQ, dG, K);
    float* dst = dlq + ((size_t)unit * N + t0) * K;
    for (int p = threadIdx.x; p < nvalid * K; p += blockDim.x) dst[p] = dG[p];
    dx_tile<IO>(xq, dG, nvalid, mu, sigma2, h, K, dQ + ((size_t)unit * N + t0) * kD);
  }
}

// Exclusive suffix scan over segments: bagg[unit][p][e] <- sum_{p' > p} bagg[unit][p'][e].
__global__ void simt_rscan_kernel(float* bagg, int P, int npairs) {
  const int unit = blockIdx.y;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= npairs) return;
  float* base = bagg + (size_t)unit * P * npairs + e;
  float run = 0.f;
  for (int p = P - 1; p >= 0; --p) {
    const float t = base[(size_t)p * npairs];
    base[(size_t)p * npairs] = run;
    run += t;
  }
}

// Key side: grid (segments, B*H).  R starts at bagg[unit][seg] (suffix-scanned) and the segment's tiles are
// walked last to first; writes dl_K, dK and dV.
template <typename IO>
__global__ void __launch_bounds__(kThreads) simt_bwd_causal_key_kernel(
    const IO* __restrict__ Q, const IO* __restrict__ Kx, const IO* __restrict__ V, float* params,
    const float* __restrict__ mu, const float* __restrict__ sigma2, int H, int N, int K, int seg_tiles, int P,
    const float* bagg, const float* uglob, float* dlk, IO* __restrict__ dK, IO* __restrict__ dV) {
  extern __shared__ float sm[];
  const int npairs = K * kStateCols;
  float* R = sm;                   // [K][65]
  float* xs = R + npairs;          // [T][64]  queries, then keys
  float* vs = xs + T * kD;         // [T][64]
  float* us = vs + T * kDv;        // [T][65]
  float* GQ = us + T * kStateCols;  // [T][K]
  float* GK = GQ + T * K;          // [T][K]
  float* dG = GK + T * K;          // [T][K]
  float* A = dG + T * K;           // [T][T]
  float* W = A + T * T;            // [T][T]
  const int unit = blockIdx.y, h = unit % H, seg = blockIdx.x;
  const SimtParams Pp = params_at(params, H, K);
  const float* R0 = bagg + ((size_t)unit * P + seg) * npairs;
  for (int p = threadIdx.x; p < npairs; p += blockDim.x) R[p] = R0[p];
  const int tiles = (N + T - 1) / T;
  const int tb = seg * seg_tiles, te = min(tiles, tb + seg_tiles);
  for (int t = te - 1; t >= tb; --t) {
    const int t0 = t * T, nvalid = min(T, N - t0);
    __syncthreads();
    load_rows<IO>(Q + (size_t)unit * N * kD, t0, nvalid, xs);
    for (int p = threadIdx.x; p < T * kStateCols; p += blockDim.x)
      us[p] = p < nvalid * kStateCols ? uglob[((size_t)unit * N + t0) * kStateCols + p] : 0.f;
    __syncthreads();
    gamma_tile(xs, nvalid, Pp, h, K, GQ);
    load_rows<IO>(Kx + (size_t)unit * N * kD, t0, nvalid, xs);
    load_rows<IO>(V + (size_t)unit * N * kDv, t0, nvalid, vs);
    __syncthreads();
    gamma_tile(xs, nvalid, Pp, h, K, GK);
    causal_tile_products(GQ, GK, us, vs, K, A, W);
    __syncthreads();
    for (int p = threadIdx.x; p < T * K; p += blockDim.x) {  // dgamma_K = R [v | 1] + sum_{i >= j} W_ij gQ_i
      const int j = p / K, k = p % K;
      float s = R[k * kStateCols + kDv];
      for (int c = 0; c < kDv; ++c) s = fmaf(R[k * kStateCols + c], vs[j * kDv + c], s);
      for (int i = j; i < T; ++i) s = fmaf(W[i * T + j], GQ[i * K + k], s);
      dG[p] = s;
    }
    IO* dv_out = dV + ((size_t)unit * N + t0) * kDv;
    for (int p = threadIdx.x; p < nvalid * kDv; p += blockDim.x) {  // dv = R^T gK + sum_{i >= j} A_ij dn_i
      const int j = p / kDv, c = p % kDv;
      float s = 0.f;
      for (int k = 0; k < K; ++k) s = fmaf(GK[j * K + k], R[k * kStateCols + c], s);
      for (int i = j; i < T; ++i) s = fmaf(A[i * T + j], us[i * kStateCols + c], s);
      st_io<IO>(dv_out + p, s);
    }
    __syncthreads();
    for (int p = threadIdx.x; p < npairs; p += blockDim.x) {  // R += gamma_Q^T u over the whole tile
      const int k = p / kStateCols, c = p % kStateCols;
      float b = 0.f;
      for (int i = 0; i < T; ++i) b = fmaf(GQ[i * K + k], us[i * kStateCols + c], b);
      R[p] += b;
    }
    __syncthreads();
    softmax_backward_tile(GK, dG, K);
    float* dst = dlk + ((size_t)unit * N + t0) * K;
    for (int p = threadIdx.x; p < nvalid * K; p += blockDim.x) dst[p] = dG[p];
    dx_tile<IO>(xs, dG, nvalid, mu, sigma2, h, K, dK + ((size_t)unit * N + t0) * kD);
  }
}

// Parameter-gradient sums: grid (ceil(K / 32), H, chunks).  Thread (k within a block of 32, group of 8
// dims) sums dl_k (x_d - mu_kd) and dl_k (x_d - mu_kd)^2 over its chunk of the head's rows (queries
// then keys of every batch entry) and adds them into pacc[h][k][d][2] (and b_k into pb[h][k]).
template <typename IO>
__global__ void __launch_bounds__(kThreads) simt_bwd_param_kernel(const IO* __restrict__ Q, const IO* __restrict__ Kx,
                                                                  const float* __restrict__ mu, const float* dlq,
                                                                  const float* dlk, int B, int H, int N, int K,
                                                                  int rows_per_chunk, float* pacc, float* pb) {
  __shared__ float xs[T * kD];
  __shared__ float ds[T * 32];
  const int h = blockIdx.y, k0 = blockIdx.x * 32;
  const int kl = threadIdx.x & 31, dg = threadIdx.x >> 5;  // 8 groups of 8 dims
  const int k = k0 + kl;
  float m[8], a1[8], a2[8], bsum = 0.f;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    m[q] = k < K ? __ldg(mu + ((size_t)h * K + k) * kD + dg * 8 + q) : 0.f;
    a1[q] = 0.f;
    a2[q] = 0.f;
  }
  const long long total = 2LL * B * N;  // rows of this head: queries then keys, batch-major
  const long long r0 = (long long)blockIdx.z * rows_per_chunk, r1 = min(total, r0 + rows_per_chunk);
  for (long long rb = r0; rb < r1; rb += T) {
    const int n = (int)min((long long)T, r1 - rb);
    __syncthreads();
    for (int p = threadIdx.x; p < T * kD; p += blockDim.x) {
      const int i = p / kD, j = p % kD;
      float x = 0.f;
      if (i < n) {
        const long long r = rb + i, side = r / ((long long)B * N), rr = r % ((long long)B * N);
        const long long b = rr / N, tok = rr % N, unit = b * H + h;
        const IO* src = side == 0 ? Q : Kx;
        x = ld_io<IO>(src + ((size_t)unit * N + tok) * kD + j);
      }
      xs[p] = x;
    }
    for (int p = threadIdx.x; p < T * 32; p += blockDim.x) {
      const int i = p / 32, kk = k0 + (p % 32);
      float v = 0.f;
      if (i < n && kk < K) {
        const long long r = rb + i, side = r / ((long long)B * N), rr = r % ((long long)B * N);
        const long long b = rr / N, tok = rr % N, unit = b * H + h;
        const float* src = side == 0 ? dlq : dlk;
        v = src[((size_t)unit * N + tok) * K + kk];
      }
      ds[p] = v;
    }
    __syncthreads();
    for (int i = 0; i < n; ++i) {
      const float dl = ds[i * 32 + kl];
      if (dg == 0) bsum += dl;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const float diff = xs[i * kD + dg * 8 + q] - m[q];
        const float t = dl * diff;
        a1[q] += t;
        a2[q] = fmaf(t, diff, a2[q]);
      }
    }
  }
  if (k < K) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float* dst = pacc + (((size_t)h * K + k) * kD + dg * 8 + q) * 2;
      atomicAdd(dst, a1[q]);
      atomicAdd(dst + 1, a2[q]);
    }
    if (dg == 0) atomicAdd(pb + (size_t)h * K + k, bsum);
  }
}

__global__ void simt_bwd_param_finish_kernel(const float* __restrict__ sigma2, const float* pacc, const float* pb, int H,
                                             int K, float* dmu, float* dsigma2, float* dlog_pi) {
  const size_t n = (size_t)H * K * kD;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const float w = 1.0f / sigma2[i], b = pb[i / kD];
    dmu[i] = pacc[2 * i] * w;
    dsigma2[i] = 0.5f * w * (pacc[2 * i + 1] * w - b);
    if (i % kD == 0) dlog_pi[i / kD] = b;
  }
}

// ----------------------------------------------------------------------------------------------- decode
// Causal decode: the recurrent form of the prefix sums ("Variants and training" item 3).  One CTA per
// (b, h) holds that head's state S [K][dv + 1] and its parameters in shared memory and takes its T new
// tokens in order:
//   S_k += gamma_K(k_t)_k [v_t | 1],   o_t = gamma_Q(q_t) . S[:, :dv] / (gamma_Q(q_t) . S[:, dv] + eps),
// so token t sees every earlier key and itself (inclusive), exactly as the causal forward does.
// Thread k < K owns component k (log-density, state row); the read splits the 64 value columns over
// four groups of components.  float32 throughout; the state is read once and written back once, and
// the parameters are folded in the prologue (one launch per call).
constexpr int kDecodeThreads = 256;

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float u = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, u) : v + u;
  }
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float r = red[0];
  for (int w = 1; w < nw; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
  __syncthreads();  // red is reused by the next reduction
  return r;
}

// Shared-memory floats of the decode kernel for K components.
__host__ __device__ constexpr size_t decode_smem_floats(int K) {
  return (size_t)K * kStateCols + 2 * (size_t)kD * (K + 1) + 2 * (size_t)K + 2 * kD + kDv + 4 * kDv + 32;
}

template <typename IO>
__global__ void __launch_bounds__(kDecodeThreads) simt_decode_kernel(const IO* __restrict__ Q, const IO* __restrict__ Kx,
                                                                     const IO* __restrict__ V,
                                                                     const float* __restrict__ mu,
                                                                     const float* __restrict__ sigma2,
                                                                     const float* __restrict__ log_pi, int H, int Tn,
                                                                     int K, float* __restrict__ state, float eps,
                                                                     IO* __restrict__ out) {
  extern __shared__ float sm[];
  const int bh = blockIdx.x, h = bh % H, k = threadIdx.x;
  const int ld = K + 1;                     // row stride of the parameter tables (conflict-free both ways)
  float* S = sm;                            // [K][kStateCols]
  float* mu_s = S + (size_t)K * kStateCols;  // [kD][K + 1]
  float* w_s = mu_s + (size_t)kD * ld;       // [kD][K + 1]  1 / sigma2
  float* c_s = w_s + (size_t)kD * ld;        // [K]
  float* gq = c_s + K;                       // [K]
  float* xq = gq + K;                        // [kD]
  float* xk = xq + kD;                       // [kD]
  float* xv = xk + kD;                       // [kDv]
  float* part = xv + kDv;                    // [4][kDv]
  float* red = part + 4 * kDv;               // [32]
  float* st = state + (size_t)bh * K * kStateCols;
  const int n_state = K * kStateCols;
  // float4 copies when this head's state starts on a 16-byte boundary (K a multiple of 4), so that
  // many loads are in flight per thread; plain floats otherwise
  const bool vec = ((reinterpret_cast<uintptr_t>(st) | reinterpret_cast<uintptr_t>(S)) & 15) == 0 && (n_state & 3) == 0;
  if (vec) {
    // all of a thread's loads in flight before the first store (one round trip to memory)
    const int n4s = n_state / 4;
    for (int i0 = threadIdx.x; i0 < n4s; i0 += 16 * kDecodeThreads) {
      float4 x[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int i = i0 + u * kDecodeThreads;
        if (i < n4s) x[u] = __ldcg(reinterpret_cast<const float4*>(st) + i);
      }
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const int i = i0 + u * kDecodeThreads;
        if (i < n4s) reinterpret_cast<float4*>(S)[i] = x[u];
      }
    }
  } else {
#pragma unroll 8
    for (int i = threadIdx.x; i < n_state; i += blockDim.x) S[i] = __ldcg(st + i);
  }
  // parameters of head h, transposed to [dim][component], and c_k = log pi_k - 1/2 sum_d log sigma2_kd:
  // each thread takes 4 dims of one component per float4 pair; the 16 threads of a component (an
  // aligned half-warp) add their log-variances with shuffles.  The trip count is warp-uniform.
  const float4* mu4 = reinterpret_cast<const float4*>(mu + (size_t)h * K * kD);
  const float4* s24 = reinterpret_cast<const float4*>(sigma2 + (size_t)h * K * kD);
  const int n4 = K * (kD / 4);
  // eight float4 of each table in flight per thread; the trip count and the 16-thread component groups
  // (aligned half-warps: n4 and the block size are multiples of 16) are warp-uniform
  for (int i0 = threadIdx.x; i0 - (int)threadIdx.x < n4; i0 += 8 * kDecodeThreads) {
    float4 m[8], v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i4 = i0 + u * kDecodeThreads;
      if (i4 < n4) {
        m[u] = __ldg(mu4 + i4);
        v[u] = __ldg(s24 + i4);
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i4 = i0 + u * kDecodeThreads;
      const bool on = i4 < n4;
      const int kk = i4 >> 4, j0 = (i4 & 15) << 2;
      float lg = 0.f;
      if (on) {
        mu_s[(size_t)(j0 + 0) * ld + kk] = m[u].x;
        mu_s[(size_t)(j0 + 1) * ld + kk] = m[u].y;
        mu_s[(size_t)(j0 + 2) * ld + kk] = m[u].z;
        mu_s[(size_t)(j0 + 3) * ld + kk] = m[u].w;
        w_s[(size_t)(j0 + 0) * ld + kk] = 1.0f / v[u].x;
        w_s[(size_t)(j0 + 1) * ld + kk] = 1.0f / v[u].y;
        w_s[(size_t)(j0 + 2) * ld + kk] = 1.0f / v[u].z;
        w_s[(size_t)(j0 + 3) * ld + kk] = 1.0f / v[u].w;
        lg = (logf(v[u].x) + logf(v[u].y)) + (logf(v[u].z) + logf(v[u].w));
      }
      if (i0 - (int)threadIdx.x + u * kDecodeThreads < n4) {  // warp-uniform: the whole warp is on or off
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) lg += __shfl_xor_sync(0xffffffffu, lg, o);
      }
      if (on && (i4 & 15) == 0) c_s[kk] = __ldg(log_pi + (size_t)h * K + kk) - 0.5f * lg;
    }
  }
  __syncthreads();
  for (int t = 0; t < Tn; ++t) {
    const size_t row = (size_t)bh * Tn + t;
    if (threadIdx.x < kD) {
      xq[threadIdx.x] = ld_io<IO>(Q + row * kD + threadIdx.x);
      xk[threadIdx.x] = ld_io<IO>(Kx + row * kD + threadIdx.x);
      xv[threadIdx.x] = ld_io<IO>(V + row * kDv + threadIdx.x);
    }
    __syncthreads();
    // log-densities of the key and the query under component k (centered form)
    float lk = -INFINITY, lq = -INFINITY;
    if (k < K) {
      float ak = 0.f, aq = 0.f;
#pragma unroll 8
      for (int j = 0; j < kD; ++j) {
        const float m = mu_s[(size_t)j * ld + k], w = w_s[(size_t)j * ld + k];
        const float dk = xk[j] - m, dq = xq[j] - m;
        ak = fmaf(dk * w, dk, ak);
        aq = fmaf(dq * w, dq, aq);
      }
      lk = c_s[k] - 0.5f * ak;
      lq = c_s[k] - 0.5f * aq;
    }
    const float mk = block_reduce(lk, true, red), mq = block_reduce(lq, true, red);
    const float ek = k < K ? expf(lk - mk) : 0.f, eq = k < K ? expf(lq - mq) : 0.f;
    const float sk = block_reduce(ek, false, red), sq = block_reduce(eq, false, red);
    // state update (own row), then the query's responsibilities for the read
    if (k < K) {
      const float g = ek / sk;
      float* Sk = S + (size_t)k * kStateCols;
#pragma unroll 8
      for (int j = 0; j < kDv; ++j) Sk[j] = fmaf(g, xv[j], Sk[j]);
      Sk[kDv] += g;
      gq[k] = eq / sq;
    }
    __syncthreads();
    // read: numerator column j over component group g4, denominator over all components
    {
      const int j = threadIdx.x & (kDv - 1), g4 = threadIdx.x >> 6;
      const int k1 = min(K, g4 * 64 + 64);
      float acc = 0.f;
#pragma unroll 8
      for (int kk = g4 * 64; kk < k1; ++kk) acc = fmaf(gq[kk], S[(size_t)kk * kStateCols + j], acc);
      part[g4 * kDv + j] = acc;
    }
    const float den = block_reduce(k < K ? gq[k] * S[(size_t)k * kStateCols + kDv] : 0.f, false, red) + eps;
    if (threadIdx.x < kDv) {
      const float num = (part[threadIdx.x] + part[kDv + threadIdx.x]) + (part[2 * kDv + threadIdx.x] + part[3 * kDv + threadIdx.x]);
      st_io<IO>(out + row * kDv + threadIdx.x, num / den);
    }
    __syncthreads();  // xq / xk / xv / gq / part are rewritten by the next token
  }
  __syncthreads();
  if (vec) {
#pragma unroll 4
    for (int i = threadIdx.x; i < n_state / 4; i += blockDim.x)
      reinterpret_cast<float4*>(st)[i] = reinterpret_cast<const float4*>(S)[i];
  } else {
#pragma unroll 8
    for (int i = threadIdx.x; i < n_state; i += blockDim.x) st[i] = S[i];
  }
}

}  // namespace

// Workspace of the backward pass.  Bidirectional: control block | parameters | Vt|Z | dVt|dZ |
// parameter sums | dl of the queries | dl of the keys (the three accumulators contiguous, zeroed
// together).  Causal: control block | parameters | segment aggregates of the keys (scanned: S at each
// segment start) | segment aggregates of the queries' gamma_Q u^T (suffix-scanned: R after each
// segment) | parameter sums | u rows | dl of the queries | dl of the keys.
struct BwdPlan {
  size_t off_params, off_state, off_dstate, off_pacc, off_pb, off_u, off_dlq, off_dlk, total;
  int splits, seg_tiles, tiles;
};
BwdPlan bwd_plan(const gma_problem_t& p, bool causal) {
  BwdPlan b{};
  const SimtPlan sp = simt_plan(p, causal ? GMA_OP_CAUSAL : GMA_OP_BIDIR);
  const size_t BH = (size_t)p.B * p.H, npairs = (size_t)p.K * kStateCols;
  const size_t nstate = causal ? BH * sp.splits * npairs : BH * npairs;
  b.splits = sp.splits;
  b.seg_tiles = sp.seg_tiles;
  b.tiles = sp.tiles;
  b.off_params = sp.off_params;
  b.off_state = align_up(sp.off_params + ((size_t)2 * p.H * kD * p.K + (size_t)p.H * p.K) * sizeof(float));
  b.off_dstate = b.off_state + nstate * sizeof(float);
  b.off_pacc = b.off_dstate + nstate * sizeof(float);
  b.off_pb = b.off_pacc + (size_t)p.H * p.K * kD * 2 * sizeof(float);
  b.off_u = align_up(b.off_pb + (size_t)p.H * p.K * sizeof(float));
  b.off_dlq = align_up(b.off_u + (causal ? BH * p.N * kStateCols * sizeof(float) : 0));
  b.off_dlk = align_up(b.off_dlq + BH * p.N * p.K * sizeof(float));
  b.total = align_up(b.off_dlk + BH * p.N * p.K * sizeof(float));
  return b;
}

template <typename IO>
gma_status_t backward_typed(const gma_problem_t& p, bool causal, const IO* Q, const IO* Kx, const IO* V,
                            const float* mu, const float* sigma2, const float* log_pi, const IO* dO, IO* dQ, IO* dK,
                            IO* dV, float* dmu, float* dsigma2, float* dlog_pi, void* ws, cudaStream_t st) {
  const BwdPlan b = bwd_plan(p, causal);
  char* base = (char*)ws;
  float* params = (float*)(base + b.off_params);
  float* state = (float*)(base + b.off_state);
  float* dstate = (float*)(base + b.off_dstate);
  float* pacc = (float*)(base + b.off_pacc);
  float* pb = (float*)(base + b.off_pb);
  float* urows = (float*)(base + b.off_u);
  float* dlq = (float*)(base + b.off_dlq);
  float* dlk = (float*)(base + b.off_dlk);
  const int BH = p.B * p.H, K = p.K, npairs = K * kStateCols;
  // bidirectional: zero Vt|Z, dVt|dZ and the parameter sums; causal: the parameter sums (the segment
  // aggregates are stored whole)
  float* zero = causal ? pacc : state;
  const size_t zero_n = (b.off_u - (causal ? b.off_pacc : b.off_state)) / sizeof(float);
  GMA_LAUNCH("simt_prep", simt_prep_kernel, 148, 256, 0, st, mu, sigma2, log_pi, p.H, K, params, (Ctrl*)base, zero,
             zero_n);
  if (gma_status_t e = check_launch("launch simt_prep", (const void*)simt_prep_kernel)) return e;
  if (p.N > 0) {
    const size_t sm_write = (size_t)(T * kD + T * kDv + T * K + npairs) * sizeof(float);
    if (set_smem_optin((const void*)simt_write_kernel<IO>, (int)sm_write, 1) != GMA_OK) return GMA_ERR_CUDA;
    GMA_LAUNCH("simt_write", simt_write_kernel<IO>, dim3(b.splits, BH), kThreads, sm_write, st, Kx, V, params, p.H,
               p.N, K, b.seg_tiles, b.splits, state, causal ? 0 : 1);
    if (gma_status_t e = check_launch("launch simt_write", (const void*)simt_write_kernel<IO>)) return e;
    if (causal) {
      GMA_LAUNCH("simt_scan", simt_scan_kernel, dim3(cdiv(npairs, 256), BH), 256, 0, st, state, b.splits, npairs);
      if (gma_status_t e = check_launch("launch simt_scan", (const void*)simt_scan_kernel)) return e;
      const size_t sm_q = (size_t)(npairs + 3 * T * kD + T * kStateCols + 3 * T * K + 2 * T * T) * sizeof(float);
      if (set_smem_optin((const void*)simt_bwd_causal_query_kernel<IO>, (int)sm_q, 7) != GMA_OK) return GMA_ERR_CUDA;
      GMA_LAUNCH("simt_bwd_causal_query", simt_bwd_causal_query_kernel<IO>, dim3(b.splits, BH), kThreads, sm_q, st, Q,
                 Kx, V, dO, params, mu, sigma2, p.H, p.N, K, b.seg_tiles, b.splits, state, p.eps, dstate, urows, dlq,
                 dQ);
      if (gma_status_t e = check_launch("launch simt_bwd_causal_query", (const void*)simt_bwd_causal_query_kernel<IO>))
        return e;
      GMA_LAUNCH("simt_rscan", simt_rscan_kernel, dim3(cdiv(npairs, 256), BH), 256, 0, st, dstate, b.splits, npairs);
      if (gma_status_t e = check_launch("launch simt_rscan", (const void*)simt_rscan_kernel)) return e;
      const size_t sm_k = (size_t)(npairs + 2 * T * kD + T * kStateCols + 3 * T * K + 2 * T * T) * sizeof(float);
      if (set_smem_optin((const void*)simt_bwd_causal_key_kernel<IO>, (int)sm_k, 8) != GMA_OK) return GMA_ERR_CUDA;
      GMA_LAUNCH("simt_bwd_causal_key", simt_bwd_causal_key_kernel<IO>, dim3(b.splits, BH), kThreads, sm_k, st, Q, Kx,
                 V, params, mu, sigma2, p.H, p.N, K, b.seg_tiles, b.splits, dstate, urows, dlk, dK, dV);
      if (gma_status_t e = check_launch("launch simt_bwd_causal_key", (const void*)simt_bwd_causal_key_kernel<IO>))
        return e;
    } else {
      const size_t sm_q = (size_t)(2 * npairs + T * kD + T * kDv + T * kStateCols + 2 * T * K) * sizeof(float);
      if (set_smem_optin((const void*)simt_bwd_query_kernel<IO>, (int)sm_q, 5) != GMA_OK) return GMA_ERR_CUDA;
      GMA_LAUNCH("simt_bwd_query", simt_bwd_query_kernel<IO>, dim3(b.splits, BH), kThreads, sm_q, st, Q, dO, params,
                 mu, sigma2, p.H, p.N, K, b.seg_tiles, state, p.eps, dstate, dlq, dQ);
      if (gma_status_t e = check_launch("launch simt_bwd_query", (const void*)simt_bwd_query_kernel<IO>)) return e;
      const size_t sm_k = (size_t)(npairs + T * kD + T * kDv + 2 * T * K) * sizeof(float);
      if (set_smem_optin((const void*)simt_bwd_key_kernel<IO>, (int)sm_k, 6) != GMA_OK) return GMA_ERR_CUDA;
      GMA_LAUNCH("simt_bwd_key", simt_bwd_key_kernel<IO>, dim3(b.tiles, BH), kThreads, sm_k, st, Kx, V, params, mu,
                 sigma2, p.H, p.N, K, dstate, dlk, dK, dV);
      if (gma_status_t e = check_launch("launch simt_bwd_key", (const void*)simt_bwd_key_kernel<IO>)) return e;
    }
    const int rows_per_chunk = 2048;
    const long long rows = 2LL * p.B * p.N;
    const dim3 grid_p(cdiv(K, 32), p.H, cdiv(rows, rows_per_chunk));
    GMA_LAUNCH("simt_bwd_param", simt_bwd_param_kernel<IO>, grid_p, kThreads, 0, st, Q, Kx, mu, dlq, dlk, p.B, p.H, p.N,
               K, rows_per_chunk, pacc, pb);
    if (gma_status_t e = check_launch("launch simt_bwd_param", (const void*)simt_bwd_param_kernel<IO>)) return e;
  }
  GMA_LAUNCH("simt_bwd_param_finish", simt_bwd_param_finish_kernel, 148, 256, 0, st, sigma2, pacc, pb, p.H, K, dmu,
             dsigma2, dlog_pi);
  return check_launch("launch simt_bwd_param_finish", (const void*)simt_bwd_param_finish_kernel);
}

size_t simt_backward_bytes(const gma_problem_t& p, bool causal) { return bwd_plan(p, causal).total; }

gma_status_t simt_backward(const gma_problem_t& p, bool causal, const void* Q, const void* K, const void* V,
                           const float* mu, const float* sigma2, const float* log_pi, const void* dO, void* dQ,
                           void* dK, void* dV, float* dmu, float* dsigma2, float* dlog_pi, void* ws, cudaStream_t st) {
  if (p.dtype == GMA_F32)
    return backward_typed<float>(p, causal, (const float*)Q, (const float*)K, (const float*)V, mu, sigma2, log_pi,
                                 (const float*)dO, (float*)dQ, (float*)dK, (float*)dV, dmu, dsigma2, dlog_pi, ws, st);
  using bf = __nv_bfloat16;
  return backward_typed<bf>(p, causal, (const bf*)Q, (const bf*)K, (const bf*)V, mu, sigma2, log_pi, (const bf*)dO,
                            (bf*)dQ, (bf*)dK, (bf*)dV, dmu, dsigma2, dlog_pi, ws, st);
}

// Decode T new tokens per (b, h) from `state` (float32 [B*H][K][dv + 1], updated in place).  One launch;
// the workspace is not used (its error word stays as the caller left it).
gma_status_t simt_decode(const gma_problem_t& p, const void* Q, const void* K, const void* V, const float* mu,
                         const float* sigma2, const float* log_pi, float* state, void* out, void* /*ws*/,
                         cudaStream_t st) {
  const size_t smem = decode_smem_floats(p.K) * sizeof(float);
  const int BH = p.B * p.H;
  if (p.dtype == GMA_F32) {
    if (set_smem_optin((const void*)simt_decode_kernel<float>, (int)smem, 4) != GMA_OK) return GMA_ERR_CUDA;
    GMA_LAUNCH("simt_decode", simt_decode_kernel<float>, BH, kDecodeThreads, smem, st, (const float*)Q,
               (const float*)K, (const float*)V, mu, sigma2, log_pi, p.H, p.N, p.K, state, p.eps, (float*)out);
    return check_launch("launch simt_decode", (const void*)simt_decode_kernel<float>);
  }
  if (set_smem_optin((const void*)simt_decode_kernel<__nv_bfloat16>, (int)smem, 4) != GMA_OK) return GMA_ERR_CUDA;
  GMA_LAUNCH("simt_decode", simt_decode_kernel<__nv_bfloat16>, BH, kDecodeThreads, smem, st,
             (const __nv_bfloat16*)Q, (const __nv_bfloat16*)K, (const __nv_bfloat16*)V, mu, sigma2, log_pi, p.H,
             p.N, p.K, state, p.eps, (__nv_bfloat16*)out);
  return check_launch("launch simt_decode", (const void*)simt_decode_kernel<__nv_bfloat16>);
}

namespace {

template <typename IO>
gma_status_t run_typed(const gma_problem_t& p, gma_op_t op, int Nk, const IO* Q, const IO* Kx, const IO* V,
                       const float* mu, const float* sigma2, const float* log_pi, void* out, void* ws,
                       cudaStream_t st) {
  const SimtPlan pl = simt_plan(p, op);
  char* base = (char*)ws;
  Ctrl* ctrl = (Ctrl*)base;
  float* params = (float*)(base + pl.off_params);
  float* state = (float*)(base + pl.off_state);
  const int BH = p.B * p.H, K = p.K;
  const int npairs = K * kStateCols;
  const bool write_only = op == GMA_OP_CAUSAL_STATE;  // state of all N keys, copied to `out`
  if (write_only) op = GMA_OP_BIDIR;
  const size_t zero_n = op == GMA_OP_BIDIR ? (size_t)BH * npairs : 0;
  GMA_LAUNCH("simt_prep", simt_prep_kernel, 148, 256, 0, st, mu, sigma2, log_pi, p.H, K, params, ctrl, state, zero_n);
  if (cudaGetLastError() != cudaSuccess) return GMA_ERR_CUDA;
  if (p.N == 0 && !write_only) return GMA_OK;
  const size_t sm_gamma = (size_t)(T * kD + T * K) * sizeof(float);
  if (op == GMA_OP_RESPONSIBILITIES) {
    if (set_smem_optin((const void*)simt_resp_kernel<IO>, (int)sm_gamma, 0) != GMA_OK) return GMA_ERR_CUDA;
    GMA_LAUNCH("simt_resp", simt_resp_kernel<IO>, dim3(pl.tiles, BH), kThreads, sm_gamma, st, Q, params, p.H, p.N, K, (float*)out);
    return cudaGetLastError() == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
  }
  const size_t sm_write = (size_t)(T * kD + T * kDv + T * K + npairs) * sizeof(float);
  if (set_smem_optin((const void*)simt_write_kernel<IO>, (int)sm_write, 1) != GMA_OK) return GMA_ERR_CUDA;
  if (op == GMA_OP_BIDIR) {
    // write over the Nk keys (its own split plan; the workspace layout does not depend on N)
    if (Nk > 0) {
      gma_problem_t pk = p;
      pk.N = Nk;
      const SimtPlan plk = simt_plan(pk, op);
      GMA_LAUNCH("simt_write", simt_write_kernel<IO>, dim3(plk.splits, BH), kThreads, sm_write, st, Kx, V, params, p.H, Nk, K,
                 plk.seg_tiles, plk.splits, state, 1);
      if (cudaGetLastError() != cudaSuccess) return GMA_ERR_CUDA;
    }
    if (write_only) {  // the accumulator already has the public state layout [B*H][K][dv + 1]
      if (cudaMemcpyAsync(out, state, (size_t)BH * npairs * sizeof(float), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return cuda_fail("copy state");
      return GMA_OK;
    }
    const size_t sm_read = (size_t)(T * kD + T * K + T * kStateCols) * sizeof(float);
    if (set_smem_optin((const void*)simt_read_kernel<IO>, (int)sm_read, 2) != GMA_OK) return GMA_ERR_CUDA;
    GMA_LAUNCH("simt_read", simt_read_kernel<IO>, dim3(pl.tiles, BH), kThreads, sm_read, st, Q, params, p.H, p.N, K, state, p.eps,
                                                                        (IO*)out);
    return cudaGetLastError() == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
  }
  // causal
  GMA_LAUNCH("simt_write", simt_write_kernel<IO>, dim3(pl.splits, BH), kThreads, sm_write, st, Kx, V, params, p.H, p.N, K, pl.seg_tiles,
                                                                         pl.splits, state, 0);
  if (cudaGetLastError() != cudaSuccess) return GMA_ERR_CUDA;
  GMA_LAUNCH("simt_scan", simt_scan_kernel, dim3(cdiv(npairs, 256), BH), 256, 0, st, state, pl.splits, npairs);
  if (cudaGetLastError() != cudaSuccess) return GMA_ERR_CUDA;
  const size_t sm_causal = (size_t)(npairs + T * kD + T * kDv + 2 * T * K + T * T + T * kStateCols) * sizeof(float);
  if (set_smem_optin((const void*)simt_causal_kernel<IO>, (int)sm_causal, 3) != GMA_OK) return GMA_ERR_CUDA;
  GMA_LAUNCH("simt_causal", simt_causal_kernel<IO>, dim3(pl.splits, BH), kThreads, sm_causal, st, Q, Kx, V, params, p.H, p.N, K,
                                                                           pl.seg_tiles, pl.splits, state, p.eps,
                                                                           (IO*)out);
  return cudaGetLastError() == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

}  // namespace

SimtPlan simt_plan(const gma_problem_t& p, gma_op_t op) {
  SimtPlan pl{};
  const int BH = p.B * p.H;
  pl.tiles = cdiv(p.N, T);
  int want = cdiv(kTargetUnits, BH);
  if (want < 1) want = 1;
  if (want > pl.tiles) want = pl.tiles;
  if (want < 1) want = 1;
  pl.seg_tiles = cdiv(pl.tiles > 0 ? pl.tiles : 1, want);
  pl.splits = cdiv(pl.tiles > 0 ? pl.tiles : 1, pl.seg_tiles);
  pl.off_params = align_up(sizeof(Ctrl));
  const size_t params_bytes = ((size_t)2 * p.H * kD * p.K + (size_t)p.H * p.K) * sizeof(float);
  pl.off_state = align_up(pl.off_params + params_bytes);
  size_t state_bytes = 0;
  if (op == GMA_OP_BIDIR || op == GMA_OP_CROSS || op == GMA_OP_CAUSAL_STATE)
    state_bytes = (size_t)BH * p.K * kStateCols * sizeof(float);
  if (op == GMA_OP_CAUSAL) state_bytes = (size_t)BH * pl.splits * p.K * kStateCols * sizeof(float);
  pl.total = align_up(pl.off_state + state_bytes);
  return pl;
}

gma_status_t simt_run(const gma_problem_t& p, gma_op_t op, int Nk, const void* Q, const void* K, const void* V,
                      const float* mu, const float* sigma2, const float* log_pi, void* out, void* ws,
                      cudaStream_t stream) {
  if (p.dtype == GMA_F32)
    return run_typed<float>(p, op, Nk, (const float*)Q, (const float*)K, (const float*)V, mu, sigma2, log_pi, out, ws,
                            stream);
  return run_typed<__nv_bfloat16>(p, op, Nk, (const __nv_bfloat16*)Q, (const __nv_bfloat16*)K, (const __nv_bfloat16*)V,
                                  mu, sigma2, log_pi, out, ws, stream);
}

}  // namespace gma

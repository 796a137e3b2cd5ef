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

#include <climits>

#include "gma_internal.h"
#include "gma_tc_common.cuh"

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
// floats at `zero` (the write-phase accumulator).  wpair (backward only, else null): the pairs
// (1 / sigma2, mu / sigma2) in the order of mu, [H][K][64][2], read by the dx step.
__global__ void simt_prep_kernel(const float* __restrict__ mu, const float* __restrict__ sigma2,
                                 const float* __restrict__ log_pi, int H, int K, float* params, Ctrl* ctrl,
                                 float* zero, size_t zero_n, float2* wpair) {
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
    const float w = 1.0f / sigma2[i];
    P.mu_t[o] = mu[i];
    P.w_t[o] = w;
    if (wpair) wpair[i] = make_float2(w, w * mu[i]);
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
// rows past `n` are zero.  rows: the matrix's row count, checked in the bounds-check build.
template <typename IO>
__device__ __forceinline__ void load_rows(const IO* __restrict__ src, int r0, int n, float* dst, int rows = INT_MAX) {
  for (int i = threadIdx.x; i < T * kD; i += blockDim.x) {
    const int r = i / kD;
    dst[i] = r < n && GMA_INB(r0 + r, rows, 201) ? ld_io<IO>(src + (size_t)(r0 + r) * kD + (i % kD)) : 0.f;
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

// ---- register-tiled pieces of the write and backward kernels ---------------------------------------
// KC is K rounded up to 32, 64, 128 or 256: the width of the shared-memory gamma tiles G[T][KC] (zero past
// K) and the row count of the state images.  A state image holds a [K][dv + 1] float32 state as S[KC][kSP]
// (the dv columns; rows past K zero) with the normaliser column apart in Z[KC].  kSP = 68 keeps the rows
// 16-byte aligned, and eight lanes whose 16-byte loads are one row apart hit disjoint groups of banks.
constexpr int kSP = 68;

__host__ __device__ constexpr int kc_class(int K) { return K <= 32 ? 32 : (K <= 64 ? 64 : (K <= 128 ? 128 : 256)); }

template <int KC>
__device__ __forceinline__ void load_state_image(const float* src, int K, float* S, float* Z) {
  for (int p = threadIdx.x; p < KC * kDv; p += blockDim.x) {
    const int k = p / kDv, c = p % kDv;
    S[k * kSP + c] = k < K ? src[(size_t)k * kStateCols + c] : 0.f;
  }
  for (int k = threadIdx.x; k < KC; k += blockDim.x) Z[k] = k < K ? src[(size_t)k * kStateCols + kDv] : 0.f;
}

// Responsibilities of the T rows in xs (first `nvalid` valid) into G[T][KC]; rows past nvalid and
// columns past K are zero.  Thread (component k, group of RPT = T KC / 256 rows) keeps RPT independent
// sums of the centered log-density, so that each parameter is read once per tile; then one warp per
// row takes the softmax.  Needs 256 threads.  UJ: unroll of the loop over dims (2 where the registers
// allow it).
template <int KC, int UJ = 1>
__device__ void gamma_tile_kc(const float* xs, int nvalid, const SimtParams& P, int h, int K, float* G) {
  constexpr int RK = KC / 32, RPT = T * KC / kThreads;
  const float* mu_t = P.mu_t + (size_t)h * kD * K;
  const float* w_t = P.w_t + (size_t)h * kD * K;
  const float* c = P.c + (size_t)h * K;
  const int k = threadIdx.x % KC, r0 = (threadIdx.x / KC) * RPT;
  if (k < K) {
    float acc[RPT];
#pragma unroll
    for (int ii = 0; ii < RPT; ++ii) acc[ii] = 0.f;
#pragma unroll UJ
    for (int j = 0; j < kD; j += 4) {
      float m[4], w[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        m[t] = __ldg(mu_t + (size_t)(j + t) * K + k);
        w[t] = __ldg(w_t + (size_t)(j + t) * K + k);
      }
#pragma unroll
      for (int ii = 0; ii < RPT; ++ii) {
        const float4 x = *reinterpret_cast<const float4*>(xs + (r0 + ii) * kD + j);
        float d = x.x - m[0];
        acc[ii] = fmaf(d * w[0], d, acc[ii]);
        d = x.y - m[1];
        acc[ii] = fmaf(d * w[1], d, acc[ii]);
        d = x.z - m[2];
        acc[ii] = fmaf(d * w[2], d, acc[ii]);
        d = x.w - m[3];
        acc[ii] = fmaf(d * w[3], d, acc[ii]);
      }
    }
    const float ck = __ldg(c + k);
#pragma unroll
    for (int ii = 0; ii < RPT; ++ii) G[(r0 + ii) * KC + k] = ck - 0.5f * acc[ii];
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  for (int i = warp; i < T; i += nwarps) {
    float* row = G + i * KC;
    if (i >= nvalid) {
#pragma unroll
      for (int r = 0; r < RK; ++r) row[lane + 32 * r] = 0.f;
      continue;
    }
    float v[RK], m = -INFINITY;
#pragma unroll
    for (int r = 0; r < RK; ++r) {
      v[r] = lane + 32 * r < K ? row[lane + 32 * r] : -INFINITY;
      m = fmaxf(m, v[r]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = 0.f;
#pragma unroll
    for (int r = 0; r < RK; ++r) {
      v[r] = lane + 32 * r < K ? expf(v[r] - m) : 0.f;
      s += v[r];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float inv = 1.0f / s;
#pragma unroll
    for (int r = 0; r < RK; ++r) row[lane + 32 * r] = v[r] * inv;
  }
  __syncthreads();
}

// acc[q][e] += sum_i G[i][k0 + q] B[i][lane + 32 e] and z += sum_i G[i][k0 + lane] b_i (lanes < KC / 8):
// warp w owns components k0 = w KC / 8 .. + KC / 8 against the 64 columns of the rows B[T][ldb];
// b_i = bz[i], or 1 where bz is null.  G has row stride LDG.  Needs 8 warps.
template <int KC, int LDG = KC>
__device__ __forceinline__ void accumulate_gt(const float* G, const float* B, int ldb, const float* bz,
                                              float (&acc)[KC / 8][2], float& z) {
  constexpr int KW = KC / 8;
  const int lane = threadIdx.x & 31, k0 = (threadIdx.x >> 5) * KW;
#pragma unroll 2
  for (int i = 0; i < T; ++i) {
    const float b0 = B[i * ldb + lane], b1 = B[i * ldb + 32 + lane];
    const float* g = G + i * LDG + k0;
#pragma unroll
    for (int q = 0; q < KW; q += 4) {
      const float4 g4 = *reinterpret_cast<const float4*>(g + q);
      acc[q][0] = fmaf(g4.x, b0, acc[q][0]);
      acc[q][1] = fmaf(g4.x, b1, acc[q][1]);
      acc[q + 1][0] = fmaf(g4.y, b0, acc[q + 1][0]);
      acc[q + 1][1] = fmaf(g4.y, b1, acc[q + 1][1]);
      acc[q + 2][0] = fmaf(g4.z, b0, acc[q + 2][0]);
      acc[q + 2][1] = fmaf(g4.z, b1, acc[q + 2][1]);
      acc[q + 3][0] = fmaf(g4.w, b0, acc[q + 3][0]);
      acc[q + 3][1] = fmaf(g4.w, b1, acc[q + 3][1]);
    }
    if (lane < KW) z = fmaf(g[lane], bz ? bz[i] : 1.f, z);
  }
}

// Copies the first nvalid rows of a tile G[T][KC] to dst[nvalid][K], and back (zero past nvalid and K).
template <int KC>
__device__ __forceinline__ void store_rows(const float* G, int nvalid, int K, float* dst) {
  for (int p = threadIdx.x; p < nvalid * K; p += blockDim.x) dst[p] = G[(p / K) * KC + p % K];
}
// (G row stride LDG; the pad columns past KC are left alone)
template <int KC, int LDG = KC>
__device__ __forceinline__ void load_tile_rows(const float* src, int nvalid, int K, float* G) {
  if ((K & 3) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0) {  // 16-byte words
    for (int p = threadIdx.x; p < T * KC / 4; p += blockDim.x) {
      const int i = p / (KC / 4), k = 4 * (p % (KC / 4));
      *reinterpret_cast<float4*>(G + i * LDG + k) =
          i < nvalid && k < K ? *reinterpret_cast<const float4*>(src + (size_t)i * K + k) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }
  for (int p = threadIdx.x; p < T * KC; p += blockDim.x) {
    const int i = p / KC, k = p % KC;
    G[i * LDG + k] = i < nvalid && k < K ? src[(size_t)i * K + k] : 0.f;
  }
}

// Writes (or adds, atomic != 0) the register blocks of accumulate_gt into a [K][dv + 1] state at dst.
// off, lim (checked in the bounds-check build): dst's offset in its buffer, and the buffer's extent.
template <int KC>
__device__ __forceinline__ void store_gt(float* dst, int K, const float (&acc)[KC / 8][2], float z, int atomic,
                                         size_t off = 0, size_t lim = ~(size_t)0) {
  constexpr int KW = KC / 8;
  const int lane = threadIdx.x & 31, k0 = (threadIdx.x >> 5) * KW;
#pragma unroll
  for (int q = 0; q < KW; ++q) {
    if (k0 + q >= K) break;
    float* row = dst + (size_t)(k0 + q) * kStateCols;
    if (!GMA_INB(off + (size_t)(k0 + q + 1) * kStateCols - 1, lim, 210)) continue;
    if (atomic) {
      atomicAdd(row + lane, acc[q][0]);
      atomicAdd(row + 32 + lane, acc[q][1]);
    } else {
      row[lane] = acc[q][0];
      row[32 + lane] = acc[q][1];
    }
  }
  if (lane < KW && k0 + lane < K && GMA_INB(off + (size_t)(k0 + lane) * kStateCols + kDv, lim, 210)) {
    float* zp = dst + (size_t)(k0 + lane) * kStateCols + kDv;
    if (atomic) atomicAdd(zp, z); else *zp = z;
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
  load_rows<IO>(X + (size_t)unit * N * kD, t0, nvalid, xs, N);
  __syncthreads();
  gamma_tile(xs, nvalid, P, h, K, G);
  float* out = gamma + ((size_t)unit * N + t0) * K;
  for (int i = threadIdx.x; i < nvalid * K; i += blockDim.x)
    if (GMA_INB(((size_t)unit * N + t0) * K + i, (size_t)gridDim.y * N * K, 213)) out[i] = G[i];
}

// Eight consecutive elements of a row as float32 (one 16-byte load for bf16, two for float32).
template <typename IO>
__device__ __forceinline__ void load8(const IO* __restrict__ p, float (&v)[8]);
template <>
__device__ __forceinline__ void load8<float>(const float* __restrict__ p, float (&v)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p)), b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* __restrict__ p, float (&v)[8]) {
  const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    v[2 * t] = __uint_as_float(w[t] << 16);
    v[2 * t + 1] = __uint_as_float(w[t] & 0xffff0000u);
  }
}

// A tile's share of one thread of 256: row r = tid / 8, elements 8 (tid % 8) .. + 7 of rows [r0, r0 + n)
// of a [rows][64] matrix (zero past n), and its store into a [T][64] shared-memory tile.
template <typename IO>
__device__ __forceinline__ void fetch_tile8(const IO* __restrict__ src, int r0, int n, float (&v)[8], int rows = INT_MAX) {
  const int r = threadIdx.x >> 3, c = 8 * (threadIdx.x & 7);
#pragma unroll
  for (int t = 0; t < 8; ++t) v[t] = 0.f;
  if (r < n && GMA_INB(r0 + r, rows, 202)) load8<IO>(src + (size_t)(r0 + r) * kD + c, v);
}
__device__ __forceinline__ void put_tile8(float* dst, const float (&v)[8]) {
  float* d = dst + (threadIdx.x >> 3) * kD + 8 * (threadIdx.x & 7);
  *reinterpret_cast<float4*>(d) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(d + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// Write phase (bidirectional) or segment aggregate (causal): grid (splits, B*H).  Each CTA covers
// tiles [split * seg_tiles, ...) of its (b,h) and keeps its partial [Vt | Z] in registers (accumulate_gt).
// atomic != 0: add into state[unit][K][65]; atomic == 0: store into state[unit][split][K][65].
// gout (backward only, else null): every key's responsibilities, [B*H][N][K].
template <typename IO, int KC>
__global__ void __launch_bounds__(kThreads, KC <= 128 ? 2 : 1) simt_write_kernel(const IO* __restrict__ Kx, const IO* __restrict__ V,
                                                              float* params, int H, int N, int K, int seg_tiles,
                                                              int splits, float* state, int atomic, float* gout,
                                                              size_t state_lim) {
  extern __shared__ float sm[];
  float* xs = sm;           // [T][64]
  float* vs = xs + T * kD;  // [T][64]
  float* G = vs + T * kDv;  // [T][KC]
  const int unit = blockIdx.y, h = unit % H, split = blockIdx.x;
  const SimtParams P = params_at(params, H, K);
  float acc[KC / 8][2], z = 0.f;
#pragma unroll
  for (int q = 0; q < KC / 8; ++q) acc[q][0] = acc[q][1] = 0.f;
  const int tiles = (N + T - 1) / T;
  const int tb = split * seg_tiles, te = min(tiles, tb + seg_tiles);
  const IO* kb = Kx + (size_t)unit * N * kD;
  const IO* vb = V + (size_t)unit * N * kDv;
  float xk[8], xv[8];  // the next tile's key and value rows, loaded while the current one is worked on
  if (tb < te) {
    fetch_tile8<IO>(kb, tb * T, min(T, N - tb * T), xk, N);
    fetch_tile8<IO>(vb, tb * T, min(T, N - tb * T), xv, N);
  }
  for (int t = tb; t < te; ++t) {
    const int t0 = t * T, nvalid = min(T, N - t0);
    put_tile8(xs, xk);
    put_tile8(vs, xv);
    __syncthreads();
    if (t + 1 < te) {
      fetch_tile8<IO>(kb, t0 + T, min(T, N - t0 - T), xk, N);
      fetch_tile8<IO>(vb, t0 + T, min(T, N - t0 - T), xv, N);
    }
    gamma_tile_kc<KC>(xs, nvalid, P, h, K, G);
    accumulate_gt<KC>(G, vs, kDv, nullptr, acc, z);
    if (gout) store_rows<KC>(G, nvalid, K, gout + ((size_t)unit * N + t0) * K);
    __syncthreads();
  }
  const size_t npairs = (size_t)K * kStateCols;
  const size_t off = atomic ? (size_t)unit * npairs : ((size_t)unit * splits + split) * npairs;
  store_gt<KC>(state + off, K, acc, z, atomic, off, state_lim);
}

// Read phase (bidirectional): grid (tiles, B*H).
template <typename IO>
__global__ void __launch_bounds__(kThreads) simt_read_kernel(const IO* __restrict__ Q, float* params, int H, int N,
                                                             int K, const float* __restrict__ state, float eps,
                                                             IO* __restrict__ O, size_t state_lim) {
  extern __shared__ float sm[];
  float* xs = sm;
  float* G = xs + T * kD;
  float* num = G + T * K;
  const int unit = blockIdx.y, h = unit % H;
  const int t0 = blockIdx.x * T, nvalid = min(T, N - t0);
  const SimtParams P = params_at(params, H, K);
  load_rows<IO>(Q + (size_t)unit * N * kD, t0, nvalid, xs, N);
  __syncthreads();
  gamma_tile(xs, nvalid, P, h, K, G);
  const float* S = state + (size_t)unit * K * kStateCols;
  for (int p = threadIdx.x; p < T * kStateCols; p += blockDim.x) {
    const int i = p / kStateCols, c = p % kStateCols;
    float s = 0.f;
    for (int k = 0; k < K; ++k)
      if (GMA_INB((size_t)unit * K * kStateCols + k * kStateCols + c, state_lim, 211))
        s = fmaf(G[i * K + k], __ldg(S + k * kStateCols + c), s);
    num[p] = s;
  }
  __syncthreads();
  IO* out = O + ((size_t)unit * N + t0) * kDv;
  for (int p = threadIdx.x; p < nvalid * kDv; p += blockDim.x) {
    const int i = p / kDv, c = p % kDv;
    if (GMA_INB(((size_t)unit * N + t0) * kDv + p, (size_t)gridDim.y * N * kDv, 212))
      st_io<IO>(out + p, num[i * kStateCols + c] / (num[i * kStateCols + kDv] + eps));
  }
}

// Deterministic reduction mode: state[unit][e] = sum over p = 0 .. P-1 of part[unit][p][e], added in the
// order of p.  grid (ceil(npairs / 256), B*H).
__global__ void simt_state_sum_kernel(const float* __restrict__ part, int P, int npairs, float* __restrict__ state,
                                      size_t part_lim, size_t state_lim) {
  const int unit = blockIdx.y;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= npairs) return;
  const float* src = part + (size_t)unit * P * npairs + e;
  float s = 0.f;
  for (int p = 0; p < P; ++p)
    if (GMA_INB(((size_t)unit * P + p) * npairs + e, part_lim, 215)) s += src[(size_t)p * npairs];
  if (GMA_INB((size_t)unit * npairs + e, state_lim, 216)) state[(size_t)unit * npairs + e] = s;
}

// Exclusive scan over segments: agg[unit][p][e] <- sum_{p' < p} agg[unit][p'][e].  grid (ceil(K*65/256), B*H).
__global__ void simt_scan_kernel(float* agg, int P, int npairs, size_t lim) {
  const int unit = blockIdx.y;
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= npairs) return;
  float* base = agg + (size_t)unit * P * npairs + e;
  float run = 0.f;
  for (int p = 0; p < P; ++p) {
    if (!GMA_INB(((size_t)unit * P + p) * npairs + e, lim, 214)) continue;
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
                                                               float eps, IO* __restrict__ O, size_t agg_lim) {
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
  for (int p = threadIdx.x; p < npairs; p += blockDim.x)
    S[p] = GMA_INB(((size_t)unit * P + seg) * npairs + p, agg_lim, 217) ? S0[p] : 0.f;
  const int tiles = (N + T - 1) / T;
  const int tb = seg * seg_tiles, te = min(tiles, tb + seg_tiles);
  for (int t = tb; t < te; ++t) {
    const int t0 = t * T, nvalid = min(T, N - t0);
    __syncthreads();
    load_rows<IO>(Q + (size_t)unit * N * kD, t0, nvalid, xs, N);
    __syncthreads();
    gamma_tile(xs, nvalid, Pp, h, K, GQ);
    load_rows<IO>(Kx + (size_t)unit * N * kD, t0, nvalid, xs, N);
    load_rows<IO>(V + (size_t)unit * N * kDv, t0, nvalid, vs, N);
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
      if (GMA_INB(((size_t)unit * N + t0) * kDv + p, (size_t)gridDim.y * N * kDv, 218))
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

// a[q][e] = sum_k G[i0 + q][k] S[k][lane + 32 e]: rows i0 .. i0 + 3 of a tile (row stride LDG) times the
// dv columns of a state image (the warp's lanes split the columns; each G row is read as a broadcast).
template <int KC, int LDG = KC>
__device__ __forceinline__ void rows_times_image(const float* G, const float* S, int i0, float (&a)[4][2]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int q = 0; q < 4; ++q) a[q][0] = a[q][1] = 0.f;
#pragma unroll 2
  for (int k = 0; k < KC; k += 4) {
    float4 g[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) g[q] = *reinterpret_cast<const float4*>(G + (i0 + q) * LDG + k);
    const float* sk = S + k * kSP + lane;
    float s0[4], s1[4];
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      s0[t] = sk[t * kSP];
      s1[t] = sk[t * kSP + 32];
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      a[q][0] = fmaf(g[q].x, s0[0], a[q][0]);
      a[q][1] = fmaf(g[q].x, s1[0], a[q][1]);
      a[q][0] = fmaf(g[q].y, s0[1], a[q][0]);
      a[q][1] = fmaf(g[q].y, s1[1], a[q][1]);
      a[q][0] = fmaf(g[q].z, s0[2], a[q][0]);
      a[q][1] = fmaf(g[q].z, s1[2], a[q][1]);
      a[q][0] = fmaf(g[q].w, s0[3], a[q][0]);
      a[q][1] = fmaf(g[q].w, s1[3], a[q][1]);
    }
  }
}

// b[q][r] = sum_c A[i0 + q][c] S[lane + 32 r][c] over the dv columns: rows i0 .. i0 + 3 of A[T][lda]
// against every component row of a state image (lane + 32 r is the component).
template <int KC>
__device__ __forceinline__ void rows_times_image_t(const float* A, int lda, const float* S, int i0,
                                                   float (&b)[4][KC / 32]) {
  constexpr int RK = KC / 32;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int r = 0; r < RK; ++r) b[q][r] = 0.f;
#pragma unroll 2
  for (int c = 0; c < kDv; c += 4) {
    float4 a4[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) a4[q] = *reinterpret_cast<const float4*>(A + (i0 + q) * lda + c);
#pragma unroll
    for (int r = 0; r < RK; ++r) {
      const float4 s4 = *reinterpret_cast<const float4*>(S + (lane + 32 * r) * kSP + c);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        b[q][r] = fmaf(a4[q].x, s4.x, b[q][r]);
        b[q][r] = fmaf(a4[q].y, s4.y, b[q][r]);
        b[q][r] = fmaf(a4[q].z, s4.z, b[q][r]);
        b[q][r] = fmaf(a4[q].w, s4.w, b[q][r]);
      }
    }
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Softmax backward of rows i0 .. i0 + 3 in registers: dg[q][r] (dgamma at component lane + 32 r) becomes
// dl = gamma (dgamma - gamma . dgamma); G has row stride LDG.
template <int KC, int LDG = KC>
__device__ __forceinline__ void softmax_backward_rows(const float* G, int i0, float (&dg)[4][KC / 32]) {
  constexpr int RK = KC / 32;
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    float g[RK], dot = 0.f;
#pragma unroll
    for (int r = 0; r < RK; ++r) {
      g[r] = G[(i0 + q) * LDG + lane + 32 * r];
      dot = fmaf(g[r], dg[q][r], dot);
    }
    dot = warp_sum(dot);
#pragma unroll
    for (int r = 0; r < RK; ++r) dg[q][r] = g[r] * (dg[q][r] - dot);
  }
}

// dx_ij = sum_k dl_ik (mu_kj - x_ij) / sigma2_kj = (dl (mu / sigma2))_ij - x_ij (dl (1 / sigma2))_ij for the
// tile's rows from dl[T][LDG] (zero past K).  The head's (1 / sigma2, mu / sigma2) pairs wp[K][64] pass
// through `stage` (2048 floats of free shared memory) 16 components at a time; thread (column j, group
// of 8 rows) then reads its pair per component and four dl values per row at a time.
template <typename IO, int KC, int LDG = KC>
__device__ void dx_tile_kc(const float* xs, const float* dl, int nvalid, const float2* __restrict__ wp, int K,
                           float* stage, IO* dst) {
  const int j = threadIdx.x % kD, rg = threadIdx.x / kD;  // 4 groups of 8 rows
  const float2* st2 = reinterpret_cast<const float2*>(stage);
  float a1[8], a2[8];
#pragma unroll
  for (int r = 0; r < 8; ++r) a1[r] = a2[r] = 0.f;
  for (int k0 = 0; k0 < K; k0 += 16) {
    const int nk = min(16, K - k0);
    __syncthreads();  // the previous chunk's readers are done
    for (int p = threadIdx.x; p < 16 * kD / 2; p += blockDim.x) {  // 512 float4 = 16 components x 64 pairs
      const int kk = p / (kD / 2);
      reinterpret_cast<float4*>(stage)[p] =
          kk < nk ? __ldg(reinterpret_cast<const float4*>(wp + (size_t)k0 * kD) + p) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
#pragma unroll 2
    for (int kk = 0; kk < 16; kk += 4) {
      float2 w[4];
#pragma unroll
      for (int t = 0; t < 4; ++t) w[t] = st2[(kk + t) * kD + j];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float4 d = *reinterpret_cast<const float4*>(dl + (rg * 8 + r) * LDG + k0 + kk);
        a1[r] = fmaf(d.x, w[0].y, a1[r]);
        a2[r] = fmaf(d.x, w[0].x, a2[r]);
        a1[r] = fmaf(d.y, w[1].y, a1[r]);
        a2[r] = fmaf(d.y, w[1].x, a2[r]);
        a1[r] = fmaf(d.z, w[2].y, a1[r]);
        a2[r] = fmaf(d.z, w[2].x, a2[r]);
        a1[r] = fmaf(d.w, w[3].y, a1[r]);
        a2[r] = fmaf(d.w, w[3].x, a2[r]);
      }
    }
  }
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    const int i = rg * 8 + r;
    if (i < nvalid) st_io<IO>(dst + (size_t)i * kD + j, a1[r] - xs[i * kD + j] * a2[r]);
  }
}

// Stores the warp's rows i0 .. i0 + 3 of dl (registers, component lane + 32 r) into the tile G[T][LDG] and,
// for valid rows and components, into the workspace rows dst[i][K].
template <int KC, int LDG = KC>
__device__ __forceinline__ void store_dl_rows(const float (&dl)[4][KC / 32], int i0, int nvalid, int K, float* G,
                                              float* dst) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int q = 0; q < 4; ++q)
#pragma unroll
    for (int r = 0; r < KC / 32; ++r) {
      const int k = lane + 32 * r;
      G[(i0 + q) * LDG + k] = dl[q][r];
      if (i0 + q < nvalid && k < K) dst[(size_t)(i0 + q) * K + k] = dl[q][r];
    }
}

// Query side: grid (splits, B*H).  Recomputes O, pushes dO back through the read, writes dQ and dl_Q, and
// adds [dVt | dZ] into dstate[unit][K][65] (dsplits = 0) or stores this CTA's share into
// dstate[unit][split][K][65] (dsplits = the grid's splits; the deterministic reduction mode).  Warp w owns tile rows 4w .. 4w + 3 in the row products and
// components w KC / 8 .. + KC / 8 of [dVt | dZ], which stay in registers across the CTA's tiles.
template <typename IO, int KC>
__global__ void __launch_bounds__(kThreads) simt_bwd_query_kernel(const IO* __restrict__ Q, const IO* __restrict__ dO,
                                                                  float* params, const float2* __restrict__ wpair,
                                                                  int H, int N, int K, int seg_tiles,
                                                                  const float* __restrict__ state, float eps,
                                                                  float* dstate, int dsplits, float* dlq,
                                                                  IO* __restrict__ dQ, int gpre) {
  constexpr int RK = KC / 32;
  extern __shared__ float sm[];
  float* S = sm;            // [KC][kSP]  Vt image
  float* Z = S + KC * kSP;  // [KC]
  float* xs = Z + KC;       // [T][64]   query rows
  float* gs = xs + T * kD;  // [T][64]   dO rows, then the dx parameter stage
  float* dn = gs + T * kDv;  // [T][kSP]  dO / den
  float* dd = dn + T * kSP;  // [T]       -(dO . O) / den
  float* G = dd + T;         // [T][KC]   gamma_Q, then dl_Q
  const int unit = blockIdx.y, h = unit % H, split = blockIdx.x;
  const int lane = threadIdx.x & 31, i0 = 4 * (threadIdx.x >> 5);
  const SimtParams P = params_at(params, H, K);
  const size_t npairs = (size_t)K * kStateCols;
  load_state_image<KC>(state + unit * npairs, K, S, Z);
  float acc[KC / 8][2], zacc = 0.f;
#pragma unroll
  for (int q = 0; q < KC / 8; ++q) acc[q][0] = acc[q][1] = 0.f;
  const int tiles = (N + T - 1) / T;
  const int tb = split * seg_tiles, te = min(tiles, tb + seg_tiles);
  for (int t = tb; t < te; ++t) {
    const int t0 = t * T, nvalid = min(T, N - t0);
    __syncthreads();
    load_rows<IO>(Q + (size_t)unit * N * kD, t0, nvalid, xs);
    load_rows<IO>(dO + (size_t)unit * N * kDv, t0, nvalid, gs);
    // gamma_Q: recomputed, or (gpre) the rows the tensor-core responsibilities kernel left in dlq, which
    // this tile overwrites with dl_Q below
    if (gpre)
      load_tile_rows<KC>(dlq + ((size_t)unit * N + t0) * K, nvalid, K, G);
    __syncthreads();
    if (!gpre) gamma_tile_kc<KC, 2>(xs, nvalid, P, h, K, G);
    __syncthreads();
    {  // numerators and denominators of the warp's rows, then dn | dd (rows past N: zero)
      float a[4][2], dp[4] = {0.f, 0.f, 0.f, 0.f};
      rows_times_image<KC>(G, S, i0, a);
#pragma unroll
      for (int r = 0; r < RK; ++r) {
        const float z = Z[lane + 32 * r];
#pragma unroll
        for (int q = 0; q < 4; ++q) dp[q] = fmaf(G[(i0 + q) * KC + lane + 32 * r], z, dp[q]);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = i0 + q;
        const float den = warp_sum(dp[q]) + eps;
        float n0 = 0.f, n1 = 0.f, dv = 0.f;
        if (i < nvalid) {
          const float g0 = gs[i * kDv + lane], g1 = gs[i * kDv + 32 + lane];
          const float go = warp_sum(g0 * (a[q][0] / den) + g1 * (a[q][1] / den));
          n0 = g0 / den;
          n1 = g1 / den;
          dv = -go / den;
        }
        dn[i * kSP + lane] = n0;
        dn[i * kSP + 32 + lane] = n1;
        if (lane == 0) dd[i] = dv;
      }
    }
    __syncthreads();
    accumulate_gt<KC>(G, dn, kSP, dd, acc, zacc);  // [dVt | dZ] += gamma_Q^T [dn | dd]
    float b[4][RK];                                // dgamma_Q = [Vt | Z] [dn | dd]
    rows_times_image_t<KC>(dn, kSP, S, i0, b);
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int r = 0; r < RK; ++r) b[q][r] = fmaf(dd[i0 + q], Z[lane + 32 * r], b[q][r]);
    softmax_backward_rows<KC>(G, i0, b);
    __syncthreads();  // every warp is done with gamma_Q
    store_dl_rows<KC>(b, i0, nvalid, K, G, dlq + ((size_t)unit * N + t0) * K);
    __syncthreads();
    dx_tile_kc<IO, KC>(xs, G, nvalid, wpair + (size_t)h * K * kD, K, gs, dQ + ((size_t)unit * N + t0) * kD);
  }
  if (dsplits > 0)
    store_gt<KC>(dstate + ((size_t)unit * dsplits + blockIdx.x) * npairs, K, acc, zacc, 0);
  else
    store_gt<KC>(dstate + unit * npairs, K, acc, zacc, 1);
}

// Key side: grid (splits, B*H).  Pushes [dVt | dZ] back through the write: dV, dK and dl_K.  Warp w owns
// tile rows 4w .. 4w + 3.  dlk holds gamma_K on entry (the write kernel's copy) and dl_K on exit.
template <typename IO, int KC>
__global__ void __launch_bounds__(kThreads) simt_bwd_key_kernel(const IO* __restrict__ Kx, const IO* __restrict__ V,
                                                                const float2* __restrict__ wpair, int H, int N, int K,
                                                                int seg_tiles,
                                                                const float* __restrict__ dstate,
                                                                float* dlk, IO* __restrict__ dK, IO* __restrict__ dV) {
  constexpr int RK = KC / 32;
  extern __shared__ float sm[];
  float* dS = sm;             // [KC][kSP]  dVt image
  float* dZ = dS + KC * kSP;  // [KC]
  float* xs = dZ + KC;        // [T][64]   key rows
  float* vs = xs + T * kD;    // [T][64]   value rows, then the dx parameter stage
  float* G = vs + T * kDv;    // [T][KC]   gamma_K, then dl_K
  const int unit = blockIdx.y, h = unit % H, split = blockIdx.x;
  const int lane = threadIdx.x & 31, i0 = 4 * (threadIdx.x >> 5);
  load_state_image<KC>(dstate + unit * (size_t)K * kStateCols, K, dS, dZ);
  const int tiles = (N + T - 1) / T;
  const int tb = split * seg_tiles, te = min(tiles, tb + seg_tiles);
  for (int t = tb; t < te; ++t) {
    const int t0 = t * T, nvalid = min(T, N - t0);
    __syncthreads();
    load_rows<IO>(Kx + (size_t)unit * N * kD, t0, nvalid, xs);
    load_rows<IO>(V + (size_t)unit * N * kDv, t0, nvalid, vs);
    load_tile_rows<KC>(dlk + ((size_t)unit * N + t0) * K, nvalid, K, G);  // gamma_K, stored by the write
    __syncthreads();
    {  // dv = dVt^T gamma_K
      float a[4][2];
      rows_times_image<KC>(G, dS, i0, a);
      IO* dv_out = dV + ((size_t)unit * N + t0) * kDv;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (i0 + q < nvalid) {
          st_io<IO>(dv_out + (i0 + q) * kDv + lane, a[q][0]);
          st_io<IO>(dv_out + (i0 + q) * kDv + 32 + lane, a[q][1]);
        }
    }
    float b[4][RK];  // dgamma_K = [dVt | dZ] [v | 1]
    rows_times_image_t<KC>(vs, kDv, dS, i0, b);
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int r = 0; r < RK; ++r) b[q][r] += dZ[lane + 32 * r];
    softmax_backward_rows<KC>(G, i0, b);
    __syncwarp();  // the warp's reads of its own gamma_K rows are done
    store_dl_rows<KC>(b, i0, nvalid, K, G, dlk + ((size_t)unit * N + t0) * K);
    __syncthreads();
    dx_tile_kc<IO, KC>(xs, G, nvalid, wpair + (size_t)h * K * kD, K, vs, dK + ((size_t)unit * N + t0) * kD);
  }
}

// ---- causal backward.  S_i = sum_{j <= i} gamma_Kj [v_j | 1] (running state), u_i = [G_i / den_i |
// -(G_i . O_i) / den_i], R_j = sum_{i >= j} gamma_Qi u_i^T (suffix sum of the queries' contributions):
//   dgamma_Qi = S_i u_i,   dgamma_Kj = R_j [v_j | 1],   dv_j = R_j[:, :dv]^T gamma_Kj.
// Chunked like the forward: segment aggregates and an exclusive scan give S at each segment start; the
// query pass walks its segment forward (intra-tile terms masked to j <= i) and leaves the segment's
// aggregate of gamma_Q u^T; an exclusive suffix scan gives R after each segment; the key pass walks its
// segment backward.

// Loads `n` valid rows (of 64) starting at row `r0` of a [rows][64] matrix into dst[T][ld] as float32;
// rows past `n` are zero.
template <typename IO>
__device__ __forceinline__ void load_rows_ld(const IO* __restrict__ src, int r0, int n, float* dst, int ld) {
  for (int i = threadIdx.x; i < T * kD; i += blockDim.x) {
    const int r = i / kD, c = i % kD;
    dst[r * ld + c] = r < n ? ld_io<IO>(src + (size_t)(r0 + r) * kD + c) : 0.f;
  }
}

// In-tile products of the causal backward for the warp's rows i0 .. i0 + 3 (lane = j), zero for j > i:
//   A_ij = gamma_Qi . gamma_Kj (GQ row stride KC, GK row stride KC + 4) into A[T][T],
//   W_ij = dn_i . v_j + dd_i (dn, vs row stride kSP) into W[T][T].
template <int KC>
__device__ __forceinline__ void causal_tile_A(const float* GQ, const float* GK, int i0, float* A) {
  constexpr int KG = KC + 4;
  const int lane = threadIdx.x & 31;
  float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
  for (int k = 0; k < KC; k += 4) {
    const float4 g = *reinterpret_cast<const float4*>(GK + lane * KG + k);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 f = *reinterpret_cast<const float4*>(GQ + (i0 + q) * KC + k);
      a[q] = fmaf(f.x, g.x, fmaf(f.y, g.y, fmaf(f.z, g.z, fmaf(f.w, g.w, a[q]))));
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) A[(i0 + q) * T + lane] = lane <= i0 + q ? a[q] : 0.f;
}

__device__ __forceinline__ void causal_tile_W(const float* dn, const float* dd, const float* vs, int i0, float* W) {
  const int lane = threadIdx.x & 31;
  float w[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) w[q] = dd[i0 + q];
#pragma unroll 2
  for (int c = 0; c < kDv; c += 4) {
    const float4 v = *reinterpret_cast<const float4*>(vs + lane * kSP + c);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 f = *reinterpret_cast<const float4*>(dn + (i0 + q) * kSP + c);
      w[q] = fmaf(f.x, v.x, fmaf(f.y, v.y, fmaf(f.z, v.z, fmaf(f.w, v.w, w[q]))));
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) W[(i0 + q) * T + lane] = lane <= i0 + q ? w[q] : 0.f;
}

// S[k][c] += sum_i G[i][k] B[i][c], Z[k] += sum_i G[i][k] b_i (b_i = bz[i], or 1 where bz is null) over one
// tile: a state image updated in place, warp w owning components w KC / 8 .. + KC / 8 (G row stride LDG).
template <int KC, int LDG>
__device__ __forceinline__ void add_gt_to_image(const float* G, const float* B, int ldb, const float* bz, float* S,
                                                float* Z) {
  constexpr int KW = KC / 8;
  const int lane = threadIdx.x & 31, k0 = (threadIdx.x >> 5) * KW;
  float z = 0.f;
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    float acc[KW];
#pragma unroll
    for (int q = 0; q < KW; ++q) acc[q] = 0.f;
#pragma unroll 2
    for (int i = 0; i < T; ++i) {
      const float bv = B[i * ldb + 32 * e + lane];
      const float* g = G + i * LDG + k0;
#pragma unroll
      for (int q = 0; q < KW; q += 4) {
        const float4 g4 = *reinterpret_cast<const float4*>(g + q);
        acc[q] = fmaf(g4.x, bv, acc[q]);
        acc[q + 1] = fmaf(g4.y, bv, acc[q + 1]);
        acc[q + 2] = fmaf(g4.z, bv, acc[q + 2]);
        acc[q + 3] = fmaf(g4.w, bv, acc[q + 3]);
      }
      if (e == 0 && lane < KW) z = fmaf(g[lane], bz ? bz[i] : 1.f, z);
    }
#pragma unroll
    for (int q = 0; q < KW; ++q) S[(k0 + q) * kSP + 32 * e + lane] += acc[q];
  }
  if (lane < KW) Z[k0 + lane] += z;
}

// Query side: grid (segments, B*H).  S starts at agg[unit][seg] (scanned) and follows the segment's tiles;
// writes u, gamma_Q (for the key side), dl_Q, dQ and the segment aggregate sum_i gamma_Qi u_i^T into
// bagg[unit][seg].  gamma_K comes from the aggregate pass (dlk).  Warp w owns tile rows 4w .. 4w + 3.
template <typename IO, int KC>
__global__ void __launch_bounds__(kThreads) simt_bwd_causal_query_kernel(
    const IO* __restrict__ Q, const IO* __restrict__ V, const IO* __restrict__ dO, float* params,
    const float2* __restrict__ wpair, int H, int N, int K, int seg_tiles, int P, const float* agg, float eps,
    float* bagg, float* uglob, float* gq, const float* dlk, float* dlq, IO* __restrict__ dQ) {
  constexpr int RK = KC / 32, KG = KC + 4;
  extern __shared__ float sm[];
  float* S = sm;              // [KC][kSP]  running state image
  float* Z = S + KC * kSP;    // [KC]
  float* xq = Z + KC;         // [T][64]    query rows
  float* gs = xq + T * kD;    // [T][64]    dO rows, then the dx parameter stage
  float* vs = gs + T * kDv;   // [T][kSP]   value rows
  float* dn = vs + T * kSP;   // [T][kSP]   dO / den
  float* dd = dn + T * kSP;   // [T]        -(dO . O) / den
  float* GQ = dd + T;         // [T][KC]    gamma_Q, then dl_Q
  float* GK = GQ + T * KC;    // [T][KG]    gamma_K
  float* A = GK + T * KG;     // [T][T]
  float* W = A + T * T;       // [T][T]
  const int unit = blockIdx.y, h = unit % H, seg = blockIdx.x;
  const int lane = threadIdx.x & 31, i0 = 4 * (threadIdx.x >> 5);
  const SimtParams Pp = params_at(params, H, K);
  const size_t npairs = (size_t)K * kStateCols;
  load_state_image<KC>(agg + ((size_t)unit * P + seg) * npairs, K, S, Z);
  float bacc[KC / 8][2], bz = 0.f;
#pragma unroll
  for (int q = 0; q < KC / 8; ++q) bacc[q][0] = bacc[q][1] = 0.f;
  const int tiles = (N + T - 1) / T;
  const int tb = seg * seg_tiles, te = min(tiles, tb + seg_tiles);
  for (int t = tb; t < te; ++t) {
    const int t0 = t * T, nvalid = min(T, N - t0);
    const size_t row0 = (size_t)unit * N + t0;
    __syncthreads();
    load_rows<IO>(Q + (size_t)unit * N * kD, t0, nvalid, xq);
    load_rows<IO>(dO + (size_t)unit * N * kDv, t0, nvalid, gs);
    load_rows_ld<IO>(V + (size_t)unit * N * kDv, t0, nvalid, vs, kSP);
    load_tile_rows<KC, KG>(dlk + row0 * K, nvalid, K, GK);
    __syncthreads();
    gamma_tile_kc<KC, 2>(xq, nvalid, Pp, h, K, GQ);
    store_rows<KC>(GQ, nvalid, K, gq + row0 * K);
    {  // A, then [num | den] = gamma_Q [S | Z] + sum_{j <= i} A_ij [v_j | 1], then u = [dn | dd]
      causal_tile_A<KC>(GQ, GK, i0, A);
      __syncwarp();
      float a[4][2], dp[4];
      rows_times_image<KC>(GQ, S, i0, a);
#pragma unroll
      for (int q = 0; q < 4; ++q) dp[q] = A[(i0 + q) * T + lane];
#pragma unroll
      for (int r = 0; r < RK; ++r) {
        const float z = Z[lane + 32 * r];
#pragma unroll
        for (int q = 0; q < 4; ++q) dp[q] = fmaf(GQ[(i0 + q) * KC + lane + 32 * r], z, dp[q]);
      }
#pragma unroll 4
      for (int j = 0; j < T; ++j) {
        const float v0 = vs[j * kSP + lane], v1 = vs[j * kSP + 32 + lane];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float aij = A[(i0 + q) * T + j];
          a[q][0] = fmaf(aij, v0, a[q][0]);
          a[q][1] = fmaf(aij, v1, a[q][1]);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = i0 + q;
        const float den = warp_sum(dp[q]) + eps;
        float n0 = 0.f, n1 = 0.f, dv = 0.f;
        if (i < nvalid) {
          const float g0 = gs[i * kDv + lane], g1 = gs[i * kDv + 32 + lane];
          const float go = warp_sum(g0 * (a[q][0] / den) + g1 * (a[q][1] / den));
          n0 = g0 / den;
          n1 = g1 / den;
          dv = -go / den;
          float* ug = uglob + (row0 + i) * kStateCols;
          ug[lane] = n0;
          ug[32 + lane] = n1;
          if (lane == 0) ug[kDv] = dv;
        }
        dn[i * kSP + lane] = n0;
        dn[i * kSP + 32 + lane] = n1;
        if (lane == 0) dd[i] = dv;
      }
    }
    __syncthreads();
    accumulate_gt<KC>(GQ, dn, kSP, dd, bacc, bz);  // segment aggregate of gamma_Q u^T
    causal_tile_W(dn, dd, vs, i0, W);
    __syncwarp();
    float b[4][RK];  // dgamma_Q = [S | Z] u + sum_{j <= i} W_ij gamma_Kj
    rows_times_image_t<KC>(dn, kSP, S, i0, b);
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int r = 0; r < RK; ++r) b[q][r] = fmaf(dd[i0 + q], Z[lane + 32 * r], b[q][r]);
#pragma unroll 4
    for (int j = 0; j < T; ++j) {
      float g[RK];
#pragma unroll
      for (int r = 0; r < RK; ++r) g[r] = GK[j * KG + lane + 32 * r];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float wij = W[(i0 + q) * T + j];
#pragma unroll
        for (int r = 0; r < RK; ++r) b[q][r] = fmaf(wij, g[r], b[q][r]);
      }
    }
    softmax_backward_rows<KC>(GQ, i0, b);
    __syncthreads();  // every warp is done with S, Z and gamma_Q
    add_gt_to_image<KC, KG>(GK, vs, kSP, nullptr, S, Z);  // S += gamma_K^T [V | 1] over the tile
    store_dl_rows<KC>(b, i0, nvalid, K, GQ, dlq + row0 * K);
    __syncthreads();
    dx_tile_kc<IO, KC>(xq, GQ, nvalid, wpair + (size_t)h * K * kD, K, gs, dQ + row0 * kD);
  }
  store_gt<KC>(bagg + ((size_t)unit * P + seg) * npairs, K, bacc, bz, 0);
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
// walked last to first; gamma_Q and u come from the query side, gamma_K from the aggregate pass (dlk, which
// holds dl_K on exit); writes dK and dV.  Warp w owns tile rows 4w .. 4w + 3 (as queries in the in-tile
// products, as keys after them).
template <typename IO, int KC>
__global__ void __launch_bounds__(kThreads) simt_bwd_causal_key_kernel(
    const IO* __restrict__ Kx, const IO* __restrict__ V, const float2* __restrict__ wpair, int H, int N, int K,
    int seg_tiles, int P, const float* bagg, const float* uglob, const float* gq, float* dlk, IO* __restrict__ dK,
    IO* __restrict__ dV) {
  constexpr int RK = KC / 32, KG = KC + 4;
  extern __shared__ float sm[];
  float* R = sm;              // [KC][kSP]  running suffix image
  float* Rz = R + KC * kSP;   // [KC]
  float* xs = Rz + KC;        // [T][64]    key rows
  float* vs = xs + T * kD;    // [T][kSP]   value rows, then the dx parameter stage
  float* dn = vs + T * kSP;   // [T][kSP]   u rows (dv part)
  float* dd = dn + T * kSP;   // [T]        u rows (normaliser part)
  float* GQ = dd + T;         // [T][KC]    gamma_Q
  float* GK = GQ + T * KC;    // [T][KG]    gamma_K, then dl_K
  float* A = GK + T * KG;     // [T][T]
  float* W = A + T * T;       // [T][T]
  const int unit = blockIdx.y, h = unit % H, seg = blockIdx.x;
  const int lane = threadIdx.x & 31, i0 = 4 * (threadIdx.x >> 5);
  const size_t npairs = (size_t)K * kStateCols;
  load_state_image<KC>(bagg + ((size_t)unit * P + seg) * npairs, K, R, Rz);
  const int tiles = (N + T - 1) / T;
  const int tb = seg * seg_tiles, te = min(tiles, tb + seg_tiles);
  for (int t = te - 1; t >= tb; --t) {
    const int t0 = t * T, nvalid = min(T, N - t0);
    const size_t row0 = (size_t)unit * N + t0;
    __syncthreads();
    load_rows<IO>(Kx + (size_t)unit * N * kD, t0, nvalid, xs);
    load_rows_ld<IO>(V + (size_t)unit * N * kDv, t0, nvalid, vs, kSP);
    load_tile_rows<KC>(gq + row0 * K, nvalid, K, GQ);
    load_tile_rows<KC, KG>(dlk + row0 * K, nvalid, K, GK);
    for (int p = threadIdx.x; p < T * kStateCols; p += blockDim.x) {
      const int i = p / kStateCols, c = p % kStateCols;
      const float u = i < nvalid ? uglob[row0 * kStateCols + p] : 0.f;
      if (c < kDv) dn[i * kSP + c] = u; else dd[i] = u;
    }
    __syncthreads();
    causal_tile_A<KC>(GQ, GK, i0, A);
    causal_tile_W(dn, dd, vs, i0, W);
    __syncthreads();
    float b[4][RK];  // dgamma_Kj = R [v_j | 1] + sum_{i >= j} W_ij gamma_Qi
    rows_times_image_t<KC>(vs, kSP, R, i0, b);
#pragma unroll
    for (int q = 0; q < 4; ++q)
#pragma unroll
      for (int r = 0; r < RK; ++r) b[q][r] += Rz[lane + 32 * r];
    float a[4][2];  // dv_j = R^T gamma_Kj + sum_{i >= j} A_ij dn_i
    rows_times_image<KC, KG>(GK, R, i0, a);
#pragma unroll 4
    for (int i = 0; i < T; ++i) {
      float g[RK];
#pragma unroll
      for (int r = 0; r < RK; ++r) g[r] = GQ[i * KC + lane + 32 * r];
      const float d0 = dn[i * kSP + lane], d1 = dn[i * kSP + 32 + lane];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float wij = W[i * T + i0 + q], aij = A[i * T + i0 + q];
#pragma unroll
        for (int r = 0; r < RK; ++r) b[q][r] = fmaf(wij, g[r], b[q][r]);
        a[q][0] = fmaf(aij, d0, a[q][0]);
        a[q][1] = fmaf(aij, d1, a[q][1]);
      }
    }
    IO* dv_out = dV + row0 * kDv;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (i0 + q < nvalid) {
        st_io<IO>(dv_out + (i0 + q) * kDv + lane, a[q][0]);
        st_io<IO>(dv_out + (i0 + q) * kDv + 32 + lane, a[q][1]);
      }
    softmax_backward_rows<KC, KG>(GK, i0, b);
    __syncthreads();  // every warp is done with R, Rz, gamma_Q and the value rows
    add_gt_to_image<KC, KC>(GQ, dn, kSP, dd, R, Rz);  // R += gamma_Q^T u over the tile
    store_dl_rows<KC, KG>(b, i0, nvalid, K, GK, dlk + row0 * K);
    __syncthreads();
    dx_tile_kc<IO, KC, KG>(xs, GK, nvalid, wpair + (size_t)h * K * kD, K, vs, dK + row0 * kD);
  }
}

// Parameter-gradient sums: grid (ceil(K / 32), H, ctas).  The rows of head h (queries then keys of every
// batch entry, 2 B N in all) are split into ranges of rows_per_cta; a CTA walks its range in tiles of at
// most T rows that stay within one (side, batch entry) and loads the next tile into registers while it
// works on the current one.  The sums are taken in the expanded form, so that one thread's row loads
// serve several components: thread (half, kq, dg) accumulates, for components 4 kq .. 4 kq + 3 of the
// block and dims 4 dg .. 4 dg + 3, sum dl_k x_d, sum dl_k x_d^2 and sum dl_k over the rows of its half
// (even or odd rows of each tile).  The halves are added in a fixed order at the end, and then
//   sum dl_k (x_d - mu_kd)   = sum dl_k x_d - mu_kd sum dl_k,
//   sum dl_k (x_d - mu_kd)^2 = sum dl_k x_d^2 - 2 mu_kd sum dl_k x_d + mu_kd^2 sum dl_k,
// added into pacc[h][k][d][2] (and sum dl_k into pb[h][k]); with zstride > 0 (the deterministic reduction
// mode) stored instead into the slice of its row range, at pacc + blockIdx.z * zstride (and pb + ...).
// In float32 the expansion loses at most about (|x| / |x - mu|)^2 ulps to cancellation.
template <typename IO>
__global__ void __launch_bounds__(kThreads) simt_bwd_param_kernel(const IO* __restrict__ Q, const IO* __restrict__ Kx,
                                                                  const float* __restrict__ mu, const float* dlq,
                                                                  const float* dlk, int B, int H, int N, int K,
                                                                  long long rows_per_cta, float* pacc, float* pb,
                                                                  size_t zstride) {
  __shared__ __align__(16) float xs[T * kD];
  __shared__ __align__(16) float ds[T * 32];
  __shared__ float part[128 * 36];  // the odd-row half's sums, handed to the even-row half
  const int h = blockIdx.y, k0 = blockIdx.x * 32;
  const int dg = threadIdx.x & 15, kq = (threadIdx.x >> 4) & 7, half = threadIdx.x >> 7;
  const int fi = threadIdx.x >> 3, fc = threadIdx.x & 7;  // fetch: row fi, dims 8 fc .. 8 fc + 7, dl 4 fc .. 4 fc + 3
  const long long total = 2LL * B * N;
  const long long r0 = (long long)blockIdx.z * rows_per_cta, r1 = min(total, r0 + rows_per_cta);
  float a1[4][4], a2[4][4], bs[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    bs[j] = 0.f;
#pragma unroll
    for (int q = 0; q < 4; ++q) a1[j][q] = a2[j][q] = 0.f;
  }
  // the tile starting at virtual row rb: its row count, and this thread's share of x and dl
  auto fetch = [&](long long rb, int& n, float (&xv)[8], float (&dv)[4]) {
    const long long sb = rb / N;  // side * B + b
    const int n0 = (int)(rb - sb * N), side = (int)(sb / B), b = (int)(sb % B);
    n = (int)min((long long)min(T, N - n0), r1 - rb);
    const size_t row = ((size_t)b * H + h) * N + n0 + fi;
    const bool ok = fi < n;
#pragma unroll
    for (int t = 0; t < 8; ++t) xv[t] = 0.f;
    if (ok) load8<IO>((side == 0 ? Q : Kx) + row * kD + 8 * fc, xv);
    const float* dsrc = (side == 0 ? dlq : dlk) + row * K;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      const int kk = k0 + 4 * fc + t;
      dv[t] = ok && kk < K ? dsrc[kk] : 0.f;
    }
  };
  int n = 0;
  float xv[8], dv[4];
  if (r0 < r1) fetch(r0, n, xv, dv);
  for (long long rb = r0; rb < r1;) {
    const int ncur = n;
    __syncthreads();  // the previous tile's readers are done
    *reinterpret_cast<float4*>(xs + fi * kD + 8 * fc) = make_float4(xv[0], xv[1], xv[2], xv[3]);
    *reinterpret_cast<float4*>(xs + fi * kD + 8 * fc + 4) = make_float4(xv[4], xv[5], xv[6], xv[7]);
    *reinterpret_cast<float4*>(ds + fi * 32 + 4 * fc) = make_float4(dv[0], dv[1], dv[2], dv[3]);
    __syncthreads();
    rb += ncur;
    if (rb < r1) fetch(rb, n, xv, dv);  // in flight while this tile is summed
#pragma unroll 2
    for (int i = half; i < ncur; i += 2) {
      const float4 x4 = *reinterpret_cast<const float4*>(xs + i * kD + 4 * dg);
      const float4 d4 = *reinterpret_cast<const float4*>(ds + i * 32 + 4 * kq);
      const float x[4] = {x4.x, x4.y, x4.z, x4.w}, d[4] = {d4.x, d4.y, d4.z, d4.w};
      float x2[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) x2[q] = x[q] * x[q];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        bs[j] += d[j];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          a1[j][q] = fmaf(d[j], x[q], a1[j][q]);
          a2[j][q] = fmaf(d[j], x2[q], a2[j][q]);
        }
      }
    }
  }
  // the odd-row half hands its sums over; the even-row half adds them (a fixed order) and finishes
  const int slot = threadIdx.x & 127;
  if (half == 1) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      part[(j * 9) * 128 + slot] = bs[j];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        part[(j * 9 + 1 + q) * 128 + slot] = a1[j][q];
        part[(j * 9 + 5 + q) * 128 + slot] = a2[j][q];
      }
    }
  }
  __syncthreads();
  if (half == 1) return;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    bs[j] += part[(j * 9) * 128 + slot];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      a1[j][q] += part[(j * 9 + 1 + q) * 128 + slot];
      a2[j][q] += part[(j * 9 + 5 + q) * 128 + slot];
    }
  }
  const size_t zo = zstride > 0 ? (size_t)blockIdx.z * zstride : 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int k = k0 + 4 * kq + j;
    if (k >= K) break;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int d = 4 * dg + q;
      const float m = __ldg(mu + ((size_t)h * K + k) * kD + d);
      const float c1 = fmaf(-m, bs[j], a1[j][q]);                        // sum dl (x - mu)
      const float c2 = fmaf(m * m, bs[j], fmaf(-2.f * m, a1[j][q], a2[j][q]));  // sum dl (x - mu)^2
      float* dst = pacc + zo + (((size_t)h * K + k) * kD + d) * 2;
      if (zstride > 0) {
        *reinterpret_cast<float2*>(dst) = make_float2(c1, c2);
      } else {
        atomicAdd(dst, c1);
        atomicAdd(dst + 1, c2);
      }
    }
    if (dg == 0) {
      if (zstride > 0)
        pb[zo + (size_t)h * K + k] = bs[j];
      else
        atomicAdd(pb + (size_t)h * K + k, bs[j]);
    }
  }
}

// The parameter gradients from the sums; Z slices of sums zstride floats apart are added in slice order
// first (Z = 1: the sums themselves).
__global__ void simt_bwd_param_finish_kernel(const float* __restrict__ sigma2, const float* pacc, const float* pb, int H,
                                             int K, int Z, size_t zstride, float* dmu, float* dsigma2,
                                             float* dlog_pi) {
  const size_t n = (size_t)H * K * kD;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    float s1 = pacc[2 * i], s2 = pacc[2 * i + 1], b = pb[i / kD];
    for (int z = 1; z < Z; ++z) {
      const size_t zo = (size_t)z * zstride;
      s1 += pacc[zo + 2 * i];
      s2 += pacc[zo + 2 * i + 1];
      b += pb[zo + i / kD];
    }
    const float w = 1.0f / sigma2[i];
    dmu[i] = s1 * w;
    dsigma2[i] = 0.5f * w * (s2 * w - b);
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

// Two block-wide reductions at once (a0 over one value, a1 over another); both max or both sum.
__device__ __forceinline__ float2 block_reduce2(float a0, float a1, bool is_max, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float u0 = __shfl_xor_sync(0xffffffffu, a0, o), u1 = __shfl_xor_sync(0xffffffffu, a1, o);
    a0 = is_max ? fmaxf(a0, u0) : a0 + u0;
    a1 = is_max ? fmaxf(a1, u1) : a1 + u1;
  }
  if (lane == 0) {
    red[2 * warp] = a0;
    red[2 * warp + 1] = a1;
  }
  __syncthreads();
  float2 r = make_float2(red[0], red[1]);
  for (int w = 1; w < nw; ++w) {
    r.x = is_max ? fmaxf(r.x, red[2 * w]) : r.x + red[2 * w];
    r.y = is_max ? fmaxf(r.y, red[2 * w + 1]) : r.y + red[2 * w + 1];
  }
  __syncthreads();  // red is reused by the next reduction
  return r;
}

// Folded parameters of one head for the decode kernel, in the order of its shared memory:
// mu_t [kD][K + 1], w_t = 1 / sigma2 [kD][K + 1] (row stride K + 1: conflict-free along either index),
// c [K] = log pi_k - 1/2 sum_d log sigma2_kd; rounded up to a multiple of 4 floats.
__host__ __device__ constexpr size_t decode_head_floats(int K) {
  return (2 * (size_t)kD * (K + 1) + (size_t)K + 3) / 4 * 4;
}

// Shared-memory floats of the decode kernel for K components: the state, one head's folded parameters,
// and the per-token rows and scratch.
__host__ __device__ constexpr size_t decode_smem_floats(int K) {
  return (size_t)K * kStateCols + decode_head_floats(K) + (size_t)K + 2 * kD + kDv + 4 * kDv + 64;
}

// The fold for every head, once per decode call: into `folded`, decode_head_floats(K) floats per head.
// Grid (ceil(K / 32), H): a block reads 32 components' rows of mu and sigma2 (coalesced), transposes them
// through shared memory and writes 32-component runs of every dim row.
__global__ void __launch_bounds__(256) simt_decode_fold_kernel(const float* __restrict__ mu,
                                                               const float* __restrict__ sigma2,
                                                               const float* __restrict__ log_pi, int H, int K,
                                                               float* __restrict__ folded) {
  __shared__ float tm[kD][33], tw[kD][33];
  tc::dep_launch_next();  // the decode kernel starts its state copy meanwhile
  const int h = blockIdx.y, k0 = blockIdx.x * 32, t = threadIdx.x;
  const int r = t >> 3, c0 = 8 * (t & 7);  // component k0 + r, dims c0 .. c0 + 7
  const size_t ld = (size_t)K + 1;
  float* f = folded + (size_t)h * decode_head_floats(K);
  float lg = 0.f;
  if (k0 + r < K) {
    const size_t o = ((size_t)h * K + k0 + r) * kD + c0;
    const float4 m0 = __ldg(reinterpret_cast<const float4*>(mu + o));
    const float4 m1 = __ldg(reinterpret_cast<const float4*>(mu + o) + 1);
    const float4 s0 = __ldg(reinterpret_cast<const float4*>(sigma2 + o));
    const float4 s1 = __ldg(reinterpret_cast<const float4*>(sigma2 + o) + 1);
    const float mv[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
    const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      tm[c0 + q][r] = mv[q];
      tw[c0 + q][r] = 1.0f / sv[q];
      lg += logf(sv[q]);
    }
  }
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) lg += __shfl_xor_sync(0xffffffffu, lg, o);  // the 8 threads of a component
  if ((t & 7) == 0 && k0 + r < K) f[2 * (size_t)kD * ld + k0 + r] = __ldg(log_pi + (size_t)h * K + k0 + r) - 0.5f * lg;
  __syncthreads();
  const int kk = t & 31;
  if (k0 + kk < K) {
#pragma unroll
    for (int j = t >> 5; j < kD; j += 8) {
      f[(size_t)j * ld + k0 + kk] = tm[j][kk];
      f[(size_t)kD * ld + (size_t)j * ld + k0 + kk] = tw[j][kk];
    }
  }
}

template <typename IO>
__global__ void __launch_bounds__(kDecodeThreads) simt_decode_kernel(const IO* __restrict__ Q, const IO* __restrict__ Kx,
                                                                     const IO* __restrict__ V,
                                                                     const float* __restrict__ folded, int H, int Tn,
                                                                     int K, float* __restrict__ state, float eps,
                                                                     IO* __restrict__ out, Ctrl* ctrl) {
  extern __shared__ __align__(16) float sm[];
  __shared__ uint64_t bar;
  __shared__ tc::Abort ab;
  const int bh = blockIdx.x, h = bh % H, k = threadIdx.x;
  const int ld = K + 1;                      // row stride of the parameter tables (conflict-free both ways)
  const size_t hs = decode_head_floats(K);
  float* S = sm;                             // [K][kStateCols]
  float* mu_s = S + (size_t)K * kStateCols;  // [kD][K + 1]  } one head's folded parameters,
  float* w_s = mu_s + (size_t)kD * ld;       // [kD][K + 1]  } copied as they lie in `folded`
  float* c_s = w_s + (size_t)kD * ld;        // [K]          }
  float* gq = mu_s + hs;                     // [K]
  float* xq = gq + K;                        // [kD]
  float* xk = xq + kD;                       // [kD]
  float* xv = xk + kD;                       // [kDv]
  float* part = xv + kDv;                    // [4][kDv]
  float* red = part + 4 * kDv;               // [64]
  float* st = state + (size_t)bh * K * kStateCols;
  const float* fh = folded + (size_t)h * hs;
  const int n_state = K * kStateCols;
  // state and parameters: bulk copies (TMA engine, 16 KB pieces on one mbarrier) when both start on a
  // 16-byte boundary (K a multiple of 4; the sizes then are multiples of 16 bytes too), else plain loads
  const uint32_t state_bytes = (uint32_t)n_state * 4u, param_bytes = (uint32_t)hs * 4u;
  const bool vec = ((reinterpret_cast<uintptr_t>(st) | reinterpret_cast<uintptr_t>(fh)) & 15) == 0 && (K & 3) == 0;
  if (vec) {
    if (threadIdx.x == 0) {
      ab.flag = 0;
      tc::mbar_init(&bar, 1);
      tc::mbar_fence_init();
      tc::mbar_expect_tx(&bar, state_bytes + param_bytes);
      constexpr uint32_t kPiece = 16384;
      for (uint32_t o = 0; o < state_bytes; o += kPiece)  // the state does not depend on the fold
        tc::bulk_load(reinterpret_cast<char*>(S) + o, reinterpret_cast<const char*>(st) + o,
                      state_bytes - o < kPiece ? state_bytes - o : kPiece, &bar);
      tc::dep_wait();  // the fold of this call is complete
      for (uint32_t o = 0; o < param_bytes; o += kPiece)
        tc::bulk_load(reinterpret_cast<char*>(mu_s) + o, reinterpret_cast<const char*>(fh) + o,
                      param_bytes - o < kPiece ? param_bytes - o : kPiece, &bar);
      if (!tc::wait_bounded(&bar, 0, &ab, ctrl, 0x20u, 1000000000ull)) {
        ab.flag = 1;
        tc::Abort again{0};  // give the copies in flight another bounded while to land before leaving
        tc::wait_bounded(&bar, 0, &again, ctrl, 0x20u, 1000000000ull);
      }
    }
    tc::dep_wait();
    __syncthreads();
    if (ab.flag) return;  // the copy did not land in time: the error word says so; the state is untouched
  } else {
    tc::dep_wait();
#pragma unroll 8
    for (int i = threadIdx.x; i < n_state; i += blockDim.x) S[i] = __ldcg(st + i);
#pragma unroll 8
    for (int i = threadIdx.x; i < (int)hs; i += blockDim.x) mu_s[i] = __ldg(fh + i);
    __syncthreads();
  }
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
    const float2 mx = block_reduce2(lk, lq, true, red);
    const float ek = k < K ? expf(lk - mx.x) : 0.f, eq = k < K ? expf(lq - mx.y) : 0.f;
    const float2 sm2 = block_reduce2(ek, eq, false, red);
    const float sk = sm2.x, sq = sm2.y;
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
  if (vec) {
    tc::fence_async_smem();  // this thread's shared-memory writes become visible to the bulk copy
    __syncthreads();
    if (threadIdx.x == 0) {
      constexpr uint32_t kPiece = 16384;
      for (uint32_t o = 0; o < state_bytes; o += kPiece)
        tc::bulk_store(reinterpret_cast<char*>(st) + o, reinterpret_cast<const char*>(S) + o,
                       state_bytes - o < kPiece ? state_bytes - o : kPiece);
      tc::bulk_commit();
      tc::bulk_wait_all();
    }
  } else {
    __syncthreads();
#pragma unroll 8
    for (int i = threadIdx.x; i < n_state; i += blockDim.x) st[i] = S[i];
  }
}

}  // namespace

// Workspace of the backward pass.  Bidirectional: control block | parameters | Vt|Z | dVt|dZ |
// parameter sums | dl of the queries | dl of the keys (gamma_K until the key side) | (1 / sigma2,
// mu / sigma2) pairs (the three accumulators contiguous, zeroed together).  Causal: control block |
// parameters | segment aggregates of the keys (scanned: S at each segment start) | segment aggregates of
// the queries' gamma_Q u^T (suffix-scanned: R after each segment) | parameter sums | u rows | dl of the
// queries | dl of the keys (gamma_K until the key side) | pairs | gamma_Q.
// Deterministic reduction mode, after these: the per-CTA partials of Vt|Z and of dVt|dZ (bidirectional
// only; one area, used by the two in turn) and pz slices of the parameter sums (pacc then pb, one slice
// per range of rows).
constexpr int kParamSlices = 16;
// bf16 I/O, bidirectional: last, the workspace of the tensor-core state write and responsibilities
// (off_tc), which compute the state and every key's gamma_K in place of the float32 write pass.
struct BwdPlan {
  size_t off_params, off_state, off_dstate, off_pacc, off_pb, off_u, off_dlq, off_dlk, off_wpair, off_gq;
  size_t off_part, off_ppart, pstride, off_tc, total;  // pstride: floats per slice of the parameter sums
  int splits, seg_tiles, tiles, pz;
  bool det, tc_front;
};
BwdPlan bwd_plan(const gma_problem_t& p, bool causal, bool det) {
  BwdPlan b{};
  const SimtPlan sp = simt_plan(p, causal ? GMA_OP_CAUSAL : GMA_OP_BIDIR);
  const size_t BH = (size_t)p.B * p.H, npairs = (size_t)p.K * kStateCols;
  b.tiles = sp.tiles;
  b.splits = sp.splits;
  b.seg_tiles = sp.seg_tiles;
  if (causal) {  // one wave of the causal query / key kernels: two CTAs per SM, one when K > 128
    const int units = kc_class(p.K) <= 128 ? kTargetUnits : kTargetUnits / 2;
    const int nt = b.tiles > 0 ? b.tiles : 1;
    int want = units / (int)(BH > 0 ? BH : 1);
    want = want < 1 ? 1 : (want > nt ? nt : want);
    b.seg_tiles = cdiv(nt, want);
    b.splits = cdiv(nt, b.seg_tiles);
  }
  const size_t nstate = causal ? BH * b.splits * npairs : BH * npairs;
  b.off_params = sp.off_params;
  b.off_state = align_up(sp.off_params + ((size_t)2 * p.H * kD * p.K + (size_t)p.H * p.K) * sizeof(float));
  b.off_dstate = b.off_state + nstate * sizeof(float);
  b.off_pacc = b.off_dstate + nstate * sizeof(float);
  b.off_pb = b.off_pacc + (size_t)p.H * p.K * kD * 2 * sizeof(float);
  b.off_u = align_up(b.off_pb + (size_t)p.H * p.K * sizeof(float));
  b.off_dlq = align_up(b.off_u + (causal ? BH * p.N * kStateCols * sizeof(float) : 0));
  b.off_dlk = align_up(b.off_dlq + BH * p.N * p.K * sizeof(float));
  b.off_wpair = align_up(b.off_dlk + BH * p.N * p.K * sizeof(float));
  b.off_gq = align_up(b.off_wpair + (size_t)p.H * p.K * kD * sizeof(float2));
  b.total = align_up(b.off_gq + (causal ? BH * p.N * p.K * sizeof(float) : 0));
  b.det = det;
  b.pz = 1;
  b.pstride = ((size_t)p.H * p.K * (2 * kD + 1) + 3) / 4 * 4;  // 16-byte slices (float2 stores)
  b.off_part = b.off_ppart = b.total;
  if (det) {
    b.off_ppart = align_up(b.off_part + (causal ? 0 : BH * b.splits * npairs * sizeof(float)));
    const long long rows = 2LL * p.B * p.N;
    b.pz = (int)std::max(1LL, std::min<long long>(kParamSlices, (rows + T - 1) / T));
    b.total = align_up(b.off_ppart + (size_t)b.pz * b.pstride * sizeof(float));
  }
  b.tc_front = p.dtype == GMA_BF16 && !causal && p.N > 0 && tc_available();
  b.off_tc = b.total;
  if (b.tc_front)
    b.total = align_up(b.off_tc + std::max(tc_plan(p, GMA_OP_CAUSAL_STATE, det).total,
                                           tc_plan(p, GMA_OP_RESPONSIBILITIES, det).total));
  return b;
}

// Splits of a per-(b, h) tile loop that fill the GPU in one wave: the resident CTAs of `func` on every SM,
// shared among the B*H units.
gma_status_t fill_splits(const void* func, size_t smem, int BH, int tiles, int* splits, int* seg_tiles) {
  int dev = 0, nsm = 0, occ = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, func, kThreads, smem) != cudaSuccess)
    return cuda_fail("occupancy query", cudaSuccess, func);
  const int nt = tiles > 0 ? tiles : 1;
  int want = nsm * (occ > 0 ? occ : 1) / (BH > 0 ? BH : 1);
  want = want < 1 ? 1 : (want > nt ? nt : want);
  *seg_tiles = cdiv(nt, want);
  *splits = cdiv(nt, *seg_tiles);
  return GMA_OK;
}

// Write phase / segment aggregates (simt_write_kernel) for the KC class of K.
template <typename IO, int KC>
gma_status_t launch_write_kc(int splits, int BH, cudaStream_t st, const IO* Kx, const IO* V, float* params, int H,
                             int N, int K, int seg_tiles, float* state, int atomic, float* gout = nullptr,
                             size_t state_lim = ~(size_t)0) {
  const size_t sm = (size_t)(T * kD + T * kDv + T * KC) * sizeof(float);
  const auto kfn = simt_write_kernel<IO, KC>;
  if (set_smem_optin((const void*)kfn, (int)sm, 1) != GMA_OK) return GMA_ERR_CUDA;
  GMA_LAUNCH("simt_write", kfn, dim3(splits, BH), kThreads, sm, st, Kx, V, params, H, N, K, seg_tiles, splits,
             state, atomic, gout, state_lim);
  return check_launch("launch simt_write", (const void*)kfn);
}

template <typename IO>
gma_status_t launch_write(int splits, int BH, cudaStream_t st, const IO* Kx, const IO* V, float* params, int H, int N,
                          int K, int seg_tiles, float* state, int atomic, size_t lim) {
  switch (kc_class(K)) {
    case 32: return launch_write_kc<IO, 32>(splits, BH, st, Kx, V, params, H, N, K, seg_tiles, state, atomic, nullptr, lim);
    case 64: return launch_write_kc<IO, 64>(splits, BH, st, Kx, V, params, H, N, K, seg_tiles, state, atomic, nullptr, lim);
    case 128:
      return launch_write_kc<IO, 128>(splits, BH, st, Kx, V, params, H, N, K, seg_tiles, state, atomic, nullptr, lim);
    default:
      return launch_write_kc<IO, 256>(splits, BH, st, Kx, V, params, H, N, K, seg_tiles, state, atomic, nullptr, lim);
  }
}

// Bidirectional backward after the parameter fold: write (Vt | Z), the query side, the key side; each
// loop sized to fill the GPU.
// part (the deterministic reduction mode, else null): the write and the query side store per-CTA partials
// there, with the plan's splits, and each is summed in a fixed order.
template <typename IO, int KC>
gma_status_t backward_bidir_kc(const gma_problem_t& p, const BwdPlan& b, const IO* Q, const IO* Kx, const IO* V,
                               const IO* dO, IO* dQ, IO* dK, IO* dV, float* params, const float2* wpair, float* state,
                               float* dstate, float* dlq, float* dlk, float* part, cudaStream_t st) {
  const bool write = !b.tc_front;  // else the state and gamma_K are already in place
  const int BH = p.B * p.H, K = p.K, tiles = cdiv(p.N, T), npairs = K * kStateCols;
  int splits = 1, seg = 1;
  const size_t sm_w = (size_t)(T * kD + T * kDv + T * KC) * sizeof(float);
  const auto wfn = simt_write_kernel<IO, KC>;
  if (!write) {
  } else if (part) {
    if (gma_status_t e = launch_write_kc<IO, KC>(b.splits, BH, st, Kx, V, params, p.H, p.N, K, b.seg_tiles, part, 0,
                                                 dlk))
      return e;
    GMA_LAUNCH("simt_state_sum", simt_state_sum_kernel, dim3(cdiv(npairs, 256), BH), 256, 0, st, part, b.splits,
               npairs, state, ~(size_t)0, ~(size_t)0);
    if (gma_status_t e = check_launch("launch simt_state_sum", (const void*)simt_state_sum_kernel)) return e;
  } else {
    if (gma_status_t e = fill_splits((const void*)wfn, sm_w, BH, tiles, &splits, &seg)) return e;
    if (gma_status_t e = launch_write_kc<IO, KC>(splits, BH, st, Kx, V, params, p.H, p.N, K, seg, state, 1, dlk))
      return e;
  }
  const size_t sm_q = (size_t)(KC * kSP + KC + T * kD + T * kDv + T * kSP + T + T * KC) * sizeof(float);
  const auto qfn = simt_bwd_query_kernel<IO, KC>;
  if (set_smem_optin((const void*)qfn, (int)sm_q, 5) != GMA_OK) return GMA_ERR_CUDA;
  if (part) {
    splits = b.splits;
    seg = b.seg_tiles;
  } else if (gma_status_t e = fill_splits((const void*)qfn, sm_q, BH, tiles, &splits, &seg)) {
    return e;
  }
  GMA_LAUNCH("simt_bwd_query", qfn, dim3(splits, BH), kThreads, sm_q, st, Q, dO, params, wpair, p.H, p.N, K, seg,
             state, p.eps, part ? part : dstate, part ? splits : 0, dlq, dQ, b.tc_front ? 1 : 0);
  if (gma_status_t e = check_launch("launch simt_bwd_query", (const void*)qfn)) return e;
  if (part) {
    GMA_LAUNCH("simt_state_sum", simt_state_sum_kernel, dim3(cdiv(npairs, 256), BH), 256, 0, st, part, splits, npairs,
               dstate, ~(size_t)0, ~(size_t)0);
    if (gma_status_t e = check_launch("launch simt_state_sum", (const void*)simt_state_sum_kernel)) return e;
  }
  const size_t sm_k = (size_t)(KC * kSP + KC + T * kD + T * kDv + T * KC) * sizeof(float);
  const auto kkfn = simt_bwd_key_kernel<IO, KC>;
  if (set_smem_optin((const void*)kkfn, (int)sm_k, 6) != GMA_OK) return GMA_ERR_CUDA;
  if (gma_status_t e = fill_splits((const void*)kkfn, sm_k, BH, tiles, &splits, &seg)) return e;
  GMA_LAUNCH("simt_bwd_key", kkfn, dim3(splits, BH), kThreads, sm_k, st, Kx, V, wpair, p.H, p.N, K, seg,
             dstate, dlk, dK, dV);
  return check_launch("launch simt_bwd_key", (const void*)kkfn);
}

// Causal backward after the parameter fold: segment aggregates (+ every key's gamma_K into dlk), scan,
// query side (u, gamma_Q, dl_Q, dQ, the queries' segment aggregates), suffix scan, key side (dl_K, dK, dV).
template <typename IO, int KC>
gma_status_t backward_causal_kc(const gma_problem_t& p, const BwdPlan& b, const IO* Q, const IO* Kx, const IO* V,
                                const IO* dO, IO* dQ, IO* dK, IO* dV, float* params, const float2* wpair, float* state,
                                float* dstate, float* urows, float* gq, float* dlq, float* dlk, cudaStream_t st) {
  constexpr int KG = KC + 4;
  const int BH = p.B * p.H, K = p.K, npairs = K * kStateCols;
  if (gma_status_t e = launch_write_kc<IO, KC>(b.splits, BH, st, Kx, V, params, p.H, p.N, K, b.seg_tiles, state, 0,
                                               dlk))
    return e;
  GMA_LAUNCH("simt_scan", simt_scan_kernel, dim3(cdiv(npairs, 256), BH), 256, 0, st, state, b.splits, npairs,
             ~(size_t)0);
  if (gma_status_t e = check_launch("launch simt_scan", (const void*)simt_scan_kernel)) return e;
  const size_t sm_q =
      (size_t)(KC * kSP + KC + T * kD + T * kDv + 2 * T * kSP + T + T * KC + T * KG + 2 * T * T) * sizeof(float);
  const auto qfn = simt_bwd_causal_query_kernel<IO, KC>;
  if (set_smem_optin((const void*)qfn, (int)sm_q, 7) != GMA_OK) return GMA_ERR_CUDA;
  GMA_LAUNCH("simt_bwd_causal_query", qfn, dim3(b.splits, BH), kThreads, sm_q, st, Q, V, dO, params, wpair, p.H, p.N,
             K, b.seg_tiles, b.splits, state, p.eps, dstate, urows, gq, dlk, dlq, dQ);
  if (gma_status_t e = check_launch("launch simt_bwd_causal_query", (const void*)qfn)) return e;
  GMA_LAUNCH("simt_rscan", simt_rscan_kernel, dim3(cdiv(npairs, 256), BH), 256, 0, st, dstate, b.splits, npairs);
  if (gma_status_t e = check_launch("launch simt_rscan", (const void*)simt_rscan_kernel)) return e;
  const size_t sm_k =
      (size_t)(KC * kSP + KC + T * kD + 2 * T * kSP + T + T * KC + T * KG + 2 * T * T) * sizeof(float);
  const auto kfn = simt_bwd_causal_key_kernel<IO, KC>;
  if (set_smem_optin((const void*)kfn, (int)sm_k, 8) != GMA_OK) return GMA_ERR_CUDA;
  GMA_LAUNCH("simt_bwd_causal_key", kfn, dim3(b.splits, BH), kThreads, sm_k, st, Kx, V, wpair, p.H, p.N, K,
             b.seg_tiles, b.splits, dstate, urows, gq, dlk, dK, dV);
  return check_launch("launch simt_bwd_causal_key", (const void*)kfn);
}

template <typename IO>
gma_status_t backward_typed(const gma_problem_t& p, bool causal, const IO* Q, const IO* Kx, const IO* V,
                            const float* mu, const float* sigma2, const float* log_pi, const IO* dO, IO* dQ, IO* dK,
                            IO* dV, float* dmu, float* dsigma2, float* dlog_pi, void* ws, cudaStream_t st, bool det) {
  const BwdPlan b = bwd_plan(p, causal, det);
  char* base = (char*)ws;
  float* params = (float*)(base + b.off_params);
  float* state = (float*)(base + b.off_state);
  float* dstate = (float*)(base + b.off_dstate);
  float* pacc = (float*)(base + b.off_pacc);
  float* pb = (float*)(base + b.off_pb);
  float* urows = (float*)(base + b.off_u);
  float* dlq = (float*)(base + b.off_dlq);
  float* dlk = (float*)(base + b.off_dlk);
  float2* wpair = (float2*)(base + b.off_wpair);
  float* gq = (float*)(base + b.off_gq);
  float* part = det && !causal ? (float*)(base + b.off_part) : nullptr;
  float* ppart = (float*)(base + b.off_ppart);
  const int K = p.K;
  // bidirectional: zero Vt|Z, dVt|dZ and the parameter sums; causal: the parameter sums (the segment
  // aggregates are stored whole)
  float* zero = causal ? pacc : state;
  const size_t zero_n = (b.off_u - (causal ? b.off_pacc : b.off_state)) / sizeof(float);
  GMA_LAUNCH("simt_prep", simt_prep_kernel, 148, 256, 0, st, mu, sigma2, log_pi, p.H, K, params, (Ctrl*)base, zero,
             zero_n, wpair);
  if (gma_status_t e = check_launch("launch simt_prep", (const void*)simt_prep_kernel)) return e;
  if (b.tc_front) {
    // bf16 I/O, bidirectional: the tensor-core kernels write the state [B*H][K][65] and every key's
    // gamma_K [B*H][N][K] (where the key side expects them), reporting into this workspace's error word
    void* tws = base + b.off_tc;
    if (gma_status_t e = tc_run(p, GMA_OP_CAUSAL_STATE, p.N, nullptr, Kx, V, mu, sigma2, log_pi, state, tws, st, false,
                                det, (Ctrl*)base))
      return e;
    if (gma_status_t e = tc_run(p, GMA_OP_RESPONSIBILITIES, p.N, Kx, nullptr, nullptr, mu, sigma2, log_pi, dlk, tws, st,
                                false, det, (Ctrl*)base))
      return e;
    if (gma_status_t e = tc_run(p, GMA_OP_RESPONSIBILITIES, p.N, Q, nullptr, nullptr, mu, sigma2, log_pi, dlq, tws, st,
                                false, det, (Ctrl*)base))  // gamma_Q, read by the query side
      return e;
  }
  int pz_used = 1;  // slices of the parameter sums the finish adds up (1: the zeroed or atomic sums)
  if (p.N > 0) {
    if (causal) {
      gma_status_t e;
      switch (kc_class(K)) {
        case 32:
          e = backward_causal_kc<IO, 32>(p, b, Q, Kx, V, dO, dQ, dK, dV, params, wpair, state, dstate, urows, gq, dlq,
                                         dlk, st);
          break;
        case 64:
          e = backward_causal_kc<IO, 64>(p, b, Q, Kx, V, dO, dQ, dK, dV, params, wpair, state, dstate, urows, gq, dlq,
                                         dlk, st);
          break;
        case 128:
          e = backward_causal_kc<IO, 128>(p, b, Q, Kx, V, dO, dQ, dK, dV, params, wpair, state, dstate, urows, gq, dlq,
                                          dlk, st);
          break;
        default:
          e = backward_causal_kc<IO, 256>(p, b, Q, Kx, V, dO, dQ, dK, dV, params, wpair, state, dstate, urows, gq, dlq,
                                          dlk, st);
      }
      if (e != GMA_OK) return e;
    } else {
      gma_status_t e;
      switch (kc_class(K)) {
        case 32:
          e = backward_bidir_kc<IO, 32>(p, b, Q, Kx, V, dO, dQ, dK, dV, params, wpair, state, dstate, dlq, dlk, part,
                                        st);
          break;
        case 64:
          e = backward_bidir_kc<IO, 64>(p, b, Q, Kx, V, dO, dQ, dK, dV, params, wpair, state, dstate, dlq, dlk, part,
                                        st);
          break;
        case 128:
          e = backward_bidir_kc<IO, 128>(p, b, Q, Kx, V, dO, dQ, dK, dV, params, wpair, state, dstate, dlq, dlk, part,
                                        st);
          break;
        default:
          e = backward_bidir_kc<IO, 256>(p, b, Q, Kx, V, dO, dQ, dK, dV, params, wpair, state, dstate, dlq, dlk, part,
                                        st);
      }
      if (e != GMA_OK) return e;
    }
    // parameter sums: one wave of CTAs over the 2 B N rows of every head (deterministic: the plan's pz
    // ranges of rows, each stored into its own slice)
    const auto pfn = simt_bwd_param_kernel<IO>;
    const long long rows = 2LL * p.B * p.N;
    long long ctas = b.pz;
    if (!det) {
      int dev = 0, nsm = 0, occ = 0;
      if (cudaGetDevice(&dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, pfn, kThreads, 0) != cudaSuccess)
        return cuda_fail("occupancy query", cudaSuccess, (const void*)pfn);
      const int per_head = cdiv(K, 32) * p.H;
      ctas = (long long)nsm * (occ > 0 ? occ : 1) / per_head;
      ctas = ctas < 1 ? 1 : (ctas > 65535 ? 65535 : ctas);
    }
    long long rows_per_cta = (rows + ctas - 1) / ctas;
    rows_per_cta = (rows_per_cta + T - 1) / T * T;
    const int zc = (int)((rows + rows_per_cta - 1) / rows_per_cta);  // <= pz when det
    const dim3 grid_p(cdiv(K, 32), p.H, (unsigned)zc);
    if (det) {
      pacc = ppart;
      pb = ppart + (size_t)p.H * K * kD * 2;
    }
    GMA_LAUNCH("simt_bwd_param", pfn, grid_p, kThreads, 0, st, Q, Kx, mu, dlq, dlk, p.B, p.H, p.N, K, rows_per_cta,
               pacc, pb, det ? b.pstride : (size_t)0);
    if (gma_status_t e = check_launch("launch simt_bwd_param", (const void*)simt_bwd_param_kernel<IO>)) return e;
    if (det) pz_used = zc;
  }
  GMA_LAUNCH("simt_bwd_param_finish", simt_bwd_param_finish_kernel, 148, 256, 0, st, sigma2, pacc, pb, p.H, K, pz_used,
             b.pstride, dmu, dsigma2, dlog_pi);
  return check_launch("launch simt_bwd_param_finish", (const void*)simt_bwd_param_finish_kernel);
}

size_t simt_backward_bytes(const gma_problem_t& p, bool causal, bool det) { return bwd_plan(p, causal, det).total; }

gma_status_t simt_backward(const gma_problem_t& p, bool causal, const void* Q, const void* K, const void* V,
                           const float* mu, const float* sigma2, const float* log_pi, const void* dO, void* dQ,
                           void* dK, void* dV, float* dmu, float* dsigma2, float* dlog_pi, void* ws, cudaStream_t st,
                           bool det) {
  if (p.dtype == GMA_F32)
    return backward_typed<float>(p, causal, (const float*)Q, (const float*)K, (const float*)V, mu, sigma2, log_pi,
                                 (const float*)dO, (float*)dQ, (float*)dK, (float*)dV, dmu, dsigma2, dlog_pi, ws, st,
                                 det);
  using bf = __nv_bfloat16;
  return backward_typed<bf>(p, causal, (const bf*)Q, (const bf*)K, (const bf*)V, mu, sigma2, log_pi, (const bf*)dO,
                            (bf*)dQ, (bf*)dK, (bf*)dV, dmu, dsigma2, dlog_pi, ws, st, det);
}

// Decode T new tokens per (b, h) from `state` (float32 [B*H][K][dv + 1], updated in place).  Two launches:
// the parameter fold of every head into the workspace (after its control block, whose error word stays as
// the caller left it), then one CTA per (b, h).
size_t simt_decode_bytes(const gma_problem_t& p) {
  return align_up(sizeof(Ctrl)) + align_up((size_t)p.H * decode_head_floats(p.K) * sizeof(float));
}

gma_status_t simt_decode_fold(const gma_problem_t& p, const float* mu, const float* sigma2, const float* log_pi,
                              void* ws, cudaStream_t st) {
  float* folded = (float*)((char*)ws + align_up(sizeof(Ctrl)));
  GMA_LAUNCH("simt_decode_fold", simt_decode_fold_kernel, dim3(cdiv(p.K, 32), p.H), 256, 0, st, mu, sigma2, log_pi,
             p.H, p.K, folded);
  return check_launch("launch simt_decode_fold", (const void*)simt_decode_fold_kernel);
}

// The decode kernel copies the state before its grid dependency wait: launched as a dependent only of
// the fold (which itself waited for everything earlier, so the previous decode's state writes are
// complete), otherwise as a plain launch.
gma_status_t simt_decode_run(const gma_problem_t& p, const void* Q, const void* K, const void* V, float* state,
                             void* out, void* ws, bool dependent, cudaStream_t st) {
  const size_t smem = decode_smem_floats(p.K) * sizeof(float);
  const int BH = p.B * p.H;
  const float* folded = (const float*)((const char*)ws + align_up(sizeof(Ctrl)));
  if (p.dtype == GMA_F32) {
    if (set_smem_optin((const void*)simt_decode_kernel<float>, (int)smem, 4) != GMA_OK) return GMA_ERR_CUDA;
    if (dependent)
      GMA_LAUNCH_DEPENDENT("simt_decode", simt_decode_kernel<float>, BH, kDecodeThreads, smem, st, (const float*)Q,
                           (const float*)K, (const float*)V, folded, p.H, p.N, p.K, state, p.eps, (float*)out,
                           (Ctrl*)ws);
    else
      GMA_LAUNCH("simt_decode", simt_decode_kernel<float>, BH, kDecodeThreads, smem, st, (const float*)Q,
                 (const float*)K, (const float*)V, folded, p.H, p.N, p.K, state, p.eps, (float*)out, (Ctrl*)ws);
    return check_launch("launch simt_decode", (const void*)simt_decode_kernel<float>);
  }
  using bf = __nv_bfloat16;
  if (set_smem_optin((const void*)simt_decode_kernel<bf>, (int)smem, 4) != GMA_OK) return GMA_ERR_CUDA;
  if (dependent)
    GMA_LAUNCH_DEPENDENT("simt_decode", simt_decode_kernel<bf>, BH, kDecodeThreads, smem, st, (const bf*)Q,
                         (const bf*)K, (const bf*)V, folded, p.H, p.N, p.K, state, p.eps, (bf*)out, (Ctrl*)ws);
  else
    GMA_LAUNCH("simt_decode", simt_decode_kernel<bf>, BH, kDecodeThreads, smem, st, (const bf*)Q, (const bf*)K,
               (const bf*)V, folded, p.H, p.N, p.K, state, p.eps, (bf*)out, (Ctrl*)ws);
  return check_launch("launch simt_decode", (const void*)simt_decode_kernel<bf>);
}

gma_status_t simt_decode(const gma_problem_t& p, const void* Q, const void* K, const void* V, const float* mu,
                         const float* sigma2, const float* log_pi, float* state, void* out, void* ws,
                         cudaStream_t st) {
  if (gma_status_t e = simt_decode_fold(p, mu, sigma2, log_pi, ws, st)) return e;
  return simt_decode_run(p, Q, K, V, state, out, ws, true, st);
}

namespace {

template <typename IO>
gma_status_t run_typed(const gma_problem_t& p, gma_op_t op, int Nk, const IO* Q, const IO* Kx, const IO* V,
                       const float* mu, const float* sigma2, const float* log_pi, void* out, void* ws,
                       cudaStream_t st, bool det) {
  const SimtPlan pl = simt_plan(p, op, det);
  char* base = (char*)ws;
  // extents of the state section and of the partial states (checked by the bounds-check build)
  const size_t state_lim = (pl.off_agg - pl.off_state) / sizeof(float), part_lim = (pl.total - pl.off_agg) / sizeof(float);
  Ctrl* ctrl = (Ctrl*)base;
  float* params = (float*)(base + pl.off_params);
  float* state = (float*)(base + pl.off_state);
  const int BH = p.B * p.H, K = p.K;
  const int npairs = K * kStateCols;
  const bool write_only = op == GMA_OP_CAUSAL_STATE;  // state of all N keys, copied to `out`
  if (write_only) op = GMA_OP_BIDIR;
  const size_t zero_n = op == GMA_OP_BIDIR ? (size_t)BH * npairs : 0;
  GMA_LAUNCH("simt_prep", simt_prep_kernel, 148, 256, 0, st, mu, sigma2, log_pi, p.H, K, params, ctrl, state, zero_n,
             nullptr);
  if (cudaGetLastError() != cudaSuccess) return GMA_ERR_CUDA;
  if (p.N == 0 && !write_only) return GMA_OK;
  const size_t sm_gamma = (size_t)(T * kD + T * K) * sizeof(float);
  if (op == GMA_OP_RESPONSIBILITIES) {
    if (set_smem_optin((const void*)simt_resp_kernel<IO>, (int)sm_gamma, 0) != GMA_OK) return GMA_ERR_CUDA;
    GMA_LAUNCH("simt_resp", simt_resp_kernel<IO>, dim3(pl.tiles, BH), kThreads, sm_gamma, st, Q, params, p.H, p.N, K, (float*)out);
    return cudaGetLastError() == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
  }
  if (op == GMA_OP_BIDIR) {
    // write over the Nk keys (its own split plan; the workspace layout does not depend on N)
    if (Nk > 0) {
      gma_problem_t pk = p;
      pk.N = Nk;
      const SimtPlan plk = simt_plan(pk, op);
      if (pl.det) {  // each write CTA stores its own state; one fixed-order sum per element
        float* part = (float*)(base + pl.off_agg);
        if (gma_status_t e =
                launch_write<IO>(plk.splits, BH, st, Kx, V, params, p.H, Nk, K, plk.seg_tiles, part, 0, part_lim))
          return e;
        GMA_LAUNCH("simt_state_sum", simt_state_sum_kernel, dim3(cdiv(npairs, 256), BH), 256, 0, st, part, plk.splits,
                   npairs, state, part_lim, state_lim);
        if (gma_status_t e = check_launch("launch simt_state_sum", (const void*)simt_state_sum_kernel)) return e;
      } else if (gma_status_t e = launch_write<IO>(plk.splits, BH, st, Kx, V, params, p.H, Nk, K, plk.seg_tiles,
                                                   state, 1, state_lim)) {
        return e;
      }
    }
    if (write_only) {  // the accumulator already has the public state layout [B*H][K][dv + 1]
      if (cudaMemcpyAsync(out, state, (size_t)BH * npairs * sizeof(float), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return cuda_fail("copy state");
      return GMA_OK;
    }
    const size_t sm_read = (size_t)(T * kD + T * K + T * kStateCols) * sizeof(float);
    if (set_smem_optin((const void*)simt_read_kernel<IO>, (int)sm_read, 2) != GMA_OK) return GMA_ERR_CUDA;
    GMA_LAUNCH("simt_read", simt_read_kernel<IO>, dim3(pl.tiles, BH), kThreads, sm_read, st, Q, params, p.H, p.N, K,
               state, p.eps, (IO*)out, state_lim);
    return cudaGetLastError() == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
  }
  // causal
  if (gma_status_t e = launch_write<IO>(pl.splits, BH, st, Kx, V, params, p.H, p.N, K, pl.seg_tiles, state, 0, state_lim))
    return e;
  GMA_LAUNCH("simt_scan", simt_scan_kernel, dim3(cdiv(npairs, 256), BH), 256, 0, st, state, pl.splits, npairs, state_lim);
  if (cudaGetLastError() != cudaSuccess) return GMA_ERR_CUDA;
  const size_t sm_causal = (size_t)(npairs + T * kD + T * kDv + 2 * T * K + T * T + T * kStateCols) * sizeof(float);
  if (set_smem_optin((const void*)simt_causal_kernel<IO>, (int)sm_causal, 3) != GMA_OK) return GMA_ERR_CUDA;
  GMA_LAUNCH("simt_causal", simt_causal_kernel<IO>, dim3(pl.splits, BH), kThreads, sm_causal, st, Q, Kx, V, params, p.H,
             p.N, K, pl.seg_tiles, pl.splits, state, p.eps, (IO*)out, state_lim);
  return cudaGetLastError() == cudaSuccess ? GMA_OK : GMA_ERR_CUDA;
}

}  // namespace

#ifdef GMA_BOUNDS_CHECK
gma_status_t simt_bounds_io(unsigned long long* h, bool clear) { return bounds_record_io(h, clear); }
#else
gma_status_t simt_bounds_io(unsigned long long*, bool) { return GMA_ERR_UNSUPPORTED; }
#endif

SimtPlan simt_plan(const gma_problem_t& p, gma_op_t op, bool det) {
  SimtPlan pl{};
  pl.det = det;
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
  pl.off_agg = align_up(pl.off_state + state_bytes);
  size_t agg_bytes = 0;
  // the write's own plan over the key length: B*H * splits <= B*H * ceil(kTargetUnits / (B*H))
  if (det && (op == GMA_OP_BIDIR || op == GMA_OP_CROSS || op == GMA_OP_CAUSAL_STATE))
    agg_bytes = ((size_t)kTargetUnits + BH) * p.K * kStateCols * sizeof(float);
  pl.total = align_up(pl.off_agg + agg_bytes);
  return pl;
}

gma_status_t simt_run(const gma_problem_t& p, gma_op_t op, int Nk, const void* Q, const void* K, const void* V,
                      const float* mu, const float* sigma2, const float* log_pi, void* out, void* ws,
                      cudaStream_t stream, bool det) {
  if (p.dtype == GMA_F32)
    return run_typed<float>(p, op, Nk, (const float*)Q, (const float*)K, (const float*)V, mu, sigma2, log_pi, out, ws,
                            stream, det);
  return run_typed<__nv_bfloat16>(p, op, Nk, (const __nv_bfloat16*)Q, (const __nv_bfloat16*)K, (const __nv_bfloat16*)V,
                                  mu, sigma2, log_pi, out, ws, stream, det);
}

}  // namespace gma

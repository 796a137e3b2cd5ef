// gma_tc.cu -- bf16-I/O path of the GMA forward pass on the sm_103a tensor cores (tcgen05 + TMEM +
// TMA), one CTA per SM, warp-specialised.
//
// Method (Gaussian Mixture Attention pages, gist.science summaries):
//   "Core mechanism" item 1: gamma_ik = softmax_k(log pi_k + log N(x_i; mu_k, diag sigma2_k)).
//     The log-density is expanded into one dense contraction per 128-token tile,
//       L'_ik = [x_i^2 , x_i , 1] . [a_k ; b_k ; c'_k]                                   (fp16 operands)
//     with a = -1/2 sigma2^-1 log2(e) and b = -2 a mu rounded consistently (the expanded form is then
//     exactly a (x - mu')^2 for a mean within 2^-12 |mu| of mu) and the component constant
//     c'_k = (log pi_k - 1/2 sum_d log sigma2) log2(e) + sum_d a mu'^2 as one extra K-step (fp16 hi / lo
//     parts of c'/256 against a constant [256 | 1] block; the causal sweep adds it from a float32 table
//     instead), followed by a base-2 softmax over k held in registers.
//   "Core mechanism" item 2: write  [Vt | Z] = Gamma_K^T [V | 1]   (bf16 operands, fp32 TMEM accumulator)
//                            read   O = Gamma_Q Vt / (Gamma_Q Z + eps)
//   Keys are normalised before packing (bf16 gamma = e / s_j, 0 past N) and used with [V | 1] as loaded
//   and a constant 1 column, in the bidirectional write, the causal aggregates and the chunked sweep.
//   Gamma_Q stays unnormalised: the read divides by gamma~_i . (Z + eps) = gamma~_i . Z + eps s_i, which
//   is the same quotient, with eps added once to the Z column of the state operand, so no query row
//   needs its sum.  No responsibility goes to global memory except through the responsibilities entry.
//
// Roles per CTA (640 threads): warps 0-3 are control warps (TMA producer; one MMA-issuing thread per
// independent contraction, since a thread issuing tcgen05.mma waits about as long as the instruction
// runs; warp 1 also owns the TMEM columns), warps 4..19 are row warps: thread (q, part) owns token
// row 32q+lane of the tile and a quarter of its components / dimensions (TMEM lane quarter q = warp % 4,
// part = warpgroup - 1).  The control warps hand registers to the row warps with setmaxnreg.
#include <algorithm>
#include <cstdio>
#include <cstdlib>
#include <mutex>

#include "gma_tc_common.cuh"
#include "gma_trace.cuh"


namespace gma {
namespace {

using namespace tc;

constexpr int kTile = 128;
constexpr int kThreadsTc = 640;  // 5 warpgroups
constexpr int kRowWarp0 = 4;     // first row warp (warpgroups 1..4 are row warps)
constexpr int kParts = 4;        // row threads sharing one token row
// Register split (setmaxnreg): launch pool 640 x 96 = 61440 >= 128 x 56 + 512 x 104 = 60416, and per SM
// sub-partition (one control warp + four row warps) 32 x (56 + 4 x 104) = 15104 <= 16384.
constexpr uint32_t kCtrlRegs = 56, kRowRegs = 104;
// The causal sweep's row code needs 112: 128 x 32 + 512 x 112 = 61440, per SM sub-partition
// 32 x (32 + 4 x 112) = 15360 (its issuers use rolled loops to fit in 32).
constexpr uint32_t kCtrlRegsC = 32, kRowRegsC = 112;
constexpr int kRowWarps = 16;  // arrival count of the barriers the row warps signal
constexpr int kStCols = 80;  // state row: [Vt (64) | Z | 15 zero]
constexpr int kStRow = 68;   // row of the accumulated state in global memory: [Vt (64) | Z | 3 zero]
constexpr int kCTable = 256;  // c' entries per head (-inf past K)
constexpr int kTargetCtas = 152;
constexpr float kLog2e = 1.4426950408889634f;

// TMEM columns (512 allocated)
constexpr uint32_t kColLog = 0;    // logits, Kp columns (<= 256)
constexpr uint32_t kColAx = 256;   // [x^2 | x] fp16 operand, 64 columns
constexpr uint32_t kColAcc = 320;  // write: state accumulators 80 per 128-component block; read: O (80)
constexpr uint32_t kColOnes = 480; // [256 | 1] fp16 A columns of the constant step of the log-density contraction

// Bytes per head of the prepared B operand of the log-density contraction: the K-major W image
// (Kp rows x 256 B, two 64-element 128-byte-swizzle blocks) followed by the constant step (Kp rows x 32 B,
// 32-byte swizzle: c'/256 rounded to fp16 and the fp16 remainder, against A columns [256, 1]).
__host__ __device__ constexpr uint32_t w_head_bytes(int Kp) { return (uint32_t)Kp * 288u; }

__host__ __device__ constexpr uint32_t align1k(uint32_t x) { return (x + 1023u) & ~1023u; }

struct SmemLayout {
  uint32_t w, g, x, v, inv, sb, c, red, total;
};

// write kernel: W | G (MN-major Gamma~, MB x 32K) | X ring | V ring | INV atom | c' | exchange
__host__ __device__ inline SmemLayout write_layout(int Kp) {
  SmemLayout s{};
  const int MB = (Kp + 127) / 128;
  s.w = 0;
  s.g = align1k(w_head_bytes(Kp));
  s.x = s.g + MB * 32768;
  s.v = s.x + 2 * 16384;
  s.inv = s.v + 2 * 16384;
  s.sb = s.inv + 16384;
  s.c = s.sb;
  s.red = s.c;
  s.total = s.red + kParts * kTile * 8;
  return s;
}
// responsibilities kernel: W | X ring | exchange
__host__ __device__ inline SmemLayout read_layout(int Kp) {
  SmemLayout s{};
  s.w = 0;
  s.g = align1k(w_head_bytes(Kp));
  s.x = s.g;
  s.v = s.x;
  s.inv = s.x;
  s.sb = s.x + 2 * 16384;
  s.c = s.sb;
  s.red = s.c;
  s.total = s.red + kParts * kTile * 8;
  return s;
}

struct Bars {
  uint64_t w_full;
  uint64_t x_full[2], x_empty[2], v_empty[2];
  uint64_t ax_full, l_full, l_empty, g_full, g_empty;
  uint64_t g_fullq[4];  // write: Gamma rows of lane quarter q (tokens 32q .. 32q+31) stored
  uint64_t done, done_l;
  uint32_t tmem_base;
  Abort ab;
};

// Extents of the workspace sections and the output, as planned on the host (checked by the bounds-check
// debug build only): state / out / c in floats, w in bytes, flags in words.
struct TcLimits {
  size_t state, out, w, c, flags;
};

struct TcArgs {
  const uint8_t* w_img;  // [H][w_head_bytes(Kp)] swizzled fp16 B operand of the log-density contraction
  const float* cbias;    // [H][256] c'_k (log2 domain); -inf past K
  const uint32_t* range_flags;  // [H][32] non-zero where a block of the parameter fold saw an fp16 overflow
  float* state;          // [BH][Kp][68] (bidir: [Vt | Z | 0 0 0]) or [BH][splits][80][Kp] (causal aggregates, column-major)
  Ctrl* ctrl;
  void* out;             // read: O bf16 [BH][N][64]; responsibilities: gamma fp32 [BH][N][K]
  int H, N, K, Kp, tiles, seg_tiles, splits;
  float eps;
  uint64_t wait_ns;
  uint32_t fault;  // bit 0: the producer never loads the first X tile (bounded-wait test hook)
#ifdef GMA_BOUNDS_CHECK
  TcLimits lim;  // only the checked build carries (and reads) the extents
#endif
};

// ----------------------------------------------------------------------------------------------- prep
// a1: fold (mu, sigma2, log_pi) of every head into the swizzled fp16 W image and the 256-entry c'
// table (-inf past K); clear the error word (unless clear_err is 0: an earlier kernel of the same call
// cleared it and may have reported into it); zero `zero_n` floats of the write accumulator.
// grid (256 / 8, H), 128 threads: 16 threads per component, thread q of a component builds the 16-byte
// chunk of W elements 8q .. 8q+7 of that component's row (x^2 coefficients for q < 8, x coefficients
// after) with one store, and the q < 8 threads sum c'_k over their 8 dims.
__global__ void __launch_bounds__(128, 16) tc_prep_kernel(const float* __restrict__ mu, const float* __restrict__ sigma2,
                                                      const float* __restrict__ log_pi, int H, int K, int Kp,
                                                      uint8_t* w_img, float* cbias, Ctrl* ctrl, float* zero,
                                                      size_t zero_n, uint32_t* range_flags, int clear_err,
                                                      TcLimits lim) {
  // Launched as a dependent of whatever precedes it on the stream: nothing is read or written before that
  // grid has completed (it may produce the parameters, or still read the previous call's W image).  The
  // 32-register bound lets a CTA of this grid sit beside a running tensor-core CTA meanwhile.
  dep_launch_next();  // the main kernel sets itself up meanwhile and waits for this grid before reading
  dep_wait();
  if (threadIdx.x == 0) GMA_SPAN_AT(8);
  const int h = blockIdx.y, k = blockIdx.x * 8 + (threadIdx.x >> 4), q = threadIdx.x & 15;
  const int d0 = 8 * (q & 7);
  uint32_t w[4] = {0u, 0u, 0u, 0u};
  float term = 0.f;
  int bad = 0;
  if (k < K) {
    const float4* m4 = reinterpret_cast<const float4*>(mu + ((size_t)h * K + k) * kD + d0);
    const float4* s4 = reinterpret_cast<const float4*>(sigma2 + ((size_t)h * K + k) * kD + d0);
    const float4 ma = __ldg(m4), mb = __ldg(m4 + 1), sa = __ldg(s4), sb = __ldg(s4 + 1);
    const float m[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
    const float s2[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
    // Consistent rounding: a = fp16(-1/2 sigma2^-1 log2 e) first, then b = fp16(-2 a mu), and the constant
    // carries b^2 / (4 a) = a mu'^2 with mu' = b / (-2 a), so a x^2 + b x + a mu'^2 = a (x - mu')^2 exactly:
    // the expanded form is the centred one for a mean within 2^-12 |mu| of mu (and a variance within 2^-12
    // relative), instead of three large terms each rounded on its own that cancel near the best component.
    // Threads q < 8 hold a (x^2 coefficients of dims d0..d0+7) and sum log sigma2; threads q >= 8 hold b and
    // sum a mu'^2.
    float val[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float af = __half2float(__float2half_rn(-0.5f / s2[i] * kLog2e));
      if (q < 8) {
        val[i] = af;
        term += logf(s2[i]);
      } else {
        const float bf = __half2float(__float2half_rn(-2.0f * af * m[i]));
        val[i] = bf;
        term += (bf * bf) / (4.0f * af);  // a mu'^2 (<= 0)
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const __half2 p2 = __floats2half2_rn(val[2 * i], val[2 * i + 1]);  // exact: val is already fp16
      w[i] = *reinterpret_cast<const uint32_t*>(&p2);
      // fp16 overflow (sigma2 too small, |mu| / sigma2 too large) or a non-finite parameter
      if (!isfinite(val[2 * i]) || !isfinite(val[2 * i + 1])) bad = 1;
    }
  }
  if (k < Kp &&
      GMA_INB((size_t)h * w_head_bytes(Kp) + sw128_off(k, 8 * q, (uint32_t)Kp * 128) + 15, lim.w, 101))
    *reinterpret_cast<uint4*>(w_img + (size_t)h * w_head_bytes(Kp) + sw128_off(k, 8 * q, (uint32_t)Kp * 128)) =
        make_uint4(w[0], w[1], w[2], w[3]);
  // c'_k = log pi_k log2(e) + sum_d a mu'^2 - 1/2 log2(e) sum_d log sigma2 (the two partial sums above, kept
  // apart by the half of the component's 16 threads that formed them; the 16 are an aligned half-warp)
  float lsum = q < 8 ? term : 0.f, qsum = q < 8 ? 0.f : term;
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) {
    lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    qsum += __shfl_xor_sync(0xffffffffu, qsum, o);
  }
  const float cprime = k < K ? log_pi[(size_t)h * K + k] * kLog2e + qsum - 0.5f * kLog2e * lsum : -INFINITY;
  if (q == 0 && k < kCTable && GMA_INB((size_t)h * kCTable + k, lim.c, 102)) cbias[(size_t)h * kCTable + k] = cprime;
  if (q == 0 && k < Kp &&
      GMA_INB((size_t)h * w_head_bytes(Kp) + (size_t)Kp * 256 + (size_t)max(sw32_chunk(k, 0), sw32_chunk(k, 1)) + 15,
              lim.w, 103)) {
    // constant step of the contraction: [256 | 1] . [fp16(c'/256) | fp16(c' - 256 fp16(c'/256))] = c' to
    // about 2^-22 |c'| (-inf past K, so the padding components never win the row maximum)
    const __half hi = __float2half_rn(k < K ? cprime * (1.0f / 256.0f) : -INFINITY);
    const __half lo = __float2half_rn(k < K ? cprime - 256.0f * __half2float(hi) : 0.0f);
    if (k < K && (!isfinite(__half2float(hi)) || !isfinite(__half2float(lo)))) bad = 1;
    const __half2 hl = __halves2half2(hi, lo);
    uint8_t* cimg = w_img + (size_t)h * w_head_bytes(Kp) + (size_t)Kp * 256;
    *reinterpret_cast<uint4*>(cimg + sw32_chunk(k, 0)) = make_uint4(*reinterpret_cast<const uint32_t*>(&hl), 0u, 0u, 0u);
    *reinterpret_cast<uint4*>(cimg + sw32_chunk(k, 1)) = make_uint4(0u, 0u, 0u, 0u);
  }
  if (clear_err && blockIdx.x == 0 && h == 0 && threadIdx.x == 0) {
    ctrl->err = kErrNone;
    ctrl->err_site = 0;
  }
  // one flag per block, rewritten every call (so nothing needs clearing); the next kernel turns it
  // into the error word after this grid has completed
  const int any_bad = __syncthreads_or(bad);
  if (threadIdx.x == 0 && GMA_INB(blockIdx.y * gridDim.x + blockIdx.x, lim.flags, 104))
    range_flags[blockIdx.y * gridDim.x + blockIdx.x] = any_bad ? 1u : 0u;
  const size_t tid = ((size_t)blockIdx.y * gridDim.x + blockIdx.x) * blockDim.x + threadIdx.x;
  const size_t nth = (size_t)gridDim.x * gridDim.y * blockDim.x;
  for (size_t i = tid; i < zero_n; i += nth)
    if (GMA_INB(i, lim.state, 105)) zero[i] = 0.f;
  if (threadIdx.x == 0) GMA_SPAN_AT(9);
}

// ----------------------------------------------------------------------------------------------- shared pieces
// Row-thread context.  Shared-memory positions are 32-bit shared-window addresses; every 128-row SW128
// tile starts on a 1 KB boundary, so chunk c of a token row sits at (tile + rowsw) ^ (c << 4).
struct RowCtx {
  int warp, lane, q, part, row;  // row warps: q = TMEM lane quarter, part = component / dimension quarter
  uint32_t lane_base;            // TMEM address bits of this warp's lane quarter
  uint32_t rowsw;                // offset of chunk 0 of this token row in a 128-row SW128 tile
  uint32_t rowq;                 // offset of chunk 2 * part (this thread's 16 of the row's 64 elements)
  uint32_t red;                  // this row's slots in the exchange area (float2 [kParts][kTile])
  uint32_t bar;                  // named barrier of the row's four part threads (the warps of quarter q)
};

__device__ __forceinline__ RowCtx row_ctx(uint32_t red_area) {
  RowCtx r;
  r.warp = threadIdx.x >> 5;
  r.lane = threadIdx.x & 31;
  r.q = r.warp & 3;
  r.part = (r.warp - kRowWarp0) >> 2;
  r.row = r.q * 32 + r.lane;
  r.lane_base = (uint32_t)(r.q * 32) << 16;
  r.rowsw = (uint32_t)(r.row >> 3) * 1024u + (uint32_t)(r.row & 7) * 128u + ((uint32_t)(r.row & 7) << 4);
  r.rowq = r.rowsw ^ ((uint32_t)(2 * r.part) << 4);
  r.red = red_area + (uint32_t)r.row * 8u;
  r.bar = 1u + (uint32_t)r.q;
  return r;
}

// Row exchanges among the four part threads of a token row (the same lane of the four warps of one
// lane quarter, so one named barrier of 128 threads).  `slot` 0 / 4 selects the .x / .y float of the
// row's float2 slots.  Named barriers have no time limit, so every row warp executes every exchange of
// every tile, also after a failed wait; the caller only skips the work around them.
__device__ __forceinline__ float xchg_max(const RowCtx& rc, uint32_t slot, float mp) {
  sts32(rc.red + (uint32_t)rc.part * (kTile * 8) + slot, mp);
  named_bar_sync(rc.bar, 128);
  const float a = lds32(rc.red + slot), b = lds32(rc.red + kTile * 8 + slot);
  const float c = lds32(rc.red + 2 * kTile * 8 + slot), d = lds32(rc.red + 3 * kTile * 8 + slot);
  return fmaxf(fmaxf(a, b), fmaxf(c, d));
}
__device__ __forceinline__ float xchg_sum(const RowCtx& rc, uint32_t slot, float sp) {
  sts32(rc.red + (uint32_t)rc.part * (kTile * 8) + slot, sp);
  named_bar_sync(rc.bar, 128);
  const float a = lds32(rc.red + slot), b = lds32(rc.red + kTile * 8 + slot);
  const float c = lds32(rc.red + 2 * kTile * 8 + slot), d = lds32(rc.red + 3 * kTile * 8 + slot);
  return (a + b) + (c + d);
}

// Builds this thread's quarter (16 dims) of the [x^2 | x] fp16 operand row from the bf16 X tile at shared
// address `xtile` and stores it to TMEM (A operand of the log-density contraction, lane = token, two
// fp16 per 32-bit column).
__device__ __forceinline__ void transform_row(uint32_t xtile, const RowCtx& rc, uint32_t tmem,
                                              uint32_t col_ax = kColAx) {
  uint32_t sq[8], lin[8];
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    const uint4 v = lds128((xtile + rc.rowq) ^ (uint32_t)(jj << 4));
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float lo = __uint_as_float(w4[i] << 16), hi = __uint_as_float(w4[i] & 0xffff0000u);
      lin[jj * 4 + i] = pack_f16x2(lo, hi);
      sq[jj * 4 + i] = pack_f16x2(lo * lo, hi * hi);
    }
  }
  tmem_st8(tmem + rc.lane_base + col_ax + 8 * rc.part, sq);
  tmem_st8(tmem + rc.lane_base + col_ax + 32 + 8 * rc.part, lin);
}

// The same quarter of the operand row into shared memory at `adst` (1 KB aligned): the x^2 block, then
// the x block 16 KB on, each 128 rows of 64 fp16 in the 128-byte swizzle of the X tile, so a chunk keeps
// its position (K-major A of the log-density contraction).
__device__ __forceinline__ void transform_row_smem(uint32_t xtile, const RowCtx& rc, uint32_t adst) {
#pragma unroll
  for (int jj = 0; jj < 2; ++jj) {
    const uint32_t off = rc.rowq ^ (uint32_t)(jj << 4);
    const uint4 v = lds128(xtile + off);
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    uint32_t sq[4], lin[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float lo = __uint_as_float(w4[i] << 16), hi = __uint_as_float(w4[i] & 0xffff0000u);
      lin[i] = pack_f16x2(lo, hi);
      sq[i] = pack_f16x2(lo * lo, hi * hi);
    }
    sts128(adst + off, make_uint4(sq[0], sq[1], sq[2], sq[3]));
    sts128(adst + 16384u + off, make_uint4(lin[0], lin[1], lin[2], lin[3]));
  }
}

// Zeroes this thread's logit columns at or beyond Kp once per CTA: the contraction (N = Kp) never
// writes them, and with c'_k = -inf there they then read as -inf without any per-element masking.
template <int NC>
__device__ __forceinline__ void zero_unused_logits(uint32_t tmem, const RowCtx& rc, int Kp) {
  uint32_t z[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll
  for (int c = 0; c < NC / 16; ++c)
    if (NC * rc.part + 16 * c >= Kp) tmem_st16(tmem + rc.lane_base + kColLog + NC * rc.part + 16 * c, z);
  tmem_st_wait();
}

// Adds c'_k (shared address cb, float32) to NC logits in pairs and returns their maximum.
template <int NC>
__device__ __forceinline__ float bias_max(float* v, uint32_t cb, float m0, float m1) {
#pragma unroll
  for (int c4 = 0; c4 < NC / 4; ++c4) {
    const uint4 b = lds128(cb + 16 * c4);
    add_f32x2(v[4 * c4], v[4 * c4 + 1], __uint_as_float(b.x), __uint_as_float(b.y));
    add_f32x2(v[4 * c4 + 2], v[4 * c4 + 3], __uint_as_float(b.z), __uint_as_float(b.w));
  }
#pragma unroll
  for (int i = 0; i < NC / 4; ++i) {
    m0 = max3(m0, v[4 * i], v[4 * i + 1]);
    m1 = max3(m1, v[4 * i + 2], v[4 * i + 3]);
  }
  return fmaxf(m0, m1);
}
// Loads this thread's NC logits (components NC*part ...) from TMEM in two batches (the bias and max of
// the first overlap the second load), adds c'_k from the 256-entry table at shared address cs (-inf past
// K), and returns the part's maximum.
template <int NC>
__device__ __forceinline__ float load_logits(uint32_t tmem, const RowCtx& rc, uint32_t cs, float* v) {
  const int kbase = NC * rc.part;
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  constexpr int C = NC / 16, C1 = (C + 1) / 2;  // 16-column chunks; first batch
  const uint32_t ta = tmem + rc.lane_base + kColLog + kbase;
#pragma unroll
  for (int c = 0; c < C1; ++c) tmem_ld16(ta + 16 * c, r + 16 * c);
#pragma unroll
  for (int c = 0; c < C1; ++c) tmem_ld_wait_tied16(r + 16 * c);
#pragma unroll
  for (int c = C1; c < C; ++c) tmem_ld16(ta + 16 * c, r + 16 * c);
  float m = bias_max<16 * C1>(v, cs + 4 * kbase, -INFINITY, -INFINITY);
  if (C > C1) {
#pragma unroll
    for (int c = C1; c < C; ++c) tmem_ld_wait_tied16(r + 16 * c);
    m = bias_max<(C > C1 ? 16 * (C - C1) : 16)>(v + 16 * C1, cs + 4 * (kbase + 16 * C1), m, -INFINITY);
  }
  return m;
}

// e_k = 2^(v_k - m) in place (float32); returns the sum of the e_k.
template <int NC>
__device__ __forceinline__ float exp_inplace(float* v, float m) {
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int i = 0; i < NC / 2; ++i) {
    float t0 = v[2 * i], t1 = v[2 * i + 1];
    add_f32x2(t0, t1, -m, -m);
    v[2 * i] = ex2_approx(t0);
    v[2 * i + 1] = ex2_approx(t1);
    if (i & 1)
      add_f32x2(s2, s3, v[2 * i], v[2 * i + 1]);
    else
      add_f32x2(s0, s1, v[2 * i], v[2 * i + 1]);
  }
  return (s0 + s1) + (s2 + s3);
}

// Shared address of this thread's first 16-byte chunk (components NC*part .. +8) in a Gamma~ tile of
// 64-component SW128 blocks 16 KB apart; its chunk cj is at the returned address ^ (cj << 4) (the
// thread's NC components never cross a block, and the chunk index of NC*part has no bit in common
// with cj < NC/8).
template <int NC>
__device__ __forceinline__ uint32_t gamma_row_addr(uint32_t gtile, const RowCtx& rc) {
  const uint32_t c0 = (uint32_t)NC * rc.part;
  return gtile + (c0 >> 6) * 16384u + (rc.rowsw ^ (((c0 & 63u) >> 3) << 4));
}

// (a, b) *= (c, d) with one packed float32x2 multiply.
__device__ __forceinline__ void mul_f32x2(float& a, float& b, float c, float d) {
  asm("{\n .reg .b64 x, y;\n mov.b64 x, {%0, %1};\n mov.b64 y, {%2, %3};\n mul.rn.f32x2 x, x, y;\n"
      " mov.b64 {%0, %1}, x;\n}\n"
      : "+f"(a), "+f"(b)
      : "f"(c), "f"(d));
}
// The NC float32 values of v times inv, rounded to bf16 pairs and stored as 16-byte chunks at ga
// (gamma_row_addr), below Kp.
template <int NC>
__device__ __forceinline__ void scale_pack_store(const float* v, float inv, uint32_t ga, const RowCtx& rc, int Kp) {
  const int nvalid = (Kp - NC * rc.part) >> 3;
#pragma unroll
  for (int cj = 0; cj < NC / 8; ++cj) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float t0 = v[8 * cj + 2 * i], t1 = v[8 * cj + 2 * i + 1];
      mul_f32x2(t0, t1, inv, inv);
      w[i] = pack_bf16x2(t0, t1);
    }
    if (cj < nvalid) sts128(ga ^ (uint32_t)(cj << 4), make_uint4(w[0], w[1], w[2], w[3]));
  }
}

// Fused pass for a TMEM-resident operand: e = 2^(v - m) packed to bf16 pairs and stored over this thread's
// NC/2 columns starting at taddr (8 words per store).  The caller waits for the stores.
template <int NC>
__device__ __forceinline__ void exp_pack_tmem(const float* v, float m, uint32_t taddr, int c0 = 0,
                                              int c1 = NC / 16) {
#pragma unroll
  for (int c = 0; c < NC / 16; ++c) {
    if (c < c0 || c >= c1) continue;
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float t0 = v[16 * c + 2 * i], t1 = v[16 * c + 2 * i + 1];
      add_f32x2(t0, t1, -m, -m);
      w[i] = pack_bf16x2(ex2_approx(t0), ex2_approx(t1));
    }
    tmem_st8(taddr + 8 * c, w);
  }
}

__device__ __forceinline__ uint16_t bf16_bits(float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<const uint16_t*>(&h);
}

// g_release_count: arrivals that free the Gamma tile / a V slot (the write issuers); x_release_count:
// arrivals that free an X slot; done_count: issuers that commit to `done`.
__device__ __forceinline__ void init_bars(Bars* B, uint32_t g_release_count, uint32_t x_release_count,
                                          uint32_t done_count) {
  mbar_init(&B->w_full, 1);
  for (int s = 0; s < 2; ++s) {
    mbar_init(&B->x_full[s], 1);
    mbar_init(&B->x_empty[s], x_release_count);
    mbar_init(&B->v_empty[s], g_release_count);
  }
  mbar_init(&B->ax_full, kRowWarps);
  mbar_init(&B->l_full, 1);
  mbar_init(&B->l_empty, kRowWarps);
  mbar_init(&B->g_full, kRowWarps);
  for (int q = 0; q < 4; ++q) mbar_init(&B->g_fullq[q], kRowWarps / 4);
  mbar_init(&B->g_empty, g_release_count);
  mbar_init(&B->done, done_count);
  mbar_init(&B->done_l, 1);
  B->ab.flag = 0;
  mbar_fence_init();
}

// Producer: W image (with its constant step) once, then per tile the X tile.  With `tmV` (write kernel), iteration u also
// brings the V tile of u - 1, on the same barrier x_full[u & 1], so a row warp that has waited for the
// X tile it builds next also has the V tile of its current key tile; an extra iteration u = T brings
// the last V tile alone.  The V ring slot of tile t is t & 1, released by the write contraction.
__device__ __forceinline__ void producer(const TcArgs& a, const CUtensorMap* tmX, const CUtensorMap* tmV,
                                         uint8_t* smem, const SmemLayout& L, Bars* B, int bh, int tile0, int T) {
  const uint32_t wbytes = w_head_bytes(a.Kp);
  const int h = bh % a.H;
  // the parameter fold of this head (complete: this grid waited for it) flagged an fp16 overflow
  uint32_t bad = 0;
  for (int i = 0; i < kCTable / 8; ++i)
    if (GMA_INB(h * (kCTable / 8) + i, a.lim.flags, 110)) bad |= a.range_flags[h * (kCTable / 8) + i];
  if (bad) atomicCAS(&a.ctrl->err, kErrNone, kErrRange);
  mbar_expect_tx(&B->w_full, wbytes);
  for (uint32_t o = 0; o < wbytes; o += 32768)
    if (GMA_INB((size_t)h * wbytes + o + min(32768u, wbytes - o) - 1, a.lim.w, 111))
      bulk_load(smem + L.w + o, a.w_img + (size_t)h * wbytes + o, min(32768u, wbytes - o), &B->w_full);
  int issued[2] = {-1, -1};  // parity of the last phase armed on x_full[0], x_full[1]
  for (int u = 0; u <= T; ++u) {
    const int s = u & 1;
    const uint32_t ph = (uint32_t)(u >> 1) & 1;
    const bool has_x = u < T, has_v = tmV != nullptr && u > 0;
    if (!has_x && !has_v) break;
    // x_full[s] is re-armed only after its previous phase has been consumed (an arrival on a phase
    // that is still pending would over-count it), also when this iteration brings V alone
    if (!wait_bounded(&B->x_empty[s], ph ^ 1, &B->ab, a.ctrl, 10, a.wait_ns)) break;
    const int sv = (u - 1) & 1;
    if (has_v && !wait_bounded(&B->v_empty[sv], ((uint32_t)((u - 1) >> 1) & 1) ^ 1, &B->ab, a.ctrl, 11, a.wait_ns)) break;
    const bool load_x = has_x && !((a.fault & 1) && u == 0);
    const uint32_t bytes = (load_x ? 16384u : 0u) + (has_v ? 16384u : 0u);
    if (bytes == 0) continue;
    mbar_expect_tx(&B->x_full[s], bytes);
    if (load_x) tma_load_3d(smem + L.x + s * 16384, tmX, 0, (tile0 + u) * kTile, bh, &B->x_full[s]);
    if (has_v) tma_load_3d(smem + L.v + sv * 16384, tmV, 0, (tile0 + u - 1) * kTile, bh, &B->x_full[s]);
    issued[s] = (int)ph;
  }
  // never leave with copies in flight: wait for the last phase armed on each barrier
  Abort none{0};
  for (int s = 0; s < 2; ++s)
    if (issued[s] >= 0) wait_bounded(&B->x_full[s], (uint32_t)issued[s], &none, a.ctrl, 12, a.wait_ns);
}

// Issues the log-density contraction of one tile: LOG[128 x Kp] = AX[128 x 128] * W^T (d_w: descriptor
// of the K-major W image at its start).
__device__ __forceinline__ void issue_logits(uint32_t tmem, uint64_t d_w, int Kp, uint32_t col_ax = kColAx) {
  const uint32_t idesc = make_idesc(128, Kp, 0, 0, 0, 0);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
    mma_ts_off(tmem + kColLog, tmem + col_ax + 8 * ks, d_w, (ks >> 2) * (uint32_t)Kp * 8 + (ks & 3) * 2, idesc,
               ks > 0 ? 1u : 0u);
}
// The same with the [x^2 | x] operand in shared memory (d_a: K-major, 128-byte swizzle, the x block 16 KB
// after the x^2 block).
__device__ __forceinline__ void issue_logits_ss(uint32_t tmem, uint64_t d_a, uint64_t d_w, int Kp) {
  const uint32_t idesc = make_idesc(128, Kp, 0, 0, 0, 0);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
    mma_ss_off(tmem + kColLog, d_a, (uint32_t)((ks >> 2) * 16384 + (ks & 3) * 32) >> 4, d_w,
               (ks >> 2) * (uint32_t)Kp * 8 + (ks & 3) * 2, idesc, ks > 0 ? 1u : 0u);
}
// The same plus the constant step (A = the [256 | 1] columns at kColOnes, B = the 32-byte-swizzled c' image
// d_c), so the logits come out with c'_k added.
__device__ __forceinline__ void issue_logits_c(uint32_t tmem, uint64_t d_w, uint64_t d_c, int Kp) {
  issue_logits(tmem, d_w, Kp);
  mma_ts(tmem + kColLog, tmem + kColOnes, d_c, make_idesc(128, Kp, 0, 0, 0, 0), 1u);
}

// Writes the [256 | 1] fp16 pair (and zeros) into the 8 constant-step A columns of this thread's TMEM lane
// (one thread per lane).
__device__ __forceinline__ void write_ones_cols(uint32_t tmem, const RowCtx& rc) {
  uint32_t w[8] = {pack_f16x2(256.0f, 1.0f), 0u, 0u, 0u, 0u, 0u, 0u, 0u};
  tmem_st8(tmem + rc.lane_base + kColOnes, w);
}

// Loads this thread's NC logits (components NC*part ..., c' already included) from TMEM in two batches
// (the maximum of the first overlaps the second load) and returns the part's maximum.
template <int NC>
__device__ __forceinline__ float load_logits_c(uint32_t tmem, const RowCtx& rc, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  constexpr int C = NC / 16, C1 = (C + 1) / 2;
  const uint32_t ta = tmem + rc.lane_base + kColLog + NC * rc.part;
#pragma unroll
  for (int c = 0; c < C1; ++c) tmem_ld16(ta + 16 * c, r + 16 * c);
#pragma unroll
  for (int c = 0; c < C1; ++c) tmem_ld_wait_tied16(r + 16 * c);
#pragma unroll
  for (int c = C1; c < C; ++c) tmem_ld16(ta + 16 * c, r + 16 * c);
  float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
  for (int i = 0; i < 4 * C1; ++i) {
    m0 = max3(m0, v[4 * i], v[4 * i + 1]);
    m1 = max3(m1, v[4 * i + 2], v[4 * i + 3]);
  }
  if (C > C1) {
#pragma unroll
    for (int c = C1; c < C; ++c) tmem_ld_wait_tied16(r + 16 * c);
#pragma unroll
    for (int i = 4 * C1; i < 4 * C; ++i) {
      m0 = max3(m0, v[4 * i], v[4 * i + 1]);
      m1 = max3(m1, v[4 * i + 2], v[4 * i + 3]);
    }
  }
  return fmaxf(m0, m1);
}

// 8 output dims normalised (acc / den) and packed to bf16 (one 16-byte chunk).
__device__ __forceinline__ uint4 pack_out8(const uint32_t* acc, float rden) {
  return make_uint4(pack_bf16x2(__uint_as_float(acc[0]) * rden, __uint_as_float(acc[1]) * rden),
                    pack_bf16x2(__uint_as_float(acc[2]) * rden, __uint_as_float(acc[3]) * rden),
                    pack_bf16x2(__uint_as_float(acc[4]) * rden, __uint_as_float(acc[5]) * rden),
                    pack_bf16x2(__uint_as_float(acc[6]) * rden, __uint_as_float(acc[7]) * rden));
}
// ----------------------------------------------------------------------------------------------- write / aggregate
// grid (splits, B*H).  CTA (split, bh) covers tiles [split * seg_tiles, ...) of head-row bh and adds
// Gamma_K^T [V | 1] over them into state[bh] (kAtomic: bulk reduce-add) or stores it to state[bh][split]
// (causal segment aggregates).  Both normalise each key's Gamma row before it is packed (bf16 gamma =
// e / s, 0 past N) and use [V | 1] as loaded, with a constant 1 column.
template <bool kAtomic, int NC>
__global__ void __launch_bounds__(kThreadsTc, 1)
    tc_write_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // 1 KB aligned, still shared
  const uint32_t sbase = smem_u32(smem);
  __shared__ Bars B;
  const SmemLayout L = write_layout(a.Kp);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y, split = blockIdx.x;
  const int tile0 = split * a.seg_tiles;
  const int T = max(0, min(a.tiles, tile0 + a.seg_tiles) - tile0);
  const int MB = (a.Kp + 127) / 128;
  if (threadIdx.x == 0) GMA_SPAN_AT(0);

  // zero Gamma~ (components beyond Kp stay zero: the M=128 blocks read them) and the [1] atom
  for (uint32_t i = threadIdx.x; i < (uint32_t)MB * 32768 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem + L.g)[i] = make_uint4(0, 0, 0, 0);
  for (uint32_t i = threadIdx.x; i < 16384 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem + L.inv)[i] = make_uint4(0, 0, 0, 0);
  __syncthreads();
  // element n = 64 of each token row of the MN-major [V | 1] operand receives 1/s of that key every tile;
  // the Gamma tile and the V slot are free again once every write issuer (one per 128-component block)
  // has read them
  if (threadIdx.x == 0) init_bars(&B, (uint32_t)MB, (uint32_t)kRowWarps, (uint32_t)MB);
  if (warp == 1) {
    tmem_alloc(&B.tmem_base, 512);
    tmem_relinquish();
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  dep_wait();  // the parameter fold (and zeroed accumulator) of this call are complete
  // the next kernel (read, scan or state export) may be scheduled as SMs free up; it waits for this grid's
  // completion before it reads anything this grid writes
  dep_launch_next();
  if (threadIdx.x == 0) GMA_SPAN_AT(1);
  const uint32_t tmem = B.tmem_base;
  if (warp < kRowWarp0) {
    setmaxnreg_dec<kCtrlRegs>();
    if (warp == 0) {
      if (lane == 0) producer(a, &tmK, &tmV, smem, L, &B, bh, tile0, T);
    } else if (warp == 1) {
      if (lane == 0) {
        // issuer 1: the log-density contraction of every tile (into L once the row warps have taken the
        // previous logits and built this tile's operand)
        const uint32_t w_addr = smem_u32(smem + L.w);
        const uint64_t d_w = make_sdesc(w_addr, 16, 1024), d_c = make_sdesc32(w_addr + (uint32_t)a.Kp * 256, 16, 256);
        bool ok = wait_bounded(&B.w_full, 0, &B.ab, a.ctrl, 20, a.wait_ns);
        for (int t = 0; ok && t < T; ++t) {
          ok = wait_bounded(&B.ax_full, t & 1, &B.ab, a.ctrl, 22, a.wait_ns) &&
               (t == 0 || wait_bounded(&B.l_empty, (t - 1) & 1, &B.ab, a.ctrl, 23, a.wait_ns));
          if (!ok) break;
          GMA_TRACE_AT(52, t);
          tc_fence_after();
          issue_logits_c(tmem, d_w, d_c, a.Kp);
          mma_commit(&B.l_full);  // also frees the [x^2 | x] columns for the next tile
          GMA_TRACE_AT(53, t);
        }
        mma_commit(&B.done_l);
        Abort none{0};
        wait_bounded(&B.done_l, 0, &none, a.ctrl, 25, a.wait_ns);
      }
    } else if (warp - 2 < MB) {
      if (lane == 0) {
        // issuers 2 / 3: component block mb = warp - 2 of the write contraction, Gamma_K^T [V | 1]
        const int mb = warp - 2;
        const uint32_t idw = make_idesc(128, kStCols, 1, 1, 1, 1);
        const uint32_t g_addr = smem_u32(smem + L.g) + (uint32_t)mb * 32768u;
        const uint32_t v_addr = smem_u32(smem + L.v), inv_addr = smem_u32(smem + L.inv);
        const uint64_t d_g = make_sdesc(g_addr, 16384, 1024);
        // [V | 1] of ring slot s: MN-major, the 1 atom one leading-dimension step past the V atom
        const uint64_t d_v0 = make_sdesc(v_addr, inv_addr - v_addr, 1024);
        const uint64_t d_v1 = make_sdesc(v_addr + 16384, inv_addr - v_addr - 16384, 1024);
        bool ok = true;
        for (int t = 0; ok && t < T; ++t) {
          const int s = t & 1;
          // the K-steps of lane quarter q (tokens 32q .. 32q+31) go in once that quarter's row warps have
          // stored their Gamma rows (they waited for this tile's V before, so V has landed as well)
          const uint64_t d_v = s ? d_v1 : d_v0;
          for (int q = 0; ok && q < 4; ++q) {
            ok = wait_bounded(&B.g_fullq[q], t & 1, &B.ab, a.ctrl, 24, a.wait_ns);
            if (!ok) break;
            if (q == 0) GMA_TRACE_AT(20 + mb, t);
            tc_fence_after();
#pragma unroll
            for (int k2 = 0; k2 < 2; ++k2) {
              const int ks = 2 * q + k2;
              mma_ss_off(tmem + kColAcc + kStCols * mb, d_g, (ks * 2048) >> 4, d_v, (ks * 2048) >> 4, idw,
                         (t > 0 || ks > 0) ? 1u : 0u);
            }
          }
          if (!ok) break;
          mma_commit(&B.g_empty);
          mma_commit(&B.v_empty[s]);
          GMA_TRACE_AT(22 + mb, t);
        }
        mma_commit(&B.done);
        Abort none{0};
        wait_bounded(&B.done, 0, &none, a.ctrl, 26, a.wait_ns);
      }
    }
  } else {
    setmaxnreg_inc<kRowRegs>();
    // ------------------------------------------------------------------ row warps
    const RowCtx rc = row_ctx(sbase + L.red);
    const uint32_t ga = gamma_row_addr<NC>(sbase + L.g, rc);
    if (rc.part == 0) write_ones_cols(tmem, rc);
    // element n = 64 of every row of the [V | 1] operand is 1 (rows past N have a zero Gamma row)
    if (rc.part == 0) sts16(sbase + L.inv + rc.rowsw, bf16_bits(1.f));
    bool ok = warp_wait(&B.w_full, 0, &B.ab, a.ctrl, 30, a.wait_ns);
    if (ok && T > 0) {
      ok = warp_wait(&B.x_full[0], 0, &B.ab, a.ctrl, 31, a.wait_ns);
      if (ok) {
        transform_row(sbase + L.x, rc, tmem);
        warp_arrive(&B.x_empty[0]);
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(&B.ax_full);
      }
    }
    float v[NC];
    // every row warp runs all T tiles and all exchanges; after a failed wait (ok = false) it skips the
    // work and the waits but still takes part in the exchanges, whose barriers have no time limit
    for (int t = 0; t < T; ++t) {
      const int tok = (tile0 + t) * kTile + rc.row;
      float mp = -INFINITY;
      if (warp == kRowWarp0) GMA_TRACE_AT(30, t);
      // logits of tile t; the [x^2 | x] columns are free again, so the operand of tile t+1 goes in first:
      // its TMEM stores drain while the logits are loaded, and one wait covers both before the operand
      // and the logit columns are handed back to the issuer
      if (ok) ok = warp_wait(&B.l_full, t & 1, &B.ab, a.ctrl, 32, a.wait_ns);
      if (warp == kRowWarp0) GMA_TRACE_AT(31, t);
      bool next_op = false;
      if (ok) {
        tc_fence_after();
        // x_full of u = t + 1 brings X(t + 1) (if any) and V(t)
        const int s1 = (t + 1) & 1;
        ok = warp_wait(&B.x_full[s1], ((t + 1) >> 1) & 1, &B.ab, a.ctrl, 33, a.wait_ns);
        if (ok && t + 1 < T) {
          transform_row(sbase + L.x + s1 * 16384, rc, tmem);
          warp_arrive(&B.x_empty[s1]);
          next_op = true;
        }
      }
      if (warp == kRowWarp0) GMA_TRACE_AT(32, t);
      if (ok) {
        mp = load_logits_c<NC>(tmem, rc, v);
        if (next_op) tmem_st_wait();
        tc_fence_before();
        if (next_op) warp_arrive(&B.ax_full);
        warp_arrive(&B.l_empty);
      }
      if (warp == kRowWarp0) GMA_TRACE_AT(33, t);
      const float m = xchg_max(rc, 0, mp);
      if (warp == kRowWarp0) GMA_TRACE_AT(34, t);
      // normalised Gamma row (0 past N) -> smem once the previous contraction has read the tile: the
      // exponentials stay in float32 registers through the sum exchange, then are scaled by 1/s, packed
      // to bf16 and stored ([V | 1] is used as loaded)
      float sp = 0.f;
      if (ok) sp = exp_inplace<NC>(v, m);
      if (warp == kRowWarp0) GMA_TRACE_AT(35, t);
      const float sum = xchg_sum(rc, 4, sp);
      if (warp == kRowWarp0) GMA_TRACE_AT(36, t);
      if (ok) {
        const float inv = tok < a.N ? rcp_approx(sum) : 0.f;
        if (t > 0) ok = warp_wait(&B.g_empty, (t - 1) & 1, &B.ab, a.ctrl, 36, a.wait_ns);
        if (warp == kRowWarp0) GMA_TRACE_AT(37, t);
        if (ok) scale_pack_store<NC>(v, inv, ga, rc, a.Kp);
      }
      if (warp == kRowWarp0) GMA_TRACE_AT(39, t);
      if (ok) {
        fence_async_smem();
        warp_arrive(&B.g_fullq[rc.q]);
      }
      if (warp == kRowWarp0) GMA_TRACE_AT(40, t);
      if (warp > kRowWarp0 && warp < kRowWarp0 + 4) GMA_TRACE_AT(40 + warp - kRowWarp0, t);
    }
    // epilogue: state rows of this CTA -> global
    if (kAtomic) {
      // bidirectional: the CTA's rows [Vt | Z] (68 floats per component) are staged in shared memory (over the
      // Gamma~ and X areas, idle once the last contraction is done) and added to state[bh] by bulk reductions
      if (T > 0 && rc.part < MB) {
        const uint32_t stage = sbase + L.g;
        if (ok && warp_wait(&B.done, 0, &B.ab, a.ctrl, 39, a.wait_ns)) {
          tc_fence_after();
          const int comp = 128 * rc.part + rc.row;
          uint32_t r[80];
#pragma unroll
          for (int c = 0; c < 5; ++c) tmem_ld16(tmem + rc.lane_base + kColAcc + kStCols * rc.part + 16 * c, r + 16 * c);
          tmem_ld_wait();
          if (comp < a.Kp) {
#pragma unroll
            for (int c = 0; c < kStRow / 4; ++c)
              sts128(stage + (uint32_t)(comp * kStRow + 4 * c) * 4u,
                     c == kDv / 4 ? make_uint4(r[kDv], 0u, 0u, 0u)
                                  : make_uint4(r[4 * c], r[4 * c + 1], r[4 * c + 2], r[4 * c + 3]));
          }
        }
        fence_async_smem();
        named_bar_sync(15, (uint32_t)MB * 128u);
        if (threadIdx.x == 32 * kRowWarp0 && ok) {
          const uint32_t bytes = (uint32_t)a.Kp * kStRow * 4u, chunk = bytes / 4u;  // 16-byte multiples
          float* dst = a.state + (size_t)bh * a.Kp * kStRow;
          if (GMA_INB(((size_t)bh + 1) * a.Kp * kStRow - 1, a.lim.state, 112))
            for (uint32_t o = 0; o < bytes; o += chunk)
              bulk_reduce_add_f32(reinterpret_cast<uint8_t*>(dst) + o, stage + o, chunk);
          bulk_commit();
          bulk_wait_read_all();
        }
      }
    } else if (ok && T > 0 && rc.part < MB) {
      if (warp_wait(&B.done, 0, &B.ab, a.ctrl, 39, a.wait_ns)) {
        tc_fence_after();
        const int comp = 128 * rc.part + rc.row;
        uint32_t r[80];
#pragma unroll
        for (int c = 0; c < 5; ++c) tmem_ld16(tmem + rc.lane_base + kColAcc + kStCols * rc.part + 16 * c, r + 16 * c);
        tmem_ld_wait();
        if (comp < a.Kp) {  // segment aggregate, column-major agg[bh][split][80][Kp]: each store covers 32 components
          const size_t i0 = ((size_t)bh * a.splits + split) * kStCols * a.Kp + comp;
          float* dst = a.state + i0;
#pragma unroll
          for (int c = 0; c < kStCols; ++c)
            if (GMA_INB(i0 + (size_t)c * a.Kp, a.lim.state, 113)) dst[(size_t)c * a.Kp] = __uint_as_float(r[c]);
        }
      }
    }
    if (threadIdx.x == 32 * kRowWarp0) GMA_SPAN_AT(2);
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) GMA_SPAN_AT(3);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ----------------------------------------------------------------------------------------------- responsibilities
// a8: grid (splits, B*H); writes the normalised Gamma (float32 [BH][N][K]) of every token: the logits
// (issuer 1, c' included by the constant step) and a float32 softmax over k in the row warps.
template <int NC>
__global__ void __launch_bounds__(kThreadsTc, 1) tc_resp_kernel(const __grid_constant__ CUtensorMap tmQ, TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // 1 KB aligned, still shared
  const uint32_t sbase = smem_u32(smem);
  __shared__ Bars B;
  const SmemLayout L = read_layout(a.Kp);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y, split = blockIdx.x;
  const int tile0 = split * a.seg_tiles;
  const int T = max(0, min(a.tiles, tile0 + a.seg_tiles) - tile0);

  if (threadIdx.x == 0) init_bars(&B, 1u, (uint32_t)kRowWarps, 1u);
  if (warp == 1) {
    tmem_alloc(&B.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  dep_wait();  // the parameter fold of this call is complete
  const uint32_t tmem = B.tmem_base;
  if (warp < kRowWarp0) {
    setmaxnreg_dec<kCtrlRegs>();
    if (warp == 0) {
      if (lane == 0) producer(a, &tmQ, nullptr, smem, L, &B, bh, tile0, T);
    } else if (warp == 1) {
      if (lane == 0) {
        const uint32_t w_addr = smem_u32(smem + L.w);
        const uint64_t d_w = make_sdesc(w_addr, 16, 1024), d_c = make_sdesc32(w_addr + (uint32_t)a.Kp * 256, 16, 256);
        bool ok = wait_bounded(&B.w_full, 0, &B.ab, a.ctrl, 40, a.wait_ns);
        for (int t = 0; ok && t < T; ++t) {
          ok = wait_bounded(&B.ax_full, t & 1, &B.ab, a.ctrl, 43, a.wait_ns) &&
               (t == 0 || wait_bounded(&B.l_empty, (t - 1) & 1, &B.ab, a.ctrl, 44, a.wait_ns));
          if (!ok) break;
          tc_fence_after();
          issue_logits_c(tmem, d_w, d_c, a.Kp);
          mma_commit(&B.l_full);  // also frees the [x^2 | x] columns for the next tile
        }
        mma_commit(&B.done_l);
        Abort none{0};
        wait_bounded(&B.done_l, 0, &none, a.ctrl, 47, a.wait_ns);
      }
    }
  } else {
    setmaxnreg_inc<kRowRegs>();
    const RowCtx rc = row_ctx(sbase + L.red);
    if (rc.part == 0) write_ones_cols(tmem, rc);
    bool ok = warp_wait(&B.w_full, 0, &B.ab, a.ctrl, 50, a.wait_ns);
    if (ok && T > 0) {
      ok = warp_wait(&B.x_full[0], 0, &B.ab, a.ctrl, 51, a.wait_ns);
      if (ok) {
        transform_row(sbase + L.x, rc, tmem);
        warp_arrive(&B.x_empty[0]);
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(&B.ax_full);
      }
    }
    float v[NC];
    // every row warp runs all T tiles and all exchanges (see the write kernel)
    for (int t = 0; t < T; ++t) {
      float mp = -INFINITY;
      if (ok) ok = warp_wait(&B.l_full, t & 1, &B.ab, a.ctrl, 52, a.wait_ns);
      if (ok) {
        tc_fence_after();
        if (t + 1 < T) {
          const int s1 = (t + 1) & 1;
          ok = warp_wait(&B.x_full[s1], ((t + 1) >> 1) & 1, &B.ab, a.ctrl, 53, a.wait_ns);
          if (ok) {
            transform_row(sbase + L.x + s1 * 16384, rc, tmem);
            warp_arrive(&B.x_empty[s1]);
            tmem_st_wait();
            tc_fence_before();
            warp_arrive(&B.ax_full);
          }
        }
      }
      if (ok) {
        mp = load_logits_c<NC>(tmem, rc, v);
        tc_fence_before();
        warp_arrive(&B.l_empty);
      }
      const int tok = (tile0 + t) * kTile + rc.row;
      // gamma = 2^(v - m) / s in float32
      const float m = xchg_max(rc, 0, mp);
      float sp = 0.f;
      if (ok) sp = exp_inplace<NC>(v, m);
      const float sum = xchg_sum(rc, 4, sp);
      if (ok && tok < a.N) {
        const float r = 1.0f / sum;
        const size_t i0 = ((size_t)bh * a.N + tok) * a.K + NC * rc.part;
        float* dst = reinterpret_cast<float*>(a.out) + i0;
        const int nk = min(max(a.K - NC * rc.part, 0), NC);
        if ((a.K & 3) == 0) {  // 16-byte aligned row segments (nk a multiple of 4 too): vector stores
#pragma unroll
          for (int k = 0; k < NC; k += 4)
            if (k < nk && GMA_INB(i0 + k + 3, a.lim.out, 120))
              *reinterpret_cast<float4*>(dst + k) = make_float4(v[k] * r, v[k + 1] * r, v[k + 2] * r, v[k + 3] * r);
        } else {
#pragma unroll
          for (int k = 0; k < NC; ++k)
            if (k < nk && GMA_INB(i0 + k, a.lim.out, 120)) dst[k] = v[k] * r;
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ----------------------------------------------------------------------------------------------- read (two groups)
// Bidirectional read with two tiles in flight.  The 16 row warps form two groups of 8; group g takes the
// tiles t with t & 1 == g and owns TMEM columns 256 g .. 256 g + 255, which hold in turn the tile's
// logits, then Gamma~_Q (bf16 pairs, compacted in place) beside the output accumulator.  Within a group
// two threads share a token row (half h owns components h NC2 .. h NC2 + NC2 - 1) and stream their
// logits from TMEM twice (maximum, then exponentials), so few registers are live and the other group's
// tile proceeds meanwhile.  The [x^2 | x] operand of the logits is built in shared memory (TMEM has no
// room for it), so the log-density contraction reads both operands from shared memory.  Issuer g
// (warp 1 + g) issues group g's logits and read contractions and its output tile stores.
struct R2Layout {
  uint32_t w, a0, ones, sb, stg0, red, total;
};
__host__ __device__ inline R2Layout read2_layout(int Kp) {
  R2Layout s{};
  const int KB = (Kp + 63) / 64;
  s.w = 0;
  s.a0 = align1k(w_head_bytes(Kp));   // two [x^2 | x] operands (x^2 block, then x block, 16 KB each)
  s.ones = s.a0 + 2 * 32768;          // the constant step's A: 128 rows x [256 | 1 | 0 ...] fp16, 32-byte swizzle
  s.sb = s.ones + 4096;               // state operand [80][Kp] bf16, K-major
  s.stg0 = align1k(s.sb + KB * (kStCols * 128));  // two 16 KB output staging tiles
  s.red = s.stg0 + 2 * 16384;         // maximum exchange: [group][slot][row][half] float
  s.total = s.red + 2 * 2 * kTile * 2 * 4;
  return s;
}

struct R2Bars {
  uint64_t w_full;
  uint64_t x_full[2], a_empty[2], a_full[2], l_full[2], g_full[2], o_full[2], r_empty[2], o_staged[2], st_done[2];
  uint64_t done[2];
  uint32_t tmem_base;
  Abort ab;
};

template <int NC2>
__global__ void __launch_bounds__(kThreadsTc, 1)
    tc_read2_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmO, TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // 1 KB aligned, still shared
  const uint32_t sbase = smem_u32(smem);
  __shared__ R2Bars B;
  const R2Layout L = read2_layout(a.Kp);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y, split = blockIdx.x;
  const int tile0 = split * a.seg_tiles;
  const int T = max(0, min(a.tiles, tile0 + a.seg_tiles) - tile0);
  const int KS = a.Kp / 16;
  constexpr int kGroupWarps = 8;
  // output accumulator columns within a group's region: past the compacted Gamma~_Q of half 0
  // (NC2 / 2 columns) and clear of half 1's (the last NC2 / 2 columns of 2 NC2)
  constexpr uint32_t kColOut = NC2 == 128 ? 64u : 128u;
  if (threadIdx.x == 0) GMA_SPAN_AT(4);

  if (threadIdx.x == 0) {
    mbar_init(&B.w_full, 1);
    for (int g = 0; g < 2; ++g) {
      mbar_init(&B.x_full[g], 1);
      mbar_init(&B.a_empty[g], 1);
      mbar_init(&B.a_full[g], kGroupWarps);
      mbar_init(&B.l_full[g], 1);
      mbar_init(&B.g_full[g], kGroupWarps);
      mbar_init(&B.o_full[g], 1);
      mbar_init(&B.r_empty[g], kGroupWarps);
      mbar_init(&B.o_staged[g], kGroupWarps);
      mbar_init(&B.st_done[g], 1);
      mbar_init(&B.done[g], 1);
    }
    B.ab.flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(&B.tmem_base, 512);
    tmem_relinquish();
  }
  dep_wait();  // the write (and before it the parameter fold) of this call are complete
  if (threadIdx.x == 0) {
    // the W image and the first X tile of each group land while the state operand is built
    const uint32_t wbytes = w_head_bytes(a.Kp);
    mbar_expect_tx(&B.w_full, wbytes);
    for (uint32_t o = 0; o < wbytes; o += 32768)
      if (GMA_INB((size_t)(bh % a.H) * wbytes + o + min(32768u, wbytes - o) - 1, a.lim.w, 130))
        bulk_load(smem + L.w + o, a.w_img + (size_t)(bh % a.H) * wbytes + o, min(32768u, wbytes - o), &B.w_full);
    for (int t = 0; t < 2 && t < T; ++t) {
      mbar_expect_tx(&B.x_full[t], 16384);
      tma_load_3d(smem + L.a0 + 32768 * t + 16384, &tmQ, 0, (tile0 + t) * kTile, bh, &B.x_full[t]);
    }
  }
  if (warp >= kRowWarp0) {
    const int i = threadIdx.x - 32 * kRowWarp0;  // 0 .. 511
    // the constant step's A rows: [256 | 1 | 0 ...] (fp16), 32-byte swizzle
    if (i < kTile) {
      *reinterpret_cast<uint4*>(smem + L.ones + sw32_chunk(i, 0)) = make_uint4(pack_f16x2(256.0f, 1.0f), 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(smem + L.ones + sw32_chunk(i, 1)) = make_uint4(0u, 0u, 0u, 0u);
    }
    // state [Kp][80] fp32 -> bf16 K-major operand SB[n][comp] (eps folded into column 64 once): one item is
    // 8 consecutive components of column n, packed into one 16-byte chunk; consecutive threads take
    // consecutive n, so each of the 8 loads of an item is coalesced across the warp
    const float* src = a.state + (size_t)bh * a.Kp * kStRow;
    const int items = kStCols * (a.Kp / 8), nt = 32 * (kThreadsTc / 32 - kRowWarp0);
    for (int i0 = i; i0 < items; i0 += 2 * nt) {
      float f[2][8];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int it = i0 + u * nt, n = it % kStCols, c8 = it / kStCols;
        if (it < items) {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            f[u][j] = n <= kDv && GMA_INB((size_t)bh * a.Kp * kStRow + (size_t)(8 * c8 + j) * kStRow + n, a.lim.state, 131)
                          ? __ldg(src + (size_t)(8 * c8 + j) * kStRow + n)
                          : 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int it = i0 + u * nt, n = it % kStCols, c8 = it / kStCols;
        if (it < items) {
          const float e = n == kDv ? a.eps : 0.f;
          const uint4 v = make_uint4(pack_bf16x2(f[u][0] + e, f[u][1] + e), pack_bf16x2(f[u][2] + e, f[u][3] + e),
                                     pack_bf16x2(f[u][4] + e, f[u][5] + e), pack_bf16x2(f[u][6] + e, f[u][7] + e));
          sts128(sbase + L.sb + sw128_off(n, 8 * c8, kStCols * 128), v);
        }
      }
    }
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x == 0) GMA_SPAN_AT(5);
  const uint32_t tmem = B.tmem_base;

  if (warp < kRowWarp0) {
    setmaxnreg_dec<kCtrlRegs>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------------- producer: X tiles 2 .. T-1 (the W
      // image and tiles 0 and 1 were issued in the prologue)
      int issued[2] = {T > 0 ? 0 : -1, T > 1 ? 0 : -1};
      for (int t = 2; t < T; ++t) {
        const int g = t & 1;
        const uint32_t k = (uint32_t)(t >> 1);
        // the x block of group g's operand once the logits of its previous tile have read it
        if (!wait_bounded(&B.a_empty[g], (k - 1) & 1, &B.ab, a.ctrl, 110, a.wait_ns)) break;
        mbar_expect_tx(&B.x_full[g], 16384);
        tma_load_3d(smem + L.a0 + 32768 * g + 16384, &tmQ, 0, (tile0 + t) * kTile, bh, &B.x_full[g]);
        issued[g] = (int)(k & 1);
      }
      Abort none{0};
      for (int g = 0; g < 2; ++g)
        if (issued[g] >= 0) wait_bounded(&B.x_full[g], (uint32_t)issued[g], &none, a.ctrl, 111, a.wait_ns);
    } else if ((warp == 1 || warp == 2) && lane == 0) {
      // ---------------------------------------------------------------- issuer of group g
      const int g = warp - 1;
      const uint32_t rg = tmem + 256u * (uint32_t)g;
      const uint32_t w_addr = smem_u32(smem + L.w), a_addr = smem_u32(smem + L.a0) + 32768u * (uint32_t)g;
      const uint64_t d_w = make_sdesc(w_addr, 16, 1024), d_c = make_sdesc32(w_addr + (uint32_t)a.Kp * 256, 16, 256);
      const uint64_t d_a = make_sdesc(a_addr, 16, 1024), d_ones = make_sdesc32(smem_u32(smem + L.ones), 16, 256);
      const uint64_t d_sb = make_sdesc(smem_u32(smem + L.sb), 16, 1024);
      const uint32_t id_log = make_idesc(128, a.Kp, 0, 0, 0, 0);
      constexpr uint32_t idr = make_idesc(128, kStCols, 1, 1, 0, 0);
      bool ok = wait_bounded(&B.w_full, 0, &B.ab, a.ctrl, 112, a.wait_ns);
      for (int t = g; ok && t < T; t += 2) {
        const uint32_t k = (uint32_t)(t >> 1), ph = k & 1;
        // logits: the group's operand is built and its region free (the previous output has been read),
        // and the previous tile's logits (the other group's) have completed.  Left to themselves, the two
        // chains settle into a rhythm in which their logits and softmax passes coincide (tile loops of
        // 108 - 114 us per CTA at B=1 H=8 N=131072 K=256); kept one logits contraction apart, each
        // group's softmax runs beside the other's contractions.  (The other group's next logits wait
        // for this group's, so the awaited phase is the last one that can have completed.)
        if (!(ok = wait_bounded(&B.a_full[g], ph, &B.ab, a.ctrl, 113, a.wait_ns) &&
                   (t < 2 || wait_bounded(&B.r_empty[g], ph ^ 1, &B.ab, a.ctrl, 114, a.wait_ns)) &&
                   (t == 0 || wait_bounded(&B.l_full[g ^ 1], (uint32_t)((t - 1) >> 1) & 1u, &B.ab, a.ctrl, 119,
                                           a.wait_ns))))
          break;
        GMA_TRACE_AT(20, t);
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma_ss_off(rg, d_a, ((ks >> 2) * 16384 + (ks & 3) * 32) >> 4, d_w, (ks >> 2) * (uint32_t)a.Kp * 8 + (ks & 3) * 2,
                     id_log, ks > 0 ? 1u : 0u);
        mma_ss(rg, d_ones, d_c, id_log, 1u);
        mma_commit(&B.l_full[g]);
        mma_commit(&B.a_empty[g]);
        GMA_TRACE_AT(21, t);
        // the previous tile's output (staged by the rows after its read) while this tile's logits run
        if (t >= 2) {
          if (!(ok = wait_bounded(&B.o_staged[g], ph ^ 1, &B.ab, a.ctrl, 116, a.wait_ns))) break;
          GMA_TRACE_AT(24, t);
          tma_store_3d(&tmO, smem_u32(smem + L.stg0) + 16384u * (uint32_t)g, 0, (tile0 + t - 2) * kTile, bh);
          bulk_commit();
          bulk_wait_read_all();
          mbar_arrive(&B.st_done[g]);
          GMA_TRACE_AT(25, t);
        }
        // read: Gamma~_Q (TMEM, compacted) [Vt | Z + eps] into the region's output columns
        if (!(ok = wait_bounded(&B.g_full[g], ph, &B.ab, a.ctrl, 115, a.wait_ns))) break;
        GMA_TRACE_AT(22, t);
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
          if (ks < KS) {
            const uint32_t acol = ks < NC2 / 16 ? 8u * ks : (uint32_t)(3 * NC2 / 2) + 8u * (ks - NC2 / 16);
            mma_ts_off(rg + kColOut, rg + acol, d_sb, ((ks >> 2) * (kStCols * 128) + (ks & 3) * 32) >> 4, idr,
                       ks > 0 ? 1u : 0u);
          }
        }
        mma_commit(&B.o_full[g]);
        GMA_TRACE_AT(23, t);
      }
      // the group's last output tile
      const int tl = g + 2 * ((T - 1 - g) / 2);  // last tile of this group (if any)
      if (ok && g < T) {
        if (wait_bounded(&B.o_staged[g], (uint32_t)(tl >> 1) & 1u, &B.ab, a.ctrl, 118, a.wait_ns)) {
          tma_store_3d(&tmO, smem_u32(smem + L.stg0) + 16384u * (uint32_t)g, 0, (tile0 + tl) * kTile, bh);
          bulk_commit();
        }
      }
      bulk_wait_all();
      mma_commit(&B.done[g]);
      Abort none{0};
      wait_bounded(&B.done[g], 0, &none, a.ctrl, 117, a.wait_ns);
    }
  } else {
    setmaxnreg_inc<kRowRegs>();
    // ------------------------------------------------------------------ row warps
    const int wi = warp - kRowWarp0;
    const int g = wi / kGroupWarps, half = (wi % kGroupWarps) / 4, q = warp & 3;
    const int row = 32 * q + lane;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    const uint32_t rg = tmem + lane_base + 256u * (uint32_t)g;
    const uint32_t rowsw = (uint32_t)(row >> 3) * 1024u + (uint32_t)(row & 7) * 128u + ((uint32_t)(row & 7) << 4);
    const uint32_t bar = 1u + 4u * (uint32_t)g + (uint32_t)q;  // the two warps sharing this quarter's rows
    const uint32_t red = sbase + L.red + (uint32_t)g * (2 * kTile * 2 * 4);
    const uint32_t a_x = sbase + L.a0 + 32768u * (uint32_t)g + 16384u;  // x block of the group's operand
    const uint32_t stg = sbase + L.stg0 + 16384u * (uint32_t)g;
    const uint32_t lcol = (uint32_t)(NC2 * half);                         // this half's logit columns
    // packed Gamma~ pairs of chunk c (32 components): half 0 compacts upwards from column 0, half 1
    // downwards into the top of its own columns, so neither overwrites logits still to be read
    const uint32_t gcol0 = half == 0 ? 0u : (uint32_t)(3 * NC2 / 2);
    // [x^2 | x] fp16 operand of this row (dims 32 half .. + 31) of tile u, built in place from its bf16 tile
    auto build_operand = [&](int u) {
      if (!warp_wait(&B.x_full[g], (uint32_t)(u >> 1) & 1u, &B.ab, a.ctrl, 121, a.wait_ns)) return false;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t ad = (a_x + rowsw) ^ ((uint32_t)(4 * half + j) << 4);
        const uint4 v = lds128(ad);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
        uint32_t sq[4], lin[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float lo = __uint_as_float(w4[e] << 16), hi = __uint_as_float(w4[e] & 0xffff0000u);
          lin[e] = pack_f16x2(lo, hi);
          sq[e] = pack_f16x2(lo * lo, hi * hi);
        }
        sts128(ad, make_uint4(lin[0], lin[1], lin[2], lin[3]));
        sts128(ad - 16384u, make_uint4(sq[0], sq[1], sq[2], sq[3]));
      }
      fence_async_smem();
      warp_arrive(&B.a_full[g]);
      return true;
    };
    bool ok = warp_wait(&B.w_full, 0, &B.ab, a.ctrl, 120, a.wait_ns);
    if (ok && g < T) ok = build_operand(g);
    for (int t = g; t < T; t += 2) {
      const uint32_t k = (uint32_t)(t >> 1), ph = k & 1;
      if (wi == 0) GMA_TRACE_AT(0, t);
      // pass 1: this half's maximum, exchanged with the partner thread of the row
      float mh = -INFINITY;
      if (wi == 0) GMA_TRACE_AT(2, t);
      if (ok) ok = warp_wait(&B.l_full[g], ph, &B.ab, a.ctrl, 122, a.wait_ns);
      if (wi == 0) GMA_TRACE_AT(3, t);
      if (ok) {
        tc_fence_after();
        // chunk c + 1's load is in flight while chunk c is reduced
        float m0 = -INFINITY, m1 = -INFINITY;
        uint32_t ra[32], rb[32];
        tmem_ld32(rg + lcol, ra);
#pragma unroll
        for (int c = 0; c < NC2 / 32; ++c) {
          uint32_t* cur = (c & 1) ? rb : ra;
          uint32_t* nxt = (c & 1) ? ra : rb;
          tmem_ld_wait_tied32(cur);
          if (c + 1 < NC2 / 32) tmem_ld32(rg + lcol + 32 * (c + 1), nxt);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            m0 = max3(m0, __uint_as_float(cur[4 * e]), __uint_as_float(cur[4 * e + 1]));
            m1 = max3(m1, __uint_as_float(cur[4 * e + 2]), __uint_as_float(cur[4 * e + 3]));
          }
        }
        mh = fmaxf(m0, m1);
      }
      if (wi == 0) GMA_TRACE_AT(4, t);
      const uint32_t slot = red + (ph * kTile + (uint32_t)row) * 8u;
      sts32(slot + 4u * (uint32_t)half, mh);
      named_bar_sync(bar, 64);
      const float m = fmaxf(mh, lds32(slot + 4u * (uint32_t)(half ^ 1)));
      if (wi == 0) GMA_TRACE_AT(5, t);
      // pass 2: unnormalised gamma~ = 2^(v - m) packed to bf16 in place (half 1 walks its chunks
      // downwards); the read divides by gamma~ . (Z + eps) = gamma~ . Z + eps s
      if (ok) {
        // chunk order: half 0 upwards, half 1 downwards; the next chunk's load is in flight while this one is
        // exponentiated (its source never overlaps this chunk's packed destination)
        uint32_t ra[32], rb[32];
        tmem_ld32(rg + lcol + 32 * (half == 0 ? 0 : NC2 / 32 - 1), ra);
#pragma unroll
        for (int cc = 0; cc < NC2 / 32; ++cc) {
          const int c = half == 0 ? cc : NC2 / 32 - 1 - cc;
          uint32_t* cur = (cc & 1) ? rb : ra;
          uint32_t* nxt = (cc & 1) ? ra : rb;
          tmem_ld_wait_tied32(cur);
          if (wi == 0) GMA_TRACE_AT(10 + cc, t);
          if (cc + 1 < NC2 / 32) tmem_ld32(rg + lcol + 32 * (half == 0 ? c + 1 : c - 1), nxt);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            float t0 = __uint_as_float(cur[2 * e]), t1 = __uint_as_float(cur[2 * e + 1]);
            add_f32x2(t0, t1, -m, -m);
            cur[e] = pack_bf16x2(ex2_approx(t0), ex2_approx(t1));
          }
          tmem_st16(rg + gcol0 + 16 * c, cur);
          if (wi == 0) GMA_TRACE_AT(14 + cc, t);
        }
        tmem_st_wait();
        if (wi == 0) GMA_TRACE_AT(18, t);
        tc_fence_before();
        warp_arrive(&B.g_full[g]);
      }
      // the next tile's operand while this tile's read contraction runs (its X tile landed long ago: the
      // producer loads it once this tile's logits have read the operand buffer)
      if (ok && t + 2 < T) ok = build_operand(t + 2);
      if (wi == 0) GMA_TRACE_AT(6, t);
      // epilogue: dims 32 half .. + 31 divided by column 64, staged as bf16 for the tensor store
      if (ok) ok = warp_wait(&B.o_full[g], ph, &B.ab, a.ctrl, 123, a.wait_ns);
      if (wi == 0) GMA_TRACE_AT(7, t);
      if (ok) {
        tc_fence_after();
        uint32_t r[32];
        tmem_ld32(rg + kColOut + 32 * half, r);
        uint32_t zc = tmem_ld1(rg + kColOut + 64);
        tmem_ld_wait_tied32(r);
        tmem_ld_wait_tied1(zc);
        tc_fence_before();
        warp_arrive(&B.r_empty[g]);
        const float rden = rcp_approx(__uint_as_float(zc));
        if (t >= 2) ok = warp_wait(&B.st_done[g], ph ^ 1, &B.ab, a.ctrl, 124, a.wait_ns);
        if (ok) {
#pragma unroll
          for (int j = 0; j < 4; ++j) sts128((stg + rowsw) ^ ((uint32_t)(4 * half + j) << 4), pack_out8(r + 8 * j, rden));
          fence_async_smem();
          warp_arrive(&B.o_staged[g]);
        }
      }
      if (wi == 0) GMA_TRACE_AT(8, t);
    }
    if (wi == 0 && lane == 0) GMA_SPAN_AT(6);
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) GMA_SPAN_AT(7);
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ----------------------------------------------------------------------------------------------- causal
// Chunked causal sweep.  CTA (segment, bh) starts from the exclusive prefix state of its segment and
// walks the segment tile by tile with the state S resident in TMEM:
//   O_i = [gq~_i . S_prev + sum_{j in tile, j <= i} (gq~_i . gk_j) [v_j | 1]] / (... + eps s_i),
//   S  += Gamma_K(tile)^T [V | 1]
// (gist.science summary, "Variants and training" item 3: prefix sums, O_i depends on j <= i only).
// Both sides of every tile are computed here from Q and K; no responsibilities are read from or
// written to global memory.
//
// TMEM: L (columns 0..255) holds, in turn, the key logits, the query logits, then Gamma~_Q (bf16 pairs,
// columns 0..127) beside P = Gamma~_Q Gamma_K^T (columns 128..255); S (256..415); OX (416..495) holds
// the [x^2 | x] operand of the query logits, then the output accumulator.  The key logits read their
// operand from shared memory: the row warps build tile t+1's, and snapshot the state for its inter-tile
// term, while P [V | 1] of tile t runs, and its key logits start as soon as that contraction is done,
// so they overlap tile t's output instead of opening tile t+1.
// Three MMA issuers run side by side (each issuing thread waits about 100 cycles per instruction, so
// the N = 80 / 128 contractions reach the tensor pipe's rate only when several threads issue):
// warp 1 the logits and the state update, warp 2 the inter-tile term and P [V | 1], warp 3 P.
constexpr uint32_t kCColP = 128;   // P (fp32 128 columns; bf16 pairs in its first 64 after masking)
constexpr uint32_t kCColS = 256;   // state accumulators, 80 columns per 128-component block
constexpr uint32_t kCColO = 416;   // query logit operand, then the output accumulator (80 columns)

struct CausalLayout {
  uint32_t w, gk, xk, xq, v, sbv, sbz, c, red, ak, total;
};
__host__ __device__ inline CausalLayout causal_layout(int Kp) {
  CausalLayout s{};
  const int MB = (Kp + 127) / 128;
  s.w = 0;
  // normalised Gamma_K tile: 64-component 128-byte-swizzle blocks 16 KB apart (MN-major A of the state
  // update, K-major B of P), written by the row warps
  s.gk = align1k(Kp * 256);
  // the key and query X tiles (bf16, 128-byte swizzle), read by the row warps into the logit operand
  s.xk = s.gk + MB * 32768;
  s.xq = s.xk + 16384;
  // [V | 1] as one MN-major B of N = 80 in the 32-byte swizzle: four 4 KB atoms of 16 value dims, then
  // the constant atom (column 0 = 1, columns 1..15 zero)
  s.v = s.xq + 16384;
  // bf16 copy of S_prev [Kp][80] (+ eps in column 64), MN-major B of N = 80, 32-byte swizzle: five
  // atoms of Kp rows x 32 bytes
  s.sbv = s.v + 5 * 4096;
  s.sbz = s.sbv + 4 * Kp * 32;  // the fifth atom (Z + eps in column 64)
  s.c = s.sbz + Kp * 32;
  s.red = s.c + 1024;
  s.total = s.red + kParts * kTile * 8;
  // the [x^2 | x] fp16 operand of the key logits (K-major, 128-byte swizzle: the x^2 block, then the x
  // block 16 KB on), built while the previous tile's P [V | 1] runs.  At Kp = 256 it takes Gamma_K
  // blocks 2 and 3, free from the moment P and the state update have read them until the key softmax
  // stores the next Gamma_K (after the key logits have read the operand); below, a region of its own.
  if (MB >= 2) {
    s.ak = s.gk + 32768;
  } else {
    s.ak = align1k(s.total);
    s.total = s.ak + 32768;
  }
  return s;
}

struct CBars {
  uint64_t w_full, xk_full, xk_empty, xq_full, xq_empty, v_full, v_empty;
  uint64_t ak_full, ax_full, lk_full, lq_full, gk_full, gk_empty, gq_half, gq_full, sb_full, s_done, p_full, pb_full,
      o_full;
  uint64_t o_staged, o_stored;
  uint64_t done[3];
  uint32_t tmem_base;
  Abort ab;
};

// Writes float32 state columns 16c .. 16c+15 of component `comp` (r) into atom c of the bf16 copy of
// S_prev (MN-major, 32-byte swizzle, atoms of Kp rows x 32 bytes at sb + c * Kp * 32); for c = 4 only
// column 64 (Z, plus eps) is kept, as element 0 of the fifth atom.
__device__ __forceinline__ void snapshot_state_chunk(uint32_t sb, int Kp, int comp, int c, const uint32_t* r,
                                                     float eps) {
  const uint32_t atom = sb + (uint32_t)c * (uint32_t)Kp * 32u;
  if (c < 4) {
    const uint4 lo = make_uint4(pack_bf16x2(__uint_as_float(r[0]), __uint_as_float(r[1])),
                                pack_bf16x2(__uint_as_float(r[2]), __uint_as_float(r[3])),
                                pack_bf16x2(__uint_as_float(r[4]), __uint_as_float(r[5])),
                                pack_bf16x2(__uint_as_float(r[6]), __uint_as_float(r[7])));
    const uint4 hi = make_uint4(pack_bf16x2(__uint_as_float(r[8]), __uint_as_float(r[9])),
                                pack_bf16x2(__uint_as_float(r[10]), __uint_as_float(r[11])),
                                pack_bf16x2(__uint_as_float(r[12]), __uint_as_float(r[13])),
                                pack_bf16x2(__uint_as_float(r[14]), __uint_as_float(r[15])));
    sts128(atom + sw32_chunk(comp, 0), lo);
    sts128(atom + sw32_chunk(comp, 1), hi);
  } else {
    sts16(atom + sw32_chunk(comp, 0), bf16_bits(__uint_as_float(r[0]) + eps));
  }
}



template <int NC>
__global__ void __launch_bounds__(kThreadsTc, 1)
    tc_causal_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO, TcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);  // 1 KB aligned, still shared
  const uint32_t sbase = smem_u32(smem);
  __shared__ CBars B;
  const CausalLayout L = causal_layout(a.Kp);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int bh = blockIdx.y, seg = blockIdx.x;
  const int tile0 = seg * a.seg_tiles;
  const int T = max(0, min(a.tiles, tile0 + a.seg_tiles) - tile0);
  const int MB = (a.Kp + 127) / 128;
  const int KS = a.Kp / 16;

  // zero the Gamma_K blocks (components past Kp stay zero: the M = 128 blocks read them), the constant
  // atom and the state copies
  for (uint32_t i = threadIdx.x; i < (uint32_t)MB * 32768 / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem + L.gk)[i] = make_uint4(0, 0, 0, 0);
  for (uint32_t i = threadIdx.x; i < (L.c - (L.v + 16384)) / 16; i += blockDim.x)
    reinterpret_cast<uint4*>(smem + L.v + 16384)[i] = make_uint4(0, 0, 0, 0);
  if (threadIdx.x == 0) {
    mbar_init(&B.w_full, 1);
    mbar_init(&B.xk_full, 1);
    mbar_init(&B.xk_empty, kRowWarps);
    mbar_init(&B.xq_full, 1);
    mbar_init(&B.xq_empty, kRowWarps);
    mbar_init(&B.v_full, 1);
    mbar_init(&B.v_empty, 2);    // the state update and P [V | 1] read V
    mbar_init(&B.ak_full, kRowWarps);
    mbar_init(&B.ax_full, kRowWarps);
    mbar_init(&B.lk_full, 1);
    mbar_init(&B.lq_full, 1);
    mbar_init(&B.gk_full, kRowWarps);
    mbar_init(&B.gk_empty, 2);   // the state update and P read Gamma_K
    mbar_init(&B.gq_half, kRowWarps);
    mbar_init(&B.gq_full, kRowWarps);
    mbar_init(&B.sb_full, kRowWarps);
    mbar_init(&B.s_done, 1);
    mbar_init(&B.p_full, 2);     // the inter-tile term and P
    mbar_init(&B.pb_full, kRowWarps);
    mbar_init(&B.o_full, 1);
    mbar_init(&B.o_staged, kRowWarps);
    mbar_init(&B.o_stored, 1);
    for (int i = 0; i < 3; ++i) mbar_init(&B.done[i], 1);
    B.ab.flag = 0;
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc(&B.tmem_base, 512);
    tmem_relinquish();
  }
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  dep_wait();  // the scan (and before it the aggregates and the parameter fold) of this call are complete
  const uint32_t tmem = B.tmem_base;

  if (warp < kRowWarp0) {
    setmaxnreg_dec<kCtrlRegsC>();
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------------- producer
      // the W image without its constant step (c' is added from the float32 table, which needs no
      // shared memory for the constant step's B operand)
      const uint32_t wbytes = (uint32_t)a.Kp * 256, cbytes = kCTable * 4;
      const int h = bh % a.H;
      mbar_expect_tx(&B.w_full, wbytes + cbytes);
      for (uint32_t o = 0; o < wbytes; o += 32768)
        if (GMA_INB((size_t)h * w_head_bytes(a.Kp) + o + min(32768u, wbytes - o) - 1, a.lim.w, 140))
          bulk_load(smem + L.w + o, a.w_img + (size_t)h * w_head_bytes(a.Kp) + o, min(32768u, wbytes - o), &B.w_full);
      if (GMA_INB((size_t)h * kCTable + kCTable - 1, a.lim.c, 141))
        bulk_load(smem + L.c, a.cbias + (size_t)h * kCTable, cbytes, &B.w_full);
      int issued[3] = {-1, -1, -1};  // parity of the last load armed on xk_full, xq_full, v_full
      for (int t = 0; t < T; ++t) {
        const uint32_t pe = (t & 1) ^ 1;
        const int row0 = (tile0 + t) * kTile;
        // each X slot once the row warps have built the previous tile's operand from it
        if (!wait_bounded_bo(&B.xk_empty, pe, &B.ab, a.ctrl, 70, a.wait_ns)) break;
        mbar_expect_tx(&B.xk_full, 16384);
        tma_load_3d(smem + L.xk, &tmK, 0, row0, bh, &B.xk_full);
        issued[0] = t & 1;
        if (!wait_bounded_bo(&B.xq_empty, pe, &B.ab, a.ctrl, 71, a.wait_ns)) break;
        mbar_expect_tx(&B.xq_full, 16384);
        tma_load_3d(smem + L.xq, &tmQ, 0, row0, bh, &B.xq_full);
        issued[1] = t & 1;
        if (!wait_bounded_bo(&B.v_empty, pe, &B.ab, a.ctrl, 72, a.wait_ns)) break;
        mbar_expect_tx(&B.v_full, 16384);
        for (int a4 = 0; a4 < 4; ++a4) tma_load_3d(smem + L.v + 4096 * a4, &tmV, 16 * a4, row0, bh, &B.v_full);
        issued[2] = t & 1;
      }
      // never leave with copies in flight
      Abort none{0};
      if (issued[0] >= 0) wait_bounded_bo(&B.xk_full, (uint32_t)issued[0], &none, a.ctrl, 73, a.wait_ns);
      if (issued[1] >= 0) wait_bounded_bo(&B.xq_full, (uint32_t)issued[1], &none, a.ctrl, 74, a.wait_ns);
      if (issued[2] >= 0) wait_bounded_bo(&B.v_full, (uint32_t)issued[2], &none, a.ctrl, 75, a.wait_ns);
    } else if (warp == 1 && lane == 0) {
      // ---------------------------------------------------------------- issuer 1: logits, state update
      const uint64_t d_w = make_sdesc(smem_u32(smem + L.w), 16, 1024);
      const uint64_t d_vb = make_sdesc32(smem_u32(smem + L.v), 4096, 256);          // [V | 1], N = 80
      const uint64_t d_gk_mn = make_sdesc(smem_u32(smem + L.gk), 16384, 1024);     // Gamma_K^T as MN-major A
      const uint64_t d_ak = make_sdesc(smem_u32(smem + L.ak), 16, 1024);           // key [x^2 | x], K-major A
      constexpr uint32_t id_s80 = make_idesc(128, kStCols, 1, 1, 1, 1);
      bool ok = wait_bounded_bo(&B.w_full, 0, &B.ab, a.ctrl, 80, a.wait_ns);
      for (int t = 0; ok && t < T; ++t) {
        const uint32_t ph = t & 1;
        // key logits: the key operand is in shared memory (the row warps build tile t's while P [V | 1]
        // of tile t-1 runs) and L is free once that contraction has read the bf16 P
        if (!(ok = wait_bounded_bo(&B.ak_full, ph, &B.ab, a.ctrl, 81, a.wait_ns) &&
                   (t == 0 || wait_bounded_bo(&B.o_full, ph ^ 1u, &B.ab, a.ctrl, 96, a.wait_ns))))
          break;
        GMA_TRACE_AT(20, t);
        tc_fence_after();
        issue_logits_ss(tmem, d_ak, d_w, a.Kp);
        mma_commit(&B.lk_full);
        GMA_TRACE_AT(21, t);
#ifdef GMA_TRACE
        { Abort none{0}; wait_bounded(&B.lk_full, ph, &none, a.ctrl, 0, a.wait_ns); }
        GMA_TRACE_AT(26, t);
#endif
        // query logits: the row warps have loaded the key logits and put the query operand in OX
        if (!(ok = wait_bounded_bo(&B.ax_full, ph, &B.ab, a.ctrl, 82, a.wait_ns))) break;
        GMA_TRACE_AT(22, t);
        tc_fence_after();
        issue_logits(tmem, d_w, a.Kp, kCColO);
        mma_commit(&B.lq_full);
        GMA_TRACE_AT(23, t);
#ifdef GMA_TRACE
        { Abort none{0}; wait_bounded(&B.lq_full, ph, &none, a.ctrl, 0, a.wait_ns); }
        GMA_TRACE_AT(27, t);
#endif
        // S += Gamma_K^T [V | 1] once Gamma_K and V are in and the snapshot of the previous S is taken
        if (!(ok = wait_bounded_bo(&B.gk_full, ph, &B.ab, a.ctrl, 83, a.wait_ns) &&
                   wait_bounded_bo(&B.v_full, ph, &B.ab, a.ctrl, 84, a.wait_ns) &&
                   wait_bounded_bo(&B.sb_full, ph, &B.ab, a.ctrl, 85, a.wait_ns)))
          break;
        GMA_TRACE_AT(24, t);
        tc_fence_after();
#pragma unroll
        for (int mb = 0; mb < 2; ++mb) {
          if (mb < MB) {
#pragma unroll
            for (int s = 0; s < 8; ++s)
              mma_ss_off(tmem + kCColS + kStCols * mb, d_gk_mn, (mb * 32768 + 2048 * s) >> 4, d_vb, (512 * s) >> 4,
                         id_s80, 1u);
          }
        }
        mma_commit(&B.s_done);
        mma_commit(&B.gk_empty);
        mma_commit(&B.v_empty);
        GMA_TRACE_AT(25, t);
      }
      mma_commit(&B.done[0]);
      Abort none{0};
      wait_bounded_bo(&B.done[0], 0, &none, a.ctrl, 86, a.wait_ns);
    } else if (warp == 2 && lane == 0) {
      // ---------------------------------------------------------------- issuer 2: O = Gq~ S_prev, O += P [V | 1]
      const uint64_t d_sb = make_sdesc32(smem_u32(smem + L.sbv), (uint32_t)a.Kp * 32, 256);
      const uint64_t d_vb = make_sdesc32(smem_u32(smem + L.v), 4096, 256);
      constexpr uint32_t id_c80 = make_idesc(128, kStCols, 1, 1, 0, 1);  // A tmem, B MN-major, N = 80
      bool ok = true;
      for (int t = 0; ok && t < T; ++t) {
        const uint32_t ph = t & 1;
        // the K-steps of the first chunks of every row part once those are written (gq_half), then the
        // rest (as for P)
        constexpr int kCpp = NC / 16, kHalf = kCpp > 1 ? kCpp / 2 : 1;
        constexpr int kRest = kCpp - kHalf > 0 ? kCpp - kHalf : 1;
        if (!(ok = wait_bounded_bo(&B.gq_half, ph, &B.ab, a.ctrl, 98, a.wait_ns) &&
                   wait_bounded_bo(&B.sb_full, ph, &B.ab, a.ctrl, 88, a.wait_ns)))
          break;
        GMA_TRACE_AT(30, t);
        tc_fence_after();
        // (the issuing thread waits ~100 cycles per instruction here, so a rolled loop costs nothing and
        // keeps this role's register footprint small)
#pragma unroll 1
        for (int i = 0; i < KS / kCpp * kHalf; ++i) {
          const int ks = (i / kHalf) * kCpp + i % kHalf;
          mma_ts_off(tmem + kCColO, tmem + kColLog + 8 * ks, d_sb, (uint32_t)(512 * ks) >> 4, id_c80, i > 0);
        }
        if (!(ok = wait_bounded_bo(&B.gq_full, ph, &B.ab, a.ctrl, 87, a.wait_ns))) break;
        tc_fence_after();
#pragma unroll 1
        for (int i = 0; i < KS / kCpp * (kCpp - kHalf); ++i) {
          const int ks = (i / kRest) * kCpp + kHalf + i % kRest;
          mma_ts_off(tmem + kCColO, tmem + kColLog + 8 * ks, d_sb, (uint32_t)(512 * ks) >> 4, id_c80, 1u);
        }
        mma_commit(&B.p_full);
        GMA_TRACE_AT(31, t);
        if (!(ok = wait_bounded_bo(&B.pb_full, ph, &B.ab, a.ctrl, 89, a.wait_ns) &&
                   wait_bounded_bo(&B.v_full, ph, &B.ab, a.ctrl, 95, a.wait_ns)))
          break;
        GMA_TRACE_AT(32, t);
        tc_fence_after();
#pragma unroll 1
        for (int s = 0; s < 8; ++s) {
          const uint32_t ap = tmem + kCColP + 32 * (s >> 1) + 8 * (s & 1);  // bf16 P of keys 16s..16s+15
          mma_ts_off(tmem + kCColO, ap, d_vb, (uint32_t)(512 * s) >> 4, id_c80, 1u);
        }
        mma_commit(&B.o_full);
        mma_commit(&B.v_empty);
        GMA_TRACE_AT(33, t);
      }
      mma_commit(&B.done[1]);
      Abort none{0};
      wait_bounded_bo(&B.done[1], 0, &none, a.ctrl, 90, a.wait_ns);
    } else if (warp == 3 && lane == 0) {
      // ---------------------------------------------------------------- issuer 3: P = Gq~ Gk^T
      const uint64_t d_gk_k = make_sdesc(smem_u32(smem + L.gk), 16, 1024);  // Gamma_K as K-major B
      constexpr uint32_t id_p = make_idesc(128, 128, 1, 1, 0, 0);
      bool ok = true;
      for (int t = 0; ok && t < T; ++t) {
        const uint32_t ph = t & 1;
        // K-step ks reads chunk ks % (NC / 16) of row part ks / (NC / 16): the first chunks of every part
        // are issued once the row warps have written them (gq_half), the rest after gq_full
        constexpr int kCpp = NC / 16, kHalf = kCpp > 1 ? kCpp / 2 : 1;
        if (!(ok = wait_bounded_bo(&B.gq_half, ph, &B.ab, a.ctrl, 97, a.wait_ns) &&
                   wait_bounded_bo(&B.gk_full, ph, &B.ab, a.ctrl, 92, a.wait_ns)))
          break;
        GMA_TRACE_AT(40, t);
        tc_fence_after();
#pragma unroll 1
        for (int i = 0; i < KS / kCpp * kHalf; ++i) {
          const int ks = (i / kHalf) * kCpp + i % kHalf;
          mma_ts_off(tmem + kCColP, tmem + kColLog + 8 * ks, d_gk_k, (uint32_t)((ks >> 2) * 16384 + (ks & 3) * 32) >> 4,
                     id_p, i > 0);
        }
        constexpr int kRest = kCpp - kHalf > 0 ? kCpp - kHalf : 1;  // the loop below is empty when kCpp == 1
        if (!(ok = wait_bounded_bo(&B.gq_full, ph, &B.ab, a.ctrl, 91, a.wait_ns))) break;
        tc_fence_after();
#pragma unroll 1
        for (int i = 0; i < KS / kCpp * (kCpp - kHalf); ++i) {
          const int ks = (i / kRest) * kCpp + kHalf + i % kRest;
          mma_ts_off(tmem + kCColP, tmem + kColLog + 8 * ks, d_gk_k, (uint32_t)((ks >> 2) * 16384 + (ks & 3) * 32) >> 4,
                     id_p, 1u);
        }
        mma_commit(&B.p_full);
        mma_commit(&B.gk_empty);
        GMA_TRACE_AT(41, t);
        // the row warps stage the normalised bf16 output tile in the (then unused) first Gamma_K block;
        // one tensor store writes it (rows past N clipped), then the block is handed back
        if (!(ok = wait_bounded_bo(&B.o_staged, ph, &B.ab, a.ctrl, 94, a.wait_ns))) break;
        tma_store_3d(&tmO, smem_u32(smem + L.gk), 0, (tile0 + t) * kTile, bh);
        bulk_commit();
        bulk_wait_read_all();
        mbar_arrive(&B.o_stored);
      }
      bulk_wait_all();
      mma_commit(&B.done[2]);
      Abort none{0};
      wait_bounded_bo(&B.done[2], 0, &none, a.ctrl, 93, a.wait_ns);
    }
  } else {
    setmaxnreg_inc<kRowRegsC>();
    // ------------------------------------------------------------------ row warps
    const RowCtx rc = row_ctx(sbase + L.red);
    const uint32_t cs = sbase + L.c;
    const uint32_t ga = gamma_row_addr<NC>(sbase + L.gk, rc);
    // S <- exclusive prefix state of this segment; SB <- its bf16 copy (eps rides in the Z column)
    if (rc.part < MB) {
      const int comp = 128 * rc.part + rc.row;
      // column-major [80][Kp]: each load of a warp covers 32 consecutive components
      const float* pre = a.state + ((size_t)bh * a.splits + seg) * kStCols * a.Kp + comp;
      // the 80 loads in two batches (columns 0..47, then 48..79): two round trips to memory, not five
#pragma unroll
      for (int hb = 0; hb < 2; ++hb) {
        const int c0 = hb ? 3 : 0, nc = hb ? 2 : 3;  // 16-column chunks of this batch
        uint32_t r[48];
#pragma unroll
        for (int i = 0; i < 48; ++i)
          if (i < 16 * nc)
            r[i] = comp < a.Kp && GMA_INB(((size_t)bh * a.splits + seg) * kStCols * a.Kp + comp + (size_t)(16 * c0 + i) * a.Kp,
                                          a.lim.state, 142)
                       ? __float_as_uint(__ldg(pre + (size_t)(16 * c0 + i) * a.Kp))
                       : 0u;
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          if (c < nc) {
            tmem_st16(tmem + rc.lane_base + kCColS + kStCols * rc.part + 16 * (c0 + c), r + 16 * c);
            if (comp < a.Kp) snapshot_state_chunk(sbase + L.sbv, a.Kp, comp, c0 + c, r + 16 * c, a.eps);
          }
        }
      }
    }
    // the constant atom of [V | 1]: column 0 is 1 for every key row (rows past N have a zero Gamma_K row)
    if (rc.part == 0) sts16(sbase + L.v + 16384 + sw32_chunk(rc.row, 0), bf16_bits(1.f));
    tmem_st_wait();
    fence_async_smem();
    tc_fence_before();
    warp_arrive(&B.sb_full);
    bool ok = warp_wait(&B.w_full, 0, &B.ab, a.ctrl, 100, a.wait_ns);
    // logit columns past Kp: never written by the logits contractions; zero (with c' = -inf they read as
    // -inf) or, at Kp <= 128, stale P values (finite, so the same)
    zero_unused_logits<NC>(tmem, rc, a.Kp);
    // the key operand of tile u -> shared memory (K-major A of the key logits)
    auto build_key = [&](int u) {
      if (!warp_wait(&B.xk_full, (uint32_t)u & 1u, &B.ab, a.ctrl, 101, a.wait_ns)) return false;
      transform_row_smem(sbase + L.xk, rc, sbase + L.ak);
      fence_async_smem();
      warp_arrive(&B.xk_empty);
      warp_arrive(&B.ak_full);
      return true;
    };
    if (ok && T > 0) ok = build_key(0);
    float v[NC];
    // every row warp runs all T tiles and all exchanges (see the write kernel); exchange e of the CTA uses
    // slot (e & 1), three per tile
    for (int t = 0; t < T; ++t) {
      const uint32_t ph = t & 1;
      const int tok = (tile0 + t) * kTile + rc.row;
      const uint32_t s0 = (uint32_t)((3 * t) & 1) * 4u, s1 = s0 ^ 4u;
      if (warp == kRowWarp0) GMA_TRACE_AT(0, t);
      // key logits -> registers; then the query operand -> OX
      float mk = -INFINITY;
      if (warp == kRowWarp0) GMA_TRACE_AT(2, t);
      if (ok) ok = warp_wait(&B.lk_full, ph, &B.ab, a.ctrl, 102, a.wait_ns);
      if (warp == kRowWarp0) GMA_TRACE_AT(3, t);
      if (ok) {
        // OX is free (this thread read its output columns at the end of the previous tile): the query
        // operand goes in first (while no logits are held in registers), then the key logits are
        // loaded and both L and OX handed over
        tc_fence_after();
        ok = warp_wait(&B.xq_full, ph, &B.ab, a.ctrl, 103, a.wait_ns);
        if (ok) {
          transform_row(sbase + L.xq, rc, tmem, kCColO);
          warp_arrive(&B.xq_empty);
          mk = load_logits<NC>(tmem, rc, cs, v);
          tmem_st_wait();
          tc_fence_before();
          warp_arrive(&B.ax_full);
        }
      }
      if (warp == kRowWarp0) GMA_TRACE_AT(4, t);
      // key softmax: the normalised Gamma_K row (0 past N) -> smem once the previous tile's readers are done
      // (state update, P, and the output tile staged in its first block); [V | 1] is used as loaded
      const float m_k = xchg_max(rc, s0, mk);
      if (warp == kRowWarp0) GMA_TRACE_AT(5, t);
      float sp = 0.f;
      if (ok) sp = exp_inplace<NC>(v, m_k);
      if (warp == kRowWarp0) GMA_TRACE_AT(6, t);
      const float sum = xchg_sum(rc, s1, sp);
      if (warp == kRowWarp0) GMA_TRACE_AT(7, t);
      if (ok && t > 0)
        ok = warp_wait(&B.gk_empty, (t - 1) & 1, &B.ab, a.ctrl, 104, a.wait_ns) &&
             warp_wait(&B.o_stored, (t - 1) & 1, &B.ab, a.ctrl, 110, a.wait_ns);
      if (warp == kRowWarp0) GMA_TRACE_AT(19, t);
      if (ok) {
        const float inv = tok < a.N ? rcp_approx(sum) : 0.f;
        scale_pack_store<NC>(v, inv, ga, rc, a.Kp);
        fence_async_smem();
        warp_arrive(&B.gk_full);
      }
      if (warp == kRowWarp0) GMA_TRACE_AT(8, t);
      // query softmax: Gamma~_Q (unnormalised) -> TMEM over its own logit columns
      float mq = -INFINITY;
      if (ok) ok = warp_wait(&B.lq_full, ph, &B.ab, a.ctrl, 105, a.wait_ns);
      if (warp == kRowWarp0) GMA_TRACE_AT(9, t);
      if (ok) {
        tc_fence_after();
        mq = load_logits<NC>(tmem, rc, cs, v);
      }
      if (warp == kRowWarp0) GMA_TRACE_AT(10, t);
      const float m_q = xchg_max(rc, s0, mq);
      if (warp == kRowWarp0) GMA_TRACE_AT(11, t);
      if (ok) {
        // in two halves of this thread's chunks: P starts on the K-steps of the first half meanwhile
        constexpr int kHalf = NC / 16 > 1 ? NC / 32 : 1;
        const uint32_t tq = tmem + rc.lane_base + kColLog + (NC / 2) * rc.part;
        exp_pack_tmem<NC>(v, m_q, tq, 0, kHalf);
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(&B.gq_half);
        exp_pack_tmem<NC>(v, m_q, tq, kHalf, NC / 16);
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(&B.gq_full);
      }
      if (warp == kRowWarp0) GMA_TRACE_AT(12, t);
      // intra-tile affinity: mask j > i, bf16 over the first half of this thread's own 32 columns
      if (ok) ok = warp_wait(&B.p_full, ph, &B.ab, a.ctrl, 106, a.wait_ns);
      if (warp == kRowWarp0) GMA_TRACE_AT(13, t);
      if (ok) {
        tc_fence_after();
        uint32_t pr[32];
        tmem_ld32(tmem + rc.lane_base + kCColP + 32 * rc.part, pr);
        tmem_ld_wait_tied32(pr);
        const int lim = rc.row - 32 * rc.part;  // columns c <= lim are keys j <= i
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float p0 = (2 * i <= lim) ? __uint_as_float(pr[2 * i]) : 0.f;
          const float p1 = (2 * i + 1 <= lim) ? __uint_as_float(pr[2 * i + 1]) : 0.f;
          pr[i] = pack_bf16x2(p0, p1);
        }
        tmem_st16(tmem + rc.lane_base + kCColP + 32 * rc.part, pr);
        tmem_st_wait();
        tc_fence_before();
        warp_arrive(&B.pb_full);
      }
      // while P [V | 1] runs: the state after this tile's update -> the bf16 copy read by the next tile's
      // inter-tile term (this tile's has completed with P), then the next tile's key operand -> shared
      // memory (P and the state update have read this tile's Gamma_K).  Every tile waits for its state
      // update, since the output below is staged in Gamma_K's first block.  Parts 0 / 1 take columns
      // 0..31 and Z of state block 0 / 1, parts 2 / 3 columns 32..63.
      if (warp == kRowWarp0) GMA_TRACE_AT(14, t);
      if (ok) ok = warp_wait(&B.s_done, ph, &B.ab, a.ctrl, 107, a.wait_ns);
      if (warp == kRowWarp0) GMA_TRACE_AT(15, t);
      if (t + 1 < T) {
        if (ok) {
          tc_fence_after();
          const int mb = rc.part & 1;
          if (mb < MB) {
            const int comp = 128 * mb + rc.row;
            const uint32_t ts = tmem + rc.lane_base + kCColS + kStCols * mb;
            const int c0 = rc.part < 2 ? 0 : 2;
            uint32_t ra[16];
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              tmem_ld16(ts + 16 * (c0 + c), ra);
              tmem_ld_wait_tied16(ra);
              if (comp < a.Kp) snapshot_state_chunk(sbase + L.sbv, a.Kp, comp, c0 + c, ra, a.eps);
            }
            if (rc.part < 2) {
              uint32_t z = tmem_ld1(ts + 64);
              tmem_ld_wait_tied1(z);
              if (comp < a.Kp) snapshot_state_chunk(sbase + L.sbv, a.Kp, comp, 4, &z, a.eps);
            }
          }
          fence_async_smem();
          tc_fence_before();
          warp_arrive(&B.sb_full);
        }
        if (ok) ok = build_key(t + 1);
      }
      if (warp == kRowWarp0) GMA_TRACE_AT(1, t);
      // output: dims 8 part + [0, 8) and 32 + 8 part + [0, 8) -- the columns this thread's part of the
      // next query operand overwrites -- normalised by gq~ . (Z + eps)
      if (warp == kRowWarp0) GMA_TRACE_AT(16, t);
      if (ok) ok = warp_wait(&B.o_full, ph, &B.ab, a.ctrl, 108, a.wait_ns);
      if (warp == kRowWarp0) GMA_TRACE_AT(17, t);
      if (ok) {
        tc_fence_after();
        uint32_t oa[8], ob[8];
        tmem_ld8(tmem + rc.lane_base + kCColO + 8 * rc.part, oa);
        tmem_ld8(tmem + rc.lane_base + kCColO + 32 + 8 * rc.part, ob);
        uint32_t z = tmem_ld1(tmem + rc.lane_base + kCColO + 64);
        tmem_ld_wait_tied8(oa);
        tmem_ld_wait_tied8(ob);
        tmem_ld_wait_tied1(z);
        const float rden = rcp_approx(__uint_as_float(z));
        // Gamma_K's readers (P, state update) have completed (p_full, s_done): its first block takes the
        // output tile in the 128-byte swizzle of the output tensor map (dims 8 part.. and 32 + 8 part..
        // are 16-byte chunks part and 4 + part of the token row)
        const uint32_t orow = sbase + L.gk + rc.rowsw;
        sts128(orow ^ ((uint32_t)rc.part << 4), pack_out8(oa, rden));
        sts128(orow ^ ((uint32_t)(4 + rc.part) << 4), pack_out8(ob, rden));
        fence_async_smem();
        warp_arrive(&B.o_staged);
      }
      if (warp == kRowWarp0) GMA_TRACE_AT(18, t);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Exclusive scan over segments: agg[bh][p][e] <- sum_{p' < p} agg[bh][p'][e].  grid (ceil(n / 128), B*H),
// one thread per element.  Its loads go in batches of eight segments, all eight in flight; a batch's
// stores may alias the next batch's loads, so each batch is one round trip to L2.
// 128 threads of at most 32 registers, so that its CTAs fit beside a running aggregate CTA and start the
// moment that grid completes.
__global__ void __launch_bounds__(128, 16) tc_scan_kernel(float* agg, int P, int n, size_t lim) {
  dep_wait();         // the aggregates are complete
  dep_launch_next();  // the sweep sets itself up meanwhile and waits for this grid before reading
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= n) return;
  float* base = agg + (size_t)blockIdx.y * P * n + e;
  float run = 0.f;
  for (int p0 = 0; p0 < P; p0 += 8) {
    float x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j)
      x[j] = (p0 + j < P) && GMA_INB(((size_t)blockIdx.y * P + p0 + j) * n + e, lim, 150)
                 ? __ldcg(base + (size_t)(p0 + j) * n)
                 : 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (p0 + j < P && GMA_INB(((size_t)blockIdx.y * P + p0 + j) * n + e, lim, 150))
        __stcg(base + (size_t)(p0 + j) * n, run);
      run += x[j];
    }
  }
}

// Deterministic reduction mode: the state state[bh][k][c] (c < 68) is the sum of the write CTAs' own
// states agg[bh][s][c][k] (column-major, s = 0 .. P-1), added in the order of s by one thread per
// element; grid (ceil(68 Kp / 128), B*H).  The pad columns 65 .. 67 are written as zero.
__global__ void __launch_bounds__(128, 16) tc_state_sum_kernel(const float* agg, int P, int Kp, float* state,
                                                               size_t lim_agg, size_t lim_state) {
  dep_wait();         // the per-CTA states are complete
  dep_launch_next();  // the read sets itself up meanwhile and waits for this grid before reading
  const int e = blockIdx.x * blockDim.x + threadIdx.x;  // c * Kp + k
  if (e >= kStRow * Kp) return;
  const int c = e / Kp, k = e - c * Kp;
  const float* src = agg + (size_t)blockIdx.y * P * kStCols * Kp + e;
  float s = 0.f;
  if (c <= kDv)
    for (int q = 0; q < P; ++q)
      if (GMA_INB((size_t)blockIdx.y * P * kStCols * Kp + e + (size_t)q * kStCols * Kp, lim_agg, 151))
        s += __ldcg(src + (size_t)q * kStCols * Kp);
  if (GMA_INB(((size_t)blockIdx.y * Kp + k) * kStRow + c, lim_state, 152))
    state[((size_t)blockIdx.y * Kp + k) * kStRow + c] = s;
}

// Public causal state [B*H][K][dv + 1] from the write accumulator [B*H][Kp][68] (columns 0..64).
__global__ void tc_state_export_kernel(const float* __restrict__ acc, int K, int Kp, size_t n, float* __restrict__ out,
                                       size_t lim_acc) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % (kDv + 1));
    const size_t rk = i / (kDv + 1);  // bh * K + k
    const int k = (int)(rk % K);
    const size_t bh = rk / K;
    if (GMA_INB((bh * Kp + k) * kStRow + c, lim_acc, 153)) out[i] = acc[(bh * Kp + k) * kStRow + c];
  }
}

// ----------------------------------------------------------------------------------------------- host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 3-D map over a [B*H][N][64] bf16 tensor, box 64 x 128 x 1, 128-byte swizzle, zero fill past N.
// 3-D map over [B*H][N][ld] bf16 (ld = 64 unless given) with 128-row boxes: 64-element boxes in the
// 128-byte swizzle, or (sw32) 16-element boxes in the 32-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int BH, int N, bool sw32 = false, int ld = kD) {
  EncodeTiledFn f = encode_fn();
  if (!f) {
    set_error_detail("cuTensorMapEncodeTiled entry point unavailable");
    return false;
  }
  cuuint64_t dims[3] = {(cuuint64_t)ld, (cuuint64_t)N, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)ld * 2, (cuuint64_t)N * ld * 2};
  cuuint32_t box[3] = {sw32 ? 16u : 64u, (cuuint32_t)kTile, 1}, es[3] = {1, 1, 1};
  const CUresult r = f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, sw32 ? CU_TENSOR_MAP_SWIZZLE_32B : CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char msg[96];
    snprintf(msg, sizeof msg, "cuTensorMapEncodeTiled returned CUresult %d", (int)r);
    set_error_detail(msg);
  }
  return r == CUDA_SUCCESS;
}

}  // namespace

// Map over a row-major bf16 matrix [rows][cols] (row pitch cols * 2 bytes) as a 3-D tensor with a unit
// outer dimension, boxes of box_cols x box_rows in the 128-byte swizzle, zero fill outside the matrix.
bool make_map_rows(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                   uint32_t box_rows) {
  EncodeTiledFn f = encode_fn();
  if (!f) {
    set_error_detail("cuTensorMapEncodeTiled entry point unavailable");
    return false;
  }
  cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, 1};
  cuuint64_t strides[2] = {(cuuint64_t)cols * 2, (cuuint64_t)cols * rows * 2};
  cuuint32_t box[3] = {box_cols, box_rows, 1}, es[3] = {1, 1, 1};
  const CUresult r = f(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char msg[96];
    snprintf(msg, sizeof msg, "cuTensorMapEncodeTiled returned CUresult %d", (int)r);
    set_error_detail(msg);
  }
  return r == CUDA_SUCCESS;
}

namespace {

// Dynamic shared memory of a launch: the layout plus alignment slack, never below 116 KB so that
// exactly one CTA (which owns all 512 TMEM columns) is resident per SM.
uint32_t smem_bytes(uint32_t layout_total) { return layout_total + 1024 > 116u * 1024 ? layout_total + 1024 : 116u * 1024; }

// Segments per head row.  Each CTA walks one segment of seg = ceil(tiles / s) tiles and owns an SM, so
// a launch of BH * s CTAs runs in ceil(BH * s / 152) waves of seg tiles.  Over the largest s that fits
// in w = 1 .. 8 waves, the count minimises waves * (seg + 1), the 1 standing for a CTA's fixed cost
// (set-up and epilogue); ties go to fewer segments.  At most 8 * 152 segments (or B*H, if larger) are
// used, so the causal aggregates stay independent of N.
int split_for(int BH, int tiles) {
  if (BH < 1 || tiles < 1) return 1;
  int best = 1;
  long long best_cost = -1;
  for (int w = 1; w <= 8; ++w) {
    const long long fit = (long long)w * kTargetCtas / BH;
    const int s = (int)std::max(1LL, std::min<long long>(fit, tiles));
    const int seg = cdiv(tiles, s);
    const int splits = cdiv(tiles, seg);
    const long long ctas = (long long)BH * splits;
    const long long cost = ((ctas + kTargetCtas - 1) / kTargetCtas) * (seg + 1);
    if (best_cost < 0 || cost < best_cost || (cost == best_cost && splits < best)) {
      best_cost = cost;
      best = splits;
    }
  }
  return best;
}

// Launches the per-tile kernels with NC components per row thread (2 * NC >= Kp).
template <int NC>
gma_status_t tc_launch(const gma_problem_t& p, gma_op_t op, int Nk, const TcPlan& pl, TcArgs a, const void* Q,
                       const void* K, const void* V, void* ws, cudaStream_t st) {
  const int BH = p.B * p.H;
  CUtensorMap mq, mk, mv;
  if (op == GMA_OP_RESPONSIBILITIES) {
    if (!make_map(&mq, Q, BH, p.N)) return GMA_ERR_CUDA;
    const uint32_t smem = smem_bytes(read_layout(pl.Kp).total);
    if (set_smem_optin((const void*)tc_resp_kernel<NC>, (int)smem, 0) != GMA_OK) return GMA_ERR_CUDA;
    a.fault = 0;
    GMA_LAUNCH_DEPENDENT("tc_resp", tc_resp_kernel<NC>, dim3(pl.splits, BH), kThreadsTc, smem, st, mq, a);
    return check_launch("launch tc_resp", (const void*)tc_resp_kernel<NC>);
  }
  if (op == GMA_OP_CAUSAL) {
    // the sweep's V tiles are four 16-dim boxes in the 32-byte swizzle
    CUtensorMap mv32, mo;
    if (!make_map(&mq, Q, BH, p.N) || !make_map(&mk, K, BH, p.N) || !make_map(&mv, V, BH, p.N) ||
        !make_map(&mv32, V, BH, p.N, true) || !make_map(&mo, a.out, BH, p.N))
      return GMA_ERR_CUDA;
    // a5: segment aggregates; a6: exclusive scan over segments; a7: chunked sweep (both sides of every
    // tile recomputed there)
    const uint32_t smem_w = smem_bytes(write_layout(pl.Kp).total);
    if (set_smem_optin((const void*)tc_write_kernel<false, NC>, (int)smem_w, 0) != GMA_OK) return GMA_ERR_CUDA;
    GMA_LAUNCH_DEPENDENT("tc_causal_aggregate", (tc_write_kernel<false, NC>), dim3(pl.splits, BH), kThreadsTc, smem_w,
                         st, mk, mv, a);
    if (gma_status_t e = check_launch("launch tc_causal_aggregate", (const void*)tc_write_kernel<false, NC>)) return e;
    a.fault = 0;
    const int n = pl.Kp * kStCols;
    if (set_carveout_max((const void*)tc_scan_kernel) != GMA_OK) return GMA_ERR_CUDA;
    GMA_LAUNCH_DEPENDENT("tc_causal_scan", tc_scan_kernel, dim3(cdiv(n, 128), BH), 128, 0, st, a.state, pl.splits, n,
                         (pl.off_agg - pl.off_state) / 4);
    if (gma_status_t e = check_launch("launch tc_causal_scan", (const void*)tc_scan_kernel)) return e;
    const uint32_t smem_c = smem_bytes(causal_layout(pl.Kp).total);
    if (set_smem_optin((const void*)tc_causal_kernel<NC>, (int)smem_c, 0) != GMA_OK) return GMA_ERR_CUDA;
    GMA_LAUNCH_DEPENDENT("tc_causal_chunk", tc_causal_kernel<NC>, dim3(pl.splits, BH), kThreadsTc, smem_c, st, mq, mk,
                         mv32, mo, a);
    return check_launch("launch tc_causal_chunk", (const void*)tc_causal_kernel<NC>);
  }
  // bidirectional / cross: write over the Nk keys with their own split plan (the state layout does not
  // depend on the sequence lengths; with Nk = 0 the zeroed state is the empty memory)
  if (Nk > 0) {
    gma_problem_t pk = p;
    pk.N = Nk;
    const TcPlan plk = tc_plan(pk, op);
    TcArgs aw = a;
    aw.N = Nk;
    aw.tiles = plk.tiles;
    aw.seg_tiles = plk.seg_tiles;
    aw.splits = plk.splits;
    if (!make_map(&mk, K, BH, Nk) || !make_map(&mv, V, BH, Nk)) return GMA_ERR_CUDA;
    const uint32_t smem_w = smem_bytes(write_layout(pl.Kp).total);
    if (pl.det) {
      // deterministic: every write CTA stores its own state, then one fixed-order sum per element; at
      // most one wave of CTAs (max(152, B*H) states in all, whatever the key length)
      const int cap = std::max(1, kTargetCtas / BH);
      if (aw.splits > cap) {
        aw.seg_tiles = cdiv(aw.tiles, cap);
        aw.splits = cdiv(aw.tiles, aw.seg_tiles);
      }
      aw.state = (float*)((char*)ws + pl.off_agg);
      const size_t agg_lim = (pl.total - pl.off_agg) / 4;
#ifdef GMA_BOUNDS_CHECK
      aw.lim.state = agg_lim;
#endif
      if (set_smem_optin((const void*)tc_write_kernel<false, NC>, (int)smem_w, 0) != GMA_OK) return GMA_ERR_CUDA;
      GMA_LAUNCH_DEPENDENT("tc_bidir_write", (tc_write_kernel<false, NC>), dim3(aw.splits, BH), kThreadsTc, smem_w,
                           st, mk, mv, aw);
      if (gma_status_t e = check_launch("launch tc_bidir_write", (const void*)tc_write_kernel<false, NC>)) return e;
      if (set_carveout_max((const void*)tc_state_sum_kernel) != GMA_OK) return GMA_ERR_CUDA;
      GMA_LAUNCH_DEPENDENT("tc_state_sum", tc_state_sum_kernel, dim3(cdiv(kStRow * pl.Kp, 128), BH), 128, 0, st,
                           (const float*)aw.state, aw.splits, pl.Kp, a.state, agg_lim, (pl.off_agg - pl.off_state) / 4);
      if (gma_status_t e = check_launch("launch tc_state_sum", (const void*)tc_state_sum_kernel)) return e;
    } else {
      if (set_smem_optin((const void*)tc_write_kernel<true, NC>, (int)smem_w, 0) != GMA_OK) return GMA_ERR_CUDA;
      GMA_LAUNCH_DEPENDENT("tc_bidir_write", (tc_write_kernel<true, NC>), dim3(plk.splits, BH), kThreadsTc, smem_w,
                           st, mk, mv, aw);
      if (gma_status_t e = check_launch("launch tc_bidir_write", (const void*)tc_write_kernel<true, NC>)) return e;
    }
  }
  if (op == GMA_OP_CAUSAL_STATE) return GMA_OK;  // the state alone
  a.fault = 0;
  CUtensorMap mo;
  if (!make_map(&mq, Q, BH, p.N) || !make_map(&mo, a.out, BH, p.N)) return GMA_ERR_CUDA;
  const uint32_t smem_r = smem_bytes(read2_layout(pl.Kp).total);
  if (set_smem_optin((const void*)tc_read2_kernel<2 * NC>, (int)smem_r, 0) != GMA_OK) return GMA_ERR_CUDA;
  GMA_LAUNCH_DEPENDENT("tc_bidir_read", tc_read2_kernel<2 * NC>, dim3(pl.splits, BH), kThreadsTc, smem_r, st, mq, mo, a);
  return check_launch("launch tc_bidir_read", (const void*)tc_read2_kernel<2 * NC>);
}

uint32_t g_fault_next = 0;  // test hook, consumed by the next launch of the write kernel
std::mutex g_fault_mu;

}  // namespace

TcPlan tc_plan(const gma_problem_t& p, gma_op_t op, bool det) {
  TcPlan t{};
  t.det = det;
  const int BH = p.B * p.H;
  t.Kp = p.K <= 64 ? 64 : (p.K <= 128 ? 128 : 256);  // = 4 NC: every row thread's logit columns are written
  t.tiles = cdiv(p.N, kTile);
  t.splits = split_for(BH, t.tiles > 0 ? t.tiles : 1);
  t.seg_tiles = cdiv(t.tiles > 0 ? t.tiles : 1, t.splits);
  t.splits = cdiv(t.tiles > 0 ? t.tiles : 1, t.seg_tiles);
  t.off_w = align_up(sizeof(Ctrl));
  t.off_c = align_up(t.off_w + (size_t)p.H * w_head_bytes(t.Kp));
  t.off_flags = align_up(t.off_c + (size_t)p.H * kCTable * 4);
  t.off_state = align_up(t.off_flags + (size_t)p.H * (kCTable / 8) * 4);
  size_t st = 0;
  if (op == GMA_OP_BIDIR || op == GMA_OP_CROSS || op == GMA_OP_CAUSAL_STATE) st = (size_t)BH * t.Kp * kStRow * 4;
  if (op == GMA_OP_CAUSAL) st = (size_t)BH * t.splits * t.Kp * kStCols * 4;  // segment aggregates
  t.off_agg = align_up(t.off_state + st);
  size_t agg = 0;
  // the deterministic write makes at most max(152, B*H) CTAs over any key length
  if (det && (op == GMA_OP_BIDIR || op == GMA_OP_CROSS || op == GMA_OP_CAUSAL_STATE))
    agg = (size_t)std::max(kTargetCtas, BH) * t.Kp * kStCols * 4;
  t.total = align_up(t.off_agg + agg);
  return t;
}

gma_status_t tc_run(const gma_problem_t& p, gma_op_t op, int Nk, const void* Q, const void* K, const void* V,
                    const float* mu, const float* sigma2, const float* log_pi, void* out, void* ws,
                    cudaStream_t st, bool clear_err, bool det, Ctrl* ctrl) {
  const TcPlan pl = tc_plan(p, op, det);
  const int BH = p.B * p.H;
  char* base = (char*)ws;
  TcArgs a{};
  a.w_img = (const uint8_t*)(base + pl.off_w);
  a.cbias = (const float*)(base + pl.off_c);
  a.range_flags = (const uint32_t*)(base + pl.off_flags);
  a.state = (float*)(base + pl.off_state);
  a.ctrl = ctrl ? ctrl : (Ctrl*)base;
  a.out = out;
  a.H = p.H;
  a.N = p.N;
  a.K = p.K;
  a.Kp = pl.Kp;
  a.tiles = pl.tiles;
  a.seg_tiles = pl.seg_tiles;
  a.splits = pl.splits;
  a.eps = p.eps;
  a.wait_ns = wait_limit_ns();
  TcLimits lim;
  lim.state = (pl.off_agg - pl.off_state) / 4;
  lim.out = op == GMA_OP_RESPONSIBILITIES ? (size_t)BH * p.N * p.K : 0;
  lim.w = pl.off_c - pl.off_w;
  lim.c = (pl.off_flags - pl.off_c) / 4;
  lim.flags = (pl.off_state - pl.off_flags) / 4;
#ifdef GMA_BOUNDS_CHECK
  a.lim = lim;
#endif
  if (op == GMA_OP_BIDIR) {
    std::lock_guard<std::mutex> lock(g_fault_mu);
    // GMA_FAULT_INJECT, read at the first bidirectional call of the process: a value other than "" or "0"
    // arms the withheld-load hook for that call
    static bool env_seen = false;
    if (!env_seen) {
      env_seen = true;
      const char* e = std::getenv("GMA_FAULT_INJECT");
      if (e && *e && !(e[0] == '0' && e[1] == 0)) g_fault_next |= 1u;
    }
    a.fault = g_fault_next;
    g_fault_next = 0;
  }
  const bool with_state = op == GMA_OP_BIDIR || op == GMA_OP_CAUSAL_STATE;  // write accumulator starts at zero
  const size_t zero_n = with_state ? (size_t)BH * pl.Kp * kStRow : 0;
  if (set_carveout_max((const void*)tc_prep_kernel) != GMA_OK) return GMA_ERR_CUDA;
  GMA_LAUNCH_DEPENDENT("tc_prep", tc_prep_kernel, dim3(kCTable / 8, p.H), 128, 0, st, mu, sigma2, log_pi, p.H, p.K, pl.Kp,
             (uint8_t*)a.w_img, (float*)a.cbias, a.ctrl, a.state, zero_n, (uint32_t*)a.range_flags, clear_err ? 1 : 0,
             lim);
  if (gma_status_t e = check_launch("launch tc_prep", (const void*)tc_prep_kernel)) return e;
  const int nc = pl.Kp <= 64 ? 16 : (pl.Kp <= 128 ? 32 : 64);  // components per row thread (4 per row)
  gma_status_t e = nc == 16   ? tc_launch<16>(p, op, Nk, pl, a, Q, K, V, ws, st)
                   : nc == 32 ? tc_launch<32>(p, op, Nk, pl, a, Q, K, V, ws, st)
                              : tc_launch<64>(p, op, Nk, pl, a, Q, K, V, ws, st);
  if (e != GMA_OK || op != GMA_OP_CAUSAL_STATE) return e;
  const size_t n = (size_t)BH * p.K * (kDv + 1);
  GMA_LAUNCH("tc_state_export", tc_state_export_kernel, (unsigned)std::min<size_t>((n + 255) / 256, 4096), 256, 0, st,
             a.state, p.K, pl.Kp, n, (float*)out, lim.state);
  return check_launch("launch tc_state_export", (const void*)tc_state_export_kernel);
}

bool tc_available() { return encode_fn() != nullptr; }

#ifdef GMA_BOUNDS_CHECK
namespace {
// An index one past an extent of three, checked and skipped: no memory is touched.
__global__ void bounds_selftest_kernel() {
  if (GMA_INB(threadIdx.x + 3, 3, 999)) asm volatile("" ::: "memory");
}
}  // namespace
gma_status_t tc_bounds_io(unsigned long long* h, bool clear) { return bounds_record_io(h, clear); }
gma_status_t bounds_selftest(cudaStream_t st) {
  GMA_LAUNCH("bounds_selftest", bounds_selftest_kernel, 1, 1, 0, st);
  return check_launch("launch bounds_selftest", (const void*)bounds_selftest_kernel);
}
#else
gma_status_t tc_bounds_io(unsigned long long*, bool) { return GMA_ERR_UNSUPPORTED; }
gma_status_t bounds_selftest(cudaStream_t) { return GMA_ERR_UNSUPPORTED; }
#endif

void tc_set_fault_injection(uint32_t mask) {
  std::lock_guard<std::mutex> lock(g_fault_mu);
  g_fault_next = mask;
}

}  // namespace gma

#ifdef GMA_TRACE
extern "C" GMA_API int gma_debug_trace_read(unsigned long long* host, size_t n) {
  if (n > (size_t)gma::kTraceIds * gma::kTraceTiles) n = (size_t)gma::kTraceIds * gma::kTraceTiles;
  return cudaMemcpyFromSymbol(host, gma::g_trace, n * sizeof(unsigned long long)) == cudaSuccess ? 0 : -1;
}
extern "C" GMA_API int gma_debug_span_read(unsigned long long* host, size_t n) {
  if (n > (size_t)gma::kSpanSlots * gma::kSpanCtas) n = (size_t)gma::kSpanSlots * gma::kSpanCtas;
  return cudaMemcpyFromSymbol(host, gma::g_span, n * sizeof(unsigned long long)) == cudaSuccess ? 0 : -1;
}
extern "C" GMA_API int gma_debug_trace_clear(void) {
  static unsigned long long zero[gma::kSpanSlots * gma::kSpanCtas];
  if (cudaMemcpyToSymbol(gma::g_span, zero, sizeof zero) != cudaSuccess) return -1;
  return cudaMemcpyToSymbol(gma::g_trace, zero, (size_t)gma::kTraceIds * gma::kTraceTiles * 8) == cudaSuccess ? 0 : -1;
}
#endif

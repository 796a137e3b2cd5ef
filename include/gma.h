/*
 * gma.h -- C ABI of libgma.so: the forward pass of Gaussian Mixture Attention
 * (GMA) on one NVIDIA GB300 (sm_103a).
 *
 * Method: "Gaussian Mixture Attention: Linear-Time Sequence Mixing via
 * Probabilistic Latent Routing" (Huang & Raza, arXiv 2606.18283), as described
 * on the gist.science technical summaries ("Core mechanism" items 1-2,
 * "Variants and training" item 3) and in the English abstract on fugumt.com.
 *
 *   gamma_ik = p(z = k | x_i)             GMM posterior over K diagonal Gaussians
 *                                         with means mu_k, variances sigma2_k and
 *                                         priors pi_k, shared by queries and keys
 *   Vt = Gamma_K^T V,  Z = Gamma_K^T 1    write phase (K-slot latent memory)
 *   O  = Gamma_Q Vt / (Gamma_Q Z + eps)   read phase
 *   causal: Vt, Z replaced by inclusive prefix sums over key positions j <= i.
 *
 * Conventions shared by every entry point:
 *   - Every pointer argument except `p` is a DEVICE pointer (cudaMalloc'd or
 *     equivalent) owned by the caller.  The library allocates and frees
 *     nothing; scratch memory is the caller's workspace `ws`.
 *   - Tensors are dense, row-major, innermost dimension last:
 *       Q, K, X : [B, H, N, d]      V, O : [B, H, N, dv]
 *       mu, sigma2 : [H, K, d] float32      log_pi : [H, K] float32
 *     Q, K, X, V, O use the I/O dtype `p->dtype`; every base pointer must be
 *     16-byte aligned, ws 256-byte aligned.
 *   - sigma2 is the variance after the caller's reparametrisation and floor
 *     (softplus + lower bound), must be > 0; log_pi is the log prior (any
 *     constant offset per head cancels).  One component set per head routes
 *     both queries and keys.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *     asynchronous on it; argument errors are returned before anything is
 *     launched.  No C++ exception crosses this interface.
 *   - A device-side wait that runs out of time sets an error word in `ws`
 *     (never a trap); gma_check_device_error() reports it.
 *   - Supported in this version: d == dv == 64, 1 <= K <= 256, N >= 0
 *     (N == 0 is a no-op), B, H >= 1, B*H*N < 2^31.
 *   - Precision: dtype GMA_F32 computes in float32 on the CUDA cores;
 *     GMA_BF16 runs the log-density contraction with fp16 operands and the
 *     write/read contractions with bf16 operands on the tcgen05 tensor cores,
 *     all accumulated in float32; the output is rounded to bf16 (RNE).
 *     For GMA_BF16, |q|, |k| must stay below 255 (fp16 range of q^2), and the folded
 *     parameters must fit fp16: sigma2 > 1.1e-5 (-1/2 sigma2^-1 log2(e) > -65504),
 *     |mu| / sigma2 < 45000 and |c'_k| < 1.6e7 for the component constant
 *     c'_k = (log pi_k - 1/2 sum_d (mu^2 / sigma2 + log sigma2)) log2(e).  A call whose
 *     parameters break these bounds (or hold NaN / inf) still runs, and sets the
 *     workspace error word: gma_check_device_error() then returns GMA_ERR_RANGE.
 *     Accuracy of GMA_BF16 (the bounds above only keep the operands finite): the
 *     expanded form a x^2 + b x + c' keeps about 2^-12 of each term's size, so the
 *     absolute log-density error grows with sigma2^-1 (x^2 + |mu x| + mu^2) summed
 *     over the dimensions.  With unit-scale q, k, mu and sigma2 = softplus(N(0, s))
 *     + 1e-2 (s <= 1), or a minority of components at the 1e-2 floor, outputs stay
 *     within 2e-2 of exact (max |error| / max |O|); when most components or
 *     dimensions sit at the floor, or |q|, |k| grow past ~3 with variances near it,
 *     the error reaches 0.03 - 0.16.  Use GMA_F32 (centred form, float32) there.
 */
#ifndef GMA_H_
#define GMA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define GMA_API __attribute__((visibility("default")))
#else
#define GMA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GMA_OK = 0,
  GMA_ERR_INVALID_ARG = 1, /* null pointer, bad shape, misalignment, eps < 0 */
  GMA_ERR_UNSUPPORTED = 2, /* d, dv, K or dtype outside what this build runs */
  GMA_ERR_WORKSPACE = 3,   /* ws_bytes smaller than gma_workspace_bytes() */
  GMA_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed */
  GMA_ERR_TIMEOUT = 5,     /* a bounded device wait gave up (see ws error word) */
  GMA_ERR_RANGE = 6        /* bf16 I/O: a folded parameter does not fit the fp16 operands (see ws error word) */
} gma_status_t;

typedef enum { GMA_F32 = 0, GMA_BF16 = 1 } gma_dtype_t;

typedef enum {
  GMA_OP_RESPONSIBILITIES = 0,
  GMA_OP_BIDIR = 1,
  GMA_OP_CAUSAL = 2,
  GMA_OP_CROSS = 3,
  GMA_OP_CAUSAL_STATE = 4,
  GMA_OP_CAUSAL_DECODE = 5,
  GMA_OP_BACKWARD_BIDIR = 6,
  GMA_OP_BACKWARD_CAUSAL = 7,
  GMA_OP_PROJECTED_BIDIR = 8,
  GMA_OP_PROJECTED_CAUSAL = 9
} gma_op_t;

typedef struct {
  int B, H, N; /* batch, heads, sequence length */
  int d, dv;   /* routing (query/key) width and value width; both 64 */
  int K;       /* mixture components per head */
  gma_dtype_t dtype;
  float eps;   /* read-phase denominator offset, >= 0 */
} gma_problem_t;

/* Bytes of device workspace `op` needs for problem `p` (0 if p is invalid). */
GMA_API size_t gma_workspace_bytes(const gma_problem_t *p, gma_op_t op);

/*
 * Responsibilities Gamma = p(z | x) of routing vectors X.
 * Passage: gist.science summary, "Core mechanism" item 1 (standard GMM
 * posterior with learned mu_k, diagonal Sigma_k, prior pi_k).
 *   X      [B,H,N,d] in p->dtype        gamma_out [B,H,N,K] float32 (written)
 * Rows of gamma_out are non-negative and sum to 1.
 */
GMA_API gma_status_t gma_responsibilities(const gma_problem_t *p, const void *X, const float *mu, const float *sigma2,
                                  const float *log_pi, float *gamma_out, void *ws, size_t ws_bytes, void *stream);

/*
 * Bidirectional GMA forward: O = Gamma_Q (Gamma_K^T V) / (Gamma_Q (Gamma_K^T 1) + eps).
 * Passage: gist.science summary, "Core mechanism" item 2 (write phase, read
 * phase); "Variants and training" item 3 (bidirectional form).
 *   Q, K [B,H,N,d], V [B,H,N,dv] in p->dtype;  O [B,H,N,dv] in p->dtype (written).
 * O may not alias any input.
 */
GMA_API gma_status_t gma_forward_bidir(const gma_problem_t *p, const void *Q, const void *K, const void *V, const float *mu,
                               const float *sigma2, const float *log_pi, void *O, void *ws, size_t ws_bytes,
                               void *stream);

/*
 * Bidirectional forward for callers that cannot allocate device memory (for example a plugin
 * whose host framework forbids allocation on its execute path, a runtime that plans every
 * device byte ahead of time, or a C program without a device allocator).  The method itself
 * has no counterpart to this entry point: it computes exactly what gma_forward_bidir computes,
 * but its scratch memory is a 16 MiB array inside the library (a file-scope __device__ array,
 * held by every GPU that loads the library until the process exits) instead of a caller
 * workspace.  Allocates nothing and calls no allocating routine.
 *   - Problems whose gma_workspace_bytes(p, GMA_OP_BIDIR) exceeds gma_static_ws_capacity()
 *     return GMA_ERR_WORKSPACE before launching anything.
 *   - The first call on a device looks up the array's device address (cudaGetSymbolAddress
 *     with that device current) and caches it together with the identity of the current CUDA
 *     context; a call in another context (for example after cudaDeviceReset) looks it up again.
 *     Make the first call on a device before any stream capture.
 *   - Every call shares the one array; each call clears what must start at zero.  Calls whose
 *     GPU work overlaps (several streams or host threads) race on it and must be serialised.
 *   - A bounded device wait that runs out sets the error word at the start of the array (the
 *     call itself has already returned GMA_OK); gma_static_ws_check_error() reads it.
 * Arguments and layouts as gma_forward_bidir, without ws / ws_bytes.
 */
GMA_API gma_status_t gma_forward_bidir_static_ws(const gma_problem_t *p, const void *Q, const void *K, const void *V,
                                                 const float *mu, const float *sigma2, const float *log_pi, void *O,
                                                 void *stream);

/* Size in bytes of the library-held scratch array used by gma_forward_bidir_static_ws(). */
GMA_API size_t gma_static_ws_capacity(void);

/*
 * gma_check_device_error() for the library-held array of gma_forward_bidir_static_ws(): synchronises
 * `stream`, then reads the array's error word into host memory (allocating nothing).  GMA_OK if no
 * device wait of the most recent call on the current device timed out, GMA_ERR_TIMEOUT if one did,
 * GMA_ERR_CUDA if the synchronisation or the copy failed.  Like the entry point it serves, it has no
 * counterpart in the method.
 */
GMA_API gma_status_t gma_static_ws_check_error(void *stream);

/*
 * Causal GMA forward: row i uses the inclusive prefix sums over keys j <= i,
 *   O_i = gamma_Qi . (sum_{j<=i} gamma_Kj v_j^T) / (gamma_Qi . sum_{j<=i} gamma_Kj + eps).
 * Passage: gist.science summary, "Variants and training" item 3 (prefix sums
 * of the latent memory and normaliser; O at position i depends on j <= i only).
 * Same arguments and layouts as gma_forward_bidir.  The workspace does not grow with N: it holds
 * the per-segment prefix states (at bf16 I/O at most 8 x 152 segments over all B*H rows, or B*H
 * segments if B*H is larger); no per-position
 * responsibilities are stored.  With bf16 I/O the key responsibilities are computed twice -- once for
 * the segment sums, once inside the chunked sweep -- and never leave the chip.
 */
GMA_API gma_status_t gma_forward_causal(const gma_problem_t *p, const void *Q, const void *K, const void *V, const float *mu,
                                const float *sigma2, const float *log_pi, void *O, void *ws, size_t ws_bytes,
                                void *stream);

/*
 * Cross-attention GMA forward: N queries of one sequence read the latent memory written by the
 * Nk keys / values of another,
 *   O = Gamma_Q (Gamma_K^T V) / (Gamma_Q (Gamma_K^T 1) + eps),  Gamma_Q [N x K], Gamma_K [Nk x K].
 * Passage: gist.science summary, "Significance and claims" (cross-attention applications named as
 * the next step beyond the self-attention setting); the write and read phases are those of
 * "Core mechanism" item 2 with the key sequence of its own length.
 *   Q [B,H,N,d] (N = p->N), K [B,H,Nk,d], V [B,H,Nk,dv] in p->dtype; O [B,H,N,dv] in p->dtype.
 * Nk >= 0; with Nk = 0 the memory is empty and O = 0 (eps > 0).  K and V may be null when
 * Nk = 0, Q and O when N = 0.  O may not alias any input.  The workspace is the bidirectional
 * one: gma_workspace_bytes(p, GMA_OP_CROSS) == gma_workspace_bytes(p, GMA_OP_BIDIR), and
 * neither depends on N or Nk.
 */
GMA_API gma_status_t gma_forward_cross(const gma_problem_t *p, int Nk, const void *Q, const void *K, const void *V,
                                       const float *mu, const float *sigma2, const float *log_pi, void *O, void *ws,
                                       size_t ws_bytes, void *stream);

/*
 * Causal state (latent memory and normaliser after a prefix of keys), the object a decode step
 * keeps between calls.  Layout: float32 [B][H][K][dv + 1]; row k of head (b, h) holds
 * sum_j gamma_jk v_j (dv values) followed by sum_j gamma_jk, over the keys seen so far.
 * Passage: gist.science summary, "Variants and training" item 3 (prefix sums of the latent memory
 * and the normaliser); "Core mechanism" item 2 (Vt = Gamma_K^T V, Z = Gamma_K^T 1).
 */
GMA_API size_t gma_state_bytes(const gma_problem_t *p); /* B*H*K*(dv+1)*4, or 0 if p is invalid */

/*
 * State after the N keys / values of a prompt: state = sum_{j < N} gamma_Kj [v_j | 1] per (b, h).
 *   K [B,H,N,d], V [B,H,N,dv] in p->dtype;  state float32 [B][H][K][dv+1] (written; N = 0 gives zeros).
 * Workspace: gma_workspace_bytes(p, GMA_OP_CAUSAL_STATE).
 */
GMA_API gma_status_t gma_causal_state(const gma_problem_t *p, const void *K, const void *V, const float *mu,
                                      const float *sigma2, const float *log_pi, float *state, void *ws,
                                      size_t ws_bytes, void *stream);

/*
 * Causal decode step: the recurrent form of the prefix sums.  For each (b, h), the N = p->N new
 * tokens are taken in order t = 0..N-1:
 *   state += gamma_K(k_t) [v_t | 1],   O_t = gamma_Q(q_t) . state[:, :dv] / (gamma_Q(q_t) . state[:, dv] + eps),
 * so O_t equals the causal forward output of that position over the whole sequence seen so far.
 * Passage: gist.science summary, "Variants and training" item 3 (causal form: O_i depends on the
 * prefix j <= i only, through running sums).
 *   Q, K [B,H,N,d], V [B,H,N,dv] in p->dtype; O [B,H,N,dv] in p->dtype (written);
 *   state float32 [B][H][K][dv+1] (read and updated in place; see gma_causal_state).
 * Computed in float32 on the CUDA cores in two launches: the parameter fold of every head (1 / sigma2,
 * the component constants) into the workspace, then one CTA per (b, h) that keeps the head's state and
 * folded parameters in shared memory; meant for small N per call.  Workspace:
 * gma_workspace_bytes(p, GMA_OP_CAUSAL_DECODE): a control block (not cleared here; its error word
 * records a copy into shared memory that did not land within 1 s, which leaves the state untouched,
 * see gma_check_device_error) and the folded parameters, 4 H (128 (K + 1) + K) bytes rounded up.
 * O may not alias any input or the state.
 */
GMA_API gma_status_t gma_causal_decode(const gma_problem_t *p, const void *Q, const void *K, const void *V,
                                       const float *mu, const float *sigma2, const float *log_pi, float *state,
                                       void *O, void *ws, size_t ws_bytes, void *stream);

/*
 * The decode step split for fixed parameters: gma_decode_prepare runs only the parameter fold of
 * gma_causal_decode into the workspace (gma_workspace_bytes(p, GMA_OP_CAUSAL_DECODE), the same layout;
 * p->N is not used), and gma_causal_decode_prepared runs only the decode with the folded parameters
 * found there, once per call, as long as the parameters have not changed.  The outputs and the state
 * are bit-identical to gma_causal_decode with the same parameters.  A prepared call is one launch,
 * ordered after everything earlier on the stream; a prepare must be ordered after any decode still
 * reading the workspace (same stream, or an event).  Errors as gma_causal_decode; a workspace that was
 * never prepared for these parameters is not detected (the outputs are then those of whatever folded
 * parameters it holds).
 */
GMA_API gma_status_t gma_decode_prepare(const gma_problem_t *p, const float *mu, const float *sigma2,
                                        const float *log_pi, void *ws, size_t ws_bytes, void *stream);
GMA_API gma_status_t gma_causal_decode_prepared(const gma_problem_t *p, const void *Q, const void *K, const void *V,
                                                float *state, void *O, void *ws, size_t ws_bytes, void *stream);

/*
 * Backward pass of the bidirectional forward: given dO = dL/dO, the gradients of L with respect to
 * every input and parameter,
 *   dQ, dK [B,H,N,d], dV [B,H,N,dv] in p->dtype (written);
 *   dmu, dsigma2 [H,K,d], dlog_pi [H,K] float32 (written; summed over the batch and over every
 *   query and key row, since one mixture per head routes both).
 * Passage: gist.science summary, "Variants and training" item 3 (the Gaussian components are
 * parameterised differentiably and trained end to end); the chain rule runs back through the read
 * and write phases of "Core mechanism" item 2 and the GMM posterior of item 1.  The gradient with
 * respect to sigma2 and log_pi is the one of this function's inputs: a caller that reparameterises
 * (softplus, log-softmax) applies its own chain rule on top.
 *   Q, K, V, mu, sigma2, log_pi, eps: as gma_forward_bidir;  dO [B,H,N,dv] in p->dtype.
 * Computed in float32 on the CUDA cores; with bf16 I/O the state Gamma_K^T [V | 1] and every key's
 * and query's gamma come from the tensor-core forward kernels (so the parameter-range check of the bf16 forward,
 * GMA_ERR_RANGE, applies).  The workspace, gma_workspace_bytes(p, GMA_OP_BACKWARD_BIDIR), grows with N
 * (it holds the per-row softmax gradients, 8 B*H*N*K bytes, and with bf16 I/O the tensor-core
 * kernels' workspace).
 * No output may alias an input.
 */
GMA_API gma_status_t gma_backward_bidir(const gma_problem_t *p, const void *Q, const void *K, const void *V,
                                        const float *mu, const float *sigma2, const float *log_pi, const void *dO,
                                        void *dQ, void *dK, void *dV, float *dmu, float *dsigma2, float *dlog_pi,
                                        void *ws, size_t ws_bytes, void *stream);

/*
 * Backward pass of the causal forward: the same outputs, arguments and layouts as
 * gma_backward_bidir, for O_i = gamma_Qi . Vt_i / (gamma_Qi . Z_i + eps) over the inclusive prefix
 * j <= i.  Passage: gist.science summary, "Variants and training" item 3 (the causal form by prefix
 * sums, trained end to end).  With S_i the running state, u_i = [G_i / den_i | -(G_i . O_i) / den_i] and
 * R_j = sum_{i >= j} gamma_Qi u_i^T: dgamma_Qi = S_i u_i, dgamma_Kj = R_j [v_j | 1], dv_j = R_j^T gamma_Kj,
 * computed per segment (forward over the queries, backward over the keys) on the CUDA cores in float32.
 * Workspace: gma_workspace_bytes(p, GMA_OP_BACKWARD_CAUSAL), growing with N (per-row softmax
 * gradients, the queries' responsibilities and the u rows: 4 B*H*N*(3K + dv + 1) bytes and more).
 */
GMA_API gma_status_t gma_backward_causal(const gma_problem_t *p, const void *Q, const void *K, const void *V,
                                         const float *mu, const float *sigma2, const float *log_pi, const void *dO,
                                         void *dQ, void *dK, void *dV, float *dmu, float *dsigma2, float *dlog_pi,
                                         void *ws, size_t ws_bytes, void *stream);

/*
 * Forward pass of a Transformer block's attention with GMA in place of softmax attention, from the
 * block input: Q, K, V are the linear projections of X (with bias), split into H heads of 64, then
 * the bidirectional (causal = 0) or causal (causal = 1) forward above runs on them.
 * Passage: gist.science summary, "Variants and training" (GMA as the sequence mixer of a
 * Transformer language model; the experiments' model has d_model = 768 and 12 heads).
 *   X     [B, N, dm] in p->dtype, dm a multiple of 8 (GMA_ERR_UNSUPPORTED otherwise)
 *   Wqkv  [dm, 3 * H * 64] in p->dtype: columns 0 .. H*64-1 give Q (head h = columns 64h .. 64h+63),
 *         the next H*64 give K, the last H*64 give V
 *   bqkv  [3 * H * 64] float32 bias, same column order
 *   O     [B, H, N, 64] in p->dtype (written)
 * bf16: the projection is one tcgen05 GEMM (float32 accumulation in tensor memory) whose epilogue
 * adds the bias in float32, rounds once to bf16 and writes Q, K, V in the [B, H, N, 64] layout
 * inside the workspace.  float32: one library GEMM (cuBLASLt, float32 accumulation and output)
 * followed by one kernel doing the same.  Q, K, V make one round trip through HBM (the forward
 * kernels hold no room for the 3 x dm-wide weight slices).  Workspace: gma_workspace_bytes(p,
 * GMA_OP_PROJECTED_BIDIR or GMA_OP_PROJECTED_CAUSAL); its first part is the forward's own workspace,
 * so gma_check_device_error(ws, ...) applies unchanged (it also reports the projection's bounded
 * waits).
 */
GMA_API gma_status_t gma_forward_projected(const gma_problem_t *p, int causal, int dm, const void *X,
                                           const void *Wqkv, const float *bqkv, const float *mu,
                                           const float *sigma2, const float *log_pi, void *O, void *ws,
                                           size_t ws_bytes, void *stream);

/*
 * Synchronises `stream`, then reads the error word kept at the start of `ws`:
 * GMA_OK if no device wait timed out since the word was last cleared (every
 * forward/responsibilities call clears it when it starts), GMA_ERR_TIMEOUT if
 * one did, GMA_ERR_RANGE if (bf16 I/O) a folded parameter did not fit the fp16
 * operands (see the precision note above), GMA_ERR_CUDA if the synchronisation
 * itself failed.  `ws` must be a
 * workspace previously passed to one of the calls above.
 */
GMA_API gma_status_t gma_check_device_error(void *ws, void *stream);

/*
 * Time limit of every bounded device wait of the bf16 (tensor-core) kernels,
 * process-wide: a wait that runs this long sets the workspace error word
 * (GMA_ERR_TIMEOUT through gma_check_device_error()) and the kernel returns.
 * The library has no counterpart in the pages; it is the failure-detection knob
 * of this implementation.  gma_set_wait_limit_ns(0) restores the default: the
 * environment variable GMA_WAIT_LIMIT_MS (milliseconds, read once, clamped to
 * [1 ms, 10 min]) if set, else 1 s.  Other values must lie in [1e6, 6e11] ns,
 * else GMA_ERR_INVALID_ARG and the limit is unchanged.  Takes effect for calls
 * made afterwards; kernels already enqueued keep the limit they were given.
 * gma_get_wait_limit_ns() returns the limit the next call will use.
 */
GMA_API gma_status_t gma_set_wait_limit_ns(uint64_t ns);
GMA_API uint64_t gma_get_wait_limit_ns(void);

/*
 * Deterministic reduction mode, process-wide.  By default the bidirectional
 * write (gma_forward_bidir / gma_forward_cross / gma_causal_state and the
 * projected bidirectional form) adds the partial states of its CTAs into one
 * [K][dv + 1] state per head with float32 atomic (bf16 path: bulk reduce-add)
 * operations, and the backward pass does the same for the state gradient and
 * the parameter sums, so repeated calls agree within rounding but not bit for
 * bit.  The pages fix no summation order: every order computes the same sums of
 * the write (the linear-time form of "Latent memory routing").  With the mode
 * on, each CTA stores its partial in the workspace and one thread per element
 * adds them up in CTA order, and the float32 projection's library GEMM uses no
 * split-K reduction, so repeated calls with the same inputs, workspace size
 * and device give bitwise-equal outputs.  The causal forward, the
 * responsibilities and the decode already sum in a fixed order in both modes.
 * The mode enlarges the workspaces of the affected calls (query
 * gma_workspace_bytes() after setting it): by max(152, B*H) x Kp x 80 floats
 * (bf16 forward, whose write then runs at most one CTA per SM; Kp = K rounded
 * up to 64, 128 or 256), (304 + B*H) x K x 65 floats (float32 forward), or the
 * backward's partials.  A call whose
 * workspace was sized with the mode off fails with GMA_ERR_WORKSPACE when the
 * mode is on.  mode: 1 on, 0 off, -1 the default, which is on when the
 * environment variable GMA_DETERMINISTIC (read once) is set to anything but
 * "" or "0".  Other values: GMA_ERR_INVALID_ARG.  gma_get_deterministic()
 * returns 1 if the next call will use the mode, else 0.
 */
GMA_API gma_status_t gma_set_deterministic(int mode);
GMA_API int gma_get_deterministic(void);

/* Static, NUL-terminated description of a status code. */
GMA_API const char *gma_status_string(gma_status_t s);

/* Static text describing the step that made the calling thread's most recent call return
 * GMA_ERR_CUDA (with CUDA's own message), or "" if none did. */
GMA_API const char *gma_last_error(void);

/* ABI version of this library: (major << 16) | minor. */
GMA_API int gma_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GMA_H_ */

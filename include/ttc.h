/*
 * libttc: forward and backward of a rank-gated tensor-train (TT) linear layer
 * on one NVIDIA GB300 GPU (sm_103a).
 *
 * The layer (CoMERA project page, "Learn the ranks while training", figure of
 * a tensor-train layer with rank-control diagonals):
 *   W (M x N), N = n_1*...*n_d, M = m_1*...*m_d, is a chain of 2d cores
 *   G_k of shape (r_{k-1}, s_k, r_k), r_0 = r_2d = 1, input modes first:
 *   s = (n_1..n_d, m_1..m_d).  A diagonal D_k sits on every internal link
 *   k = 1..2d-1; the rank of a link is the number of nonzeros of D_k, and a
 *   zero entry drops the matching slice of both neighbouring cores.
 *   With j = (j_1..j_d), i = (i_1..i_d) row-major (first mode most
 *   significant):
 *     W[i,j] = G_1[0,j_1,:] D_1 G_2[:,j_2,:] ... D_d ... G_2d[:,i_d,0]
 *   forward   y[t,i] = sum_j W[i,j] x[t,j]                (no bias)
 *   backward  for L = sum dy[t,i] y[t,i]:  dx = dy W,  dG_k = dL/dG_k,
 *             dD_k = dL/dD_k, except that dD_k[a] is returned as 0 where
 *             D_k[a] == 0 (the rank-truncated layer has no such parameter).
 * The contraction order is the one of the project page, "Making small tensor
 * operations fast on GPUs", bullet "One contraction order for both passes":
 * the input-side cores are merged into A (N x r_d), the output-side cores
 * into B (r_d x M), and x is contracted through them
 * (y = ((x A) diag(D_d)) B).
 *
 * Conventions for every call:
 *  - All device pointers are plain CUDA device addresses owned by the caller.
 *    The library allocates no device memory at run time; it uses the
 *    caller's workspace.  It does hold a few module-scope device arrays,
 *    which every GPU that loads the library keeps until the process exits,
 *    whether or not it calls the functions that use them: the
 *    tt_forward_noalloc scratch (32 MiB), the status words and the TT-matrix
 *    lookup's unit constants (a few bytes).
 *  - Calls on different streams may overlap on the GPU when each has its own
 *    workspace: everything a call writes (grid-barrier counters included)
 *    lives in its workspace or its outputs.  Calls that share a workspace
 *    must be ordered (one stream, or events).
 *  - stream is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Calls only enqueue work; none synchronises, except
 *    tt_get_device_status.
 *  - Argument errors are reported before anything is enqueued.  A failed
 *    launch returns TT_ERR_CUDA.  Errors found on the device (a bounded wait
 *    that ran out, a failed consistency check) are recorded in a status word
 *    that the library keeps in device memory, one per GPU (a module-scope
 *    variable, zero at load), and read back by tt_get_device_status.
 *  - Activations: x is (T, N), y is (T, M), dy is (T, M), dx is (T, N), all
 *    row-major, dense, in the plan's activation type (f32 or bf16), 16-byte
 *    aligned.  Cores, diagonals and their gradients are f32.
 *  - Packed parameters: one f32 buffer holding G_1..G_2d, each
 *    (r_{k-1}, s_k, r_k) row-major, followed by D_1..D_{2d-1}
 *    (tt_param_layout gives the offsets).  dparams has the same layout.
 */
#ifndef TTC_H
#define TTC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TT_MAX_D 4 /* order 2d <= 8 */

typedef enum tt_status {
  TT_OK = 0,
  TT_ERR_INVALID_ARG = 1, /* bad descriptor, NULL or misaligned pointer, T < 0 */
  TT_ERR_UNSUPPORTED = 2, /* valid layer the library has no kernel for */
  TT_ERR_WORKSPACE = 3,   /* workspace missing or smaller than tt_workspace_size */
  TT_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
  TT_ERR_TIMEOUT = 5,     /* a bounded device-side wait ran out (device status) */
  TT_ERR_DEVICE = 6       /* a device-side consistency check failed (device status) */
} tt_status;

/* Activation types.  TT_DT_E4M3: x and dy are one-byte OCP FP8 E4M3
 * ("e4m3fn": bias 7, 3 mantissa bits, largest finite 448, NaN 0x7F/0xFF)
 * codes, y and dx are bf16; the cores, diagonals and gradients stay fp32 and
 * every product accumulates in fp32.  This is the FP8/FP32 mixed precision of
 * the CoMERA poster digest (its FP8-mix speedup table and the mixed-precision
 * DLRM results), read as FP8 storage of the activations. */
typedef enum tt_dtype { TT_DT_F32 = 0, TT_DT_BF16 = 1, TT_DT_E4M3 = 2 } tt_dtype;

/* flags of tt_desc */
#define TT_ACCUMULATE 1u /* backward adds into dparams instead of overwriting */
/* The backward reuses the merged cores that the forward left in the
 * workspace, as the CoMERA project page describes for its contraction path
 * (the forward keeps its intermediate results for the backward pass).  The
 * caller guarantees that a tt_forward call with the same plan, the same
 * params and the same workspace came before, with nothing else using the
 * workspace in between; then tt_backward skips re-merging the cores (a
 * backward of T == 0 tokens ignores the flag: a forward of none does no work).  In an
 * FFN plan (both descs must carry the same flags) each layer then keeps its
 * merges in a workspace region of its own. */
#define TT_REUSE_MERGE 2u
/* Implies TT_REUSE_MERGE.  On the tensor-core path (bf16 or E4M3 activations)
 * the forward also keeps z' = (x A) diag(D_d) for every token in the
 * workspace (bf16, T x 64 values: 128 more bytes a token, counted by
 * tt_workspace_size), and the backward reads it instead of computing x A
 * again, so it streams x once instead of twice.  The caller guarantees in
 * addition that the backward gets the forward's x and T.  The f32 path
 * ignores it.  In a bf16 FFN plan (and a bf16 multi-layer plan) every layer
 * keeps its z' the same way; without the flag the fused FFN and multi-layer
 * backward compute them first (one more pass over x). */
#define TT_REUSE_Z 4u
/* Bit-reproducible gradients: the same inputs give the same dx and dparams
 * bit for bit, run after run, on a given GPU model.  Every sum over tokens
 * is taken in a fixed order: 128-token tiles, each CTA adding its tiles in
 * order into a slot of its own (TMA bulk add with completion awaited between
 * tiles), the slots then summed in CTA order by one more kernel; the merge
 * backward runs without atomic K splits (split partials reduced in split
 * order, one more engine phase); the f32 path reduces without atomics; a
 * bf16 FFN pair runs layer by layer.  Costs workspace (up to 160 slots of
 * (N + M + 4) x 64 floats, counted by tt_workspace_size) and time.  The
 * CoMERA pages do not discuss reproducibility; this is the training
 * requirement of a library boundary. */
#define TT_DETERMINISTIC 8u

typedef struct tt_desc {
  int d;                        /* 1..TT_MAX_D: number of input (= output) modes */
  int in_modes[TT_MAX_D];       /* n_1..n_d, each >= 1 */
  int out_modes[TT_MAX_D];      /* m_1..m_d, each >= 1 */
  int ranks[2 * TT_MAX_D + 1];  /* r_0..r_2d; r_0 = r_2d = 1, others >= 1 */
  int act;                      /* tt_dtype of x, y, dx, dy (E4M3: y, dx bf16) */
  unsigned flags;               /* TT_ACCUMULATE | TT_REUSE_MERGE | TT_REUSE_Z | TT_DETERMINISTIC */
} tt_desc;

typedef struct tt_plan_s tt_plan_t; /* opaque, immutable host object */

/* Rank caps read off the printed rank table (project page, "Results",
 * "Internal tensor-train ranks of each layer in one encoder block"):
 * r_k = min(R, prod s_<=k, prod s_>k), r_0 = r_2d = 1.  ranks receives 2d+1
 * values.  Host only. */
tt_status tt_default_ranks(int d, const int* in_modes, const int* out_modes, int R,
                           int* ranks);

/* Validate desc and build a plan (host only; no device work, no allocation on
 * the device).  *out is owned by the caller and freed with tt_destroy.
 * TT_ERR_INVALID_ARG for a malformed desc (a rank outside 1..4096 among
 * them); TT_ERR_UNSUPPORTED for N or M above 2^20 or a merged intermediate
 * (the packed parameters, a prefix product of the cores, the merged A or B)
 * of 2^31 elements or more; TT_ERR_UNSUPPORTED as well for an E4M3 layer
 * outside the fused tensor-core kernels' shapes (N, M multiples of 16 and at
 * least 128, middle rank r_d <= 64): E4M3 has no other path. */
tt_status tt_plan(const tt_desc* desc, tt_plan_t** out);

/* FFN pair y = TT_down(GELU(TT_up(x))) with GELU(h) = h Phi(h).  Up's
 * output width must equal down's input width and both must use the same act
 * type and flags (F32 or BF16; E4M3 gives TT_ERR_UNSUPPORTED).  A bf16 pair
 * whose layers fit the tensor-core kernels runs fused, h never leaving the
 * SM, with Phi(h) = (1 + tanh(sqrt(2/pi)(h + 0.044715 h^3))) / 2 (Hendrycks
 * and Gimpel's tanh form; |Phi error| <= 1.8e-4, below a bf16 rounding of
 * h); every other pair evaluates erf to within 1.5e-7 (Abramowitz and
 * Stegun 7.1.26). */
tt_status tt_ffn_plan(const tt_desc* up, const tt_desc* down, tt_plan_t** out);

void tt_destroy(tt_plan_t* plan);

/* Offsets (in floats) of every core and diagonal inside the packed parameter
 * buffer: core_off receives 2d values, diag_off 2d-1, *n_floats the total.
 * For an FFN plan these describe the up layer (use tt_ffn_param_layout), for
 * a multi-layer plan its first layer (use tt_multi_param_layout). */
tt_status tt_param_layout(const tt_plan_t* plan, size_t* core_off, size_t* diag_off,
                          size_t* n_floats);
tt_status tt_ffn_param_layout(const tt_plan_t* plan, int layer /*0 up, 1 down*/,
                              size_t* core_off, size_t* diag_off, size_t* n_floats);

/* Bytes of device workspace a forward or backward call with T tokens needs
 * (the same value serves both).  The workspace must be 256-byte aligned. */
tt_status tt_workspace_size(const tt_plan_t* plan, int64_t T, size_t* bytes);

/* y = x W^T for T tokens.  T == 0 is a no-op. */
tt_status tt_forward(const tt_plan_t* plan, int64_t T, const void* x, const float* params,
                     void* y, void* ws, size_t ws_bytes, void* stream);

/* dx = dy W and dparams = dL/dparams (overwritten, or added to under
 * TT_ACCUMULATE).  Recomputes what the forward computed; needs no state from
 * a forward call.  T == 0 writes zero gradients (or leaves them under
 * TT_ACCUMULATE). */
tt_status tt_backward(const tt_plan_t* plan, int64_t T, const void* x, const void* dy,
                      const float* params, void* dx, float* dparams, void* ws,
                      size_t ws_bytes, void* stream);

/* The forward above for callers that cannot allocate device memory (a
 * plain-C host or plugin without a device allocator of its own, or a process
 * that must not call cudaMalloc once running).  The CoMERA pages have no
 * counterpart of this call; it only changes where scratch comes from.
 * Scratch is a fixed 32 MiB device array inside the library, held on every
 * GPU that loads it until exit; the caller passes only inputs and outputs.
 * Returns TT_ERR_WORKSPACE when tt_workspace_size(plan, T) exceeds 32 MiB.
 * The first call on a device looks the array's address up (once per device)
 * and should come before any stream capture.  All calls share the array:
 * calls that overlap on the GPU race on it.  Nothing in it needs to start at
 * zero.  Otherwise behaves like tt_forward. */
tt_status tt_forward_noalloc(const tt_plan_t* plan, int64_t T, const void* x,
                             const float* params, void* y, void* stream);

/* FFN pair: params_up / params_down are the two packed buffers. */
tt_status tt_ffn_forward(const tt_plan_t* plan, int64_t T, const void* x,
                         const float* params_up, const float* params_down, void* y, void* ws,
                         size_t ws_bytes, void* stream);
tt_status tt_ffn_backward(const tt_plan_t* plan, int64_t T, const void* x, const void* dy,
                          const float* params_up, const float* params_down, void* dx,
                          float* dparams_up, float* dparams_down, void* ws, size_t ws_bytes,
                          void* stream);

/* ---- several layers on one input --------------------------------------------
 * Up to TT_MULTI_MAX layers that read the same x: the Q, K and V projections
 * of an encoder block's attention (CoMERA project page, "Results", rank
 * table: the attention rows, 768 x 768 at rank 30 each).  The results are
 * those of one tt_forward / tt_backward per layer, except that the backward
 * returns the sum dx = sum_g dy_g W_g (the gradient of x, which feeds every
 * layer).  A bf16 plan whose layers all fit the tensor-core kernels (and
 * without TT_DETERMINISTIC) runs every token pass as one kernel over all
 * layers, streaming x once for all of them (twice in a backward without
 * TT_REUSE_Z); otherwise the layers run one after another and dx is their
 * sum, taken in layer order.  params, y, dy, dparams are host arrays of n
 * device pointers, one per layer, in the descs' order. */
#define TT_MULTI_MAX 3
/* descs: n (1..TT_MULTI_MAX) layers with the same input modes, act type and
 * flags (else TT_ERR_INVALID_ARG); other errors as tt_plan. */
tt_status tt_multi_plan(const tt_desc* descs, int n, tt_plan_t** out);
/* The packed parameter layout of layer `layer` (0..n-1) of a multi plan. */
tt_status tt_multi_param_layout(const tt_plan_t* plan, int layer, size_t* core_off,
                                size_t* diag_off, size_t* n_floats);
tt_status tt_multi_forward(const tt_plan_t* plan, int64_t T, const void* x,
                           const float* const* params, void* const* y, void* ws,
                           size_t ws_bytes, void* stream);
tt_status tt_multi_backward(const tt_plan_t* plan, int64_t T, const void* x,
                            const void* const* dy, const float* const* params, void* dx,
                            float* const* dparams, void* ws, size_t ws_bytes, void* stream);

/* Rank-adaptive step [CoMERA project page, "Learn the ranks while
 * training": the early-stage objective L(G, D) + gamma S_hat(D) + beta ||G||^2,
 * with S_hat an l1 penalty on the diagonals (read here as sum_k |D_k|_1 over
 * every internal link) and ||G||^2 = sum_k ||G_k||_F^2].  Works in place on
 * one layer's packed params / dparams (the tt_param_layout layout, fp32,
 * device pointers), enqueued on `stream`:
 *   lr == 0: dparams += the penalty's sub-gradient:
 *            dG_k += (2 beta) G_k,  dD_k += gamma sign(D_k), sign(0) = 0;
 *            params untouched.
 *   lr > 0:  one proximal gradient step on the whole objective:
 *            G_k <- G_k - lr (dG_k + (2 beta) G_k),
 *            D_k <- soft_threshold(D_k - lr dD_k, lr gamma),
 *            soft_threshold(v, t) = sign(v) max(|v| - t, 0) (entries with
 *            |v| <= t become exactly +0: pruned, and compacted out by the
 *            next forward / backward); dparams untouched.
 * Every step is one float32 operation, rounded to nearest, in the order
 * written (no fused multiply-add).  TT_ERR_INVALID_ARG for a null pointer,
 * an FFN plan (update each layer with its own single-layer plan), or a
 * negative or non-finite gamma, beta or lr.  The CoMERA pages give no
 * optimiser; this is the plainest step on the objective they state. */
typedef struct tt_rank_opts {
  float gamma; /* weight of the l1 penalty on the diagonals, >= 0 */
  float beta;  /* weight of the squared l2 penalty on the cores, >= 0 */
  float lr;    /* step size, >= 0; 0 selects the gradient-only form */
} tt_rank_opts;
tt_status tt_rank_update(const tt_plan_t* plan, float* params, float* dparams,
                         const tt_rank_opts* opts, void* stream);

/* tt_backward followed by tt_rank_update on the same params / dparams, with
 * the step run as the last phase of the backward's merge program (after a
 * grid barrier that follows every read of params) instead of a launch of its
 * own: the early-stage objective's gradient (lr == 0: dparams = dL/dparams +
 * the penalty's sub-gradient) or one proximal step (lr > 0: params updated in
 * place, dparams = dL/dparams).  Arguments and errors as tt_backward and
 * tt_rank_update (params is written when lr > 0); a single-layer plan only.
 * The result equals the two calls in a row. */
tt_status tt_backward_rank_update(const tt_plan_t* plan, int64_t T, const void* x,
                                  const void* dy, float* params, void* dx, float* dparams,
                                  const tt_rank_opts* opts, void* ws, size_t ws_bytes,
                                  void* stream);

/* ---- TT-matrix (TTM) embedding lookup ---------------------------------------
 * [CoMERA project page, "Making small tensor operations fast on GPUs", bullet
 * "Embedding lookup without repeated work": keep only the unique rows of a
 * batch, contract neighbouring cores in pairs so each shared part is computed
 * once, and assemble the rows with one batched product; the table is in
 * tensor-train-matrix format (project page, "Learn the ranks while training";
 * poster digest, TT/TTM figure)].
 * The table E (V x Dm), V = prod m_k rows, Dm = prod n_k columns, is
 *     E[i, j] = F_1[0, i_1, j_1, :] D_1 F_2[:, i_2, j_2, :] D_2 ... F_d[:, i_d, j_d, 0]
 * with i = (i_1..i_d) and j = (j_1..j_d) row-major (first mode most
 * significant).  Packed params: F_1..F_d, each (r_{k-1}, m_k, n_k, r_k)
 * row-major, then D_1..D_{d-1}, fp32 (tt_param_layout describes a TTM plan
 * too: d core offsets, d-1 diagonal offsets).  d is 2 or 3; ranks 1..64;
 * n_1 n_2 r_2 <= 8192, r_1 n_2 r_2 <= 16384 and Dm <= 8192 (else
 * TT_ERR_UNSUPPORTED). */
typedef struct tt_ttm_desc {
  int d;               /* 2 or 3 cores */
  int row_modes[4];    /* m_1..m_d (the vocabulary V = prod m_k, <= 2^24) */
  int col_modes[4];    /* n_1..n_d (the embedding width Dm = prod n_k) */
  int ranks[5];        /* r_0..r_d, r_0 = r_d = 1 */
  unsigned flags;      /* TT_ACCUMULATE (backward adds into dparams),
                          TT_REUSE_MERGE (see tt_ttm_lookup_backward) */
} tt_ttm_desc;
tt_status tt_ttm_plan(const tt_ttm_desc* desc, tt_plan_t** out);

/* out[b, :] = E[idx[b], :] for b < B (out: B x Dm fp32, row-major; idx:
 * int32 device array).  Each distinct row and each distinct (i_1, i_2)
 * prefix is computed once.  An index outside [0, V) is skipped (its output
 * row is left unwritten) and recorded in the device status word
 * (TT_ERR_DEVICE from tt_get_device_status).  Workspace: tt_workspace_size
 * with T = B.  B == 0 is a no-op. */
tt_status tt_ttm_lookup(const tt_plan_t* plan, int64_t B, const int32_t* idx,
                        const float* params, float* out, void* ws, size_t ws_bytes,
                        void* stream);

/* Gradients of L = <dout, lookup(idx)> (dout: B x Dm fp32): every dF_k and
 * dD_k into dparams (overwritten, or added to under TT_ACCUMULATE); repeated
 * indices add up.  dD_k[a] is 0 where D_k[a] == 0 (as for the TT layers).
 * Recomputes the forward's unique rows; needs no state from a lookup call.
 * Under TT_REUSE_MERGE it also takes the batch's distinct rows and prefixes
 * from the workspace instead of finding them again: the caller guarantees
 * that a tt_ttm_lookup with the same plan, the same idx and B and the same
 * workspace came before, with nothing but such backward calls using the
 * workspace in between.
 * Gradient sums are reduced with atomics (summation order not fixed). */
tt_status tt_ttm_lookup_backward(const tt_plan_t* plan, int64_t B, const int32_t* idx,
                                 const float* dout, const float* params, float* dparams,
                                 void* ws, size_t ws_bytes, void* stream);

/* After a lookup or backward on ws (synchronises stream): the number of
 * distinct rows and of distinct (i_1, i_2) prefixes of that batch. */
tt_status tt_ttm_stats(const tt_plan_t* plan, const void* ws, int64_t* unique_rows,
                       int64_t* unique_pairs, void* stream);

/* ---- the device-side error path ---------------------------------------------
 * Every wait inside the library's kernels (on a TMA transfer, on another warp
 * of the CTA, on a grid barrier) is bounded: after the limit it records
 * TT_ERR_TIMEOUT in the device status word, tells the CTA's other warps to
 * stop, waits (bounded) for its own copies and MMAs, frees its tensor memory
 * and returns, leaving the context usable.  Not part of the CoMERA method. */

/* The limit of those waits on the current device, in nanoseconds of the
 * global timer (default 2e9, at least 1000).  Applies to kernels launched
 * afterwards; call it with no library work in flight on the device and
 * outside stream capture.  TT_ERR_INVALID_ARG below 1000 ns. */
tt_status tt_set_wait_limit_ns(uint64_t ns);

/* Test hook: the next launch on the current device of the named kernel skips
 * one arrival in its first CTA, so that a bounded wait of that launch runs
 * out (the launch then reports TT_ERR_TIMEOUT through tt_get_device_status
 * and its outputs are undefined).  It faults nothing and hangs nothing: it is
 * for testing the error path above.  Same calling rules as
 * tt_set_wait_limit_ns. */
#define TT_DEBUG_NONE 0
#define TT_DEBUG_FWD_TOKENS 1    /* forward token kernel: first stage never loaded */
#define TT_DEBUG_BWD_TOKENS 2    /* backward token kernel: first stage never loaded */
#define TT_DEBUG_MERGE_BARRIER 3 /* merge engine (programs of 2+ phases): one grid-barrier arrival */
tt_status tt_debug_skip_arrival(int site);

/* Synchronise stream, then read and clear the status word of the current
 * device.  The word is sticky: it holds the first error any libttc kernel
 * on this device recorded since the last read.  Returns TT_OK,
 * TT_ERR_TIMEOUT or TT_ERR_DEVICE (or TT_ERR_CUDA). */
tt_status tt_get_device_status(void* stream);

const char* tt_status_string(tt_status s);

/* ---- measurement hooks (host side, not thread-safe) ------------------------
 * When enabled, every kernel phase the library enqueues is bracketed by CUDA
 * events on the caller's stream, and every kernel launch is counted.  Phases:
 * 0 merge (chain merges, forward), 1 forward token pass, 2 backward token pass,
 * 3 merge backward, 4 elementwise (GELU).  Not part of the CoMERA method:
 * it lets a benchmark time the library's own kernels with CUDA events. */
#define TT_NUM_PHASES 5
void tt_profile_enable(int on); /* on != 0: clear records and start; 0: stop */
/* Synchronise on the recorded events and return the summed milliseconds and
 * the number of bracketed intervals of one phase since the last enable.
 * Calls captured into a CUDA graph record external event nodes: after each
 * replay of that graph this returns the times of that replay. */
tt_status tt_profile_phase(int phase, double* total_ms, int64_t* intervals);
const char* tt_profile_phase_name(int phase);
/* Total kernels this library has launched in this process (monotonic). */
uint64_t tt_launch_count(void);
/* Throughput probe of the fused FFN kernels' GELU arithmetic: `blocks`
 * blocks of 256 threads each carry 16 values through `iters` rounds of the
 * same packed tanh-form GELU (mode 0) or GELU and GELU' (mode 1), in
 * registers, and write one float each to out (device, blocks * 256 floats).
 * Evaluations = blocks * 256 * 16 * iters; time it with CUDA events on
 * `stream`. */
tt_status tt_gelu_rate(int mode, int iters, int blocks, float* out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TTC_H */

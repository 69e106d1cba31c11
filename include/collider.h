/*
 * libcollider -- filtered transformer backward on one GB300 (sm_103a).
 *
 * The method ("Enhancing Token Filtering Efficiency in Large Language Model
 * Training with Collider", arXiv 2502.00340):
 *   - the forward stays dense; a token filter marks each token kept or
 *     filtered and drops the loss of filtered tokens (Fig. 2b);
 *   - in backward, the activations and output gradients of filtered tokens
 *     are dropped in EVERY layer, not only at the loss (abstract; TL;DR);
 *   - inside attention the softmax of filtered tokens is filtered as well, so
 *     that G_V -- and the activations used for the Q and K gradients -- stay
 *     sparse (Fig. 3, Fig. 5);
 *   - each would-be sparse GEMM runs as a dimension-reduced dense GEMM over
 *     the kept rows only (abstract).
 *
 * Conventions shared by every entry point
 *   Ownership   The caller owns every buffer and the stream.  Pointers are
 *               DEVICE pointers unless a parameter says otherwise.  Entry
 *               points allocate no device memory, except that the first call
 *               on a device allocates a 256-byte status word for that device.
 *               Scratch comes from the caller's workspace `ws` (`ws_bytes`
 *               long, 256-byte aligned), sized by the *_workspace_size calls.
 *   Asynchrony  Every call enqueues work on `stream` (a cudaStream_t, may be
 *               NULL for the legacy default stream) and returns without
 *               synchronising.  n_kept stays on the device.
 *   Errors      Argument errors are detected on the host and returned at
 *               once; nothing is enqueued then.  A CUDA launch error is
 *               COLLIDER_ERR_CUDA.  Every wait inside a kernel is bounded;
 *               a wait that runs out sets the device status word, the kernel
 *               returns early, and collider_check() reports
 *               COLLIDER_ERR_TIMEOUT.  collider_last_error() gives a
 *               thread-local message for the last failing call.  No C++
 *               exception crosses this interface.
 *   Layouts     Row-major.  Tokens are M = B*T rows in sequence order
 *               (token t of sequence b is row b*T + t).  Linear weights are
 *               stored [in, out] (Y = X.W).  bf16 = IEEE bfloat16 storage,
 *               f32 = IEEE binary32.  "FULL" token rows means one row per
 *               token (M rows; filtered rows of an output are written 0);
 *               "COMPACT" means one row per kept token, in kept order
 *               (n_kept rows, row r is token idx[r]).  COMPACT outputs are
 *               written with zero rows from n_kept up to the next multiple
 *               of 128 (within the M-row capacity).
 *   Keep-mask   uint8 [B, T]; nonzero = kept.
 */
#ifndef COLLIDER_H
#define COLLIDER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  COLLIDER_OK = 0,
  COLLIDER_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, workspace too small */
  COLLIDER_ERR_UNSUPPORTED = 2, /* shape or option the library does not handle */
  COLLIDER_ERR_CUDA = 3,        /* a CUDA call failed (incl. an earlier asynchronous error) */
  COLLIDER_ERR_TIMEOUT = 4      /* a bounded in-kernel wait ran out (see collider_check) */
} collider_status;

typedef enum { COLLIDER_F32 = 0, COLLIDER_BF16 = 1 } collider_dtype;
typedef enum { COLLIDER_ROWS_FULL = 0, COLLIDER_ROWS_COMPACT = 1 } collider_rows;
typedef enum { COLLIDER_ARCH_LLAMA = 0, COLLIDER_ARCH_PHI = 1 } collider_arch;
typedef enum { COLLIDER_NORM_RMS = 0, COLLIDER_NORM_LAYER = 1 } collider_norm;
typedef enum { COLLIDER_ACT_SWIGLU = 0, COLLIDER_ACT_GELU_TANH = 1 } collider_act;

/* ------------------------------------------------------------------------ */
/* Status                                                                    */
/* ------------------------------------------------------------------------ */

/* Message describing the last failing call made by this host thread
 * ("" if none).  The string stays valid until the thread's next call. */
const char* collider_last_error(void);

/* Synchronises `stream`, then reports (and clears) the device status word:
 * COLLIDER_ERR_TIMEOUT if a kernel's bounded wait ran out since the last
 * check, COLLIDER_ERR_INVALID_ARG if a kernel met a kept index outside its
 * buffer (and skipped it), COLLIDER_ERR_CUDA if the stream holds an
 * asynchronous CUDA error. */
collider_status collider_check(void* stream);

/* Self-test of the failure path (the pages have no counterpart): one thread
 * waits on an mbarrier that nothing arrives on, through the same bounded wait
 * every kernel of the library uses.  After about 2 s the wait gives up, the
 * timeout (site 999) lands in the status word and the kernel returns; the
 * next collider_check reports COLLIDER_ERR_TIMEOUT and clears the word, and
 * the device stays usable.  Returns the launch status. */
collider_status collider_selftest_wait_timeout(void* stream);

/* Number of kernels this library has launched on the calling host thread
 * since the last reset (reset=1 returns the count and zeroes it). */
long long collider_launch_count(int reset);

/* Launch profiler (per host thread).  While enabled, every kernel launch of
 * the library is bracketed by a pair of CUDA events recorded on the launch
 * stream.  collider_profile_enable(1) clears earlier records and turns
 * recording on; (0) turns it off and keeps the records.  collider_profile_get
 * returns record i: the kernel's name (static string), for GEMM launches
 * mnk_dyn = {M, N, K, dyn} (dyn 1: M is the device-resident kept count, 2: K
 * is; all 0 for other kernels), and the elapsed milliseconds between the two
 * events (waits for them).  Returns -1 for an index out of range. */
int collider_profile_enable(int on);
int collider_profile_count(void);
int collider_profile_get(int i, const char** name, long long* mnk_dyn, float* ms);
/* Record i on a timeline: the milliseconds from record 0's first event to
 * record i's two events (the launch reaching the head of its stream, and the
 * kernel done), and its stream, numbered 0, 1, ... in the order the records'
 * streams first appear.  Waits for the events.  -1 for an index out of range. */
int collider_profile_get_span(int i, float* start_ms, float* end_ms, int* stream_index);

/* ------------------------------------------------------------------------ */
/* a1. Compaction  (abstract: the dimension-reduced GEMM runs over the kept  */
/*     tokens; this is the index list it runs over)                          */
/* ------------------------------------------------------------------------ */

/* The token filter's decision (Fig. 2b: the filter drops the loss of the
 * tokens it filters), from per-token scores: in every sequence the n_filter
 * lowest scores are filtered -- equal scores lower position first, NaN above
 * every number, -0.0 equal to +0.0 -- and mask[b, t] = 1 for the kept tokens.
 * scores f32 [B, T], mask u8 [B, T], both device.  Bit-exact, deterministic.
 * 0 <= n_filter <= T.  The scoring model itself is outside this library. */
collider_status collider_select_keep(const float* scores, int B, int T, int n_filter, uint8_t* mask,
                                     void* stream);

/* Workspace bytes collider_compact needs for B*T tokens (0 when B*T <=
 * 4,194,304: a single thread block scans the mask). */
size_t collider_compact_workspace_size(int B, int T);

/* mask [B,T] u8 -> idx i32 [capacity B*T] (ascending flat indices of kept
 * tokens, first n_kept entries written), cu_kept i32 [B+1] (kept tokens
 * before sequence b; cu_kept[B] = n_kept), n_kept i32 [1].  All device.
 * Bit-exact; deterministic.  B >= 1, T >= 1, B*T < 2^31. */
collider_status collider_compact(const uint8_t* mask, int B, int T, int32_t* idx,
                                 int32_t* cu_kept, int32_t* n_kept, void* ws,
                                 size_t ws_bytes, void* stream);

/* Compaction that allocates nothing, for callers that cannot allocate device
 * memory: programs whose device memory is handed out by their own pool
 * allocator (a raw cudaMalloc would bypass it, or fail once the pool has
 * reserved the device), and latency-critical paths, since cudaMalloc and
 * cudaFree can synchronise the device.  The pages have no counterpart: this is
 * an interface convenience, not part of the method.
 * Same arguments and results as collider_compact (bit-identical), without the
 * workspace.  Its scratch (one int per 16,384 tokens) is a fixed 256 KB array
 * of device memory inside the library, held by every device that loads the
 * library until the process exits; so B*T may be at most 1,073,741,824
 * (2^30) tokens, and larger sizes return COLLIDER_ERR_INVALID_ARG.  All calls
 * share that array: calls whose work can overlap on the GPU (different
 * streams without ordering between them) race and must be serialised by the
 * caller; calls on one stream are fine.  The first call on each device looks
 * up the array's device address (cudaGetSymbolAddress, with that device
 * current) and keeps it for the life of the process; make that first call
 * before any stream capture.  The kept address belongs to the device's primary
 * context: do not call this after cudaDeviceReset on that device, or with
 * another (non-primary) context current.  Nothing is allocated, and no earlier
 * call's contents need clearing: every entry a call reads is written by that
 * call first. */
collider_status collider_compact_noalloc(const uint8_t* mask, int B, int T, int32_t* idx,
                                         int32_t* cu_kept, int32_t* n_kept, void* stream);

/* ------------------------------------------------------------------------ */
/* a2. Row gather / scatter (abstract: the activations of filtered tokens   */
/*     are dropped in every layer)                                           */
/* ------------------------------------------------------------------------ */

/* dst[r, :] = src[idx[r], :] for r < n_kept; dst rows n_kept .. next
 * multiple of 128 (below M) are zeroed.  row_bytes, src_ld_bytes and
 * dst_ld_bytes are multiples of 16 and both pointers 16-byte aligned.  src
 * has M rows, dst has room for M rows. */
collider_status collider_gather_rows(const void* src, size_t src_ld_bytes, void* dst,
                                     size_t dst_ld_bytes, size_t row_bytes, int M,
                                     const int32_t* idx, const int32_t* n_kept, void* stream);

/* full[t, :] = compact[r, :] where idx[r] == t, and full[t, :] = 0 for every
 * filtered token t < M.  Same alignment rules as collider_gather_rows. */
collider_status collider_scatter_rows(const void* compact, size_t compact_ld_bytes, void* full,
                                      size_t full_ld_bytes, size_t row_bytes, int M,
                                      const int32_t* idx, const int32_t* n_kept, void* stream);

/* ------------------------------------------------------------------------ */
/* a3/a4. Linear backward (abstract: sparse GEMM -> dimension-reduced dense  */
/*        GEMM)                                                              */
/* ------------------------------------------------------------------------ */

/* Y = X.W (+b) with X [M,K], W [K,N] (stored [in=K, out=N]), dY [M,N] rows:
 *   dX_k = dY_k . W^T        (only kept rows; filtered rows of a FULL dX = 0)
 *   dW   = X_k^T . dY_k      ([K,N] f32, overwritten)
 *   db   = column sums of dY_k ([N] f32, overwritten; may be NULL)
 * dtype COLLIDER_F32: X, W, dY, dX are f32 and the arithmetic is f32 FMA
 * (no TF32).  COLLIDER_BF16: X, W, dY, dX are bf16, products accumulate in
 * f32 on the tensor cores.  x_rows / dy_rows say whether X and dY hold M
 * (FULL, read through idx) or n_kept (COMPACT) rows; dx_rows likewise for
 * the output.  dX may be NULL (skip), dW may be NULL (skip).
 * bf16 needs K % 8 == 0 and N % 8 == 0 and 16-byte aligned pointers.
 * Workspace: collider_linear_workspace_size(). */
size_t collider_linear_workspace_size(collider_dtype dtype, int M, int K, int N);
collider_status collider_linear_bwd(collider_dtype dtype, int M, int K, int N,
                                    const void* X, collider_rows x_rows, const void* W,
                                    const void* dY, collider_rows dy_rows,
                                    const int32_t* idx, const int32_t* n_kept,
                                    void* dX, collider_rows dx_rows, float* dW, float* db,
                                    void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* a7/a8. Attention backward over the compacted sequences (Figs. 3 and 5)    */
/* ------------------------------------------------------------------------ */

/* Causal (or not) GQA attention backward with filtered probabilities:
 *   P_ij  = exp(S_ij - lse_i), S = Q K^T * scale, on pairs with pos_j <= pos_i
 *           inside one sequence (original positions; P is not renormalised)
 *   P'_ij = P_ij for kept i and kept j, else 0
 *   dV = P'^T dO;  dP = dO V^T;  D_i = sum_j P'_ij dP_ij;
 *   dS = P' * (dP - D);  dQ = dS K * scale;  dK = dS^T Q * scale
 * summed over each group of H/Hkv query heads for dK and dV (query head h
 * reads kv head h*Hkv/H).
 * Q [rows, H, dh], K and V [rows, Hkv, dh], dO [rows, H, dh], all bf16 with
 * row strides q_ld, kv_ld, do_ld (elements); `rows` is M (in_rows FULL, read
 * through idx) or n_kept (COMPACT).  O is not read (D is taken over P', not
 * from the forward output) and may be NULL.  lse f32 [B, H, T] (natural
 * log, from the dense forward).  Outputs dQ [*, H, dh], dK, dV [*, Hkv, dh]
 * bf16 with the same row strides as the inputs, FULL or COMPACT per
 * out_rows.  rotary_dim > 0 additionally applies the RoPE backward
 * (rotate-half pairing on the first rotary_dim dims, angle pos*base^(-2i/r))
 * to dQ and dK so they are gradients with respect to the pre-rotation q, k.
 * dh in {64, 128}; H % Hkv == 0.  Bit-identical from run to run: dQ tiles
 * are added in key-block order, each dK / dV tile gets at most two additions.
 * Workspace: collider_attn_workspace_size(). */
size_t collider_attn_workspace_size(int B, int T, int H, int Hkv, int dh);
collider_status collider_attn_bwd(int B, int T, int H, int Hkv, int dh, int causal, float scale,
                                  int rotary_dim, float rope_base,
                                  const void* Q, const void* K, const void* V, const void* O,
                                  const void* dO, int q_ld, int kv_ld, int do_ld,
                                  collider_rows in_rows, const float* lse,
                                  const int32_t* idx, const int32_t* cu_kept,
                                  const int32_t* n_kept, void* dQ, void* dK, void* dV,
                                  collider_rows out_rows, void* ws, size_t ws_bytes,
                                  void* stream);

/* ------------------------------------------------------------------------ */
/* Whole decoder block                                                       */
/* ------------------------------------------------------------------------ */

typedef struct {
  int arch;          /* collider_arch: LLAMA (sequential, SwiGLU) or PHI (parallel block) */
  int B, T;          /* batch, sequence length */
  int D;             /* model width */
  int H, Hkv, dh;    /* query heads, kv heads, head dim (64 or 128) */
  int F;             /* MLP hidden width */
  int rotary_dim;    /* RoPE dims per head (== dh for full, 32 for Phi-style partial) */
  float rope_base;
  int norm;          /* collider_norm */
  float eps;         /* norm epsilon (informational: the saved rstd already includes it) */
  int act;           /* collider_act: SWIGLU (llama) or GELU_TANH (phi) */
  int qkv_bias, out_bias, mlp_bias; /* which bias gradients to produce */
} collider_layer_desc;

/* Weights the backward reads (bf16).  Biases and LayerNorm beta are not
 * read by the backward.  w_up is [D, 2F] = [gate | up] for SwiGLU and
 * [D, F] (fc1) for GELU; w_down [F, D]; w_qkv [D, (H+2Hkv)dh] with columns
 * [q heads | k heads | v heads]; w_o [H*dh, D]. norm2_w unused for PHI. */
typedef struct {
  const void* norm1_w;
  const void* w_qkv;
  const void* w_o;
  const void* norm2_w;
  const void* w_up;
  const void* w_down;
} collider_layer_weights;

/* Saved forward activations, FULL rows (M = B*T), bf16 unless noted (device
 * memory; for a filtered collider_layer_bwd call also pinned host memory the
 * device addresses at the same pointer, see there):
 *   x [M,D] block input; a [M,D] = norm1(x); mean1 f32 [M] (LayerNorm only);
 *   rstd1 f32 [M]; qkv [M,(H+2Hkv)dh] with q and k AFTER RoPE; o [M,H*dh]
 *   attention output; lse f32 [B,H,T].
 *   LLAMA: h [M,D] = x + attn; b [M,D] = norm2(h); rstd2 f32 [M];
 *          up [M,2F] = [g | u]; s [M,F] = silu(g)*u.
 *   PHI:   up [M,F] = fc1 output before GELU; h, b, rstd2, s unused.
 * LLAMA: a, b and s may be NULL in a filtered call: the backward then
 * recomputes them for the kept rows from x and rstd1 (a = norm1(x)), h and
 * rstd2 (b), and up (s), with the same roundings as collider_layer_fwd, so
 * the gradients are bit-identical to those from that forward's a, b and s.
 * This shrinks what a training loop keeps (or uploads) by 2D + F values a
 * token.  The dense call (NULL index) needs all three. */
typedef struct {
  const void* x;
  const void* a;
  const float* mean1;
  const float* rstd1;
  const void* qkv;
  const void* o;
  const float* lse;
  const void* h;
  const void* b;
  const float* rstd2;
  const void* up;
  const void* s;
} collider_layer_saved;

/* Gradients (all overwritten).  dx bf16 [M or n_kept, D] per dx_rows; every
 * other gradient f32 with its weight's shape.  Pointers for gradients the
 * block does not have (e.g. dnorm1_b for RMSNorm, biases when the desc says
 * none) are ignored and may be NULL. */
typedef struct {
  void* dx;
  float* dnorm1_w;
  float* dnorm1_b;
  float* dw_qkv;
  float* db_qkv;
  float* dw_o;
  float* db_o;
  float* dnorm2_w;
  float* dw_up;
  float* db_up;
  float* dw_down;
  float* db_down;
} collider_layer_grads;

/* Filtered backward of one block: dOut (FULL or COMPACT rows, bf16 [*, D])
 * -> every gradient of the block.  Gathers the kept rows of the saved set,
 * runs the dimension-reduced GEMMs, the filtered attention backward, the
 * norm/activation/RoPE backward and the bias/norm-weight column sums on
 * kept rows only.  Every output is bit-identical from run to run: each
 * weight-gradient tile has one owner with a fixed reduction order, column
 * sums reduce fixed partials in a fixed order, and inside the attention
 * backward dQ tiles are added in key-block order and dK / dV get at most two
 * additions each.
 * idx, cu_kept and n_kept all NULL: every token is kept, and this is the
 * unfiltered dense backward (the baseline the filtered one is measured
 * against): dOut and the saved rows are read where they are, nothing is
 * gathered, dx is written in place (dout_rows / dx_rows do not matter, the
 * COMPACT rows being the FULL rows); the library writes the identity index
 * into its workspace for the kernels that read one.  Giving only some of the
 * three is COLLIDER_ERR_INVALID_ARG.  Workspace: collider_layer_workspace_size.
 * Where the inputs may live: a filtered call reads dOut and the saved set only
 * at the kept rows, with plain loads, so they may also be pinned host memory
 * (cudaHostAlloc / cudaHostRegister) that the device addresses at the same
 * pointer under unified addressing: then only the kept rows cross the host
 * link.  The dense call needs them in device memory, and the weights and
 * gradients always do.  Any other memory (pageable host memory, or host
 * memory where device memory is needed) is COLLIDER_ERR_INVALID_ARG, checked
 * before any launch. */
size_t collider_layer_workspace_size(const collider_layer_desc* desc);
collider_status collider_layer_bwd(const collider_layer_desc* desc,
                                   const collider_layer_weights* w,
                                   const collider_layer_saved* saved,
                                   const void* dOut, collider_rows dout_rows,
                                   const int32_t* idx, const int32_t* cu_kept,
                                   const int32_t* n_kept, const collider_layer_grads* grads,
                                   collider_rows dx_rows, void* ws, size_t ws_bytes,
                                   void* stream);

/* ------------------------------------------------------------------------ */
/* Dense forward of one block (Fig. 2b: the forward stays dense; it saves    */
/* what the filtered backward reads)                                         */
/* ------------------------------------------------------------------------ */

/* Every parameter of a block, bf16, layouts as collider_layer_weights.
 * Biases are read only where the desc asks for them: b_qkv [(H+2Hkv)dh]
 * (qkv_bias), b_o [D] (out_bias), b_up [F] and b_down [D] (mlp_bias, PHI
 * only: LLAMA MLPs have no bias, as in the backward).  norm1_b is the
 * LayerNorm beta (PHI). */
typedef struct {
  const void* norm1_w;
  const void* norm1_b;
  const void* w_qkv;
  const void* b_qkv;
  const void* w_o;
  const void* b_o;
  const void* norm2_w;
  const void* w_up;
  const void* b_up;
  const void* w_down;
  const void* b_down;
} collider_layer_params;

/* Where the forward writes the saved set: the buffers of collider_layer_saved
 * without x (the block input), same shapes and types.  LLAMA writes a, rstd1,
 * qkv, o, lse, h, b, rstd2, up, s (mean1 unused); PHI writes a, mean1, rstd1,
 * qkv, o, lse, up (h, b, rstd2, s unused and may be NULL). */
typedef struct {
  void* a;
  float* mean1;
  float* rstd1;
  void* qkv;
  void* o;
  float* lse;
  void* h;
  void* b;
  float* rstd2;
  void* up;
  void* s;
} collider_layer_acts;

/* y = block(x) for all M = B*T tokens (x, y bf16 [M, D], FULL rows), causal
 * attention inside each sequence of T tokens, and the saved set in `acts`:
 *   LLAMA: a = RMSNorm1(x); qkv = rope(a W_qkv (+ b_qkv)); o = attn(qkv);
 *          h = x + o W_o (+ b_o); b = RMSNorm2(h); up = b W_up = [g | u];
 *          s = silu(g) u; y = h + s W_down
 *   PHI:   a = LayerNorm(x); qkv, o as above (partial RoPE); up = a W1 + b1;
 *          y = x + (o W_o + b_o) + (gelu_tanh(up) W2 + b2)
 * Products accumulate in f32 (tcgen05 GEMMs; attention as two passes, the
 * log-sum-exp of each query row then O = exp(S - lse) V); each saved tensor
 * is rounded to its storage type once, and the projection sums (with their
 * bias) are rounded to bf16 before RoPE, the activation and the second norm.
 * lse is the natural-log log-sum-exp of the scaled logits, [B, H, T].
 * x stays part of the saved set, so y must not alias x; the acts buffers are
 * distinct from each other and from x and y.  Pointers 16-byte aligned;
 * workspace (256-byte aligned) of collider_layer_fwd_workspace_size bytes.
 * Deterministic (no atomics).  Asynchronous on the stream; errors as for
 * collider_layer_bwd (arguments synchronously, kernel-side failures through
 * collider_check). */
size_t collider_layer_fwd_workspace_size(const collider_layer_desc* desc);
collider_status collider_layer_fwd(const collider_layer_desc* desc, const collider_layer_params* w,
                                   const void* x, void* y, const collider_layer_acts* acts,
                                   void* ws, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------ */
/* Whole stack: embedding -> L blocks -> final RMSNorm -> LM head -> CE      */
/* ------------------------------------------------------------------------ */

/* Loss = mean over kept tokens of cross-entropy(logits_t, targets_t) (the
 * token filter drops the loss of filtered tokens, Fig. 2b).  The same keep
 * mask applies in every block.  Inputs (FULL rows): logits bf16 [M,V] (saved
 * by the forward), targets i32 [M], ids i32 [M] (input token ids), y bf16
 * [M,D] final-norm output, xL bf16 [M,D] final-norm input, rstdf f32 [M],
 * normf_w bf16 [D], w_lm bf16 [D,V]; per-block weights and saved sets
 * (arrays of L, block 0 first).  Outputs: the weight gradients of each block
 * in grads[l] (grads[l].dx is not used: gradients between blocks stay in the
 * workspace, COMPACT), dnormf_w f32 [D], dw_lm f32 [D,V], dE f32 [V,D] (rows
 * of token ids never seen at a kept position are 0).  LLAMA blocks, D <= 2048,
 * V % 8 == 0.  idx, cu_kept and n_kept all NULL: every token is kept -- the
 * unfiltered dense backward, as for collider_layer_bwd (the saved rows and y
 * are read in place, nothing is gathered).  Workspace:
 * collider_stack_workspace_size. */
size_t collider_stack_workspace_size(const collider_layer_desc* desc, int L, int V);
collider_status collider_stack_bwd(const collider_layer_desc* desc, int L, int V,
                                   const collider_layer_weights* w,
                                   const collider_layer_saved* saved,
                                   const void* logits, const int32_t* targets,
                                   const int32_t* ids, const void* y, const void* xL,
                                   const float* rstdf, const void* normf_w, const void* w_lm,
                                   const int32_t* idx, const int32_t* cu_kept,
                                   const int32_t* n_kept, const collider_layer_grads* grads,
                                   float* dnormf_w, float* dw_lm, float* dE, void* ws,
                                   size_t ws_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* COLLIDER_H */

// Internal launcher interface between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"

namespace collider {

// Per-call launch context.
struct Ctx {
  cudaStream_t stream;
  DevStatus* st;   // device status word of the current device
  int num_sms;
  // launch the next kernel with programmatic stream serialisation (it is
  // scheduled as the kernel ahead of it exits, and waits for that kernel's
  // completion with grid_dep_wait).  Set only where the operation ahead in
  // the stream is a kernel (not an event wait or a copy) that was launched
  // without the attribute or calls grid_dep_wait in every CTA.
  bool pdl = false;
};

// Whether programmatic dependent launch is used at all (COLLIDER_PDL=0 turns
// it off; read once).
bool pdl_allowed();

// Launch kernel k on c.stream, with the programmatic stream-serialisation
// attribute when pdl is set, and a cluster of cluster_x CTAs when > 1.
template <typename... P, typename... A>
cudaError_t launch_k(const Ctx& c, bool pdl, void (*k)(P...), dim3 grid, dim3 block, size_t smem, int cluster_x,
                     A&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (cluster_x > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  if (pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, k, static_cast<A&&>(args)...);
}

// The error of a launch made with launch_k, the runtime's last error cleared.
inline cudaError_t launched(cudaError_t e) {
  const cudaError_t last = cudaGetLastError();
  return e != cudaSuccess ? e : last;
}

// Launch accounting (per host thread) and optional per-kernel event timing.
void count_launch(int n = 1);
// Message returned by collider_last_error() on this host thread.
void set_last_error(const char* msg);
// Kernel timing hooks used by the profiler: bracket a launch with events when
// profiling is on.  `name` must be a string literal; m, n, k, dyn describe a
// GEMM launch (dyn: which extent is the device-resident kept count).
void prof_begin(const Ctx& c, const char* name, long long m = 0, long long n = 0, long long k = 0,
                int dyn = 0);
void prof_end(const Ctx& c);

// ---- keep-mask selection and compaction -------------------------------------
cudaError_t launch_select_keep(const Ctx& c, const float* scores, int B, int T, int n_filter, uint8_t* mask);
constexpr long long kCompactOneBlockMax = 4194304;  // 2^22 tokens: one block scans it all
size_t compact_ws_bytes(long long M);
cudaError_t launch_compact(const Ctx& c, const uint8_t* mask, int B, int T, int32_t* idx,
                           int32_t* cu_kept, int32_t* n_kept, void* ws);

// ---- row kernels (rows.cu) -------------------------------------------------
struct GatherJob {
  const char* src;
  char* dst;
  long long src_ld;   // bytes
  long long dst_ld;   // bytes
  int row_bytes;      // multiple of 16
  int op;             // 0 copy, 1 gelu_tanh(bf16 row) -> bf16, 2 RMSNorm output of a bf16 row (below)
  // op 2: dst = bf16(src * rstd[t] * gamma), the forward's norm_affine with
  // mean 0 and no bias (t: the FULL row read)
  const float* rstd;
  const __nv_bfloat16* gamma;
};
constexpr int kMaxGatherJobs = 8;
// idx may be null: identity (copy the first n_kept rows, zero the padding).
// cap: row capacity of every dst (rows n_kept .. min(next multiple of 128, cap) are zeroed).
cudaError_t launch_gather(const Ctx& c, const GatherJob* jobs, int njobs, int M, long long cap, const int32_t* idx,
                          const int32_t* n_kept);
// (compact null: only zero the filtered rows of full)
cudaError_t launch_scatter(const Ctx& c, const char* compact, long long compact_ld, char* full,
                           long long full_ld, int row_bytes, int M, const int32_t* idx,
                           const int32_t* n_kept);

// Column sums over the first n_kept rows of a COMPACT matrix X [rows, N] (bf16
// or f32), deterministic: per-row-block partials in `part` then a fixed-order
// reduction.  Writes out[N] f32.  part needs colsum_part_floats(M, N) floats.
// When gidx is non-null, row r is read at row gidx[r] (FULL storage).
size_t colsum_part_floats(int M, int N);
cudaError_t launch_colsum(const Ctx& c, const void* X, int x_is_bf16, long long ld, int M, int N,
                          const int32_t* gidx, const int32_t* n_kept, float* part, float* out);

// Norm backward on kept rows, plus residual:
//   out[r] = res[r] + norm_bwd(dy1[r] (+ dy2[r]))   (COMPACT rows, bf16 out)
// x, mean, rstd are FULL rows read through idx.  gamma bf16 [D].
// dgamma (and dbeta for LayerNorm) f32 [D] via deterministic partials.
struct NormBwdArgs {
  int layer_norm;       // 0 RMSNorm, 1 LayerNorm
  int M, D;
  const float* dy1;     // COMPACT f32 [*, D]
  const float* dy2;     // optional second COMPACT f32 input, summed
  const __nv_bfloat16* res;  // COMPACT bf16 residual gradient (may be null)
  long long res_ld;
  const __nv_bfloat16* x;    // FULL bf16 [M, D]
  const float* mean;    // FULL f32 [M] (LayerNorm)
  const float* rstd;    // FULL f32 [M]
  const __nv_bfloat16* gamma;
  __nv_bfloat16* out;   // COMPACT bf16 [*, D], or FULL [M, D] rows idx[r] when out_full
  __nv_bfloat16* xn_out;   // optional COMPACT bf16 [*, D]: the forward's norm output of each kept row
                           // (RMSNorm: norm_affine(x, 0, rstd, gamma, 0)), padding rows zero
  long long cap;        // row capacity of out (zero padding stops there; COMPACT only)
  int out_full;         // 1: write row r to out row idx[r], no padding (filtered rows are the caller's)
  float* dgamma;
  float* dbeta;         // LayerNorm only
  float* part;          // scratch: norm_part_floats(M, D)
  const int32_t* idx;
  const int32_t* n_kept;
};
size_t norm_part_floats(int M, int D);
cudaError_t launch_norm_bwd(const Ctx& c, const NormBwdArgs& a);
// the two halves of launch_norm_bwd: the input gradient (rows), and dgamma /
// dbeta (column partials + fixed-order reduction), which only reads dy and x
cudaError_t launch_norm_rows(const Ctx& c, const NormBwdArgs& a);
cudaError_t launch_norm_cols(const Ctx& c, const NormBwdArgs& a);

// SwiGLU backward: dgu[r] = [ds*u*sig(g)*(1+g*(1-sig(g))) | ds*silu(g)]
// ds COMPACT (bf16 or f32) [*, F]; gu FULL bf16 [M, 2F] via idx; dgu COMPACT bf16 [*, 2F];
// s_out (optional) COMPACT bf16 [*, F]: the forward's s = silu_mul(g, u) of each kept row.
cudaError_t launch_swiglu_bwd(const Ctx& c, const void* ds, int ds_is_bf16, int F,
                              const __nv_bfloat16* gu, __nv_bfloat16* dgu, int M, long long cap,
                              const int32_t* idx, const int32_t* n_kept, __nv_bfloat16* s_out = nullptr);
// GELU-tanh backward: df1[r] = df2[r] * gelu'(f1[idx[r]]); df2 COMPACT, f1 FULL.
cudaError_t launch_gelu_bwd(const Ctx& c, const void* df2, int df2_is_bf16, int F,
                            const __nv_bfloat16* f1, __nv_bfloat16* df1, int M, long long cap,
                            const int32_t* idx, const int32_t* n_kept);

// LM head: dz[r] = (softmax(z[idx[r]]) - onehot(targets[idx[r]])) / n_kept, bf16 COMPACT.
cudaError_t launch_ce_bwd(const Ctx& c, const __nv_bfloat16* logits, const int32_t* targets, int V,
                          int M, long long cap, const int32_t* idx, const int32_t* n_kept,
                          __nv_bfloat16* dz);
// Embedding gradient: dE[v] = sum of dx rows of kept tokens with id v (ascending
// kept order, deterministic); rows of unseen ids zeroed by the caller.
cudaError_t launch_embed_bwd(const Ctx& c, const __nv_bfloat16* dx, long long ld, int D,
                             const int32_t* ids, int V, int M, const int32_t* idx,
                             const int32_t* n_kept, float* dE);

// ---- fp32 SIMT GEMM (gemm_simt.cu) -----------------------------------------
// C[m, n] = sum_k A(m, k) * B(k, n), f32 FMA.  Operands addressed by
//   A(m,k) = A[rowA(m) * lda + k]     (a_trans = 0)   or  A[rowA(k) * lda + m] (a_trans = 1)
//   B(k,n) = B[n * ldb + k]           (b_trans = 0)   or  B[rowB(k) * ldb + n] (b_trans = 1)
// where row maps go through idx when the *_gather flag is set.  The dynamic
// extent (n_kept) limits M (dyn = 1) or K (dyn = 2).  When c_scatter is set,
// output row m is stored at row idx[m].
struct SimtGemm {
  int M, N, K;
  const float* A; long long lda; int a_trans, a_gather;
  const float* B; long long ldb; int b_trans, b_gather;
  float* C; long long ldc; int c_scatter;
  const int32_t* idx;
  const int32_t* n_kept;
  int dyn;
};
cudaError_t launch_simt_gemm(const Ctx& c, const SimtGemm& g);

// ---- bf16 tcgen05 GEMM (gemm_tc.cu) ----------------------------------------
// C[m, n] (+)= sum_k A(m,k) B(n,k), bf16 operands through TMA, f32 in TMEM.
//   A: a_mn_major = 0 -> stored [M rows, K] (K contiguous), else [K rows, M].
//   B: b_mn_major = 0 -> stored [N rows, K], else [K rows, N].
// dyn = 1: M is limited by *n_kept (rows beyond are not computed; rows from
// n_kept up to the next multiple of 128 are written 0 when zero_pad).
// dyn = 2: K is limited by *n_kept (operand rows beyond must be 0 or finite
// and are multiplied by 0-padded rows of the other operand -- callers keep
// COMPACT buffers zero-padded to 128 rows).
struct TcGemm {
  int M, N, K;
  const void* A; long long lda; int a_mn_major;  // lda in elements
  long long a_rows;   // rows of A's storage (M or K capacity)
  const void* B; long long ldb; int b_mn_major;
  long long b_rows;
  void* C; long long ldc; int c_bf16; int accumulate; int zero_pad;
  long long c_rows;   // row capacity of C (zero padding stops there)
  const int32_t* n_kept; int dyn;
  int bn;             // 128 or 256 (0 = choose)
  // stream-K scratch (both null: whole tiles only).  partial holds
  // kSkMaxCtas * 2 tiles of 128 x 256 f32; counters hold counter_cap ints,
  // zero before the launch (the kernel leaves them zero).
  float* partial;
  int* counters;
  long long counter_cap;
};
constexpr int kSkMaxCtas = 256;
constexpr size_t kSkPartialFloats = (size_t)kSkMaxCtas * 2 * 128 * 256;
cudaError_t launch_tc_gemm(const Ctx& c, const TcGemm& g);
bool tc_gemm_supported(const TcGemm& g);

// ---- attention backward (attn.cu) ------------------------------------------
struct AttnArgs {
  int B, T, H, Hkv, dh, causal;
  float scale;
  int rotary_dim; float rope_base;
  const __nv_bfloat16* q; const __nv_bfloat16* k; const __nv_bfloat16* v;   // COMPACT rows
  const __nv_bfloat16* dO;
  long long q_ld, kv_ld, do_ld;        // elements
  const float* lse;                    // [B, H, T] (FULL positions)
  const int32_t* idx; const int32_t* cu_kept; const int32_t* n_kept;
  __nv_bfloat16* dq; __nv_bfloat16* dk; __nv_bfloat16* dv;   // COMPACT rows, same strides as inputs
  long long dq_ld, dkv_ld;
  float* dq_acc;   // scratch f32 [M, H, dh]
  float* dk_acc;   // scratch f32 [M, Hkv, dh] (tcgen05 path)
  float* dv_acc;
  long long in_cap;  // row capacity of the COMPACT q/k/v/dO buffers (TMA extent)
  float* Dvec;     // scratch f32 [H, M]
  float* lse_k;    // scratch f32 [H, M] (lse gathered to kept order, pre-scaled)
  float2* rope;    // scratch [T, rotary_dim/2] (cos, sin)
  int* order;      // scratch [attn_order_ints(B, T, H)]: work tickets and dQ accumulation turns
  int M;
  long long cap;   // row capacity of dq, dk, dv (zero padding stops there)
  int stage;       // 0: the whole backward; 1: only the preparation (lse in kept
                   // order, zeroed accumulators and ordering scratch, RoPE table:
                   // it reads only lse, idx and cu_kept, so it may run ahead on
                   // another stream); 2: everything after it
};
// ints of the attention backward's ordering scratch: one work-item ticket and
// a dQ accumulation turn per (sequence, query head, 64-row query block)
__host__ __device__ inline size_t attn_order_ints(int B, int T, int H) { return 1 + (size_t)B * H * ((T + 63) / 64); }
cudaError_t launch_attn_bwd(const Ctx& c, const AttnArgs& a);

// ---- dense forward of one block (attn.cu, fwd.cu) ---------------------------
// Causal GQA attention over whole sequences (every token kept), two passes:
// the log-sum-exp of every query row, then O = exp(S - lse) V.
struct AttnFwdArgs {
  int B, T, H, Hkv, dh;
  float scale;
  const __nv_bfloat16* q; const __nv_bfloat16* k; const __nv_bfloat16* v;   // FULL rows [M, ...]
  long long q_ld, kv_ld;   // elements
  __nv_bfloat16* o; long long o_ld;    // [M, H*dh]
  float* lse;    // out: [B, H, T] natural log
  float* lse2;   // scratch [H, M] (log2 units)
  const int32_t* cu;   // [B+1] = b*T
  int M;
};
cudaError_t launch_attn_fwd(const Ctx& c, const AttnFwdArgs& a);
// RoPE table [T, rot_half] of (cos, sin), the same values the backward uses.
cudaError_t launch_rope_table(const Ctx& c, int T, int rot_half, float rope_base, float2* rope);

// Norm forward, one row per CTA (D a multiple of 8, D <= 4096):
//   v = x, or bf16(x + add + add_bias) (written to sum_out when given);
//   out = bf16(norm(v) * gamma (+ beta));  mean (LayerNorm) and rstd f32.
struct NormFwdArgs {
  int layer_norm;   // 0 RMSNorm, 1 LayerNorm
  int M, D;
  float eps;
  const __nv_bfloat16* x;
  const float* add; long long add_ld;   // optional f32 [M, D]
  const __nv_bfloat16* add_bias;        // optional bf16 [D] (with add)
  __nv_bfloat16* sum_out;               // optional bf16 [M, D]
  const __nv_bfloat16* gamma;
  const __nv_bfloat16* beta;            // LayerNorm
  __nv_bfloat16* out;
  float* mean;                          // LayerNorm
  float* rstd;
};
cudaError_t launch_norm_fwd(const Ctx& c, const NormFwdArgs& a);
// qkv = bf16(acc + bias), then the first rot_heads heads (q then k) rotated on
// their first 2*rot_half dims at position row % T; [M, N] f32 (acc_bf16 = 0)
// or bf16 already rounded (acc_bf16 = 1, no bias) -> bf16.
cudaError_t launch_qkv_rope_fwd(const Ctx& c, int M, int N, int rot_heads, int dh, int rot_half, int T,
                                const void* acc, int acc_bf16, const __nv_bfloat16* bias, const float2* rope,
                                __nv_bfloat16* qkv);
// gelu == 0: up = bf16(acc + bias) [M, 2F] = [g | u], act = bf16(silu(g) u) [M, F]
// gelu == 1: up = bf16(acc + bias) [M, F],            act = bf16(gelu_tanh(up)) [M, F]
cudaError_t launch_act_fwd(const Ctx& c, int gelu, int M, int F, const float* acc, const __nv_bfloat16* bias,
                           __nv_bfloat16* up, __nv_bfloat16* act);
// act = bf16(silu(g) u) from the bf16 up [M, 2F] = [g | u]
cudaError_t launch_swiglu_fwd(const Ctx& c, int M, int F, const __nv_bfloat16* up, __nv_bfloat16* act);
// y = bf16(res + acc1 (+ bias1) (+ acc2 (+ bias2))), all [M, D]
cudaError_t launch_residual_out(const Ctx& c, int M, int D, const __nv_bfloat16* res, const float* acc1,
                                const __nv_bfloat16* bias1, const float* acc2, const __nv_bfloat16* bias2,
                                __nv_bfloat16* y);
// cu[b] = b * T for b <= B
cudaError_t launch_iota_cu(const Ctx& c, int B, int T, int32_t* cu);
// the index of "every token kept": idx[i] = i (i < B*T), cu[b] = b*T, *nk = B*T
cudaError_t launch_identity_index(const Ctx& c, int B, int T, int32_t* idx, int32_t* cu, int32_t* nk);

}  // namespace collider

// Row-wise kernels of the filtered backward: gather/scatter of kept rows,
// deterministic column sums, norm / activation backward on kept rows, the
// LM-head cross-entropy backward and the embedding gradient.  All are
// HBM-bound: 16-byte vector accesses, one warp (or block) per row, grids a
// multiple of the SM count.  Collider (abstract): the activations of filtered
// tokens are dropped in every layer, so every kernel here touches kept rows
// only, and COMPACT outputs are zero-padded to the GEMM tile height.
#include "internal.h"

namespace collider {

namespace {

__device__ __forceinline__ float gelu_tanh_f(float x) {
  const float c = 0.7978845608028654f, a = 0.044715f;
  return 0.5f * x * (1.f + tanhf(c * (x + a * x * x * x)));
}
__device__ __forceinline__ float gelu_tanh_grad(float x) {
  const float c = 0.7978845608028654f, a = 0.044715f;
  float t = tanhf(c * (x + a * x * x * x));
  return 0.5f * (1.f + t) + 0.5f * x * (1.f - t * t) * c * (1.f + 3.f * a * x * x);
}
__device__ __forceinline__ float sigmoid_f(float x) { return 1.f / (1.f + __expf(-x)); }

__device__ __forceinline__ uint4 gelu8(uint4 u) {
  float f[8];
  unpack8(u, f);
#pragma unroll
  for (int i = 0; i < 8; ++i) f[i] = gelu_tanh_f(f[i]);
  return pack8(f);
}

// 8 consecutive values of a bf16 or f32 row as floats
__device__ __forceinline__ void load8(const void* base, int is_bf16, long long off, float* f) {
  if (is_bf16) {
    uint4 u = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + off);
    unpack8(u, f);
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
    float4 a = p[0], b = p[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
}

struct GatherBatch {
  GatherJob j[kMaxGatherJobs];
};

__global__ void __launch_bounds__(256) gather_kernel(GatherBatch jb, int M, long long cap,
                                                     const int32_t* __restrict__ idx,
                                                     const int32_t* __restrict__ n_kept, DevStatus* st) {
  grid_dep_wait();
  const GatherJob J = jb.j[blockIdx.y];
  const int nk = *n_kept;
  const int pad = padded_rows(nk, cap);
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int vecs = J.row_bytes >> 4;
  for (int r = blockIdx.x * wpb + (threadIdx.x >> 5); r < pad; r += gridDim.x * wpb) {
    uint4* d = reinterpret_cast<uint4*>(J.dst + (long long)r * J.dst_ld);
    if (r < nk) {
      int t = idx ? idx[r] : r;
      if ((unsigned)t >= (unsigned)M) {
        if (lane == 0) report_error(st, kErrBadIndex, 100);
        continue;
      }
      const uint4* s = reinterpret_cast<const uint4*>(J.src + (long long)t * J.src_ld);
      int v = lane;
      if (J.op == 2) {
        // the forward's RMSNorm output of row t, recomputed
        const float rs = J.rstd[t];
        for (; v < vecs; v += 32) {
          float x[8], g[8], o[8];
          unpack8(s[v], x);
          unpack8(reinterpret_cast<const uint4*>(J.gamma)[v], g);
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = norm_affine(x[e], 0.f, rs, g[e], 0.f);
          d[v] = pack8(o);
        }
        continue;
      }
      // four 16-byte loads in flight per lane before their stores
      for (; v + 96 < vecs; v += 128) {
        uint4 x0 = s[v], x1 = s[v + 32], x2 = s[v + 64], x3 = s[v + 96];
        if (J.op == 1) { x0 = gelu8(x0); x1 = gelu8(x1); x2 = gelu8(x2); x3 = gelu8(x3); }
        d[v] = x0; d[v + 32] = x1; d[v + 64] = x2; d[v + 96] = x3;
      }
      for (; v < vecs; v += 32) {
        uint4 x = s[v];
        if (J.op == 1) x = gelu8(x);
        d[v] = x;
      }
    } else {
      for (int v = lane; v < vecs; v += 32) d[v] = make_uint4(0, 0, 0, 0);
    }
  }
}

// lower_bound of key in the ascending idx[0..n)
__device__ __forceinline__ int lower_bound(const int32_t* __restrict__ a, int n, int key) {
  int lo = 0, hi = n;
  while (lo < hi) {
    int mid = (lo + hi) >> 1;
    if (a[mid] < key) lo = mid + 1; else hi = mid;
  }
  return lo;
}

__global__ void __launch_bounds__(256) scatter_kernel(const char* __restrict__ compact, long long cld,
                                                      char* __restrict__ full, long long fld, int row_bytes,
                                                      int M, const int32_t* __restrict__ idx,
                                                      const int32_t* __restrict__ n_kept) {
  const int nk = *n_kept;
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int vecs = row_bytes >> 4;
  for (int t = blockIdx.x * wpb + (threadIdx.x >> 5); t < M; t += gridDim.x * wpb) {
    int r = 0;
    if (lane == 0) r = lower_bound(idx, nk, t);
    r = __shfl_sync(0xffffffffu, r, 0);
    bool kept = (r < nk) && (idx[r] == t);
    uint4* d = reinterpret_cast<uint4*>(full + (long long)t * fld);
    if (kept && !compact) continue;   // zero the filtered rows only
    if (kept) {
      const uint4* s = reinterpret_cast<const uint4*>(compact + (long long)r * cld);
      for (int v = lane; v < vecs; v += 32) d[v] = s[v];
    } else {
      for (int v = lane; v < vecs; v += 32) d[v] = make_uint4(0, 0, 0, 0);
    }
  }
}

// ---------------------------------------------------------------------------
// column sums: pass 1 over blocks of kColRows rows, pass 2 fixed-order reduce
constexpr int kColRows = 16;

__global__ void __launch_bounds__(256) colsum_part_kernel(const void* __restrict__ X, int is_bf16, long long ld,
                                                          int N, const int32_t* __restrict__ gidx,
                                                          const int32_t* __restrict__ n_kept,
                                                          float* __restrict__ part) {
  const int nk = *n_kept;
  const int r0 = blockIdx.y * kColRows;
  if (r0 >= nk) return;
  const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (c >= N) return;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const int r1 = min(nk, r0 + kColRows);
  for (int r = r0; r < r1; ++r) {
    float f[8];
    const long long row = gidx ? gidx[r] : r;
    load8(X, is_bf16, row * ld + c, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += f[i];
  }
  float4* p = reinterpret_cast<float4*>(part + (long long)blockIdx.y * N + c);
  p[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  p[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
}

// out[c] = sum over partial rows i < ceil(n_kept / rows_per_part) of
// part[i * stride + c].  A block covers 32 columns with 8 row groups: group g
// sums rows g, g+8, ... in ascending order, then the 8 group sums are added
// in group order -- a fixed summation order, so the result is deterministic.
__global__ void __launch_bounds__(256) colsum_reduce_kernel(const float* __restrict__ part, int N, long long stride,
                                                            int rows_per_part, const int32_t* __restrict__ n_kept,
                                                            float* __restrict__ out) {
  __shared__ float acc[8][33];
  const int cl = threadIdx.x & 31, g = threadIdx.x >> 5;
  const int c = blockIdx.x * 32 + cl;
  const int nk = *n_kept;
  const int nparts = (nk + rows_per_part - 1) / rows_per_part;
  float s = 0.f;
  if (c < N)
    for (int i = g; i < nparts; i += 8) s += part[(long long)i * stride + c];
  acc[g][cl] = s;
  __syncthreads();
  if (g == 0 && c < N) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) t += acc[k][cl];
    out[c] = t;
  }
}

// ---------------------------------------------------------------------------
// norm backward (+ residual) on kept rows.
//   rows:    one warp per row, two passes over the row (the second re-reads it
//            from L1/L2): out = res + rstd * (g - xh * mean(g xh) [- mean(g)])
//   columns: dgamma = sum_r dy xh, dbeta = sum_r dy, as per-64-row partials
//            (thread = 8 columns) then a fixed-order reduction: deterministic.
constexpr int kNormWarps = 8;
constexpr int kNormColRows = 16;

__device__ __forceinline__ void norm_dy8(const NormBwdArgs& a, long long off, float* dy) {
  load8(a.dy1, 0, off, dy);
  if (a.dy2) {
    float d2[8];
    load8(a.dy2, 0, off, d2);
#pragma unroll
    for (int k = 0; k < 8; ++k) dy[k] += d2[k];
  }
}

__global__ void __launch_bounds__(kNormWarps * 32) norm_rows_kernel(NormBwdArgs a, DevStatus* st) {
  grid_dep_wait();
  const int D = a.D;
  const int nk = *a.n_kept;
  const int pad = a.out_full ? nk : padded_rows(nk, a.cap);
  const int lane = threadIdx.x & 31;
  for (int r = blockIdx.x * kNormWarps + (threadIdx.x >> 5); r < pad; r += gridDim.x * kNormWarps) {
    if (r >= nk) {
      __nv_bfloat16* orow = a.out + (long long)r * D;
      for (int c = lane * 8; c < D; c += 256) {
        *reinterpret_cast<uint4*>(orow + c) = make_uint4(0, 0, 0, 0);
        if (a.xn_out) *reinterpret_cast<uint4*>(a.xn_out + (long long)r * D + c) = make_uint4(0, 0, 0, 0);
      }
      continue;
    }
    const int t = a.idx[r];
    if ((unsigned)t >= (unsigned)a.M) {
      if (lane == 0) report_error(st, kErrBadIndex, 200);
      continue;
    }
    __nv_bfloat16* orow = a.out + (long long)(a.out_full ? t : r) * D;
    const float rstd = a.rstd[t];
    const float mu = a.layer_norm ? a.mean[t] : 0.f;
    const __nv_bfloat16* xr = a.x + (long long)t * D;
    float s_gx = 0.f, s_g = 0.f;
    for (int c = lane * 8; c < D; c += 256) {
      float dy[8], xv[8], gm[8];
      norm_dy8(a, (long long)r * D + c, dy);
      load8(xr, 1, c, xv);
      load8(a.gamma, 1, c, gm);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float g = dy[k] * gm[k];
        s_gx += g * (xv[k] - mu) * rstd;
        s_g += g;
      }
    }
    s_gx = warp_sum(s_gx) / (float)D;
    s_g = a.layer_norm ? warp_sum(s_g) / (float)D : 0.f;
    for (int c = lane * 8; c < D; c += 256) {
      float dy[8], xv[8], gm[8], o[8];
      norm_dy8(a, (long long)r * D + c, dy);
      load8(xr, 1, c, xv);
      load8(a.gamma, 1, c, gm);
      if (a.res) {
        load8(a.res, 1, (long long)r * a.res_ld + c, o);
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) o[k] = 0.f;
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) o[k] += rstd * (dy[k] * gm[k] - (xv[k] - mu) * rstd * s_gx - s_g);
      *reinterpret_cast<uint4*>(orow + c) = pack8(o);
      if (a.xn_out) {
        float xn[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) xn[k] = norm_affine(xv[k], mu, rstd, gm[k], 0.f);
        *reinterpret_cast<uint4*>(a.xn_out + (long long)r * D + c) = pack8(xn);
      }
    }
  }
}

__global__ void __launch_bounds__(256) norm_cols_kernel(NormBwdArgs a) {
  const int nk = *a.n_kept;
  const int r0 = blockIdx.y * kNormColRows;
  if (r0 >= nk) return;
  const int c = (blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (c >= a.D) return;
  float dg[8] = {0, 0, 0, 0, 0, 0, 0, 0}, db[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  const int r1 = min(nk, r0 + kNormColRows);
  for (int r = r0; r < r1; ++r) {
    const int t = a.idx[r];
    if ((unsigned)t >= (unsigned)a.M) continue;   // reported by the row kernel
    const float rstd = a.rstd[t];
    const float mu = a.layer_norm ? a.mean[t] : 0.f;
    float dy[8], xv[8];
    norm_dy8(a, (long long)r * a.D + c, dy);
    load8(a.x, 1, (long long)t * a.D + c, xv);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      dg[k] += dy[k] * (xv[k] - mu) * rstd;
      db[k] += dy[k];
    }
  }
  const int nsets = a.layer_norm ? 2 : 1;
  float4* p = reinterpret_cast<float4*>(a.part + ((long long)blockIdx.y * nsets) * a.D + c);
  p[0] = make_float4(dg[0], dg[1], dg[2], dg[3]);
  p[1] = make_float4(dg[4], dg[5], dg[6], dg[7]);
  if (nsets == 2) {
    float4* q = reinterpret_cast<float4*>(a.part + ((long long)blockIdx.y * nsets + 1) * a.D + c);
    q[0] = make_float4(db[0], db[1], db[2], db[3]);
    q[1] = make_float4(db[4], db[5], db[6], db[7]);
  }
}

// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) swiglu_bwd_kernel(const void* __restrict__ ds, int ds_bf16, int F,
                                                         const __nv_bfloat16* __restrict__ gu,
                                                         __nv_bfloat16* __restrict__ dgu, int M, long long cap,
                                                         const int32_t* __restrict__ idx,
                                                         const int32_t* __restrict__ n_kept, DevStatus* st,
                                                         __nv_bfloat16* __restrict__ s_out) {
  grid_dep_wait();
  const int nk = *n_kept;
  const int pad = padded_rows(nk, cap);
  const int vpr = F >> 3;   // 8-wide vectors per row
  const long long total = (long long)pad * vpr;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(e / vpr), c = (int)(e % vpr) * 8;
    __nv_bfloat16* o = dgu + (long long)r * 2 * F;
    if (r >= nk) {
      *reinterpret_cast<uint4*>(o + c) = make_uint4(0, 0, 0, 0);
      *reinterpret_cast<uint4*>(o + F + c) = make_uint4(0, 0, 0, 0);
      if (s_out) *reinterpret_cast<uint4*>(s_out + (long long)r * F + c) = make_uint4(0, 0, 0, 0);
      continue;
    }
    const int t = idx[r];
    if ((unsigned)t >= (unsigned)M) { report_error(st, kErrBadIndex, 300); continue; }
    float d[8], g[8], u[8], dg[8], du[8];
    load8(ds, ds_bf16, (long long)r * F + c, d);
    load8(gu, 1, (long long)t * 2 * F + c, g);
    load8(gu, 1, (long long)t * 2 * F + F + c, u);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float sg = sigmoid_f(g[i]);
      dg[i] = d[i] * u[i] * sg * (1.f + g[i] * (1.f - sg));
      du[i] = d[i] * g[i] * sg;
    }
    *reinterpret_cast<uint4*>(o + c) = pack8(dg);
    *reinterpret_cast<uint4*>(o + F + c) = pack8(du);
    if (s_out) {
      // the forward's s = silu(g) u of this kept row, recomputed
      float sv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) sv[i] = silu_mul(g[i], u[i]);
      *reinterpret_cast<uint4*>(s_out + (long long)r * F + c) = pack8(sv);
    }
  }
}

__global__ void __launch_bounds__(256) gelu_bwd_kernel(const void* __restrict__ df2, int df2_bf16, int F,
                                                       const __nv_bfloat16* __restrict__ f1,
                                                       __nv_bfloat16* __restrict__ df1, int M, long long cap,
                                                       const int32_t* __restrict__ idx,
                                                       const int32_t* __restrict__ n_kept, DevStatus* st) {
  grid_dep_wait();
  const int nk = *n_kept;
  const int pad = padded_rows(nk, cap);
  const int vpr = F >> 3;
  const long long total = (long long)pad * vpr;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(e / vpr), c = (int)(e % vpr) * 8;
    __nv_bfloat16* o = df1 + (long long)r * F + c;
    if (r >= nk) { *reinterpret_cast<uint4*>(o) = make_uint4(0, 0, 0, 0); continue; }
    const int t = idx[r];
    if ((unsigned)t >= (unsigned)M) { report_error(st, kErrBadIndex, 301); continue; }
    float d[8], x[8];
    load8(df2, df2_bf16, (long long)r * F + c, d);
    load8(f1, 1, (long long)t * F + c, x);
#pragma unroll
    for (int i = 0; i < 8; ++i) d[i] *= gelu_tanh_grad(x[i]);
    *reinterpret_cast<uint4*>(o) = pack8(d);
  }
}

// ---------------------------------------------------------------------------
constexpr int kCeThreads = 512;

__global__ void __launch_bounds__(kCeThreads) ce_bwd_kernel(const __nv_bfloat16* __restrict__ z,
                                                            const int32_t* __restrict__ targets, int V, int M,
                                                            long long cap, const int32_t* __restrict__ idx,
                                                            const int32_t* __restrict__ n_kept,
                                                            __nv_bfloat16* __restrict__ dz, DevStatus* st) {
  __shared__ float red[32];
  const int nk = *n_kept;
  const int pad = padded_rows(nk, cap);
  const int r = blockIdx.x;
  if (r >= pad) return;
  __nv_bfloat16* o = dz + (long long)r * V;
  if (r >= nk) {
    for (int c = threadIdx.x * 8; c < V; c += kCeThreads * 8)
      *reinterpret_cast<uint4*>(o + c) = make_uint4(0, 0, 0, 0);
    return;
  }
  const int t = idx[r];
  if ((unsigned)t >= (unsigned)M) { if (threadIdx.x == 0) report_error(st, kErrBadIndex, 400); return; }
  const __nv_bfloat16* zr = z + (long long)t * V;
  float mx = -INFINITY;
  for (int c = threadIdx.x * 8; c < V; c += kCeThreads * 8) {
    float f[8];
    load8(zr, 1, c, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) mx = fmaxf(mx, f[i]);
  }
  mx = block_max(mx, red);
  float s = 0.f;
  for (int c = threadIdx.x * 8; c < V; c += kCeThreads * 8) {
    float f[8];
    load8(zr, 1, c, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) s += __expf(f[i] - mx);
  }
  s = block_sum(s, red);
  const float inv = 1.f / (s * (float)nk);
  const float invn = 1.f / (float)nk;
  const int tgt = targets[t];
  for (int c = threadIdx.x * 8; c < V; c += kCeThreads * 8) {
    float f[8];
    load8(zr, 1, c, f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      f[i] = __expf(f[i] - mx) * inv;
      if (c + i == tgt) f[i] -= invn;
    }
    *reinterpret_cast<uint4*>(o + c) = pack8(f);
  }
}

// dE[v] = sum over kept rows r with ids[idx[r]] == v of dx[r], in ascending r.
// The block of the first such r owns v; later duplicates exit.
__global__ void __launch_bounds__(256) embed_bwd_kernel(const __nv_bfloat16* __restrict__ dx, long long ld, int D,
                                                        const int32_t* __restrict__ ids, int V, int M,
                                                        const int32_t* __restrict__ idx,
                                                        const int32_t* __restrict__ n_kept,
                                                        float* __restrict__ dE, DevStatus* st) {
  __shared__ int list[256];
  __shared__ int nlist;
  __shared__ int wsum[9];
  const int nk = *n_kept;
  const int r = blockIdx.x;
  if (r >= nk) return;
  const int t = idx[r];
  if ((unsigned)t >= (unsigned)M) { if (threadIdx.x == 0) report_error(st, kErrBadIndex, 500); return; }
  const int id = ids[t];
  if ((unsigned)id >= (unsigned)V) { if (threadIdx.x == 0) report_error(st, kErrBadIndex, 501); return; }
  int dup = 0;
  for (int q = threadIdx.x; q < r; q += blockDim.x) dup |= (ids[idx[q]] == id);
  if (__syncthreads_or(dup)) return;
  // this block owns id; accumulate its rows in ascending order
  const int c0 = threadIdx.x * 8;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int base = r; base < nk; base += blockDim.x) {
    const int q = base + threadIdx.x;
    const int hit = (q < nk) && (ids[idx[q]] == id);
    // ordered compaction of this chunk's hits
    const unsigned bal = __ballot_sync(0xffffffffu, hit);
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    if (lane == 0) wsum[w] = __popc(bal);
    __syncthreads();
    if (threadIdx.x == 0) {
      int s = 0;
      for (int i = 0; i < (int)(blockDim.x >> 5); ++i) { int v = wsum[i]; wsum[i] = s; s += v; }
      nlist = s;
    }
    __syncthreads();
    if (hit) list[wsum[w] + __popc(bal & ((1u << lane) - 1u))] = q;
    __syncthreads();
    if (c0 < D)
      for (int i = 0; i < nlist; ++i) {
        float f[8];
        load8(dx, 1, (long long)list[i] * ld + c0, f);
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] += f[k];
      }
    __syncthreads();
  }
  if (c0 < D) {
    float4* p = reinterpret_cast<float4*>(dE + (long long)id * D + c0);
    p[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
    p[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

inline int grid_rows(const Ctx& c, long long rows, int per_block) {
  long long g = (rows + per_block - 1) / per_block;
  long long cap = (long long)c.num_sms * 8;
  if (g > cap) g = cap;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_gather(const Ctx& c, const GatherJob* jobs, int njobs, int M, long long cap,
                          const int32_t* idx, const int32_t* n_kept) {
  if (njobs <= 0) return cudaSuccess;
  GatherBatch b{};
  for (int i = 0; i < njobs; ++i) b.j[i] = jobs[i];
  dim3 grid(grid_rows(c, cap, 8), njobs);
  double bytes = 0;
  for (int i = 0; i < njobs; ++i) bytes += 2.0 * jobs[i].row_bytes;  // per kept row
  prof_begin(c, "gather_rows");
  const cudaError_t e = launch_k(c, c.pdl, gather_kernel, grid, dim3(256), 0, 1, b, M, cap, idx, n_kept, c.st);
  prof_end(c);
  count_launch();
  return launched(e);
}

cudaError_t launch_scatter(const Ctx& c, const char* compact, long long compact_ld, char* full,
                           long long full_ld, int row_bytes, int M, const int32_t* idx,
                           const int32_t* n_kept) {
  prof_begin(c, "scatter_rows");
  scatter_kernel<<<grid_rows(c, M, 8), 256, 0, c.stream>>>(compact, compact_ld, full, full_ld, row_bytes, M,
                                                           idx, n_kept);
  prof_end(c);
  count_launch();
  return cudaGetLastError();
}

size_t colsum_part_floats(int M, int N) {
  return (size_t)((M + kColRows - 1) / kColRows) * (size_t)N;
}

cudaError_t launch_colsum(const Ctx& c, const void* X, int x_is_bf16, long long ld, int M, int N,
                          const int32_t* gidx, const int32_t* n_kept, float* part, float* out) {
  dim3 g1((N / 8 + 255) / 256, (M + kColRows - 1) / kColRows);
  prof_begin(c, "colsum");
  colsum_part_kernel<<<g1, 256, 0, c.stream>>>(X, x_is_bf16, ld, N, gidx, n_kept, part);
  colsum_reduce_kernel<<<(N + 31) / 32, 256, 0, c.stream>>>(part, N, N, kColRows, n_kept, out);
  prof_end(c);
  count_launch(2);
  return cudaGetLastError();
}

size_t norm_part_floats(int M, int D) {
  return (size_t)((M + kNormColRows - 1) / kNormColRows) * 2 * (size_t)D;
}

cudaError_t launch_norm_rows(const Ctx& c, const NormBwdArgs& a) {
  prof_begin(c, "norm_bwd");
  const cudaError_t e = launch_k(c, c.pdl, norm_rows_kernel, dim3(grid_rows(c, a.cap, kNormWarps)),
                                 dim3(kNormWarps * 32), 0, 1, a, c.st);
  count_launch(1);
  prof_end(c);
  return launched(e);
}

cudaError_t launch_norm_cols(const Ctx& c, const NormBwdArgs& a) {
  const int nsets = a.layer_norm ? 2 : 1;
  prof_begin(c, "norm_bwd");
  norm_cols_kernel<<<dim3((a.D / 8 + 255) / 256, (unsigned)((a.cap + kNormColRows - 1) / kNormColRows)), 256, 0,
                     c.stream>>>(a);
  // partials are laid out [part][set][D] with set 0 = dgamma, set 1 = dbeta
  const int g = (a.D + 31) / 32;
  colsum_reduce_kernel<<<g, 256, 0, c.stream>>>(a.part, a.D, (long long)nsets * a.D, kNormColRows, a.n_kept,
                                                a.dgamma);
  if (a.layer_norm)
    colsum_reduce_kernel<<<g, 256, 0, c.stream>>>(a.part + a.D, a.D, (long long)nsets * a.D, kNormColRows,
                                                  a.n_kept, a.dbeta);
  count_launch(1 + nsets);
  prof_end(c);
  return cudaGetLastError();
}

cudaError_t launch_norm_bwd(const Ctx& c, const NormBwdArgs& a) {
  cudaError_t e = launch_norm_rows(c, a);
  return e == cudaSuccess ? launch_norm_cols(c, a) : e;
}

cudaError_t launch_swiglu_bwd(const Ctx& c, const void* ds, int ds_is_bf16, int F, const __nv_bfloat16* gu,
                              __nv_bfloat16* dgu, int M, long long cap, const int32_t* idx, const int32_t* n_kept,
                              __nv_bfloat16* s_out) {
  prof_begin(c, "swiglu_bwd");
  const cudaError_t e = launch_k(c, c.pdl, swiglu_bwd_kernel, dim3(grid_rows(c, cap * (F / 8), 256)), dim3(256), 0,
                                 1, ds, ds_is_bf16, F, gu, dgu, M, cap, idx, n_kept, c.st, s_out);
  prof_end(c);
  count_launch();
  return launched(e);
}

cudaError_t launch_gelu_bwd(const Ctx& c, const void* df2, int df2_is_bf16, int F, const __nv_bfloat16* f1,
                            __nv_bfloat16* df1, int M, long long cap, const int32_t* idx, const int32_t* n_kept) {
  prof_begin(c, "gelu_bwd");
  const cudaError_t e = launch_k(c, c.pdl, gelu_bwd_kernel, dim3(grid_rows(c, cap * (F / 8), 256)), dim3(256), 0, 1,
                                 df2, df2_is_bf16, F, f1, df1, M, cap, idx, n_kept, c.st);
  prof_end(c);
  count_launch();
  return launched(e);
}

cudaError_t launch_ce_bwd(const Ctx& c, const __nv_bfloat16* logits, const int32_t* targets, int V, int M,
                          long long cap, const int32_t* idx, const int32_t* n_kept, __nv_bfloat16* dz) {
  prof_begin(c, "ce_bwd");
  ce_bwd_kernel<<<(int)cap, kCeThreads, 0, c.stream>>>(logits, targets, V, M, cap, idx, n_kept, dz, c.st);
  prof_end(c);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_embed_bwd(const Ctx& c, const __nv_bfloat16* dx, long long ld, int D, const int32_t* ids,
                             int V, int M, const int32_t* idx, const int32_t* n_kept, float* dE) {
  prof_begin(c, "embed_bwd");
  embed_bwd_kernel<<<M, 256, 0, c.stream>>>(dx, ld, D, ids, V, M, idx, n_kept, dE, c.st);
  prof_end(c);
  count_launch();
  return cudaGetLastError();
}

}  // namespace collider

// f32 linear backward on the CUDA cores (f32 FMA, no TF32), for layers whose
// gradients must stay in binary32.  The gather of kept rows is fused into the
// operand loads (rows addressed through the kept-index list) and the scatter
// into the store, so the dimension-reduced GEMM (Collider, abstract) needs no
// compacted copies.  64 x 64 output tile per block, 16-deep k slices staged
// in shared memory, 4 x 4 outputs per thread.
#include "internal.h"

namespace collider {

namespace {

constexpr int TM = 64, TN = 64, TK = 16;

__global__ void __launch_bounds__(256) simt_gemm_kernel(SimtGemm g, DevStatus* st) {
  int M = g.M, K = g.K;
  if (g.dyn) {
    int nk = *g.n_kept;
    nk = nk < 0 ? 0 : nk;
    if (g.dyn == 1) M = min(M, nk);
    else K = min(K, nk);
  }
  const int m0 = blockIdx.y * TM, n0 = blockIdx.x * TN;
  if (m0 >= M) return;
  __shared__ float As[TK][TM + 4];
  __shared__ float Bs[TK][TN + 4];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += TK) {
    for (int i = threadIdx.x; i < TM * TK; i += 256) {
      // A tile: element (m, k)
      int mm, kk;
      if (!g.a_trans) { mm = i / TK; kk = i % TK; } else { kk = i / TM; mm = i % TM; }
      const int m = m0 + mm, k = k0 + kk;
      float v = 0.f;
      if (m < M && k < K) {
        long long row, col;
        if (!g.a_trans) { row = g.a_gather ? g.idx[m] : m; col = k; }
        else { row = g.a_gather ? g.idx[k] : k; col = m; }
        v = g.A[row * g.lda + col];
      }
      As[kk][mm] = v;
      // B tile: element (k, n)
      int nn;
      if (!g.b_trans) { nn = i / TK; kk = i % TK; } else { kk = i / TN; nn = i % TN; }
      const int n = n0 + nn, k2 = k0 + kk;
      float w = 0.f;
      if (n < g.N && k2 < K) {
        if (!g.b_trans) w = g.B[(long long)n * g.ldb + k2];
        else w = g.B[(long long)(g.b_gather ? g.idx[k2] : k2) * g.ldb + n];
      }
      Bs[kk][nn] = w;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= M) continue;
    const long long orow = g.c_scatter ? g.idx[m] : m;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n < g.N) g.C[orow * g.ldc + n] = acc[i][j];
    }
  }
  (void)st;
}

}  // namespace

cudaError_t launch_simt_gemm(const Ctx& c, const SimtGemm& g) {
  dim3 grid((g.N + TN - 1) / TN, (g.M + TM - 1) / TM);
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  prof_begin(c, "simt_gemm_f32", g.M, g.N, g.K, g.dyn);
  simt_gemm_kernel<<<grid, 256, 0, c.stream>>>(g, c.st);
  prof_end(c);
  count_launch();
  return cudaGetLastError();
}

}  // namespace collider

// Dense forward of one decoder block: the row kernels around the GEMMs and the
// attention (norms, bias + RoPE, activations, residual sums).  Collider keeps
// the forward dense (Fig. 2b: filtering acts on the backward only); this pass
// produces the saved set the filtered backward reads.  Every kernel works on
// FULL rows and rounds to bf16 exactly where the saved set is stored: the
// projection outputs (with their bias) before RoPE and before the activation,
// the residual sum before the second norm, and each saved tensor.
#include "internal.h"

namespace collider {

namespace {

constexpr int kNormThreads = 128;
constexpr int kNormMaxChunks = 4;   // 8 columns a chunk: D <= 128 * 4 * 8 = 4096

__device__ __forceinline__ float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

__device__ __forceinline__ void load8_f32(const float* p, float* v) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// One CTA per row: the row (after the optional residual sum) stays in
// registers, 8 columns per chunk.
__global__ void __launch_bounds__(kNormThreads) norm_fwd_kernel(NormFwdArgs a) {
  __shared__ float red[32];
  const int row = blockIdx.x;
  const int nch = a.D / 8;
  const __nv_bfloat16* xr = a.x + (long long)row * a.D;
  float v[kNormMaxChunks][8];
  float s1 = 0.f;
#pragma unroll
  for (int u = 0; u < kNormMaxChunks; ++u) {
    const int ch = threadIdx.x + u * kNormThreads;
#pragma unroll
    for (int e = 0; e < 8; ++e) v[u][e] = 0.f;
    if (ch < nch) {
      unpack8(*reinterpret_cast<const uint4*>(xr + 8 * ch), v[u]);
      if (a.add) {
        float t[8], bb[8];
        load8_f32(a.add + (long long)row * a.add_ld + 8 * ch, t);
        if (a.add_bias) unpack8(*reinterpret_cast<const uint4*>(a.add_bias + 8 * ch), bb);
#pragma unroll
        for (int e = 0; e < 8; ++e) v[u][e] = bf16_round(v[u][e] + t[e] + (a.add_bias ? bb[e] : 0.f));
        if (a.sum_out) *reinterpret_cast<uint4*>(a.sum_out + (long long)row * a.D + 8 * ch) = pack8(v[u]);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) s1 += a.layer_norm ? v[u][e] : v[u][e] * v[u][e];
    }
  }
  const float inv_d = 1.f / (float)a.D;
  float mean = 0.f, var;
  if (a.layer_norm) {
    mean = block_sum(s1, red) * inv_d;
    float s2 = 0.f;
#pragma unroll
    for (int u = 0; u < kNormMaxChunks; ++u) {
      const int ch = threadIdx.x + u * kNormThreads;
      if (ch < nch)
#pragma unroll
        for (int e = 0; e < 8; ++e) s2 += (v[u][e] - mean) * (v[u][e] - mean);
    }
    var = block_sum(s2, red) * inv_d;
  } else {
    var = block_sum(s1, red) * inv_d;   // mean of squares
  }
  const float rstd = 1.f / sqrtf(var + a.eps);
  if (threadIdx.x == 0) {
    a.rstd[row] = rstd;
    if (a.layer_norm && a.mean) a.mean[row] = mean;
  }
#pragma unroll
  for (int u = 0; u < kNormMaxChunks; ++u) {
    const int ch = threadIdx.x + u * kNormThreads;
    if (ch < nch) {
      float g[8], bt[8], o[8];
      unpack8(*reinterpret_cast<const uint4*>(a.gamma + 8 * ch), g);
      if (a.layer_norm) unpack8(*reinterpret_cast<const uint4*>(a.beta + 8 * ch), bt);
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] = norm_affine(v[u][e], mean, rstd, g[e], a.layer_norm ? bt[e] : 0.f);
      *reinterpret_cast<uint4*>(a.out + (long long)row * a.D + 8 * ch) = pack8(o);
    }
  }
}

// One CTA per row; thread per column.  Column j of head j / dh, dim d = j % dh:
// for the rotated heads and d < r (r = 2 * rot_half) it pairs with d +- r/2:
//   d <  r/2:  x_d c - x_{d+r/2} s        d >= r/2:  x_d c + x_{d-r/2} s
// with (c, s) of angle pos * base^(-2i/r), i = d mod r/2.
// The projection arrives as f32 (plus bias, rounded here) or already as bf16.
template <bool IN_BF16>
__global__ void qkv_rope_kernel(int N, int rot_heads, int dh, int rot_half, int T, const void* acc,
                                const __nv_bfloat16* bias, const float2* rope, __nv_bfloat16* qkv) {
  const int row = blockIdx.x;
  const int pos = row % T;
  const float* in = static_cast<const float*>(acc) + (long long)row * N;
  const __nv_bfloat16* in16 = static_cast<const __nv_bfloat16*>(acc) + (long long)row * N;
  auto value = [&](int j) {
    return IN_BF16 ? __bfloat162float(in16[j]) : bf16_round(in[j] + (bias ? __bfloat162float(bias[j]) : 0.f));
  };
  __nv_bfloat16* out = qkv + (long long)row * N;
  for (int j = threadIdx.x; j < N; j += blockDim.x) {
    float x = value(j);
    const int head = j / dh, d = j % dh;
    if (head < rot_heads && d < 2 * rot_half) {
      const bool lo = d < rot_half;
      const int jp = lo ? j + rot_half : j - rot_half;
      const float y = value(jp);
      const float2 cs = rope[(long long)pos * rot_half + (lo ? d : d - rot_half)];
      x = lo ? x * cs.x - y * cs.y : x * cs.x + y * cs.y;
    }
    out[j] = __float2bfloat16_rn(x);
  }
}

// SwiGLU from the saved bf16 [g | u] (the GEMM wrote it rounded): s = bf16(silu(g) u).
__global__ void swiglu_fwd_kernel(int M, int F, const __nv_bfloat16* up, __nv_bfloat16* act) {
  const int nch = F / 8;
  const long long total = (long long)M * nch;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int row = (int)(e / nch), c = 8 * (int)(e % nch);
    const __nv_bfloat16* in = up + (long long)row * 2 * F;
    float g[8], u[8], o[8];
    unpack8(*reinterpret_cast<const uint4*>(in + c), g);
    unpack8(*reinterpret_cast<const uint4*>(in + F + c), u);
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i] = silu_mul(g[i], u[i]);
    *reinterpret_cast<uint4*>(act + (long long)row * F + c) = pack8(o);
  }
}

// Thread per 8 columns of the F-wide half.
__global__ void act_fwd_kernel(int gelu, int M, int F, const float* acc, const __nv_bfloat16* bias,
                               __nv_bfloat16* up, __nv_bfloat16* act) {
  const int nch = F / 8;
  const long long total = (long long)M * nch;
  const int Nup = gelu ? F : 2 * F;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int row = (int)(e / nch), c = 8 * (int)(e % nch);
    const float* in = acc + (long long)row * Nup;
    float g[8], bb[8], o[8];
    load8_f32(in + c, g);
    if (bias) unpack8(*reinterpret_cast<const uint4*>(bias + c), bb);
#pragma unroll
    for (int i = 0; i < 8; ++i) g[i] = bf16_round(g[i] + (bias ? bb[i] : 0.f));
    *reinterpret_cast<uint4*>(up + (long long)row * Nup + c) = pack8(g);
    if (gelu) {
      const float k0 = 0.7978845608028654f, k1 = 0.044715f;   // sqrt(2/pi), cubic coefficient
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = 0.5f * g[i] * (1.f + tanhf(k0 * (g[i] + k1 * g[i] * g[i] * g[i])));
    } else {
      float u[8], ub[8];
      load8_f32(in + F + c, u);
      if (bias) unpack8(*reinterpret_cast<const uint4*>(bias + F + c), ub);
#pragma unroll
      for (int i = 0; i < 8; ++i) u[i] = bf16_round(u[i] + (bias ? ub[i] : 0.f));
      *reinterpret_cast<uint4*>(up + (long long)row * Nup + F + c) = pack8(u);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = silu_mul(g[i], u[i]);
    }
    *reinterpret_cast<uint4*>(act + (long long)row * F + c) = pack8(o);
  }
}

__global__ void residual_out_kernel(int M, int D, const __nv_bfloat16* res, const float* acc1,
                                    const __nv_bfloat16* bias1, const float* acc2, const __nv_bfloat16* bias2,
                                    __nv_bfloat16* y) {
  const int nch = D / 8;
  const long long total = (long long)M * nch;
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < total;
       e += (long long)gridDim.x * blockDim.x) {
    const int row = (int)(e / nch), c = 8 * (int)(e % nch);
    const long long off = (long long)row * D + c;
    float v[8], t[8], b[8];
    unpack8(*reinterpret_cast<const uint4*>(res + off), v);
    load8_f32(acc1 + off, t);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] += t[i];
    if (bias1) {
      unpack8(*reinterpret_cast<const uint4*>(bias1 + c), b);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] += b[i];
    }
    if (acc2) {
      load8_f32(acc2 + off, t);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] += t[i];
    }
    if (bias2) {
      unpack8(*reinterpret_cast<const uint4*>(bias2 + c), b);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] += b[i];
    }
    *reinterpret_cast<uint4*>(y + off) = pack8(v);
  }
}

__global__ void iota_cu_kernel(int B, int T, int32_t* cu) {
  for (int b = threadIdx.x; b <= B; b += blockDim.x) cu[b] = b * T;
}

// every token kept: idx[i] = i, cu[b] = b*T, n_kept = B*T
__global__ void identity_index_kernel(int B, int T, int32_t* idx, int32_t* cu, int32_t* nk) {
  const long long M = (long long)B * T;
  const long long tid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long i = tid; i < M; i += stride) idx[i] = (int32_t)i;
  for (long long b = tid; b <= B; b += stride) cu[b] = (int32_t)(b * T);
  if (tid == 0) nk[0] = (int32_t)M;
}

int grid_for(const Ctx& c, long long work) {
  const long long want = (work + 255) / 256, cap = (long long)c.num_sms * 8;
  return (int)(want < 1 ? 1 : (want < cap ? want : cap));
}

}  // namespace

cudaError_t launch_norm_fwd(const Ctx& c, const NormFwdArgs& a) {
  if (a.D % 8 || a.D > kNormThreads * kNormMaxChunks * 8 || a.M < 0) return cudaErrorInvalidValue;
  if (a.M == 0) return cudaSuccess;
  prof_begin(c, "norm_fwd");
  norm_fwd_kernel<<<a.M, kNormThreads, 0, c.stream>>>(a);
  prof_end(c);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_qkv_rope_fwd(const Ctx& c, int M, int N, int rot_heads, int dh, int rot_half, int T,
                                const void* acc, int acc_bf16, const __nv_bfloat16* bias, const float2* rope,
                                __nv_bfloat16* qkv) {
  if (M <= 0) return cudaSuccess;
  if ((rot_half > 0 && !rope) || (acc_bf16 && bias)) return cudaErrorInvalidValue;
  prof_begin(c, "qkv_rope_fwd");
  if (acc_bf16)
    qkv_rope_kernel<true><<<M, 256, 0, c.stream>>>(N, rot_heads, dh, rot_half, T, acc, nullptr, rope, qkv);
  else
    qkv_rope_kernel<false><<<M, 256, 0, c.stream>>>(N, rot_heads, dh, rot_half, T, acc, bias, rope, qkv);
  prof_end(c);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_act_fwd(const Ctx& c, int gelu, int M, int F, const float* acc, const __nv_bfloat16* bias,
                           __nv_bfloat16* up, __nv_bfloat16* act) {
  if (F % 8) return cudaErrorInvalidValue;
  if (M <= 0) return cudaSuccess;
  prof_begin(c, "act_fwd");
  act_fwd_kernel<<<grid_for(c, (long long)M * (F / 8)), 256, 0, c.stream>>>(gelu, M, F, acc, bias, up, act);
  prof_end(c);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_swiglu_fwd(const Ctx& c, int M, int F, const __nv_bfloat16* up, __nv_bfloat16* act) {
  if (F % 8) return cudaErrorInvalidValue;
  if (M <= 0) return cudaSuccess;
  prof_begin(c, "act_fwd");
  swiglu_fwd_kernel<<<grid_for(c, (long long)M * (F / 8)), 256, 0, c.stream>>>(M, F, up, act);
  prof_end(c);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_residual_out(const Ctx& c, int M, int D, const __nv_bfloat16* res, const float* acc1,
                                const __nv_bfloat16* bias1, const float* acc2, const __nv_bfloat16* bias2,
                                __nv_bfloat16* y) {
  if (D % 8) return cudaErrorInvalidValue;
  if (M <= 0) return cudaSuccess;
  prof_begin(c, "residual_out");
  residual_out_kernel<<<grid_for(c, (long long)M * (D / 8)), 256, 0, c.stream>>>(M, D, res, acc1, bias1, acc2,
                                                                                 bias2, y);
  prof_end(c);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_iota_cu(const Ctx& c, int B, int T, int32_t* cu) {
  iota_cu_kernel<<<1, 256, 0, c.stream>>>(B, T, cu);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_identity_index(const Ctx& c, int B, int T, int32_t* idx, int32_t* cu, int32_t* nk) {
  identity_index_kernel<<<grid_for(c, (long long)B * T), 256, 0, c.stream>>>(B, T, idx, cu, nk);
  count_launch();
  return cudaGetLastError();
}

}  // namespace collider

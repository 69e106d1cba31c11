// Shared device helpers for libcollider kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace collider {

// ---------------------------------------------------------------------------
// device status word: kernels record the first failure here (host reads it
// in collider_check).  Codes:
constexpr unsigned kErrTimeout = 1u;  // a bounded wait ran out
constexpr unsigned kErrBadIndex = 2u; // an index outside its buffer was seen and skipped

struct DevStatus {
  unsigned code;   // first error code (0 = ok)
  unsigned site;   // which wait / check gave up
  unsigned block;  // blockIdx.x of the reporter
  unsigned pad;
};

__device__ __forceinline__ void report_error(DevStatus* st, unsigned code, unsigned site) {
  if (st != nullptr && atomicCAS(&st->code, 0u, code) == 0u) {
    st->site = site;
    st->block = blockIdx.x;
  }
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Wait budget for any spin inside a kernel: generous against any legitimate
// wait (kernels here run for at most milliseconds), short enough that a
// broken pipeline gives the GPU back within seconds.
constexpr uint64_t kWaitBudgetNs = 2000000000ull;  // 2 s

// ---------------------------------------------------------------------------
// programmatic dependent launch.  A kernel launched with the programmatic
// stream-serialisation attribute is scheduled as soon as the kernel ahead of
// it in the stream has exited, without waiting for that kernel's completion
// to be processed; it must not touch memory that kernel (or any earlier one)
// reads or writes before grid_dep_wait() returns, which happens once those
// grids have completed and their writes are visible.  Every kernel that may
// be launched so calls it in every CTA before it exits, so the wait reaches
// back along the whole stream.  No kernel here lets its dependents be
// scheduled before it exits (griddepcontrol.launch_dependents): measured on
// the layer backward, the chain's next kernel then parked on SMs that the
// side stream's persistent weight-gradient GEMMs were waiting for, and the
// step was 10% slower; scheduled at exit it is 2% faster than without the
// attribute.  For a kernel launched without the attribute the wait returns
// at once.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------------------
// The forward's elementwise outputs that the backward may recompute instead of
// reading them from the saved set (SwiGLU's s = silu(g) u, an RMSNorm output).
// Forward and backward both call these, every rounding spelled out (no
// contraction into a fused multiply-add the compiler might choose differently
// at the two sites), so a recomputed value is the forward's bit for bit.
__device__ __forceinline__ float silu_mul(float g, float u) {
  // g * sigmoid(g) * u; the hardware exponential is plenty for a bf16 result
  return __fmul_rn(__fmul_rn(g, __frcp_rn(__fadd_rn(1.f, __expf(-g)))), u);
}
__device__ __forceinline__ float norm_affine(float v, float mean, float rstd, float gamma, float beta) {
  return __fmaf_rn(__fmul_rn(__fsub_rn(v, mean), rstd), gamma, beta);
}

// ---------------------------------------------------------------------------
// small math / conversion helpers

__device__ __forceinline__ void unpack8(const uint4& u, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

__device__ __forceinline__ uint4 pack8(const float* f) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}

// two floats as bf16 (round to nearest even), a in the low half
__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum for blockDim.x a multiple of 32 (<= 1024); every thread
// gets the result.  `red` must hold 32 floats of shared memory.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = (lane < nw) ? red[lane] : 0.f;
  return warp_sum(t);
}

__device__ __forceinline__ float block_max(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  v = warp_max(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float t = (lane < nw) ? red[lane] : -INFINITY;
  return warp_max(t);
}

// Rows a COMPACT buffer must hold valid data or zeros for: n_kept rounded up
// to the GEMM tile height, capped at the buffer capacity.
__device__ __forceinline__ int padded_rows(int n, long long cap) {
  long long p = ((long long)n + 127) & ~127ll;
  return (int)(p < cap ? p : cap);
}

}  // namespace collider

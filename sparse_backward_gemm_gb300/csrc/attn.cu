// Filtered attention backward over the compacted sequences (Collider, Figs. 3
// and 5): the probabilities of filtered tokens are zeroed so G_V, G_Q and G_K
// stay sparse.  Working on the COMPACT rows does exactly that: only kept
// queries and kept keys exist, and because compaction keeps token order,
// causality on compacted indices equals causality on original positions.
//
//   P_ij = exp(S_ij * scale - lse_i)   (lse from the dense forward; no
//                                       renormalisation over kept keys)
//   D_i  = sum_j P_ij dP_ij = dO_i . O'_i,  O'_i = sum_j P_ij V_j  (pre-pass)
//   dV   = P^T dO;  dS = P * (dP - D);  dK = dS^T Q * scale;  dQ = dS K * scale
//
// Kernels: prep (lse in kept order, RoPE table, dQ accumulator reset), the
// D pre-pass (one block per sequence x head x 64 queries), the main pass
// (one block per sequence x kv head x 64 keys; loops over the group's query
// heads and the causal query blocks; dK, dV accumulate in registers; dQ
// accumulates in f32 with atomics), and a finalize pass (dQ scale + RoPE
// backward, bf16, zero padding rows).  Tensor-core math is mma.sync
// m16n8k16 bf16 with f32 accumulation.
#include "internal.h"

namespace collider {

namespace {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

constexpr int kBlk = 64;   // queries per query block and keys per key block

// Shared-memory tile of 64 rows x DH bf16, padded by 8 to keep ldmatrix rows
// on distinct banks.
template <int DH>
struct Tile {
  static constexpr int kLd = DH + 8;
};

// Load 64 rows (rows >= nrows zero-filled) of a head slice into a padded tile.
template <int DH>
__device__ __forceinline__ void load_tile(__nv_bfloat16* s, const __nv_bfloat16* g, long long ld, int nrows) {
  constexpr int kVec = DH / 8;
  for (int i = threadIdx.x; i < kBlk * kVec; i += blockDim.x) {
    const int r = i / kVec, c = (i % kVec) * 8;
    __nv_bfloat16* d = s + r * Tile<DH>::kLd + c;
    if (r < nrows) cp_async16(d, g + (long long)r * ld + c);
    else *reinterpret_cast<uint4*>(d) = make_uint4(0, 0, 0, 0);
  }
}

struct AttnK {
  int B, T, H, Hkv, G, causal;
  float scale, scale_log2;
  int rot_half;      // rotary_dim / 2 (0 = no RoPE backward)
  const __nv_bfloat16 *q, *k, *v, *dO;
  long long q_ld, kv_ld, do_ld;
  const float* lse;
  const int32_t *idx, *cu_kept, *n_kept;
  __nv_bfloat16 *dq, *dk, *dv;
  long long dq_ld, dkv_ld;
  float* dq_acc;     // [M, H, DH]
  float* Dvec;       // [H, M]
  float* lse2;       // [H, M]  lse * log2(e), kept order
  const float2* rope;  // [T, rot_half] (cos, sin)
  int M;
  long long cap;     // row capacity of dq, dk, dv
  DevStatus* st;
};

// ---------------------------------------------------------------------------
// prep: lse in kept order (log2 units), dQ accumulator reset, RoPE table
__global__ void attn_prep_kernel(AttnK p, int DH, float rope_base, float2* rope) {
  const int nk = *p.n_kept;
  const long long tid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  for (long long e = tid; e < (long long)p.H * nk; e += stride) {
    const int h = (int)(e / nk), r = (int)(e % nk);
    const int t = p.idx[r];
    const int b = t / p.T, ti = t % p.T;
    p.lse2[(long long)h * p.M + r] = p.lse[((long long)b * p.H + h) * p.T + ti] * kLog2e;
  }
  const long long nacc = (long long)nk * p.H * DH / 4;
  float4* acc4 = reinterpret_cast<float4*>(p.dq_acc);
  for (long long e = tid; e < nacc; e += stride) acc4[e] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (p.rot_half > 0) {
    const int rd = 2 * p.rot_half;
    for (long long e = tid; e < (long long)p.T * p.rot_half; e += stride) {
      const int pos = (int)(e / p.rot_half), i = (int)(e % p.rot_half);
      const double inv = pow((double)rope_base, -(2.0 * i) / (double)rd);
      const double ang = (double)pos * inv;
      rope[e] = make_float2((float)cos(ang), (float)sin(ang));
    }
  }
}

// ---------------------------------------------------------------------------
// D pre-pass: O'_i = sum_{j<=i} P_ij V_j over kept keys; D_i = dO_i . O'_i
template <int DH>
__global__ void __launch_bounds__(128) attn_dprep_kernel(AttnK p) {
  constexpr int LD = Tile<DH>::kLd;
  extern __shared__ __align__(16) uint8_t smraw[];
  __nv_bfloat16* sQ = reinterpret_cast<__nv_bfloat16*>(smraw);
  __nv_bfloat16* sdO = sQ + kBlk * LD;
  __nv_bfloat16* sK = sdO + kBlk * LD;
  __nv_bfloat16* sV = sK + kBlk * LD;
  const int nqb = (p.T + kBlk - 1) / kBlk;
  const int ib = blockIdx.x % nqb;
  const int h = (blockIdx.x / nqb) % p.H;
  const int b = blockIdx.x / (nqb * p.H);
  const int s0 = p.cu_kept[b], len = p.cu_kept[b + 1] - s0;
  const int i0 = ib * kBlk;
  if (i0 >= len) return;
  const int hk = h / p.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int qrows = min(kBlk, len - i0);
  load_tile<DH>(sQ, p.q + (long long)(s0 + i0) * p.q_ld + h * DH, p.q_ld, qrows);
  load_tile<DH>(sdO, p.dO + (long long)(s0 + i0) * p.do_ld + h * DH, p.do_ld, qrows);
  // per-thread rows: g and g+8 of this warp's 16
  const int qr0 = warp * 16 + g, qr1 = qr0 + 8;
  const float L0 = (qr0 < qrows) ? p.lse2[(long long)h * p.M + s0 + i0 + qr0] : 0.f;
  const float L1 = (qr1 < qrows) ? p.lse2[(long long)h * p.M + s0 + i0 + qr1] : 0.f;
  float o[DH / 8][4];
#pragma unroll
  for (int n = 0; n < DH / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  const int jend = p.causal ? ib : (len - 1) / kBlk;
  for (int jb = 0; jb <= jend; ++jb) {
    const int j0 = jb * kBlk;
    const int krows = min(kBlk, len - j0);
    __syncthreads();
    load_tile<DH>(sK, p.k + (long long)(s0 + j0) * p.kv_ld + hk * DH, p.kv_ld, krows);
    load_tile<DH>(sV, p.v + (long long)(s0 + j0) * p.kv_ld + hk * DH, p.kv_ld, krows);
    cp_async_wait_all();
    __syncthreads();
    // S = Q K^T : 16 queries x 64 keys for this warp
    float s[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int kt = 0; kt < DH / 16; ++kt) {
      uint32_t a[4];
      ldsm_x4(smem_addr(sQ + (warp * 16 + (lane & 15)) * LD + kt * 16 + (lane >> 4) * 8), a[0], a[1], a[2], a[3]);
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(smem_addr(sK + (np * 16 + (lane & 7) + ((lane >> 4) << 3)) * LD + kt * 16 + ((lane >> 3) & 1) * 8),
                b0, b1, b2, b3);
        mma16816(s[2 * np], a, b0, b1);
        mma16816(s[2 * np + 1], a, b2, b3);
      }
    }
    // P (zero outside the causal / sequence range)
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int qi = (e < 2 ? qr0 : qr1);
        const int kj = n * 8 + 2 * t4 + (e & 1);
        const bool ok = (qi < qrows) && (kj < krows) && (!p.causal || j0 + kj <= i0 + qi);
        s[n][e] = ok ? exp2f(s[n][e] * p.scale_log2 - (e < 2 ? L0 : L1)) : 0.f;
      }
    // O' += P V
#pragma unroll
    for (int kt = 0; kt < 4; ++kt) {
      uint32_t a[4] = {pack_bf2(s[2 * kt][0], s[2 * kt][1]), pack_bf2(s[2 * kt][2], s[2 * kt][3]),
                       pack_bf2(s[2 * kt + 1][0], s[2 * kt + 1][1]), pack_bf2(s[2 * kt + 1][2], s[2 * kt + 1][3])};
#pragma unroll
      for (int np = 0; np < DH / 16; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(smem_addr(sV + (kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LD + np * 16 + (lane >> 4) * 8),
                  b0, b1, b2, b3);
        mma16816(o[2 * np], a, b0, b1);
        mma16816(o[2 * np + 1], a, b2, b3);
      }
    }
  }
  // D_i = dO_i . O'_i
  float d0 = 0.f, d1 = 0.f;
#pragma unroll
  for (int n = 0; n < DH / 8; ++n) {
    const int c = n * 8 + 2 * t4;
    const __nv_bfloat162 x0 = *reinterpret_cast<const __nv_bfloat162*>(sdO + qr0 * LD + c);
    const __nv_bfloat162 x1 = *reinterpret_cast<const __nv_bfloat162*>(sdO + qr1 * LD + c);
    const float2 f0 = __bfloat1622float2(x0), f1 = __bfloat1622float2(x1);
    d0 += f0.x * o[n][0] + f0.y * o[n][1];
    d1 += f1.x * o[n][2] + f1.y * o[n][3];
  }
  d0 += __shfl_xor_sync(0xffffffffu, d0, 1);
  d0 += __shfl_xor_sync(0xffffffffu, d0, 2);
  d1 += __shfl_xor_sync(0xffffffffu, d1, 1);
  d1 += __shfl_xor_sync(0xffffffffu, d1, 2);
  if (t4 == 0) {
    if (qr0 < qrows) p.Dvec[(long long)h * p.M + s0 + i0 + qr0] = d0;
    if (qr1 < qrows) p.Dvec[(long long)h * p.M + s0 + i0 + qr1] = d1;
  }
}

// ---------------------------------------------------------------------------
// main pass: one block per (sequence, kv head, 64 keys)
template <int DH>
__global__ void __launch_bounds__(128) attn_main_kernel(AttnK p) {
  constexpr int LD = Tile<DH>::kLd;
  constexpr int LDS = kBlk + 8;
  extern __shared__ __align__(16) uint8_t smraw[];
  __nv_bfloat16* sK = reinterpret_cast<__nv_bfloat16*>(smraw);
  __nv_bfloat16* sV = sK + kBlk * LD;
  __nv_bfloat16* sQ = sV + kBlk * LD;
  __nv_bfloat16* sdO = sQ + kBlk * LD;
  __nv_bfloat16* sdS = sdO + kBlk * LD;     // [key][query]
  float* sL = reinterpret_cast<float*>(sdS + kBlk * LDS);
  float* sD = sL + kBlk;

  const int nkb = (p.T + kBlk - 1) / kBlk;
  const int jb = blockIdx.x % nkb;          // small key blocks (most work) launch first
  const int hk = (blockIdx.x / nkb) % p.Hkv;
  const int b = blockIdx.x / (nkb * p.Hkv);
  const int s0 = p.cu_kept[b], len = p.cu_kept[b + 1] - s0;
  const int j0 = jb * kBlk;
  if (j0 >= len) return;
  const int krows = min(kBlk, len - j0);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
  const int kr0 = warp * 16 + g, kr1 = kr0 + 8;   // this thread's key rows

  load_tile<DH>(sK, p.k + (long long)(s0 + j0) * p.kv_ld + hk * DH, p.kv_ld, krows);
  load_tile<DH>(sV, p.v + (long long)(s0 + j0) * p.kv_ld + hk * DH, p.kv_ld, krows);

  float dk[DH / 8][4], dv[DH / 8][4];
#pragma unroll
  for (int n = 0; n < DH / 8; ++n)
#pragma unroll
    for (int e = 0; e < 4; ++e) dk[n][e] = dv[n][e] = 0.f;

  for (int hg = 0; hg < p.G; ++hg) {
    const int h = hk * p.G + hg;
    for (int ib = p.causal ? jb : 0; ib * kBlk < len; ++ib) {
      const int i0 = ib * kBlk;
      const int qrows = min(kBlk, len - i0);
      __syncthreads();   // previous iteration is done with sQ, sdO, sdS
      load_tile<DH>(sQ, p.q + (long long)(s0 + i0) * p.q_ld + h * DH, p.q_ld, qrows);
      load_tile<DH>(sdO, p.dO + (long long)(s0 + i0) * p.do_ld + h * DH, p.do_ld, qrows);
      if (threadIdx.x < kBlk) {
        const int r = threadIdx.x;
        sL[r] = (r < qrows) ? p.lse2[(long long)h * p.M + s0 + i0 + r] : 0.f;
        sD[r] = (r < qrows) ? p.Dvec[(long long)h * p.M + s0 + i0 + r] : 0.f;
      }
      cp_async_wait_all();
      __syncthreads();

      // S^T = K Q^T : this warp's 16 keys x 64 queries
      float s[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
      for (int kt = 0; kt < DH / 16; ++kt) {
        uint32_t a[4];
        ldsm_x4(smem_addr(sK + (warp * 16 + (lane & 15)) * LD + kt * 16 + (lane >> 4) * 8), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(smem_addr(sQ + (np * 16 + (lane & 7) + ((lane >> 4) << 3)) * LD + kt * 16 + ((lane >> 3) & 1) * 8),
                  b0, b1, b2, b3);
          mma16816(s[2 * np], a, b0, b1);
          mma16816(s[2 * np + 1], a, b2, b3);
        }
      }
      // P^T
#pragma unroll
      for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kj = (e < 2 ? kr0 : kr1);
          const int qi = n * 8 + 2 * t4 + (e & 1);
          const bool ok = (qi < qrows) && (kj < krows) && (!p.causal || j0 + kj <= i0 + qi);
          s[n][e] = ok ? exp2f(s[n][e] * p.scale_log2 - sL[qi]) : 0.f;
        }
      // dP^T = V dO^T
      float dp[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) dp[n][0] = dp[n][1] = dp[n][2] = dp[n][3] = 0.f;
#pragma unroll
      for (int kt = 0; kt < DH / 16; ++kt) {
        uint32_t a[4];
        ldsm_x4(smem_addr(sV + (warp * 16 + (lane & 15)) * LD + kt * 16 + (lane >> 4) * 8), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int np = 0; np < 4; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(smem_addr(sdO + (np * 16 + (lane & 7) + ((lane >> 4) << 3)) * LD + kt * 16 + ((lane >> 3) & 1) * 8),
                  b0, b1, b2, b3);
          mma16816(dp[2 * np], a, b0, b1);
          mma16816(dp[2 * np + 1], a, b2, b3);
        }
      }
      // dV += P^T dO  (k = queries)
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
        uint32_t a[4] = {pack_bf2(s[2 * kt][0], s[2 * kt][1]), pack_bf2(s[2 * kt][2], s[2 * kt][3]),
                         pack_bf2(s[2 * kt + 1][0], s[2 * kt + 1][1]), pack_bf2(s[2 * kt + 1][2], s[2 * kt + 1][3])};
#pragma unroll
        for (int np = 0; np < DH / 16; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(smem_addr(sdO + (kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LD + np * 16 + (lane >> 4) * 8),
                    b0, b1, b2, b3);
          mma16816(dv[2 * np], a, b0, b1);
          mma16816(dv[2 * np + 1], a, b2, b3);
        }
      }
      // dS^T = P^T (dP^T - D_query), kept in s[]
#pragma unroll
      for (int n = 0; n < 8; ++n)
#pragma unroll
        for (int e = 0; e < 4; ++e) s[n][e] = s[n][e] * (dp[n][e] - sD[n * 8 + 2 * t4 + (e & 1)]);
      // dK += dS^T Q  (k = queries)
#pragma unroll
      for (int kt = 0; kt < 4; ++kt) {
        uint32_t a[4] = {pack_bf2(s[2 * kt][0], s[2 * kt][1]), pack_bf2(s[2 * kt][2], s[2 * kt][3]),
                         pack_bf2(s[2 * kt + 1][0], s[2 * kt + 1][1]), pack_bf2(s[2 * kt + 1][2], s[2 * kt + 1][3])};
#pragma unroll
        for (int np = 0; np < DH / 16; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(smem_addr(sQ + (kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LD + np * 16 + (lane >> 4) * 8),
                    b0, b1, b2, b3);
          mma16816(dk[2 * np], a, b0, b1);
          mma16816(dk[2 * np + 1], a, b2, b3);
        }
      }
      // dS^T -> shared (bf16) for the dQ product
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const int c = n * 8 + 2 * t4;
        *reinterpret_cast<uint32_t*>(sdS + kr0 * LDS + c) = pack_bf2(s[n][0], s[n][1]);
        *reinterpret_cast<uint32_t*>(sdS + kr1 * LDS + c) = pack_bf2(s[n][2], s[n][3]);
      }
      __syncthreads();
      // dQ_i += dS K: this warp's 16 queries x DH, in 64-column halves
      const int q0 = warp * 16 + g, q1 = q0 + 8;
#pragma unroll
      for (int half = 0; half < DH / 64; ++half) {
        float dq[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) dq[n][0] = dq[n][1] = dq[n][2] = dq[n][3] = 0.f;
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {   // k = keys
          uint32_t a[4];
          ldsm_x4_t(smem_addr(sdS + (kt * 16 + (lane & 7) + ((lane >> 4) << 3)) * LDS + warp * 16 + ((lane >> 3) & 1) * 8),
                    a[0], a[1], a[2], a[3]);
#pragma unroll
          for (int np = 0; np < 4; ++np) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(smem_addr(sK + (kt * 16 + (lane & 7) + ((lane >> 3) & 1) * 8) * LD + half * 64 + np * 16 +
                                (lane >> 4) * 8),
                      b0, b1, b2, b3);
            mma16816(dq[2 * np], a, b0, b1);
            mma16816(dq[2 * np + 1], a, b2, b3);
          }
        }
#pragma unroll
        for (int n = 0; n < 8; ++n) {
          const int c = half * 64 + n * 8 + 2 * t4;
          if (q0 < qrows) {
            float* d = p.dq_acc + ((long long)(s0 + i0 + q0) * p.H + h) * DH + c;
            atomicAdd(d, dq[n][0]);
            atomicAdd(d + 1, dq[n][1]);
          }
          if (q1 < qrows) {
            float* d = p.dq_acc + ((long long)(s0 + i0 + q1) * p.H + h) * DH + c;
            atomicAdd(d, dq[n][2]);
            atomicAdd(d + 1, dq[n][3]);
          }
        }
      }
    }
  }

  // epilogue: dK (scaled, RoPE backward) and dV, bf16, kept rows only
  const int rh = p.rot_half;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int kr = half ? kr1 : kr0;
    if (kr >= krows) continue;
    const long long row = s0 + j0 + kr;
    const int pos = p.idx[row] % p.T;
    float kv[DH / 8][2];
#pragma unroll
    for (int n = 0; n < DH / 8; ++n) {
      kv[n][0] = dk[n][2 * half] * p.scale;
      kv[n][1] = dk[n][2 * half + 1] * p.scale;
    }
    if (rh > 0) {
#pragma unroll
      for (int n = 0; n < DH / 8; ++n) {
        const int c = n * 8 + 2 * t4;
        if (c < rh) {
          const int n2 = n + rh / 8;   // partner columns c + rh live in tile n2 of this thread
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float2 cs = p.rope[(long long)pos * rh + c + e];
            const float d1 = kv[n][e], d2 = kv[n2][e];
            kv[n][e] = d1 * cs.x + d2 * cs.y;
            kv[n2][e] = d2 * cs.x - d1 * cs.y;
          }
        }
      }
    }
#pragma unroll
    for (int n = 0; n < DH / 8; ++n) {
      const int c = n * 8 + 2 * t4;
      *reinterpret_cast<uint32_t*>(p.dk + row * p.dkv_ld + hk * DH + c) = pack_bf2(kv[n][0], kv[n][1]);
      *reinterpret_cast<uint32_t*>(p.dv + row * p.dkv_ld + hk * DH + c) =
          pack_bf2(dv[n][2 * half], dv[n][2 * half + 1]);
    }
  }
}

// ---------------------------------------------------------------------------
// finalize: dQ = scale * acc, RoPE backward, bf16; zero rows n_kept..pad of dQ, dK, dV
__global__ void attn_finalize_kernel(AttnK p, int DH) {
  const int nk = *p.n_kept;
  const int pad = padded_rows(nk, p.cap);
  const int rh = p.rot_half;
  const long long tid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  // one thread per (row, head, column pair (c, c+half) or single column beyond the rotary dims)
  const int per_head = DH / 2;   // each thread handles columns c and c + DH/2
  const long long total = (long long)nk * p.H * per_head;
  for (long long e = tid; e < total; e += stride) {
    const int c = (int)(e % per_head);
    const int h = (int)((e / per_head) % p.H);
    const int r = (int)(e / ((long long)per_head * p.H));
    const float* a = p.dq_acc + ((long long)r * p.H + h) * DH;
    __nv_bfloat16* o = p.dq + (long long)r * p.dq_ld + h * DH;
    // handle the pair (c, c + DH/2) when RoPE is off or for the pass-through
    // dims; with RoPE pair (i, i + rh) for i < rh
    if (rh == 0) {
      o[c] = f2bf(a[c] * p.scale);
      o[c + per_head] = f2bf(a[c + per_head] * p.scale);
    } else {
      // map thread c in [0, DH/2) to: rotary pair i = c if c < rh, else two
      // pass-through columns starting at 2*rh + 2*(c - rh)
      if (c < rh) {
        const int pos = p.idx[r] % p.T;
        const float2 cs = p.rope[(long long)pos * rh + c];
        const float d1 = a[c] * p.scale, d2 = a[c + rh] * p.scale;
        o[c] = f2bf(d1 * cs.x + d2 * cs.y);
        o[c + rh] = f2bf(d2 * cs.x - d1 * cs.y);
      } else {
        const int cc = 2 * rh + 2 * (c - rh);
        if (cc < DH) {
          o[cc] = f2bf(a[cc] * p.scale);
          o[cc + 1] = f2bf(a[cc + 1] * p.scale);
        }
      }
    }
  }
  // zero padding rows
  const long long zq = (long long)(pad - nk) * p.H * DH, zk = (long long)(pad - nk) * p.Hkv * DH;
  for (long long e = tid; e < zq; e += stride) {
    const int r = nk + (int)(e / ((long long)p.H * DH));
    const int c = (int)(e % ((long long)p.H * DH));
    p.dq[(long long)r * p.dq_ld + c] = f2bf(0.f);
  }
  for (long long e = tid; e < zk; e += stride) {
    const int r = nk + (int)(e / ((long long)p.Hkv * DH));
    const int c = (int)(e % ((long long)p.Hkv * DH));
    p.dk[(long long)r * p.dkv_ld + c] = f2bf(0.f);
    p.dv[(long long)r * p.dkv_ld + c] = f2bf(0.f);
  }
}

template <int DH>
cudaError_t run(const Ctx& c, const AttnK& k, float rope_base) {
  constexpr int LD = Tile<DH>::kLd;
  const size_t smem_prep = 4 * kBlk * LD * sizeof(__nv_bfloat16);
  const size_t smem_main = 4 * kBlk * LD * sizeof(__nv_bfloat16) + kBlk * (kBlk + 8) * sizeof(__nv_bfloat16) +
                           2 * kBlk * sizeof(float);
  static int seen[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !seen[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_dprep_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem_prep));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_main_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem_main));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) seen[dev] = 1;
  }
  const int nb = (k.T + kBlk - 1) / kBlk;
  prof_begin(c, "attn_prep");
  attn_prep_kernel<<<c.num_sms * 4, 256, 0, c.stream>>>(k, DH, rope_base, const_cast<float2*>(k.rope));
  prof_end(c);
  prof_begin(c, "attn_dprep");
  attn_dprep_kernel<DH><<<k.B * k.H * nb, 128, smem_prep, c.stream>>>(k);
  prof_end(c);
  prof_begin(c, "attn_main");
  attn_main_kernel<DH><<<k.B * k.Hkv * nb, 128, smem_main, c.stream>>>(k);
  prof_end(c);
  prof_begin(c, "attn_finalize");
  attn_finalize_kernel<<<c.num_sms * 4, 256, 0, c.stream>>>(k, DH);
  prof_end(c);
  count_launch(4);
  return cudaGetLastError();
}

}  // namespace

size_t attn_ws_bytes(int B, int T, int H, int Hkv, int dh) {
  const size_t M = (size_t)B * T;
  size_t b = 0;
  auto add = [&](size_t n) { b += (n + 255) & ~size_t(255); };
  add(M * H * dh * sizeof(float));      // dq_acc
  add(M * H * sizeof(float));           // Dvec
  add(M * H * sizeof(float));           // lse2
  add((size_t)T * (dh / 2) * sizeof(float2));   // RoPE table
  (void)Hkv;
  return b;
}

cudaError_t launch_attn_bwd(const Ctx& c, const AttnArgs& a) {
  AttnK k{};
  k.B = a.B; k.T = a.T; k.H = a.H; k.Hkv = a.Hkv; k.G = a.H / a.Hkv; k.causal = a.causal;
  k.scale = a.scale; k.scale_log2 = a.scale * kLog2e;
  k.rot_half = a.rotary_dim / 2;
  k.q = a.q; k.k = a.k; k.v = a.v; k.dO = a.dO;
  k.q_ld = a.q_ld; k.kv_ld = a.kv_ld; k.do_ld = a.do_ld;
  k.lse = a.lse; k.idx = a.idx; k.cu_kept = a.cu_kept; k.n_kept = a.n_kept;
  k.dq = a.dq; k.dk = a.dk; k.dv = a.dv; k.dq_ld = a.dq_ld; k.dkv_ld = a.dkv_ld;
  k.dq_acc = a.dq_acc; k.Dvec = a.Dvec; k.lse2 = a.lse_k;
  k.M = a.M; k.cap = a.cap > 0 ? a.cap : a.M; k.st = c.st;
  k.rope = a.rope;
  if (a.dh == 64) return run<64>(c, k, a.rope_base);
  if (a.dh == 128) return run<128>(c, k, a.rope_base);
  return cudaErrorInvalidValue;
}

}  // namespace collider

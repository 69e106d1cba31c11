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
// Kernels: prep (lse in kept order, RoPE table, accumulator reset), the D
// pre-pass (tcgen05, one CTA per sequence x head x 128 queries), the main pass
// (tcgen05, one CTA per 128 kept keys x sequence x kv head x chunk of the
// group's query heads; head dim 64 and 128 have their own kernels), and a
// finalize pass (scale, RoPE backward, bf16, zero padding rows).  dQ, dK and
// dV are summed in f32 by TMA bulk reduce-adds.
//
// The dense forward's attention (every token kept) reuses the D pre-pass
// pipeline in two passes: the log-sum-exp of each query row, then
// O = exp(S - lse) V.
#include "internal.h"
#include "tc_ptx.cuh"

namespace collider {

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

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
  float* dk_acc;     // [M, Hkv, DH]  (tcgen05 path: dK, dV reduced here, then finalized)
  float* dv_acc;
  int kv_acc;        // 1: dK / dV come from dk_acc / dv_acc
  float* Dvec;       // [H, M]
  float* lse2;       // [H, M]  lse * log2(e), kept order
  const float2* rope;  // [T, rot_half] (cos, sin)
  int* order;        // [1 + B * H * ceil(T / 64)]: work-item ticket, dQ accumulation turns
  int M;
  long long cap;     // row capacity of dq, dk, dv
  DevStatus* st;
};

// ---------------------------------------------------------------------------
// RoPE table [T, rot_half] of (cos, sin): theta_i = base^(-2i/r) once per
// block in fp64; the angle pos * theta_i and its reduction mod 2 pi in fp64,
// then sin / cos of the reduced angle.  Called by every thread of the block
// (rot_half <= 256).
__device__ __forceinline__ void fill_rope_table(int T, int rot_half, float rope_base, float2* rope, long long tid,
                                                long long stride) {
  __shared__ double inv[256];
  const int rd = 2 * rot_half;
  for (int i = threadIdx.x; i < rot_half && i < 256; i += blockDim.x)
    inv[i] = pow((double)rope_base, -(2.0 * i) / (double)rd);
  __syncthreads();
  const double two_pi = 6.283185307179586476925;
  for (long long e = tid; e < (long long)T * rot_half; e += stride) {
    const int pos = (int)(e / rot_half), i = (int)(e % rot_half);
    const double ang = (double)pos * inv[i];
    const float red = (float)(ang - rint(ang / two_pi) * two_pi);
    float sn, cs;
    sincosf(red, &sn, &cs);
    rope[e] = make_float2(cs, sn);
  }
}

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
  if (p.kv_acc) {
    const long long nkv = (long long)nk * p.Hkv * DH / 4;
    float4* k4 = reinterpret_cast<float4*>(p.dk_acc);
    float4* v4 = reinterpret_cast<float4*>(p.dv_acc);
    for (long long e = tid; e < nkv; e += stride) {
      k4[e] = make_float4(0.f, 0.f, 0.f, 0.f);
      v4[e] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  // work-item ticket and dQ turns start at zero
  const long long nord = (long long)attn_order_ints(p.B, p.T, p.H);
  for (long long e = tid; e < nord; e += stride) p.order[e] = 0;
  if (p.rot_half > 0) fill_rope_table(p.T, p.rot_half, rope_base, rope, tid, stride);
}

__global__ void rope_table_kernel(int T, int rot_half, float rope_base, float2* rope) {
  fill_rope_table(T, rot_half, rope_base, rope, blockIdx.x * (long long)blockDim.x + threadIdx.x,
                  (long long)gridDim.x * blockDim.x);
}

// ---------------------------------------------------------------------------
// finalize: gradients from the f32 accumulators, times `scale`, RoPE backward
// where asked, to bf16; zero rows n_kept..pad of dQ, dK, dV.
// One thread per (row, head, column pair): the rotary pair (i, i + r/2) for
// i < r/2, else two adjacent pass-through columns.
// One unit of work = 8 columns of one (row, head): the rotary pairs
// (c..c+7, c+r/2..c+r/2+7) for c < r/2, else 8 pass-through columns.
__device__ __forceinline__ void load8f(const float* a, float* v) {
  const float4 x = *reinterpret_cast<const float4*>(a), y = *reinterpret_cast<const float4*>(a + 4);
  v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w; v[4] = y.x; v[5] = y.y; v[6] = y.z; v[7] = y.w;
}

__device__ __forceinline__ void finalize_unit(const float* a, __nv_bfloat16* o, int u, int rh,
                                              const float2* rope_row, float scale) {
  const int pairs = rh / 8;
  if (u < pairs) {
    const int c = 8 * u;
    float d1[8], d2[8], o1[8], o2[8];
    load8f(a + c, d1);
    load8f(a + c + rh, d2);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float2 cs = rope_row[c + e];
      const float x1 = d1[e] * scale, x2 = d2[e] * scale;
      o1[e] = x1 * cs.x + x2 * cs.y;
      o2[e] = x2 * cs.x - x1 * cs.y;
    }
    *reinterpret_cast<uint4*>(o + c) = pack8(o1);
    *reinterpret_cast<uint4*>(o + c + rh) = pack8(o2);
  } else {
    const int c = 2 * rh + 8 * (u - pairs);
    float d[8];
    load8f(a + c, d);
#pragma unroll
    for (int e = 0; e < 8; ++e) d[e] *= scale;
    *reinterpret_cast<uint4*>(o + c) = pack8(d);
  }
}

__global__ void attn_finalize_kernel(AttnK p, int DH) {
  grid_dep_wait();
  const int nk = *p.n_kept;
  const int pad = padded_rows(nk, p.cap);
  const int rh = p.rot_half;
  const long long tid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long stride = (long long)gridDim.x * blockDim.x;
  const int units = rh / 8 + (DH - 2 * rh) / 8;            // per (row, head)
  const long long tq = (long long)nk * p.H * units;
  const long long tk = p.kv_acc ? (long long)nk * p.Hkv * units : 0;
  const int vunits = DH / 8;                                // dV: no rotation
  const long long tv = p.kv_acc ? (long long)nk * p.Hkv * vunits : 0;
  for (long long e = tid; e < tq + tk + tv; e += stride) {
    long long f = e;
    int which = 0;   // 0 dQ, 1 dK, 2 dV
    if (f >= tq) {
      f -= tq;
      which = 1;
      if (f >= tk) { f -= tk; which = 2; }
    }
    const int nh = which == 0 ? p.H : p.Hkv;
    const int per = which == 2 ? vunits : units;
    const int u = (int)(f % per);
    const int h = (int)((f / per) % nh);
    const int r = (int)(f / ((long long)per * nh));
    const float* acc = which == 0 ? p.dq_acc : (which == 1 ? p.dk_acc : p.dv_acc);
    const float* a = acc + ((long long)r * nh + h) * DH;
    __nv_bfloat16* o = which == 0 ? p.dq + (long long)r * p.dq_ld + h * DH
                                  : (which == 1 ? p.dk : p.dv) + (long long)r * p.dkv_ld + h * DH;
    const int use_rh = which == 2 ? 0 : rh;
    const float2* rope_row = use_rh ? p.rope + (long long)(p.idx[r] % p.T) * rh : nullptr;
    finalize_unit(a, o, u, use_rh, rope_row, which == 2 ? 1.f : p.scale);
  }
  // zero padding rows, 16 bytes at a time
  const int qv = p.H * DH / 8, kvv = p.Hkv * DH / 8;
  const long long zq = (long long)(pad - nk) * qv, zk = (long long)(pad - nk) * kvv;
  for (long long e = tid; e < zq; e += stride) {
    const int r = nk + (int)(e / qv);
    *reinterpret_cast<uint4*>(p.dq + (long long)r * p.dq_ld + 8 * (e % qv)) = make_uint4(0, 0, 0, 0);
  }
  for (long long e = tid; e < zk; e += stride) {
    const int r = nk + (int)(e / kvv);
    const long long off = (long long)r * p.dkv_ld + 8 * (e % kvv);
    *reinterpret_cast<uint4*>(p.dk + off) = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(p.dv + off) = make_uint4(0, 0, 0, 0);
  }
}

// ---------------------------------------------------------------------------
// tcgen05 main pass, head dim 64.  One CTA per work item (sequence, kv head,
// 128 keys, a chunk of hc query heads of the group); items are numbered key
// block first, so the heavy (early) key blocks start first.
//   warp 0      TMA: K, V once; Q_i, dO_i per iteration (2 stages)
//   warp 1      TMEM owner; the converged warp waits, one elected lane issues
//               the MMAs, per 64-query half g:
//                 S^T = K Q_g^T, dP^T = V dO_g^T       (M 128 keys, N 64 queries)
//                 dV += P_g^T dO_g, dK += dS_g^T Q_g   (M 128 keys, N 64; A
//                                                       = P^T, dS^T from TMEM)
//               and per block dQ = dS K                (M 128 queries, N 64)
//   warps 2-9   query half 0, warps 10-17 query half 1: one key row and 32
//               of the half's 64 queries per thread: P^T, dS^T from TMEM ->
//               bf16 -> back into TMEM over the consumed S^T / dP^T columns;
//               dS^T also to shared (double-buffered by block) for dQ
//   warps 18-21 one query row per thread: dQ from TMEM into two staging
//               boxes (the TMEM buffer is handed back once read); at the end
//               dK, dV through the dS^T buffers into their accumulators
//   warps 22-23 one lane each, even / odd blocks: the dQ reduce-adds, in
//               key-block order, each turn passed on once its add completed
// TMEM columns: half 0 S^T 0-63 (P^T of its queries 0-31 in 0-15, of 32-63
// in 32-47, once formed), dP^T 64-127 (dS^T likewise); half 1 the same from
// 128; dV 256-319, dK 320-383, dQ 384-447 and 448-511 (double-buffered by
// block).
// P never goes through shared memory and dS^T has a buffer per block parity,
// so a softmax half waits only for the dQ of two blocks back.  The dQ adds
// of consecutive blocks overlap: a reducer waits for its add to complete
// (the next key block may add only then) while the other adds the next one.
namespace tcattn {
constexpr int kQ = 128, kK = 128, kD = 64;
constexpr uint32_t kTile = kQ * kD * 2;                 // 16 KB: 128 rows x 128 bytes
constexpr int kQS = 2;                                  // Q / dO stages
// Q and dO: kQS stages of one kTile each; dS^T buffers: two (block parity),
// each two halves of one kTile; dQ staging: two [128 rows x 32 f32] boxes.
// At the end of the item the dS^T buffers take dK and dV for their adds.
constexpr uint32_t OFF_K = 0, OFF_V = kTile, OFF_Q = 2 * kTile, OFF_DO = OFF_Q + kQS * kTile,
                   OFF_DS = OFF_DO + kQS * kTile, OFF_ST = OFF_DS + 4 * kTile, OFF_LD = OFF_ST + 2 * kTile,
                   OFF_BAR = OFF_LD + 2048;
constexpr size_t kSmem = 1024 + OFF_BAR + 256;
static_assert(kSmem <= 232448, "shared memory");
constexpr uint32_t TM_S = 0, TM_DV = 256, TM_DK = 320, TM_DQ = 384;
constexpr int kSoftWarps = 16;                      // four per TMEM lane quadrant
constexpr int kThreads = 32 * (2 + kSoftWarps + 4 + 2);
}  // namespace tcattn

struct MainTc {
  int B, T, H, Hkv, G, hc, nhc, nkb, causal;
  float scale_log2;
  const int32_t* cu_kept;
  const float* lse2;
  const float* Dvec;
  long long M;
  int* order;        // [0]: next work item; then the dQ turn of (sequence, head, query block)
  int nqb_max;       // query blocks per sequence at most (turn array stride)
  DevStatus* st;
};

// Work items are taken in ticket order, so an item only ever waits (for its
// dQ turn) on items that hold smaller tickets: items already running or done.
__device__ __forceinline__ int take_item(int* ticket) {
  __shared__ int s_item;
  if (threadIdx.x == 0) s_item = atomicAdd(ticket, 1);
  __syncthreads();
  return s_item;
}

// Key-block-ordered dQ accumulation.  The dQ tile of (sequence b, head h,
// query block ib) is added into the f32 accumulator by key block 0, 1, ... in
// turn, so the sum is the same every run.  The reducer thread of key block j
// waits for the tile's turn counter to reach j (dq_turn_wait), issues its TMA
// reduce-add, and once that add has completed passes the turn on to j + 1
// (dq_turn_flush).  A wait that runs out is recorded (COLLIDER_ERR_TIMEOUT)
// and the chain goes on unordered rather than stall.
__device__ __forceinline__ void dq_turn_flush(int*& pending, int j) {
  if (!pending) return;
  tc::bulk_wait_all();              // the previous add has completed
  tc::fence_proxy_async_global();
  tc::release_turn(pending, j + 1);
  pending = nullptr;
}
__device__ __forceinline__ int* dq_turn_wait(const MainTc& p, int b, int h, int ib, int j, bool& broken,
                                             unsigned site) {
  int* turn = p.order + 1 + ((long long)b * p.H + h) * p.nqb_max + ib;
  if (!broken && !tc::wait_turn(turn, j, p.st, site)) broken = true;
  tc::fence_proxy_async_global();
  return turn;
}

__global__ void __launch_bounds__(tcattn::kThreads, 1)
    attn_main_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                        const __grid_constant__ CUtensorMap tmdQ, const __grid_constant__ CUtensorMap tmdK,
                        const __grid_constant__ CUtensorMap tmdV, MainTc p) {
  using namespace tc;
  using namespace tcattn;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  grid_dep_wait();   // the work ticket, D', lse and the accumulators come from the kernels ahead
  const int item = take_item(p.order);
  const int per_j = p.B * p.Hkv * p.nhc;
  const int j = item / per_j;
  const int rem = item % per_j;
  const int b = rem / (p.Hkv * p.nhc);
  const int hk = (rem / p.nhc) % p.Hkv;
  const int hci = rem % p.nhc;
  const int s0 = p.cu_kept[b], len = p.cu_kept[b + 1] - s0;
  const int j0 = j * kK;
  if (j0 >= len) return;   // uniform: nothing initialised yet
  const int nqb = (len + kQ - 1) / kQ;
  const int i_start = p.causal ? j : 0;
  const int nq_head = nqb - i_start;
  const int n_iter = p.hc * nq_head;

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  // [kQS] = one per Q/dO stage (qfull, qempty, qready); [2] = one per query
  // half (sfull, pfull) or per block parity (dsempty: the dS^T buffer, handed
  // back by the epilogue; dqfull, dqempty: the dQ accumulator)
  const uint32_t b_kv = smem_u32(bars + 0), b_qfull = smem_u32(bars + 1), b_qempty = smem_u32(bars + 4),
                 b_sfull = smem_u32(bars + 7), b_pfull = smem_u32(bars + 9), b_dsempty = smem_u32(bars + 11),
                 b_dqfull = smem_u32(bars + 13), b_dqempty = smem_u32(bars + 15), b_kvready = smem_u32(bars + 17),
                 b_qready = smem_u32(bars + 18), b_staged = smem_u32(bars + 23), b_boxfree = smem_u32(bars + 25);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 21);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* sL = reinterpret_cast<float*>(sm + OFF_LD);   // [2][128]
  float* sD = sL + 256;                                // [2][128]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(b_kv, 1);
    for (int s = 0; s < kQS; ++s) {
      mbar_init(b_qfull + 8 * s, 1);
      mbar_init(b_qempty + 8 * s, 1);
      mbar_init(b_qready + 8 * s, 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(b_sfull + 8 * g, 1);
      mbar_init(b_pfull + 8 * g, 16 * kSoftWarps);
      mbar_init(b_dsempty + 8 * g, 1);
      mbar_init(b_dqfull + 8 * g, 1);
      mbar_init(b_dqempty + 8 * g, 128);
    }
    mbar_init(b_kvready, 1);
    for (int r = 0; r < 2; ++r) {
      mbar_init(b_staged + 8 * r, 1);
      mbar_init(b_boxfree + 8 * r, 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t sbase = smem_u32(sm);
  // The consumer groups below synchronise with named barriers, so they must
  // leave together: their waits give up only on their own timeout, which every
  // thread of the group reaches on the same barrier phase.
  volatile int no_abort = 0;

  if (warp == 0) {
    // ---------------- TMA producer (lane 0) + tile finishing (whole warp) ----------------
    // A tile may reach past its sequence into rows that hold anything; rows
    // past the sequence are zeroed in shared memory before the MMAs see the
    // tile (a masked probability of 0 times a non-finite row would leak).
    auto zero_rows = [&](uint32_t off, int from) {
      for (int i = lane; i < (128 - from) * 8; i += 32)
        *reinterpret_cast<uint4*>(sm + off + (from + i / 8) * 128 + (i % 8) * 16) = make_uint4(0, 0, 0, 0);
    };
    auto issue = [&](int it) -> bool {
      const int st = it % kQS, use = it / kQS;
      if (!mbar_wait(b_qempty + 8 * st, (use & 1) ^ 1, abort_flag, p.st, 20)) return false;
      const int h = hk * p.G + hci * p.hc + it % p.hc;
      const int i0 = (nqb - 1 - it / p.hc) * kQ;
      mbar_expect_tx(b_qfull + 8 * st, 2 * kTile);
      tma_load_2d(sbase + OFF_Q + st * kTile, &tmQ, b_qfull + 8 * st, h * kD, s0 + i0);
      tma_load_2d(sbase + OFF_DO + st * kTile, &tmdO, b_qfull + 8 * st, h * kD, s0 + i0);
      return true;
    };
    const int krows = min(kK, len - j0);
    bool ok = true;
    if (lane == 0) {
      mbar_expect_tx(b_kv, 2 * kTile);
      tma_load_2d(sbase + OFF_K, &tmK, b_kv, hk * kD, s0 + j0);
      tma_load_2d(sbase + OFF_V, &tmV, b_kv, hk * kD, s0 + j0);
    }
    if (mbar_wait(b_kv, 0, &no_abort, p.st, 28)) {
      if (krows < kK) {
        zero_rows(OFF_K, krows);
        zero_rows(OFF_V, krows);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_kvready);
    } else {
      ok = false;
    }
    // Block it+kQS-1 is requested once block it is handed over: its stage is
    // the one of block it-1, which the MMA thread frees (after dV, dK of
    // block it-1) without waiting for any later block, so the hand-over of
    // block it never waits on that stage.
    for (int i = 0; i < kQS - 1; ++i)
      if (lane == 0 && ok && n_iter > i) ok = issue(i);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    for (int it = 0; ok && it < n_iter; ++it) {
      const int st = it % kQS, use = it / kQS;
      if (!mbar_wait(b_qfull + 8 * st, use & 1, &no_abort, p.st, 29)) break;
      const int i0 = (nqb - 1 - it / p.hc) * kQ;
      const int qrows = min(kQ, len - i0);
      if (qrows < kQ) {
        zero_rows(OFF_Q + st * kTile, qrows);
        zero_rows(OFF_DO + st * kTile, qrows);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_qready + 8 * st);
      int nxt = 1;
      if (lane == 0 && it + kQS - 1 < n_iter) nxt = issue(it + kQS - 1) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, nxt, 0)) break;
    }
  } else if (warp == 1) {
    {
      // ---------------- MMA issuer: the converged warp waits, one elected lane issues ----------------
      // Query half g of iteration it has its own S^T / dP^T columns in TMEM
      // (buffer g), where its P^T lands too, so the MMAs of one half run while
      // the softmax warps of the other half work:
      //   S, dP (it, 0) | S, dP (it, 1) | [P(it, 0)] dV, dK (it, 0) | S, dP (it+1, 0)
      //   | [P(it, 1)] dV, dK (it, 1) | dQ (it) | S, dP (it+1, 1) | ...
      // MMAs issued by this thread run in issue order, so S (it+1, g) cannot
      // overwrite P (it, g) before dV (it, g) has read it.  (dQ (it) reads dS^T
      // from shared memory, so S, dP (it+1, 1) could go first; measured, the
      // order above was as fast.)
      const bool leader = elect_one();
      auto wait = [&](uint32_t bar, uint32_t parity, unsigned site) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.st, site)) != 0;
      };
      constexpr uint32_t id_s = idesc_bf16(128, 64, false, false);
      constexpr uint32_t id_kv = idesc_bf16(128, 64, false, true);
      constexpr uint32_t id_q = idesc_bf16(128, 64, true, true);
      // Shared-memory descriptors are built once; a k-step moves the start
      // address (bits 0-13, in 16-byte units) by a constant: +2 (32 bytes)
      // inside a K-major swizzle row, +128 (2 KB, 16 rows) down an MN-major tile.
      const uint64_t d_k = sdesc(sbase + OFF_K, 16, 1024), d_v = sdesc(sbase + OFF_V, 16, 1024);
      const uint64_t d_kmn = sdesc(sbase + OFF_K, 8192, 1024);            // K as the MN-major B of dQ
      const uint64_t d_ds_mn = sdesc(sbase + OFF_DS, kTile, 1024);        // dS^T as the MN-major A of dQ
      // per Q/dO stage (stage st is st kTiles on); per dS buffer and half
      const uint64_t d_q0 = sdesc(sbase + OFF_Q, 16, 1024), d_do0 = sdesc(sbase + OFF_DO, 16, 1024);
      const uint64_t d_qmn0 = sdesc(sbase + OFF_Q, 8192, 1024), d_domn0 = sdesc(sbase + OFF_DO, 8192, 1024);
      constexpr uint64_t kTileStep = kTile / 16;   // one tile further on, in descriptor units
      auto sdp = [&](int it, int g) {   // S^T, dP^T of half g: M 128 keys, N 64 queries
        const int st = it % kQS;
        const uint64_t bq = d_q0 + st * kTileStep + g * (kTileStep / 2),
                       bdo = d_do0 + st * kTileStep + g * (kTileStep / 2);
        const uint32_t ts = tbase + TM_S + g * 128, tdp = ts + 64;
        if (!leader) return;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) mma_bf16(ts, d_k + 2 * kk, bq + 2 * kk, id_s, kk > 0);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) mma_bf16(tdp, d_v + 2 * kk, bdo + 2 * kk, id_s, kk > 0);
        mma_commit(b_sfull + 8 * g);
      };
      auto dvdk = [&](int it, int g) {  // dV += P^T dO, dK += dS^T Q over the 64 queries of half g
        const int st = it % kQS;
        if (!leader) return;
        // P^T (dS^T) of this half: queries 0-31 packed in columns 0-15, 32-63
        // in 32-47 of its S^T (dP^T) columns; a k-step of 16 queries is 8 columns
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int kk = 4 * g + k4;
          mma_bf16_ts(tbase + TM_DV, tbase + TM_S + g * 128 + 32 * (k4 >> 1) + 8 * (k4 & 1),
                      d_domn0 + st * kTileStep + 128 * kk, id_kv, (it > 0) || (kk > 0));
        }
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4) {
          const int kk = 4 * g + k4;
          mma_bf16_ts(tbase + TM_DK, tbase + TM_S + g * 128 + 64 + 32 * (k4 >> 1) + 8 * (k4 & 1),
                      d_qmn0 + st * kTileStep + 128 * kk, id_kv, (it > 0) || (kk > 0));
        }
      };
      bool ok = wait(b_kvready, 0, 21);
      if (ok && n_iter > 0) {
        ok = wait(b_qready, 0, 22);
        if (ok) {
          fence_after();
          sdp(0, 0);
          sdp(0, 1);
        }
      }
      for (int it = 0; ok && it < n_iter; ++it) {
        const int st = it % kQS, a = it & 1, use = it >> 1;
        const bool more = it + 1 < n_iter;
        if (!wait(b_pfull, it & 1, 23)) break;
        fence_after();
        dvdk(it, 0);
        if (more) {
          if (!wait(b_qready + 8 * ((it + 1) % kQS), ((it + 1) / kQS) & 1, 22)) break;
          fence_after();
          sdp(it + 1, 0);
        }
        if (!wait(b_pfull + 8, it & 1, 23)) break;
        fence_after();
        dvdk(it, 1);
        if (leader) mma_commit(b_qempty + 8 * st);   // Q, dO of this block are read for the last time
        // dQ accumulator a was drained of block it-2
        if (use > 0 && !wait(b_dqempty + 8 * a, (use - 1) & 1, 24)) break;
        fence_after();
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kK / 16; ++kk)     // k = keys; dS read MN-major from the dS^T tiles
            mma_bf16(tbase + TM_DQ + 64 * a, d_ds_mn + 2 * a * kTileStep + 128 * kk, d_kmn + 128 * kk, id_q, kk > 0);
          mma_commit(b_dqfull + 8 * a);
          mma_commit(b_dsempty + 8 * a);   // dS^T buffer a is read for the last time
        }
        if (more) sdp(it + 1, 1);
      }
    }
  } else if (warp < 2 + kSoftWarps) {
    // ---------------- softmax warps: one key row, 32 queries per thread ----------------
    // Warps 2-9 own query half 0 of every block, warps 10-17 half 1; within
    // a half, its first four warps take the half's first 32 queries and the
    // other four the last 32.  The halves run independently, each on its own
    // TMEM buffer; the eight warps of a half meet at a named barrier per block.
    const int w = warp - 2;
    const int g = w >> 3;                       // query half
    const int cc = (w >> 2) & 1;                // which 32 queries of the half
    const int tg = threadIdx.x - 64 - 256 * g;  // 0..255 within the half's group
    const int q = warp & 3;
    const int kr = q * 32 + lane;
    const int key = j0 + kr;
    const bool kvalid = key < len;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    // lse (tg 0-63) and D (tg 64-127) of this half's queries for the block
    // after the current one are fetched one iteration early, so the
    // global-load latency hides behind the current block
    auto fetch = [&](int it) -> float {
      if (tg >= 128) return 0.f;
      const int h = hk * p.G + hci * p.hc + it % p.hc;
      const int i0 = (nqb - 1 - it / p.hc) * kQ;
      const int qq = 64 * g + (tg & 63);
      if (qq >= min(kQ, len - i0)) return 0.f;
      const float* src = tg < 64 ? p.lse2 : p.Dvec;
      return src[(long long)h * p.M + s0 + i0 + qq];
    };
    float nxt = n_iter > 0 ? fetch(0) : 0.f;
    for (int it = 0; it < n_iter; ++it) {
      const int i0 = (nqb - 1 - it / p.hc) * kQ;
      const int qrows = min(kQ, len - i0);
      const int buf = it & 1;
      if (tg < 128) (tg < 64 ? sL : sD)[buf * 128 + 64 * g + (tg & 63)] = nxt;
      if (it + 1 < n_iter) nxt = fetch(it + 1);
      named_bar(1 + 2 * g, 256);
      if (!mbar_wait(b_sfull + 8 * g, it & 1, &no_abort, p.st, 25)) break;
      fence_after();
      const float* L = sL + buf * 128;
      const float* Dd = sD + buf * 128;
      // 32 queries strictly below the diagonal, all inside the sequence, need no masking
      const bool interior = (!p.causal || i0 > j0) && qrows >= 64 * g + 32 * (cc + 1) && len - j0 >= kK;
      // 16 queries at a time (few registers live: this kernel runs 24 warps)
      const uint32_t col = TM_S + g * 128 + cc * 32;
      const uint32_t rowoff = g * kTile + kr * 128;
      bool failed = false;
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t sr[16], dr[16];
        tmem_ld16_async(tbase + lane_off + col + 16 * hh, sr);
        tmem_ld16_async(tbase + lane_off + col + 64 + 16 * hh, dr);
        // dS^T buffer (it & 1) is free once dQ of block it-2 has read it
        // (checked while the first loads are in flight)
        if (hh == 0 && it >= 2 && !mbar_wait(b_dsempty + 8 * (it & 1), ((it >> 1) - 1) & 1, &no_abort, p.st, 26))
          failed = true;
        tmem_wait_ld();
        if (failed) break;
        uint32_t pk[8], dk[8];   // bf16 pairs of P^T and dS^T
        if (interior) {
          // lse and D of these 16 queries, four at a time (16-byte shared loads)
          const float4* L4 = reinterpret_cast<const float4*>(L + 64 * g + cc * 32 + 16 * hh);
          const float4* D4 = reinterpret_cast<const float4*>(Dd + 64 * g + cc * 32 + 16 * hh);
#pragma unroll
          for (int e4 = 0; e4 < 4; ++e4) {
            const float4 l4 = L4[e4], d4 = D4[e4];
            const float lq[4] = {l4.x, l4.y, l4.z, l4.w}, dq[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
            for (int e2 = 0; e2 < 2; ++e2) {
              const int e = 2 * e4 + e2;
              const float p0 = exp2_approx(__uint_as_float(sr[2 * e]) * p.scale_log2 - lq[2 * e2]);
              const float p1 = exp2_approx(__uint_as_float(sr[2 * e + 1]) * p.scale_log2 - lq[2 * e2 + 1]);
              pk[e] = pack_bf16x2(p0, p1);
              dk[e] = pack_bf16x2(p0 * (__uint_as_float(dr[2 * e]) - dq[2 * e2]),
                                  p1 * (__uint_as_float(dr[2 * e + 1]) - dq[2 * e2 + 1]));
            }
          }
        } else {
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            float pv[2], dv[2];
#pragma unroll
            for (int k = 0; k < 2; ++k) {
              const int qi = 64 * g + cc * 32 + 16 * hh + 2 * e + k;
              const bool valid = kvalid && qi < qrows && (!p.causal || key <= i0 + qi);
              pv[k] = valid ? exp2_approx(__uint_as_float(sr[2 * e + k]) * p.scale_log2 - L[qi]) : 0.f;
              dv[k] = valid ? pv[k] * (__uint_as_float(dr[2 * e + k]) - Dd[qi]) : 0.f;
            }
            pk[e] = pack_bf16x2(pv[0], pv[1]);
            dk[e] = pack_bf16x2(dv[0], dv[1]);
          }
        }
        // P^T and dS^T into TMEM over S^T / dP^T columns already read: this
        // thread's 32 queries (columns 32 cc .. 32 cc + 31 of the half) pack
        // into the first 16 of those, these 16 queries into 8 at 32 cc + 8 hh
        // -- columns whose S / dP it loaded in sub-step 0.  The other
        // sub-group (the same TMEM lanes) reads and writes only its own 32.
        tmem_st8(tbase + lane_off + TM_S + g * 128 + 32 * cc + 8 * hh, pk);
        tmem_st8(tbase + lane_off + TM_S + g * 128 + 64 + 32 * cc + 8 * hh, dk);
        // and dS^T to shared: 16 queries = 32 bytes = two 16-byte chunks of the swizzled row
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint32_t phys = (((cc * 4 + 2 * hh + u) ^ (kr & 7)) * 16);
          *reinterpret_cast<uint4*>(sm + OFF_DS + (it & 1) * 2 * kTile + rowoff + phys) =
              make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
        }
      }
      if (failed) break;
      tmem_wait_st();
      fence_before();
      fence_async_smem();
      mbar_arrive(b_pfull + 8 * g);
    }
  } else if (warp < 2 + kSoftWarps + 4) {
    // ---------------- dQ / dK / dV epilogue: one row per thread ----------------
    const int t = threadIdx.x - 32 * (2 + kSoftWarps);
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    bool ok = true;
    // one row of 32 f32 into box `box` (128 rows x 128 bytes, 128-byte swizzle)
    auto stage32 = [&](uint32_t box, const float* v) {
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        const uint32_t phys = ((g ^ (r & 7)) * 16);
        *reinterpret_cast<float4*>(sm + box + r * 128 + phys) =
            make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
      }
    };
    for (int it = 0; it < n_iter; ++it) {
      const int h = hk * p.G + hci * p.hc + it % p.hc;
      const int i0 = (nqb - 1 - it / p.hc) * kQ;
      const int a = it & 1;
      if (!mbar_wait(b_dqfull + 8 * a, (it >> 1) & 1, &no_abort, p.st, 27)) { ok = false; break; }
      fence_after();
      // dQ through the two staging boxes (32 columns each); the boxes are free
      // once the previous block's adds have read them
      // the boxes are free once the reducer of the previous block saw its adds read them
      if (it > 0 && !mbar_wait(b_boxfree + 8 * ((it - 1) & 1), ((it - 1) >> 1) & 1, &no_abort, p.st, 31)) {
        ok = false;
        break;
      }
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        float v[32];
        tmem_ld32(tbase + lane_off + TM_DQ + 64 * a + 32 * half, v);
        if (half == 1) {
          fence_before();
          mbar_arrive(b_dqempty + 8 * a);
        }
        stage32(OFF_ST + half * kTile, v);
      }
      fence_async_smem();
      named_bar(2, 128);
      if (t == 0) mbar_arrive(b_staged + 8 * a);
    }
    if (ok) {
      // Every MMA has completed (the last dQ commit covers them all), so the
      // dS^T buffers are free: dK into buffer 0, dV into buffer 1.
#pragma unroll 1
      for (int pass = 0; pass < 4; ++pass) {   // dK then dV, 32 columns at a time
        const uint32_t col = (pass < 2 ? TM_DK : TM_DV) + 32 * (pass & 1);
        float v[32];
        tmem_ld32(tbase + lane_off + col, v);
        stage32(OFF_DS + pass * kTile, v);
      }
      fence_async_smem();
      named_bar(2, 128);
      if (t == 0) {
#pragma unroll 1
        for (int pass = 0; pass < 4; ++pass)
          tma_reduce_add_2d(pass < 2 ? &tmdK : &tmdV, sbase + OFF_DS + pass * kTile, hk * kD + 32 * (pass & 1),
                            s0 + j0);
        bulk_commit();
      }
    }
    if (t == 0) bulk_wait_all();
  } else if (lane == 0) {
    // ---------------- dQ reducers: warp 22 even blocks, warp 23 odd ----------------
    // Each adds its blocks' dQ tiles in key-block order (the tile's turn),
    // hands the staging boxes back once the adds have read them, and passes
    // the turn on as soon as its adds have completed: the two reducers
    // overlap one block's completion with the next block's adds.
    const int rr = warp - (2 + kSoftWarps + 4);
    bool broken = false;
    for (int it = rr; it < n_iter; it += 2) {
      const int h = hk * p.G + hci * p.hc + it % p.hc;
      const int i0 = (nqb - 1 - it / p.hc) * kQ;
      const int a = it & 1;
      if (!mbar_wait(b_staged + 8 * a, (it >> 1) & 1, abort_flag, p.st, 32)) break;
      int* turn = dq_turn_wait(p, b, h, i0 / kQ, j, broken, 30);
      tma_reduce_add_2d(&tmdQ, sbase + OFF_ST, h * kD, s0 + i0);
      tma_reduce_add_2d(&tmdQ, sbase + OFF_ST + kTile, h * kD + 32, s0 + i0);
      bulk_commit();
      bulk_wait_read_all();
      mbar_arrive(b_boxfree + 8 * a);
      dq_turn_flush(turn, j);
    }
    bulk_wait_all();
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ---------------------------------------------------------------------------
// tcgen05 main pass, head dim 128.  One CTA per work item (128 kept keys,
// sequence, kv head, a chunk of hc query heads), iterating over blocks of 64
// queries.  The TMEM budget sets the shape: S^T and dP^T (64 columns each),
// dV and dK (128 each) leave 64 columns, so dQ is formed transposed,
// dQ^T = K^T dS^T (M = 128 head dims, N = 64 queries).
//   warp 0      TMA: K, V once; Q_i, dO_i per iteration (2 stages)
//   warp 1      TMEM owner; one lane issues the MMAs:
//                 S^T = K Q^T, dP^T = V dO^T          (M 128 keys, N 64 queries)
//                 dV += P^T dO, dK += dS^T Q          (M 128 keys, N 128; A
//                                                      = P^T, dS^T from TMEM)
//                 dQ^T = K^T dS^T                     (M 128 head dims, N 64 queries)
//               in the order S, dP (it) | dV, dK (it) | S, dP (it+1) | dQ^T (it),
//               so the softmax of block it+1 overlaps dQ^T of block it
//   warps 2-9   one key row and 32 of the 64 queries per thread: P^T, dS^T
//               from TMEM -> bf16 -> back into TMEM over the consumed S^T /
//               dP^T columns; dS^T also to shared (double-buffered by block)
//               for dQ^T
//   warps 10-13 one head-dim row of dQ^T per thread: TMEM -> shared (as dQ
//               rows) -> TMA reduce-add into the f32 dQ accumulator; at the
//               end dK, dV likewise, 64 columns at a time
// Tiles are 64-column (128-byte) swizzle chunks.
// TMEM columns: S^T 0-63 (P^T of queries 32 g .. 32 g + 31 in 32 g .. 32 g +
// 15), dP^T 64-127 (dS^T likewise from 64), dV 128-255, dK 256-383, dQ^T
// 384-447.
namespace tcattn128 {
constexpr int kQ = 64, kK = 128, kD = 128;
constexpr uint32_t kKChunk = 16384;                 // 128 rows x 128 bytes
constexpr uint32_t kQChunk = 8192;                  // 64 rows x 128 bytes
// dS^T: two buffers (block parity) of one kKChunk
constexpr uint32_t OFF_K = 0, OFF_V = 2 * kKChunk, OFF_Q = 4 * kKChunk, OFF_DO = OFF_Q + 4 * kQChunk,
                   OFF_DS = OFF_DO + 4 * kQChunk, OFF_ST = OFF_DS + 2 * kKChunk,
                   OFF_LD = OFF_ST + 2 * kKChunk, OFF_BAR = OFF_LD + 1024;
constexpr size_t kSmem = 1024 + OFF_BAR + 256;
constexpr uint32_t TM_S = 0, TM_DP = 64, TM_DV = 128, TM_DK = 256, TM_DQ = 384;
constexpr int kSoftWarps = 8;                       // two per TMEM lane quadrant
constexpr int kThreads = 32 * (2 + kSoftWarps + 4 + 2);
static_assert(kSmem <= 232448, "shared memory");
}  // namespace tcattn128

__global__ void __launch_bounds__(tcattn128::kThreads, 1)
    attn_main_tc128_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                           const __grid_constant__ CUtensorMap tmdQ, const __grid_constant__ CUtensorMap tmdK,
                           const __grid_constant__ CUtensorMap tmdV, MainTc p) {
  using namespace tc;
  using namespace tcattn128;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  grid_dep_wait();   // the work ticket, D', lse and the accumulators come from the kernels ahead
  const int item = take_item(p.order);
  const int per_j = p.B * p.Hkv * p.nhc;
  const int j = item / per_j;
  const int rem = item % per_j;
  const int b = rem / (p.Hkv * p.nhc);
  const int hk = (rem / p.nhc) % p.Hkv;
  const int hci = rem % p.nhc;
  const int s0 = p.cu_kept[b], len = p.cu_kept[b + 1] - s0;
  const int j0 = j * kK;
  if (j0 >= len) return;   // uniform: nothing initialised yet
  const int nqb = (len + kQ - 1) / kQ;
  const int i_start = p.causal ? j0 / kQ : 0;
  const int nq_head = nqb - i_start;
  const int n_iter = p.hc * nq_head;

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  const uint32_t b_kv = smem_u32(bars + 0), b_qfull = smem_u32(bars + 1), b_qempty = smem_u32(bars + 3),
                 b_sfull = smem_u32(bars + 5), b_pfull = smem_u32(bars + 6), b_dsempty = smem_u32(bars + 7),
                 b_dqfull = smem_u32(bars + 9), b_dqempty = smem_u32(bars + 10), b_kvready = smem_u32(bars + 11),
                 b_qready = smem_u32(bars + 12), b_staged = smem_u32(bars + 16), b_boxfree = smem_u32(bars + 18);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 14);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* sL = reinterpret_cast<float*>(sm + OFF_LD);   // [2][64]
  float* sD = sL + 128;                                // [2][64]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(b_kv, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(b_qfull + 8 * s, 1);
      mbar_init(b_qempty + 8 * s, 1);
      mbar_init(b_qready + 8 * s, 1);
    }
    mbar_init(b_sfull, 1);
    mbar_init(b_pfull, 32 * kSoftWarps);
    mbar_init(b_dsempty, 1);
    mbar_init(b_dsempty + 8, 1);
    mbar_init(b_dqfull, 1);
    mbar_init(b_dqempty, 128);
    mbar_init(b_kvready, 1);
    for (int r = 0; r < 2; ++r) {
      mbar_init(b_staged + 8 * r, 1);
      mbar_init(b_boxfree + 8 * r, 1);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t sbase = smem_u32(sm);
  // The consumer groups below synchronise with named barriers, so they must
  // leave together: their waits give up only on their own timeout, which every
  // thread of the group reaches on the same barrier phase.
  volatile int no_abort = 0;

  if (warp == 0) {
    // ---------------- TMA producer (lane 0) + tile finishing (whole warp) ----------------
    // rows past the sequence are zeroed in shared memory before the MMAs see
    // a tile (a masked probability of 0 times a non-finite row would leak)
    auto zero_rows = [&](uint32_t off, int rows, int from) {
      for (int i = lane; i < (rows - from) * 8; i += 32)
        *reinterpret_cast<uint4*>(sm + off + (from + i / 8) * 128 + (i % 8) * 16) = make_uint4(0, 0, 0, 0);
    };
    auto issue = [&](int it) -> bool {
      const int st = it & 1, use = it >> 1;
      if (!mbar_wait_call(b_qempty + 8 * st, (use & 1) ^ 1, abort_flag, p.st, 50)) return false;
      const int h = hk * p.G + hci * p.hc + it % p.hc;
      const int i0 = (nqb - 1 - it / p.hc) * kQ;
      mbar_expect_tx(b_qfull + 8 * st, 4 * kQChunk);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        tma_load_2d(sbase + OFF_Q + st * 2 * kQChunk + c * kQChunk, &tmQ, b_qfull + 8 * st, h * kD + 64 * c, s0 + i0);
        tma_load_2d(sbase + OFF_DO + st * 2 * kQChunk + c * kQChunk, &tmdO, b_qfull + 8 * st, h * kD + 64 * c,
                    s0 + i0);
      }
      return true;
    };
    const int krows = min(kK, len - j0);
    bool ok = true;
    if (lane == 0) {
      mbar_expect_tx(b_kv, 4 * kKChunk);
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        tma_load_2d(sbase + OFF_K + c * kKChunk, &tmK, b_kv, hk * kD + 64 * c, s0 + j0);
        tma_load_2d(sbase + OFF_V + c * kKChunk, &tmV, b_kv, hk * kD + 64 * c, s0 + j0);
      }
    }
    if (mbar_wait_call(b_kv, 0, &no_abort, p.st, 58)) {
      if (krows < kK)
        for (int c = 0; c < 4; ++c) zero_rows(OFF_K + c * kKChunk, kK, krows);   // K chunks then V chunks
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_kvready);
    } else {
      ok = false;
    }
    // block it+1 is loaded once block it is handed over (the MMA thread frees
    // the stage block it+1 reuses only after it has taken block it)
    if (lane == 0 && ok && n_iter > 0) ok = issue(0);
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    for (int it = 0; ok && it < n_iter; ++it) {
      const int st = it & 1, use = it >> 1;
      if (!mbar_wait_call(b_qfull + 8 * st, use & 1, &no_abort, p.st, 59)) break;
      const int i0 = (nqb - 1 - it / p.hc) * kQ;
      const int qrows = min(kQ, len - i0);
      if (qrows < kQ)
        for (int c = 0; c < 2; ++c) {
          zero_rows(OFF_Q + st * 2 * kQChunk + c * kQChunk, kQ, qrows);
          zero_rows(OFF_DO + st * 2 * kQChunk + c * kQChunk, kQ, qrows);
        }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_qready + 8 * st);
      int nxt = 1;
      if (lane == 0 && it + 1 < n_iter) nxt = issue(it + 1) ? 1 : 0;
      if (!__shfl_sync(0xffffffffu, nxt, 0)) break;
    }
  } else if (warp == 1) {
    {
      // ---------------- MMA issuer: the converged warp waits, one elected lane issues ----------------
      const bool leader = elect_one();
      auto wait = [&](uint32_t bar, uint32_t parity, unsigned site) {
        return __all_sync(0xffffffffu, mbar_wait_call(bar, parity, abort_flag, p.st, site)) != 0;
      };
      constexpr uint32_t id_s = idesc_bf16(128, 64, false, false);
      constexpr uint32_t id_kv = idesc_bf16(128, 128, false, true);
      constexpr uint32_t id_q = idesc_bf16(128, 64, true, true);
      // descriptors built once; a k-step moves the start address by a constant
      const uint64_t d_k = sdesc(sbase + OFF_K, 16, 1024), d_v = sdesc(sbase + OFF_V, 16, 1024);
      const uint64_t d_q = sdesc(sbase + OFF_Q, 16, 1024), d_do = sdesc(sbase + OFF_DO, 16, 1024);
      const uint64_t d_qmn = sdesc(sbase + OFF_Q, kQChunk, 1024), d_domn = sdesc(sbase + OFF_DO, kQChunk, 1024);
      const uint64_t d_kmn = sdesc(sbase + OFF_K, kKChunk, 1024);   // K^T: MN-major A, head-dim chunks
      const uint64_t d_dsmn = sdesc(sbase + OFF_DS, kKChunk, 1024); // dS^T: MN-major B (buffer 0)
      constexpr uint64_t kQStep = 2 * kQChunk / 16, kKCh = kKChunk / 16, kQCh = kQChunk / 16;
      auto sdp = [&](int it) {   // S^T, dP^T: M 128 keys, N 64 queries
        const int st = it & 1;
        if (!leader) return;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {   // k = head dims: chunk kk / 4, 32 bytes a step inside it
          const uint64_t ko = (kk >> 2) * kKCh + 2 * (kk & 3), qo = st * kQStep + (kk >> 2) * kQCh + 2 * (kk & 3);
          mma_bf16(tbase + TM_S, d_k + ko, d_q + qo, id_s, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint64_t ko = (kk >> 2) * kKCh + 2 * (kk & 3), qo = st * kQStep + (kk >> 2) * kQCh + 2 * (kk & 3);
          mma_bf16(tbase + TM_DP, d_v + ko, d_do + qo, id_s, kk > 0);
        }
        mma_commit(b_sfull);
      };
      bool ok = wait(b_kvready, 0, 51);
      if (ok && n_iter > 0) {
        ok = wait(b_qready, 0, 52);
        if (ok) {
          fence_after();
          sdp(0);
        }
      }
      for (int it = 0; ok && it < n_iter; ++it) {
        const int st = it & 1, buf = it & 1;
        if (!wait(b_pfull, it & 1, 53)) break;
        fence_after();
        // P^T / dS^T of queries 16 kk .. 16 kk + 15: 8 packed columns, the
        // first 16 of each 32-query group's 32
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kQ / 16; ++kk)     // k = queries, 16 rows (2 KB) a step
            mma_bf16_ts(tbase + TM_DV, tbase + TM_S + 32 * (kk >> 1) + 8 * (kk & 1),
                        d_domn + st * kQStep + 128 * kk, id_kv, (it > 0) || (kk > 0));
#pragma unroll
          for (int kk = 0; kk < kQ / 16; ++kk)
            mma_bf16_ts(tbase + TM_DK, tbase + TM_DP + 32 * (kk >> 1) + 8 * (kk & 1),
                        d_qmn + st * kQStep + 128 * kk, id_kv, (it > 0) || (kk > 0));
          mma_commit(b_qempty + 8 * st);          // Q, dO of this block are read for the last time
        }
        // S, dP of the next block overwrite P, dS of this one, which the MMAs
        // above (issued first, run first) have read
        if (it + 1 < n_iter) {
          if (!wait(b_qready + 8 * ((it + 1) & 1), ((it + 1) >> 1) & 1, 52)) break;
          fence_after();
          sdp(it + 1);
        }
        if (it > 0 && !wait(b_dqempty, (it - 1) & 1, 54)) break;
        fence_after();
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kK / 16; ++kk)     // k = keys, 16 rows (2 KB) a step
            mma_bf16(tbase + TM_DQ, d_kmn + 128 * kk, d_dsmn + buf * kKCh + 128 * kk, id_q, kk > 0);
          mma_commit(b_dqfull);
          mma_commit(b_dsempty + 8 * buf);        // dS^T buffer buf is read for the last time
        }
      }
    }
  } else if (warp < 2 + kSoftWarps) {
    // ---------------- softmax warps: one key row, 32 queries per thread ----------------
    const int g = (warp - 2) >> 2;              // which 32 queries of the block
    const int tg = threadIdx.x - 64 - 128 * g;  // 0..127 within the group
    const int q = warp & 3;
    const int kr = q * 32 + lane;
    const int key = j0 + kr;
    const bool kvalid = key < len;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    // lse (tg 0-31) and D (tg 32-63) of this group's queries of the block
    // after the current one are fetched one iteration early
    auto fetch = [&](int it) -> float {
      if (tg >= 64) return 0.f;
      const int h = hk * p.G + hci * p.hc + it % p.hc;
      const int i0 = (nqb - 1 - it / p.hc) * kQ;
      const int qq = 32 * g + (tg & 31);
      if (qq >= min(kQ, len - i0)) return 0.f;
      const float* src = tg < 32 ? p.lse2 : p.Dvec;
      return src[(long long)h * p.M + s0 + i0 + qq];
    };
    float nxt = n_iter > 0 ? fetch(0) : 0.f;
    for (int it = 0; it < n_iter; ++it) {
      const int i0 = (nqb - 1 - it / p.hc) * kQ;
      const int qrows = min(kQ, len - i0);
      const int buf = it & 1;
      if (tg < 64) (tg < 32 ? sL : sD)[buf * 64 + 32 * g + (tg & 31)] = nxt;
      if (it + 1 < n_iter) nxt = fetch(it + 1);
      named_bar(1, 32 * kSoftWarps);
      if (!mbar_wait_call(b_sfull, it & 1, &no_abort, p.st, 55)) break;
      // dS^T buffer (it & 1) is free once dQ^T of block it-2 has read it
      if (it >= 2 && !mbar_wait_call(b_dsempty + 8 * (it & 1), ((it >> 1) - 1) & 1, &no_abort, p.st, 56)) break;
      fence_after();
      const float* L = sL + buf * 64;
      const float* Dd = sD + buf * 64;
      // all 32 queries past the whole key block (and inside the sequence) need no mask
      const bool interior = (!p.causal || i0 >= j0 + kK) && qrows >= 32 * (g + 1) && len - j0 >= kK;
      uint32_t sr[32], dr[32];
      tmem_ld32_async(tbase + lane_off + TM_S + 32 * g, sr);
      tmem_ld32_async(tbase + lane_off + TM_DP + 32 * g, dr);
      tmem_wait_ld();
      uint32_t pk[16], dk[16];
      if (interior) {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const int qi = 32 * g + 2 * e;
          const float p0 = exp2_approx(__uint_as_float(sr[2 * e]) * p.scale_log2 - L[qi]);
          const float p1 = exp2_approx(__uint_as_float(sr[2 * e + 1]) * p.scale_log2 - L[qi + 1]);
          pk[e] = pack_bf16x2(p0, p1);
          dk[e] = pack_bf16x2(p0 * (__uint_as_float(dr[2 * e]) - Dd[qi]),
                              p1 * (__uint_as_float(dr[2 * e + 1]) - Dd[qi + 1]));
        }
      } else {
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          float pv[2], dv[2];
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int qi = 32 * g + 2 * e + k;
            const bool valid = kvalid && qi < qrows && (!p.causal || key <= i0 + qi);
            pv[k] = valid ? exp2_approx(__uint_as_float(sr[2 * e + k]) * p.scale_log2 - L[qi]) : 0.f;
            dv[k] = valid ? pv[k] * (__uint_as_float(dr[2 * e + k]) - Dd[qi]) : 0.f;
          }
          pk[e] = pack_bf16x2(pv[0], pv[1]);
          dk[e] = pack_bf16x2(dv[0], dv[1]);
        }
      }
      // P^T, dS^T into TMEM over this group's S^T / dP^T columns (read above;
      // the other group's 32 columns are not touched)
      tmem_st16(tbase + lane_off + TM_S + 32 * g, pk);
      tmem_st16(tbase + lane_off + TM_DP + 32 * g, dk);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint32_t phys = (((4 * g + u) ^ (kr & 7)) * 16);
        *reinterpret_cast<uint4*>(sm + OFF_DS + (it & 1) * kKChunk + kr * 128 + phys) =
            make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
      }
      tmem_wait_st();
      fence_before();
      fence_async_smem();
      mbar_arrive(b_pfull);
    }
  } else if (warp < 2 + kSoftWarps + 4) {
    // ---------------- dQ / dK / dV epilogue ----------------
    const int t = threadIdx.x - 32 * (2 + kSoftWarps);
    const int q = warp & 3;
    const int r = q * 32 + lane;                // TMEM lane: head dim (dQ^T) or key (dK, dV)
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t stage = sbase + OFF_ST;
    bool ok = true;
    for (int it = 0; it < n_iter; ++it) {
      if (!mbar_wait_call(b_dqfull, it & 1, &no_abort, p.st, 57)) { ok = false; break; }
      fence_after();
      float v[64];                               // dQ[query c][head dim r], c = 0..63
      tmem_ld32(tbase + lane_off + TM_DQ, v);
      tmem_ld32(tbase + lane_off + TM_DQ + 32, v + 32);
      fence_before();
      mbar_arrive(b_dqempty);
      // the boxes are free once the reducer of the previous block saw its adds read them
      if (it > 0 && !mbar_wait_call(b_boxfree + 8 * ((it - 1) & 1), ((it - 1) >> 1) & 1, &no_abort, p.st, 61)) {
        ok = false;
        break;
      }
      // staging: four 32-column boxes of [64 query rows x 128 bytes]; head dim r
      // sits in box q, column lane
#pragma unroll
      for (int c = 0; c < kQ; ++c) {
        const uint32_t off = q * 8192 + c * 128 + ((((lane >> 2) ^ (c & 7)) * 16)) + (lane & 3) * 4;
        *reinterpret_cast<float*>(sm + OFF_ST + off) = v[c];
      }
      fence_async_smem();
      named_bar(2, 128);
      if (t == 0) mbar_arrive(b_staged + 8 * (it & 1));
    }
    // the staging boxes take dK, dV once the last dQ adds have read them
    if (ok && n_iter > 0 &&
        !mbar_wait_call(b_boxfree + 8 * ((n_iter - 1) & 1), ((n_iter - 1) >> 1) & 1, &no_abort, p.st, 62))
      ok = false;
    if (ok) {
      // every MMA has completed (the last dQ commit covers them all): drain
      // dK, dV 64 columns at a time through two [128 x 32] f32 boxes
#pragma unroll 1
      for (int pass = 0; pass < 4; ++pass) {
        const uint32_t col = (pass < 2 ? TM_DK : TM_DV) + 64 * (pass & 1);
        float v[64];
        tmem_ld32(tbase + lane_off + col, v);
        tmem_ld32(tbase + lane_off + col + 32, v + 32);
        if (t == 0) bulk_wait_read_all();
        named_bar(2, 128);
#pragma unroll
        for (int bx = 0; bx < 2; ++bx)
#pragma unroll
          for (int g8 = 0; g8 < 8; ++g8) {
            const uint32_t phys = ((g8 ^ (r & 7)) * 16);
            *reinterpret_cast<float4*>(sm + OFF_ST + bx * kKChunk + r * 128 + phys) =
                make_float4(v[bx * 32 + 4 * g8], v[bx * 32 + 4 * g8 + 1], v[bx * 32 + 4 * g8 + 2],
                            v[bx * 32 + 4 * g8 + 3]);
          }
        fence_async_smem();
        named_bar(2, 128);
        if (t == 0) {
          const CUtensorMap* m = pass < 2 ? &tmdK : &tmdV;
#pragma unroll
          for (int bx = 0; bx < 2; ++bx)
            tma_reduce_add_2d(m, stage + bx * kKChunk, hk * kD + 64 * (pass & 1) + 32 * bx, s0 + j0);
          bulk_commit();
        }
      }
    }
    if (t == 0) bulk_wait_all();
  } else if (lane == 0) {
    // ---------------- dQ reducers: warp 14 even blocks, warp 15 odd ----------------
    // Each adds its blocks' dQ^T tiles in key-block order (the tile's turn),
    // hands the staging boxes back once the adds have read them, and passes
    // the turn on as soon as its adds have completed.
    const int rr = warp - (2 + kSoftWarps + 4);
    const uint32_t stage = sbase + OFF_ST;
    bool broken = false;
    for (int it = rr; it < n_iter; it += 2) {
      const int h = hk * p.G + hci * p.hc + it % p.hc;
      const int i0 = (nqb - 1 - it / p.hc) * kQ;
      if (!mbar_wait_call(b_staged + 8 * (it & 1), (it >> 1) & 1, abort_flag, p.st, 63)) break;
      int* turn = dq_turn_wait(p, b, h, i0 / kQ, j, broken, 60);
#pragma unroll
      for (int bx = 0; bx < 4; ++bx) tma_reduce_add_2d(&tmdQ, stage + bx * 8192, h * kD + 32 * bx, s0 + i0);
      bulk_commit();
      bulk_wait_read_all();
      mbar_arrive(b_boxfree + 8 * (it & 1));
      dq_turn_flush(turn, j);
    }
    bulk_wait_all();
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ---------------------------------------------------------------------------
// tcgen05 D pre-pass, head dim 64 or 128.  One CTA per (sequence, 128 queries,
// HPC query heads of one kv head): O'_h = sum over kept causal keys of P_h V,
// D_h = rowsum(dO_h * O'_h).  With HPC > 1 the heads share each K/V block: it
// is loaded once, and the HPC (head, key block) iterations run back to back
// through the double-buffered S and P.  Tiles are 64-column (128-byte)
// swizzle chunks.
//   warp 0     TMA: the HPC Q tiles once; K_j, V_j per key block
//   warp 1     TMEM owner; one lane issues S = Q_h K_j^T (into one of two TMEM
//              buffers, so the next S overlaps the softmax of this one) and
//              O'_h += P V_j
//   warps 2-9  one query row and 64 of the 128 keys per thread: P from TMEM
//              -> bf16 -> back into TMEM, over the first 32 of the 64 S
//              columns the thread has read (so O'_h += P V_j reads A from
//              TMEM); at the end D_h from O'_h (TMEM) and dO_h (global), each
//              half of the row's columns summed separately
// TMEM columns: S buffers 0-127 and 128-255 (P of keys 0-63 in 0-31 and of
// keys 64-127 in 64-95 of its buffer), O'_h from 256 + h * head dim.
//
// The same pipeline also serves the dense attention forward over whole
// sequences (every token kept), as two passes (MODE):
//   2  log-sum-exp: S = Q_h K_j^T only (no V); each thread keeps a running
//      max and sum of exp2 over its 64 keys, the two halves of a row are
//      merged at the end -> lse (log2 units for pass 1, natural log [B,H,T])
//   1  output: exactly the D pre-pass's O'_h with the lse of pass 2, so
//      O'_h = softmax(Q_h K^T scale) V; written as bf16 instead of D.
// MODE 0 is the D pre-pass of the backward.
template <int DH, int HPC, int MODE = 0>
struct DprepCfg {
  static constexpr int kQ = 128, kK = 128, kD = DH, kCh = DH / 64;   // 64-column chunks
  static constexpr uint32_t kTile = 16384;                           // 128 rows x 64 columns
  static constexpr int kKV = DH == 64 && HPC == 1 ? 3 : 2;           // K/V stages
  static constexpr uint32_t kKVBytes = 2 * kCh * kTile;              // K and V of one stage
  static constexpr int kSoftWarps = 16;                              // four per TMEM lane quadrant
  // OFF_P: the lse pass's per-key-group maxima and sums, [2][HPC][4][128] f32
  static constexpr uint32_t OFF_Q = 0, OFF_K = HPC * kCh * kTile, OFF_P = OFF_K + kKV * kKVBytes,
                            OFF_BAR = OFF_P + HPC * (kSoftWarps / 4) * 1024;
  static constexpr uint32_t OFF_PART = OFF_BAR + 256;                // [HPC][4][128] f32 partial dot products
  static constexpr size_t kSmem = 1024 + OFF_PART + HPC * (kSoftWarps / 4) * 512;
  static constexpr uint32_t TM_S = 0, TM_O = 256;
  static constexpr int kThreads = 32 * (2 + kSoftWarps);
  static_assert(kSmem <= 232448, "shared memory");
  static_assert(TM_O + HPC * DH <= 512, "TMEM columns");
};

struct DprepTc {
  int B, T, H, G, causal, nqb;
  float scale_log2;
  const int32_t* cu_kept;
  const float* lse2;
  float* Dvec;
  const __nv_bfloat16* dO;   // COMPACT rows, head h at columns h * DH
  long long do_ld;
  long long M;
  DevStatus* st;
  // forward passes (every token kept: row s0 + i is position i)
  __nv_bfloat16* O;          // MODE 1: attention output rows, head h at columns h * DH
  long long o_ld;
  float* lse2_out;           // MODE 2: [H, M] log2 units
  float* lse_out;            // MODE 2: [B, H, T] natural log
};

template <int DH, int HPC, int MODE>
__device__ __forceinline__ void dprep_body(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                                           const DprepTc& p) {
  using namespace tc;
  using Cfg = DprepCfg<DH, HPC, MODE>;
  constexpr int kQ = Cfg::kQ, kK = Cfg::kK, kD = Cfg::kD, kCh = Cfg::kCh, kKV = Cfg::kKV, kSoftWarps = Cfg::kSoftWarps;
  constexpr uint32_t kTile = Cfg::kTile, kKVBytes = Cfg::kKVBytes, OFF_Q = Cfg::OFF_Q, OFF_K = Cfg::OFF_K,
                     OFF_P = Cfg::OFF_P, OFF_BAR = Cfg::OFF_BAR, OFF_PART = Cfg::OFF_PART, TM_S = Cfg::TM_S,
                     TM_O = Cfg::TM_O;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  grid_dep_wait();   // the kept offsets, Q, K, V and dO come from the kernels ahead
  // items: query block descending (most key blocks first), then sequence, head group
  const int ngroups = p.H / HPC;
  const int per_i = p.B * ngroups;
  const int ib = p.nqb - 1 - (int)(blockIdx.x / per_i);
  const int b = (blockIdx.x % per_i) / ngroups;
  const int h0 = (blockIdx.x % ngroups) * HPC;   // the HPC heads share kv head h0 / G
  const int s0 = p.cu_kept[b], len = p.cu_kept[b + 1] - s0;
  const int i0 = ib * kQ;
  if (i0 >= len) return;
  const int hk = h0 / p.G;
  const int nj = p.causal ? ib + 1 : (len + kK - 1) / kK;
  const int n_it = nj * HPC;                     // iteration it: key block it / HPC, head it % HPC
  const int qrows = min(kQ, len - i0);

  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + OFF_BAR);
  // kv_full/kv_empty/kv_ready: one per K/V stage; s_full/p_full/p_empty: one
  // per S / P buffer.  Every barrier's next phase needs the waiter to have
  // seen the previous one (p_full of iteration t+2 needs p_empty of t, which
  // the MMA commits only after its wait on p_full of t), so no parity wait can
  // miss a phase.  A single p_full for both buffers would not have that: the
  // softmax could finish iterations t and t+1 before the MMA looks at t.
  const uint32_t b_q = smem_u32(bars + 0), b_kvfull = smem_u32(bars + 1), b_kvempty = smem_u32(bars + 4),
                 b_kvready = smem_u32(bars + 7), b_sfull = smem_u32(bars + 10), b_pempty = smem_u32(bars + 12),
                 b_pfull = smem_u32(bars + 14), b_ofull = smem_u32(bars + 16);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    mbar_init(b_q, 1);
    for (int s = 0; s < kKV; ++s) {
      mbar_init(b_kvfull + 8 * s, 1);
      mbar_init(b_kvempty + 8 * s, 1);
      mbar_init(b_kvready + 8 * s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(b_sfull + 8 * s, 1);
      mbar_init(b_pempty + 8 * s, 1);
      mbar_init(b_pfull + 8 * s, 32 * kSoftWarps);
    }
    mbar_init(b_ofull, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_u32(tmem_slot), 512);
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tbase = *tmem_slot;
  const uint32_t sbase = smem_u32(sm);
  volatile int no_abort = 0;

  if (warp == 0) {
    // TMA producer (lane 0); the whole warp zeroes K / V rows past the
    // sequence before the MMAs read a block (0 * non-finite would leak)
    auto issue = [&](int j) -> bool {
      const int st = j % kKV, use = j / kKV;
      if (!mbar_wait(b_kvempty + 8 * st, (use & 1) ^ 1, abort_flag, p.st, 40)) return false;
      mbar_expect_tx(b_kvfull + 8 * st, MODE == 2 ? kCh * kTile : kKVBytes);   // the lse pass reads no V
      const uint32_t kb = sbase + OFF_K + st * kKVBytes;
#pragma unroll
      for (int c = 0; c < kCh; ++c) {
        tma_load_2d(kb + c * kTile, &tmK, b_kvfull + 8 * st, hk * kD + 64 * c, s0 + j * kK);
        if (MODE != 2)
          tma_load_2d(kb + (kCh + c) * kTile, &tmV, b_kvfull + 8 * st, hk * kD + 64 * c, s0 + j * kK);
      }
      return true;
    };
    int ok = 1;
    if (lane == 0) {
      mbar_expect_tx(b_q, HPC * kCh * kTile);
#pragma unroll
      for (int hh = 0; hh < HPC; ++hh)
#pragma unroll
        for (int c = 0; c < kCh; ++c)
          tma_load_2d(sbase + OFF_Q + (hh * kCh + c) * kTile, &tmQ, b_q, (h0 + hh) * kD + 64 * c, s0 + i0);
      ok = issue(0) ? 1 : 0;
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    // With three stages block j+1 can be requested before block j is
    // released: the request waits for the last P V of block j-2, which the
    // MMA issues once block j-1 is released.  With two stages the request
    // waits for the last P V of block j-1, which the MMA issues only after it
    // has taken block j, so block j is released first.
    for (int j = 0; ok && j < nj; ++j) {
      const int st = j % kKV, use = j / kKV;
      int nxt = 1;
      if (kKV >= 3) {
        if (lane == 0 && j + 1 < nj) nxt = issue(j + 1) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, nxt, 0)) break;
      }
      if (!mbar_wait(b_kvfull + 8 * st, use & 1, &no_abort, p.st, 47)) break;
      const int krows = min(kK, len - j * kK);
      if (krows < kK) {
        const uint32_t base = OFF_K + st * kKVBytes;
        for (int i = lane; i < (kK - krows) * 8; i += 32) {
          const uint32_t off = (krows + i / 8) * 128 + (i % 8) * 16;
#pragma unroll
          for (int c = 0; c < 2 * kCh; ++c) *reinterpret_cast<uint4*>(sm + base + c * kTile + off) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(b_kvready + 8 * st);
      if (kKV < 3) {
        if (lane == 0 && j + 1 < nj) nxt = issue(j + 1) ? 1 : 0;
        if (!__shfl_sync(0xffffffffu, nxt, 0)) break;
      }
    }
  } else if (warp == 1) {
    {
      // the converged warp waits, one elected lane issues
      const bool leader = elect_one();
      auto wait = [&](uint32_t bar, uint32_t parity, unsigned site) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.st, site)) != 0;
      };
      constexpr uint32_t id_s = idesc_bf16(128, 128, false, false);
      constexpr uint32_t id_o = idesc_bf16(128, kD, false, true);
      bool ok = wait(b_q, 0, 41);
      // O'_h += P V_j for the iteration whose P the softmax has finished; the
      // last head of a key block releases its K/V stage
      auto pv = [&](int t) -> bool {
        const int jj = t / HPC, hh = t % HPC;
        const int kst = jj % kKV, pb = t & 1;
        if (!wait(b_pfull + 8 * pb, (t >> 1) & 1, 42)) return false;
        fence_after();
        const uint32_t sv = sbase + OFF_K + kst * kKVBytes + kCh * kTile;
        if (MODE != 2 && leader) {   // the lse pass only releases the buffers
#pragma unroll
          for (int kk = 0; kk < kK / 16; ++kk) {   // V as the MN-major B: head-dim chunks kTile apart
            // P of keys 16 kk .. 16 kk + 15: 8 columns, in the 32-key chunk kk / 2 of the S buffer
            const uint32_t pa = tbase + TM_S + pb * 128 + 32 * (kk >> 1) + 8 * (kk & 1);
            mma_bf16_ts(tbase + TM_O + hh * kD, pa, sdesc(sv + kk * 2048, kTile, 1024), id_o, (jj > 0) || (kk > 0));
          }
        }
        if (leader) {
          if (hh == HPC - 1) mma_commit(b_kvempty + 8 * kst);
          mma_commit(b_pempty + 8 * pb);
        }
        __syncwarp();
        return true;
      };
      for (int it = 0; ok && it < n_it; ++it) {
        const int j = it / HPC, hh = it % HPC;
        const int kst = j % kKV, kuse = j / kKV, sb = it & 1;
        if (hh == 0) {
          if (!wait(b_kvready + 8 * kst, kuse & 1, 43)) { ok = false; break; }
          fence_after();
        }
        const uint32_t sk = sbase + OFF_K + kst * kKVBytes, sq = sbase + OFF_Q + hh * kCh * kTile;
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kTile + (kk & 3) * 32;
            mma_bf16(tbase + TM_S + sb * 128, sdesc(sq + off, 16, 1024), sdesc(sk + off, 16, 1024), id_s, kk > 0);
          }
          mma_commit(b_sfull + 8 * sb);
        }
        __syncwarp();
        if (it > 0 && !pv(it - 1)) { ok = false; break; }
      }
      if (ok && n_it > 0 && pv(n_it - 1) && leader) mma_commit(b_ofull);
    }
  } else {
    // softmax: one query row, kKT of the 128 keys of a block per thread
    // (four warps per TMEM lane quadrant, sub-group `sub` of the row's keys)
    constexpr int kSubs = kSoftWarps / 4, kKT = kK / kSubs, kDT = kD / kSubs;
    const int q = warp & 3;
    const int sub = (warp - 2) >> 2;
    const int r = q * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
    float Lh[HPC];
#pragma unroll
    for (int hh = 0; hh < HPC; ++hh)
      Lh[hh] = (MODE != 2 && r < qrows) ? p.lse2[(long long)(h0 + hh) * p.M + s0 + i0 + r] : 0.f;
    // lse pass: running max and sum of exp2 (log2 units) per head
    float mrun[HPC], lrun[HPC];
#pragma unroll
    for (int hh = 0; hh < HPC; ++hh) {
      mrun[hh] = -INFINITY;
      lrun[hh] = 0.f;
    }
    // with one head, this thread's kDT head-dim columns of its dO row are
    // loaded now so the latency hides behind the key loop; with several
    // heads at the end
    constexpr int kDoVec = HPC == 1 ? kDT / 8 : 1;
    uint4 dov[kDoVec];
    if (HPC == 1 && MODE == 0) {
#pragma unroll
      for (int u = 0; u < kDoVec; ++u) {
        dov[u] = make_uint4(0, 0, 0, 0);
        if (r < qrows)
          dov[u] = *reinterpret_cast<const uint4*>(p.dO + (long long)(s0 + i0 + r) * p.do_ld + h0 * kD +
                                                   sub * kDT + 8 * u);
      }
    }
    bool ok = true;
    for (int it = 0; it < n_it; ++it) {
      const int st = it & 1, use = it >> 1;
      const int j = it / HPC, hh = it % HPC;
      if (!mbar_wait(b_sfull + 8 * st, use & 1, &no_abort, p.st, 44)) { ok = false; break; }
      if (it >= 2 && !mbar_wait(b_pempty + 8 * st, (use - 1) & 1, &no_abort, p.st, 45)) { ok = false; break; }
      fence_after();
      const int j0 = j * kK;
      float L = Lh[0];
#pragma unroll
      for (int x = 1; x < HPC; ++x)
        if (hh == x) L = Lh[x];
      uint32_t sr[kKT];
#pragma unroll
      for (int c = 0; c < kKT / 32; ++c)
        tmem_ld32_async(tbase + lane_off + TM_S + st * 128 + sub * kKT + 32 * c, sr + 32 * c);
      tmem_wait_ld();
      // a full key block strictly before the query block needs no masking
      const bool interior = (!p.causal || j0 + kK <= i0) && qrows == kQ && len - j0 >= kK;
      if (MODE == 2) {
        // keys j0 + sub * kKT + e of this row, e < kKT.  The block maximum is
        // taken on the raw scores (scaling by c > 0 is monotone, so max(S) c
        // = max(S c) exactly) and each exponent is one fma; eight independent
        // partial maxima and sums keep the dependency chains short.
        float sv[kKT], bm8[8], a8[8];
#pragma unroll
        for (int q8 = 0; q8 < 8; ++q8) {
          bm8[q8] = -INFINITY;
          a8[q8] = 0.f;
        }
        if (interior) {
#pragma unroll
          for (int e = 0; e < kKT; ++e) {
            sv[e] = __uint_as_float(sr[e]);
            bm8[e & 7] = fmaxf(bm8[e & 7], sv[e]);
          }
        } else {
#pragma unroll
          for (int e = 0; e < kKT; ++e) {
            const int kj = j0 + sub * kKT + e;
            const bool valid = r < qrows && kj < len && (!p.causal || kj <= i0 + r);
            sv[e] = valid ? __uint_as_float(sr[e]) : -INFINITY;
            bm8[e & 7] = fmaxf(bm8[e & 7], sv[e]);
          }
        }
        const float bm = fmaxf(fmaxf(fmaxf(bm8[0], bm8[1]), fmaxf(bm8[2], bm8[3])),
                               fmaxf(fmaxf(bm8[4], bm8[5]), fmaxf(bm8[6], bm8[7]))) * p.scale_log2;
        float m = mrun[0], l = lrun[0];
#pragma unroll
        for (int x = 1; x < HPC; ++x)
          if (hh == x) { m = mrun[x]; l = lrun[x]; }
        const float mn = fmaxf(m, bm);
        if (mn != -INFINITY) {
#pragma unroll
          for (int e = 0; e < kKT; ++e) a8[e & 7] += exp2_approx(fmaf(sv[e], p.scale_log2, -mn));
          const float acc = ((a8[0] + a8[1]) + (a8[2] + a8[3])) + ((a8[4] + a8[5]) + (a8[6] + a8[7]));
          l = l * exp2_approx(m - mn) + acc;
          m = mn;
        }
#pragma unroll
        for (int x = 0; x < HPC; ++x)
          if (hh == x) { mrun[x] = m; lrun[x] = l; }
      }
#pragma unroll
      for (int cc = 0; cc < (MODE == 2 ? 0 : kKT / 32); ++cc) {
        const int c32 = sub * (kKT / 32) + cc;   // 32-key chunk of the block
        float sv[32];
        if (interior) {
#pragma unroll
          for (int e = 0; e < 32; ++e) sv[e] = exp2_approx(__uint_as_float(sr[cc * 32 + e]) * p.scale_log2 - L);
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const int kj = j0 + c32 * 32 + e;
            const bool valid = r < qrows && kj < len && (!p.causal || kj <= i0 + r);
            sv[e] = valid ? exp2_approx(__uint_as_float(sr[cc * 32 + e]) * p.scale_log2 - L) : 0.f;
          }
        }
        // these 32 keys' P, packed in pairs: the first 16 of the chunk's 32
        // columns (this thread has read all of them already)
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(sv[2 * e], sv[2 * e + 1]);
        tmem_st16(tbase + lane_off + TM_S + st * 128 + 32 * c32, pk);
      }
      tmem_wait_st();
      fence_before();
      mbar_arrive(b_pfull + 8 * st);
    }
    float* part = reinterpret_cast<float*>(sm + OFF_PART);   // [HPC][kSubs][128]
    // this thread's kDT head-dim columns of head hh's O' (or O), 16 at a time
    auto load_o16 = [&](int hh, int c16, float* o) {
      uint32_t u[16];
      tmem_ld16_async(tbase + lane_off + TM_O + hh * kD + sub * kDT + 16 * c16, u);
      tmem_wait_ld();
#pragma unroll
      for (int e = 0; e < 16; ++e) o[e] = __uint_as_float(u[e]);
    };
    if (MODE == 1) {
      // the attention output: this thread's columns of the row
      if (ok && mbar_wait(b_ofull, 0, &no_abort, p.st, 48)) {
        fence_after();
#pragma unroll
        for (int hh = 0; hh < HPC; ++hh) {
#pragma unroll
          for (int c16 = 0; c16 < kDT / 16; ++c16) {
            float o[16];
            load_o16(hh, c16, o);
            if (r < qrows) {
              __nv_bfloat16* dst = p.O + (long long)(s0 + i0 + r) * p.o_ld + (h0 + hh) * kD + sub * kDT + 16 * c16;
#pragma unroll
              for (int g = 0; g < 2; ++g) *reinterpret_cast<uint4*>(dst + 8 * g) = pack8(o + 8 * g);
            }
          }
        }
      }
    } else if (MODE == 2) {
      // merge the row's key groups: lse2 = max + log2(sum exp2(x - max)),
      // the groups taken in a fixed order
      if (!(ok && mbar_wait(b_ofull, 0, &no_abort, p.st, 49))) ok = false;
      float* pm = reinterpret_cast<float*>(sm + OFF_P);   // no P tile is written in this pass
      float* pl = pm + HPC * kSubs * 128;
#pragma unroll
      for (int hh = 0; hh < HPC; ++hh) {
        pm[(hh * kSubs + sub) * 128 + r] = mrun[hh];
        pl[(hh * kSubs + sub) * 128 + r] = lrun[hh];
      }
      named_bar(1, 32 * kSoftWarps);
      if (ok && sub == 0 && r < qrows) {
#pragma unroll
        for (int hh = 0; hh < HPC; ++hh) {
          float mm = -INFINITY;
#pragma unroll
          for (int x = 0; x < kSubs; ++x) mm = fmaxf(mm, pm[(hh * kSubs + x) * 128 + r]);
          float lsum = 0.f;
#pragma unroll
          for (int x = 0; x < kSubs; ++x)
            lsum += pl[(hh * kSubs + x) * 128 + r] * exp2f(pm[(hh * kSubs + x) * 128 + r] - mm);
          const float lse2 = mm + log2f(lsum);
          p.lse2_out[(long long)(h0 + hh) * p.M + s0 + i0 + r] = lse2;
          p.lse_out[((long long)b * p.H + h0 + hh) * p.T + i0 + r] = lse2 * kLn2;
        }
      }
    }
    float d[HPC];
#pragma unroll
    for (int hh = 0; hh < HPC; ++hh) d[hh] = 0.f;
    if (MODE != 0) {
      // the forward passes are done
    } else if (ok && mbar_wait(b_ofull, 0, &no_abort, p.st, 46)) {
      fence_after();
#pragma unroll
      for (int hh = 0; hh < HPC; ++hh) {
#pragma unroll
        for (int c16 = 0; c16 < kDT / 16; ++c16) {
          float o[16];
          load_o16(hh, c16, o);
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            float x[8];
            if (HPC == 1) {
              unpack8(dov[(2 * c16 + g) % kDoVec], x);
            } else {
              uint4 u = make_uint4(0, 0, 0, 0);
              if (r < qrows)
                u = *reinterpret_cast<const uint4*>(p.dO + (long long)(s0 + i0 + r) * p.do_ld + (h0 + hh) * kD +
                                                    sub * kDT + 16 * c16 + 8 * g);
              unpack8(u, x);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) d[hh] += x[e] * o[8 * g + e];
          }
        }
      }
    } else {
      ok = false;
    }
    if (MODE == 0) {
#pragma unroll
      for (int hh = 0; hh < HPC; ++hh) part[(hh * kSubs + sub) * 128 + r] = d[hh];
      named_bar(1, 32 * kSoftWarps);
      if (ok && sub == 0 && r < qrows)
#pragma unroll
        for (int hh = 0; hh < HPC; ++hh) {
          float dd = d[hh];
#pragma unroll
          for (int x = 1; x < kSubs; ++x) dd += part[(hh * kSubs + x) * 128 + r];
          p.Dvec[(long long)(h0 + hh) * p.M + s0 + i0 + r] = dd;
        }
    }
  }
  fence_before();
  __syncthreads();
  if (warp == 1) {
    fence_after();
    tmem_dealloc(tbase, 512);
  }
}

template <int DH, int HPC>
__global__ void __launch_bounds__(DprepCfg<DH, HPC>::kThreads, 1)
    attn_dprep_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, DprepTc p) {
  dprep_body<DH, HPC, 0>(tmQ, tmK, tmV, p);
}

// dense forward, pass 1: log-sum-exp of every query row
template <int DH, int HPC>
__global__ void __launch_bounds__(DprepCfg<DH, HPC, 2>::kThreads, 1)
    attn_fwd_lse_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, DprepTc p) {
  dprep_body<DH, HPC, 2>(tmQ, tmK, tmV, p);
}

// dense forward, pass 2: O = exp(S - lse) V
template <int DH, int HPC>
__global__ void __launch_bounds__(DprepCfg<DH, HPC, 1>::kThreads, 1)
    attn_fwd_o_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, DprepTc p) {
  dprep_body<DH, HPC, 1>(tmQ, tmK, tmV, p);
}

template <int DH>
cudaError_t run(const Ctx& c, const AttnK& k, float rope_base, const AttnArgs& a) {
  if (!k.kv_acc) return cudaErrorInvalidValue;   // the dK / dV accumulators are required
  static int seen[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !seen[dev]) {
    cudaError_t e = cudaSuccess;
    if (DH == 64)
      e = cudaFuncSetAttribute(attn_main_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(tcattn::kSmem));
    if (e == cudaSuccess && DH == 128)
      e = cudaFuncSetAttribute(attn_main_tc128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(tcattn128::kSmem));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_dprep_tc_kernel<DH, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(DprepCfg<DH, 1>::kSmem));
    if (e == cudaSuccess && DH == 64)
      e = cudaFuncSetAttribute(attn_dprep_tc_kernel<64, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(DprepCfg<64, 4>::kSmem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) seen[dev] = 1;
  }
  if (a.stage != 2) {
    prof_begin(c, "attn_prep");
    attn_prep_kernel<<<c.num_sms * 4, 256, 0, c.stream>>>(k, DH, rope_base, const_cast<float2*>(k.rope));
    prof_end(c);
    count_launch(1);
    if (a.stage == 1) return cudaGetLastError();
  }
  {
    // work items: (key block, sequence, kv head, chunk of hc query heads).
    // The group's heads are split in at most two chunks: a key block's dK
    // and dV then get at most two reduce-adds into a zeroed accumulator, and
    // 0 + a + b = 0 + b + a exactly, so they are the same every run.
    const int nkb = (k.T + tcattn::kK - 1) / tcattn::kK;
    int hc = k.G;
    if (hc % 2 == 0 && (long long)k.B * k.Hkv * nkb < 3LL * c.num_sms) hc /= 2;
    MainTc m{};
    m.B = k.B; m.T = k.T; m.H = k.H; m.Hkv = k.Hkv; m.G = k.G; m.hc = hc; m.nhc = k.G / hc; m.nkb = nkb;
    m.causal = k.causal; m.scale_log2 = k.scale_log2; m.cu_kept = k.cu_kept; m.lse2 = k.lse2; m.Dvec = k.Dvec;
    m.M = k.M; m.st = c.st;
    m.order = k.order; m.nqb_max = (k.T + 63) / 64;
    // Q / dO tiles: 128 query rows for head dim 64, 64 for head dim 128
    constexpr int kQRows = DH == 64 ? tcattn::kQ : tcattn128::kQ;
    CUtensorMap tq, tk, tv, tdo, tdq, tdk, tdv, tq_pre;
    bool ok = make_tensor_map(&tq, k.q, false, (long long)k.H * DH, a.in_cap, k.q_ld, 64, kQRows) &&
              make_tensor_map(&tq_pre, k.q, false, (long long)k.H * DH, a.in_cap, k.q_ld, 64, 128) &&
              make_tensor_map(&tk, k.k, false, (long long)k.Hkv * DH, a.in_cap, k.kv_ld, 64, 128) &&
              make_tensor_map(&tv, k.v, false, (long long)k.Hkv * DH, a.in_cap, k.kv_ld, 64, 128) &&
              make_tensor_map(&tdo, k.dO, false, (long long)k.H * DH, a.in_cap, k.do_ld, 64, kQRows) &&
              make_tensor_map(&tdq, k.dq_acc, true, (long long)k.H * DH, k.M, (long long)k.H * DH, 32, kQRows) &&
              make_tensor_map(&tdk, k.dk_acc, true, (long long)k.Hkv * DH, k.M, (long long)k.Hkv * DH, 32, 128) &&
              make_tensor_map(&tdv, k.dv_acc, true, (long long)k.Hkv * DH, k.M, (long long)k.Hkv * DH, 32, 128);
    if (!ok) return cudaErrorInvalidValue;
    DprepTc dp{};
    dp.B = k.B; dp.T = k.T; dp.H = k.H; dp.G = k.G; dp.causal = k.causal; dp.nqb = nkb;
    dp.scale_log2 = k.scale_log2; dp.cu_kept = k.cu_kept; dp.lse2 = k.lse2; dp.Dvec = k.Dvec; dp.M = k.M;
    dp.dO = k.dO; dp.do_ld = k.do_ld;
    dp.st = c.st;
    // (programmatic dependent launch: the pre-pass follows the preparation
    // kernel, or whatever the caller's context allows; the main pass and the
    // finalisation follow a kernel of this launcher, so they always may)
    const bool pdl = pdl_allowed();
    cudaError_t e;
    prof_begin(c, "attn_dprep_tc");
    // four query heads of one kv head per CTA share each K/V block (head dim 64, groups of 4+)
    if (DH == 64 && k.G % 4 == 0)
      e = launch_k(c, c.pdl || (a.stage != 2 && pdl), attn_dprep_tc_kernel<64, 4>, dim3(k.B * (k.H / 4) * nkb),
                   dim3(DprepCfg<64, 4>::kThreads), DprepCfg<64, 4>::kSmem, 1, tq_pre, tk, tv, dp);
    else
      e = launch_k(c, c.pdl || (a.stage != 2 && pdl), attn_dprep_tc_kernel<DH, 1>, dim3(k.B * k.H * nkb),
                   dim3(DprepCfg<DH, 1>::kThreads), DprepCfg<DH, 1>::kSmem, 1, tq_pre, tk, tv, dp);
    prof_end(c);
    if (e != cudaSuccess) return launched(e);
    prof_begin(c, "attn_main_tc");
    if (DH == 64)
      e = launch_k(c, pdl, attn_main_tc_kernel, dim3(k.B * k.Hkv * nkb * m.nhc), dim3(tcattn::kThreads),
                   tcattn::kSmem, 1, tq, tk, tv, tdo, tdq, tdk, tdv, m);
    else
      e = launch_k(c, pdl, attn_main_tc128_kernel, dim3(k.B * k.Hkv * nkb * m.nhc), dim3(tcattn128::kThreads),
                   tcattn128::kSmem, 1, tq, tk, tv, tdo, tdq, tdk, tdv, m);
    prof_end(c);
    if (e != cudaSuccess) return launched(e);
    prof_begin(c, "attn_finalize");
    e = launch_k(c, pdl, attn_finalize_kernel, dim3(c.num_sms * 4), dim3(256), 0, 1, k, DH);
    prof_end(c);
    count_launch(3);
    return launched(e);
  }
}

template <int DH>
cudaError_t run_fwd(const Ctx& c, const AttnFwdArgs& a) {
  static int seen[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !seen[dev]) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_lse_kernel<DH, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(DprepCfg<DH, 1, 2>::kSmem));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(attn_fwd_o_kernel<DH, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(DprepCfg<DH, 1, 1>::kSmem));
    if (e == cudaSuccess && DH == 64)
      e = cudaFuncSetAttribute(attn_fwd_lse_kernel<64, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(DprepCfg<64, 4, 2>::kSmem));
    if (e == cudaSuccess && DH == 64)
      e = cudaFuncSetAttribute(attn_fwd_o_kernel<64, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(DprepCfg<64, 4, 1>::kSmem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) seen[dev] = 1;
  }
  const int G = a.H / a.Hkv;
  CUtensorMap tq, tk, tv;
  bool ok = make_tensor_map(&tq, a.q, false, (long long)a.H * DH, a.M, a.q_ld, 64, 128) &&
            make_tensor_map(&tk, a.k, false, (long long)a.Hkv * DH, a.M, a.kv_ld, 64, 128) &&
            make_tensor_map(&tv, a.v, false, (long long)a.Hkv * DH, a.M, a.kv_ld, 64, 128);
  if (!ok) return cudaErrorInvalidValue;
  DprepTc dp{};
  dp.B = a.B; dp.T = a.T; dp.H = a.H; dp.G = G; dp.causal = 1; dp.nqb = (a.T + 127) / 128;
  dp.scale_log2 = a.scale * kLog2e; dp.cu_kept = a.cu; dp.lse2 = a.lse2; dp.M = a.M; dp.st = c.st;
  dp.O = a.o; dp.o_ld = a.o_ld; dp.lse2_out = a.lse2; dp.lse_out = a.lse;
  const bool multi = DH == 64 && G % 4 == 0;   // four query heads of a kv group per CTA
  const int grid = a.B * (multi ? a.H / 4 : a.H) * dp.nqb;
  prof_begin(c, "attn_fwd_lse");
  if (multi)
    attn_fwd_lse_kernel<64, 4><<<grid, DprepCfg<64, 4, 2>::kThreads, DprepCfg<64, 4, 2>::kSmem, c.stream>>>(
        tq, tk, tv, dp);
  else
    attn_fwd_lse_kernel<DH, 1><<<grid, DprepCfg<DH, 1, 2>::kThreads, DprepCfg<DH, 1, 2>::kSmem, c.stream>>>(
        tq, tk, tv, dp);
  prof_end(c);
  prof_begin(c, "attn_fwd_o");
  if (multi)
    attn_fwd_o_kernel<64, 4><<<grid, DprepCfg<64, 4, 1>::kThreads, DprepCfg<64, 4, 1>::kSmem, c.stream>>>(
        tq, tk, tv, dp);
  else
    attn_fwd_o_kernel<DH, 1><<<grid, DprepCfg<DH, 1, 1>::kThreads, DprepCfg<DH, 1, 1>::kSmem, c.stream>>>(
        tq, tk, tv, dp);
  prof_end(c);
  count_launch(2);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rope_table(const Ctx& c, int T, int rot_half, float rope_base, float2* rope) {
  if (rot_half <= 0) return cudaSuccess;
  if (rot_half > 256) return cudaErrorInvalidValue;
  const long long n = (long long)T * rot_half;
  const long long want = (n + 255) / 256, cap = (long long)c.num_sms * 4;
  const int grid = (int)(want < cap ? want : cap);
  rope_table_kernel<<<grid, 256, 0, c.stream>>>(T, rot_half, rope_base, rope);
  count_launch();
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd(const Ctx& c, const AttnFwdArgs& a) {
  if (a.H < 1 || a.Hkv < 1 || a.H % a.Hkv || a.B < 1 || a.T < 1 || !a.cu || !a.lse || !a.lse2 || !a.o)
    return cudaErrorInvalidValue;
  if (a.dh == 64) return run_fwd<64>(c, a);
  if (a.dh == 128) return run_fwd<128>(c, a);
  return cudaErrorInvalidValue;
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
  k.order = a.order;
  k.dk_acc = a.dk_acc; k.dv_acc = a.dv_acc;
  k.kv_acc = ((a.dh == 64 || a.dh == 128) && a.dk_acc && a.dv_acc && a.in_cap > 0) ? 1 : 0;
  if (!a.order) return cudaErrorInvalidValue;
  if (a.dh == 64) return run<64>(c, k, a.rope_base, a);
  if (a.dh == 128) return run<128>(c, k, a.rope_base, a);
  return cudaErrorInvalidValue;
}

}  // namespace collider

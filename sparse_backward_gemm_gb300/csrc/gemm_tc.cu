// Dimension-reduced dense GEMM on the 5th-generation tensor cores (sm_103a).
//
// Collider (abstract) turns every would-be sparse GEMM of the filtered
// backward into a dense GEMM over the kept rows.  Two shapes occur:
//   dX_k = dY_k . W^T   -> A = dY_k [Mk, out] (K-major), B = W [in, out]
//                          (K-major); the M extent is n_kept (device-resident)
//   dW   = X_k^T . dY_k -> A = X_k [Mk, in], B = dY_k [Mk, out], both
//                          MN-major; the reduction extent is n_kept
// Both run here: TMA (cp.async.bulk.tensor, 128-byte swizzle) stages
// 128 x 64 A tiles and BN x 64 B tiles through a multi-stage shared-memory
// ring; one thread issues tcgen05.mma (kind::f16, bf16 in, f32 accumulate)
// into a double-buffered TMEM accumulator; four epilogue warps drain TMEM
// with tcgen05.ld while the next tile's MMAs run.  Persistent grid (one CTA
// per SM); every mbarrier wait is bounded.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"

namespace collider {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;          // 64 bf16 = 128 bytes = one swizzle row
constexpr int kTcThreads = 192; // warp 0 TMA, warp 1 MMA + TMEM owner, warps 2-5 epilogue

struct TcParams {
  int M, N, K;       // static extents (M / K capped by *n_kept when dyn)
  int dyn;           // 0 none, 1 M = n_kept, 2 K = n_kept
  const int32_t* n_kept;
  void* C;
  long long ldc;
  int c_bf16;
  int accumulate;
  int zero_pad;
  long long c_rows;
  DevStatus* st;
};

// ---------------------------------------------------------------------------
// PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity to complete.  Returns
// false when the budget ran out (recorded in the status word) or another role
// of this CTA already gave up.
__device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                       DevStatus* st, unsigned site) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try(bar, parity)) return true;
    if ((n & 63) == 0) {
      if (*abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitBudgetNs) {
        report_error(st, kErrTimeout, site);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// tcgen05 shared-memory matrix descriptor, 128-byte swizzle, sm_100 version.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
         (static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accum) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accum)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// instruction descriptor: f32 accumulate, bf16 A and B, M = 128, N = BN
template <int BN, bool A_MN, bool B_MN>
__device__ __forceinline__ constexpr uint32_t make_idesc() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((A_MN ? 1u : 0u) << 15) | ((B_MN ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(BM >> 4) << 24);
}

template <int BN>
struct TcCfg {
  static constexpr uint32_t kABytes = BM * BK * 2;
  static constexpr uint32_t kBBytes = BN * BK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr int kStages = BN == 256 ? 4 : 6;
  static constexpr uint32_t kTmemCols = 2 * BN;   // two accumulators
  static constexpr size_t kSmem = 1024 + kStages * kStageBytes + 256;
};

template <int BN, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, TcParams p) {
  using Cfg = TcCfg<BN>;
  constexpr int S = Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * Cfg::kStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S), tfull0 = smem_u32(bars + 2 * S),
                 tempty0 = smem_u32(bars + 2 * S + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int M = p.M, K = p.K;
  if (p.dyn) {
    int nk = *p.n_kept;
    nk = nk < 0 ? 0 : nk;
    if (p.dyn == 1) M = min(M, nk);
    else K = min(K, nk);
  }
  const int m_tiles = (M + BM - 1) / BM, n_tiles = (p.N + BN - 1) / BN;
  const int num_tiles = m_tiles * n_tiles;
  const int num_kb = (K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, 128);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(Cfg::kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer ----------------
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;   // stages with copies issued, and the phase parity armed
      for (int tile = blockIdx.x; tile < num_tiles && !*abort_flag; tile += gridDim.x) {
        const int m0 = (tile % m_tiles) * BM, n0 = (tile / m_tiles) * BN;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(empty0 + 8 * stage, phase ^ 1u, abort_flag, p.st, 1)) break;
          const uint32_t fb = full0 + 8 * stage;
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          mbar_expect_tx(fb, Cfg::kStageBytes);
          const uint32_t sa = smem_u32(smem + stage * Cfg::kStageBytes), sb = sa + Cfg::kABytes;
          const int k0 = kb * BK;
          if (!A_MN) {
            tma_load_2d(sa, &tmA, fb, k0, m0);
          } else {
            tma_load_2d(sa, &tmA, fb, m0, k0);
            tma_load_2d(sa + 8192, &tmA, fb, m0 + 64, k0);
          }
          if (!B_MN) {
            tma_load_2d(sb, &tmB, fb, k0, n0);
          } else {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j) tma_load_2d(sb + 8192 * j, &tmB, fb, n0 + 64 * j, k0);
          }
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      if (*abort_flag) {
        // another role gave up: let this thread's copies still in flight land
        // (bounded, 10 ms per stage) before the CTA releases its shared memory
        for (int s = 0; s < S; ++s) {
          if (!((armed >> s) & 1u)) continue;
          const uint64_t t0 = globaltimer_ns();
          while (!mbar_try(full0 + 8 * s, (armed_parity >> s) & 1u) && globaltimer_ns() - t0 < 10000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer ----------------
      constexpr uint32_t idesc = make_idesc<BN, A_MN, B_MN>();
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      for (int tile = blockIdx.x; tile < num_tiles && !*abort_flag; tile += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t aph = (it >> 1) & 1;
        if (!mbar_wait(tempty0 + 8 * acc, aph ^ 1u, abort_flag, p.st, 2)) break;
        tc_fence_after();
        const uint32_t d = tmem_base + acc * BN;
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, p.st, 3)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * Cfg::kStageBytes), sb = sa + Cfg::kABytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = A_MN ? sdesc(sa + kk * 2048, 8192, 1024) : sdesc(sa + kk * 32, 16, 1024);
            const uint64_t bd = B_MN ? sdesc(sb + kk * 2048, 8192, 1024) : sdesc(sb + kk * 32, 16, 1024);
            mma_bf16(d, ad, bd, idesc, (kb | kk) != 0);
          }
          mma_commit(empty0 + 8 * stage);
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        mma_commit(tfull0 + 8 * acc);
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    const int q = warp & 3;   // TMEM lane quadrant this warp may access
    int it = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++it) {
      const int acc = it & 1;
      const uint32_t aph = (it >> 1) & 1;
      if (!mbar_wait(tfull0 + 8 * acc, aph, abort_flag, p.st, 4)) break;
      tc_fence_after();
      const int m0 = (tile % m_tiles) * BM, n0 = (tile / m_tiles) * BN;
      const int row = m0 + q * 32 + lane;
      const bool row_ok = row < M;
      const bool row_zero = !row_ok && p.zero_pad && row < padded_rows(M, p.c_rows);
      for (int c = 0; c < BN; c += 32) {
        float v[32];
        if (num_kb > 0) {
          tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + c, v);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        if (!(row_ok || row_zero)) continue;
        if (row_zero) {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
        }
        const int col = n0 + c;
        if (p.c_bf16) {
          __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.C) + (long long)row * p.ldc + col;
#pragma unroll
          for (int g = 0; g < 4; ++g)
            if (col + 8 * g + 8 <= p.N) *reinterpret_cast<uint4*>(out + 8 * g) = pack8(v + 8 * g);
        } else {
          float* out = static_cast<float*>(p.C) + (long long)row * p.ldc + col;
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            if (col + 4 * g + 4 <= p.N) {
              float4 o = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
              if (p.accumulate && row_ok) {
                float4 old = *reinterpret_cast<const float4*>(out + 4 * g);
                o.x += old.x; o.y += old.y; o.z += old.z; o.w += old.w;
              }
              *reinterpret_cast<float4*>(out + 4 * g) = o;
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(tempty0 + 8 * acc);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(Cfg::kTmemCols)
                 : "memory");
  }
}

// ---------------------------------------------------------------------------
// host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor map over a row-major [rows, inner] matrix with leading
// dimension ld (elements); box {64, box_rows}; 128-byte swizzle; zero fill.
bool make_map(CUtensorMap* m, const void* base, long long inner, long long rows, long long ld, int box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2};
  cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int BN, bool A_MN, bool B_MN>
cudaError_t launch_variant(const Ctx& c, const TcGemm& g, const CUtensorMap& ma, const CUtensorMap& mb,
                           const TcParams& p) {
  using Cfg = TcCfg<BN>;
  // the shared-memory opt-in is a per-device function attribute: set it the
  // first time each device uses this variant
  static int seen[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || !seen[dev]) {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<BN, A_MN, B_MN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(Cfg::kSmem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) seen[dev] = 1;
  }
  const long long tiles = ((long long)(g.M + BM - 1) / BM) * ((g.N + BN - 1) / BN);
  int grid = static_cast<int>(tiles < c.num_sms ? tiles : c.num_sms);
  if (grid < 1) grid = 1;
  tc_gemm_kernel<BN, A_MN, B_MN><<<grid, kTcThreads, Cfg::kSmem, c.stream>>>(ma, mb, p);
  return cudaGetLastError();
}

}  // namespace

bool tc_gemm_supported(const TcGemm& g) {
  if (g.N % 8 || g.K % 8 || g.M % 8) return false;
  if (g.lda % 8 || g.ldb % 8 || g.ldc % 8) return false;
  auto al = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; };
  return al(g.A) && al(g.B) && al(g.C);
}

cudaError_t launch_tc_gemm(const Ctx& c, const TcGemm& g) {
  int bn = g.bn;
  if (bn == 0) {
    const long long t256 = ((long long)(g.M + BM - 1) / BM) * ((g.N + 255) / 256);
    bn = (t256 >= c.num_sms || g.N % 256 == 0) && g.N >= 256 ? 256 : 128;
  }
  CUtensorMap ma, mb;
  // A: K-major [M rows, K] or MN-major [K rows, M]
  bool ok = g.a_mn_major ? make_map(&ma, g.A, g.M, g.a_rows, g.lda, 64)
                         : make_map(&ma, g.A, g.K, g.a_rows, g.lda, BM);
  ok = ok && (g.b_mn_major ? make_map(&mb, g.B, g.N, g.b_rows, g.ldb, 64)
                           : make_map(&mb, g.B, g.K, g.b_rows, g.ldb, bn));
  if (!ok) return cudaErrorInvalidValue;
  TcParams p{g.M, g.N, g.K, g.dyn, g.n_kept, g.C, g.ldc, g.c_bf16, g.accumulate, g.zero_pad,
             g.c_rows > 0 ? g.c_rows : g.M, c.st};
  prof_begin(c, "tc_gemm", g.M, g.N, g.K, g.dyn);
  cudaError_t e;
  const int key = (bn == 256 ? 4 : 0) | (g.a_mn_major ? 2 : 0) | (g.b_mn_major ? 1 : 0);
  switch (key) {
    case 0: e = launch_variant<128, false, false>(c, g, ma, mb, p); break;
    case 3: e = launch_variant<128, true, true>(c, g, ma, mb, p); break;
    case 4: e = launch_variant<256, false, false>(c, g, ma, mb, p); break;
    case 7: e = launch_variant<256, true, true>(c, g, ma, mb, p); break;
    case 1: e = launch_variant<128, false, true>(c, g, ma, mb, p); break;
    case 2: e = launch_variant<128, true, false>(c, g, ma, mb, p); break;
    case 5: e = launch_variant<256, false, true>(c, g, ma, mb, p); break;
    default: e = launch_variant<256, true, false>(c, g, ma, mb, p); break;
  }
  prof_end(c);
  count_launch();
  return e;
}

}  // namespace collider

// Dimension-reduced dense GEMM on the 5th-generation tensor cores (sm_103a).
//
// Collider (abstract) turns every would-be sparse GEMM of the filtered
// backward into a dense GEMM over the kept rows.  Two shapes occur:
//   dX_k = dY_k . W^T   -> A = dY_k [Mk, out] (K-major), B = W [in, out]
//                          (K-major); the M extent is n_kept (device-resident)
//   dW   = X_k^T . dY_k -> A = X_k [Mk, in], B = dY_k [Mk, out], both
//                          MN-major; the reduction extent is n_kept
// The dense forward's Y = X . W (A = X K-major, B = W [in, out] MN-major)
// uses the same kernel with static extents.
// All run here: TMA (cp.async.bulk.tensor, 128-byte swizzle) stages
// 128 x 64 A tiles and BN x 64 B tiles through a multi-stage shared-memory
// ring; one thread issues tcgen05.mma (kind::f16, bf16 in, f32 accumulate)
// into a double-buffered TMEM accumulator; four epilogue warps drain TMEM
// with tcgen05.ld while the next tile's MMAs run.  Persistent grid (one CTA
// per SM); every mbarrier wait is bounded.
#include <cstdlib>
#include <mutex>

#include "internal.h"
#include "tc_ptx.cuh"

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
  float* partial;    // stream-K: [2 * gridDim.x][BM][BN] f32 partial tiles (null: whole tiles only)
  int* counters;     // stream-K: per-(tile, pair rank) arrival counts, zero on entry and left zero
  int split_mode;    // 0 whole tiles, 1 stream-K, 2 hybrid, 3 auto (see Split)
  DevStatus* st;
};

using namespace tc;

// instruction descriptor: f32 accumulate, bf16 A and B, M = 128, N = BN
template <int BN, bool A_MN, bool B_MN>
__device__ __forceinline__ constexpr uint32_t make_idesc() {
  return idesc_bf16(BM, BN, A_MN, B_MN);
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
// 2-SM mode (BN = 256): a stage holds this CTA's 128 x 64 A slice and half of
// the 256 x 64 B slice, 32 KB, so seven stages fit
constexpr int kTwoStages = 7;
constexpr uint32_t kTwoStageBytes = BM * BK * 2 + 128 * BK * 2;
constexpr size_t kTwoSmem = 1024 + kTwoStages * kTwoStageBytes + 256;

// Work split over the workers: lone CTAs, or CTA pairs (a pair works on one
// 256-row tile, each CTA on its 128 rows, in step).
//   whole tiles  (mode 0): tiles round-robin over the workers.
//   stream-K     (mode 1): the num_tiles * num_kb (tile, k-slice) iterations
//                are cut into equal contiguous ranges, one per worker.
//   hybrid       (mode 2): whole tiles round-robin for all but the last full
//                wave, stream-K over the remaining tiles (between one and two
//                waves' worth), so the tail wave is as full as the others
//                while the bulk keeps the round-robin tile order.
//   auto         (mode 3): hybrid only where whole tiles would leave the
//                workers idle much of the time -- the waves' fill below 60%,
//                or below 90% on a long reduction (>= 128 k-slices, where a
//                tile's k-loop dwarfs the fix-up) -- else whole tiles.
//                Decided on the device, where the real tile count is known.
//                (Measured on the block shapes: a stream-K tail costs more
//                than a 70%-full last wave on a short reduction.)
// A tile cut between workers is finished by whichever of them arrives last,
// summing the partial tiles in worker order (deterministic); in a pair each
// CTA parks and finishes its own 128 rows.
struct Split {
  int m_tiles, num_tiles, num_kb;
  int m_units;         // tile rows of the schedule: m_tiles, or pairs of them for a CTA pair
  int W, wid;          // workers (CTAs or CTA pairs) and this CTA's worker
  int unit0, ustride;  // whole-tile phase: first tile and stride (per worker)
  int dp_tiles;        // tiles handled whole, round-robin, first
  long long total;     // stream-K iterations (over tiles dp_tiles..num_tiles-1)
  bool sk;
  int G;               // workers sharing the stream-K part: min(W, total), no empty range
  __device__ long long begin(int c) const { return (long long)c * total / G; }
  // the CTA whose range holds stream-K iteration x
  __device__ int owner(long long x) const { return (int)(((x + 1) * (long long)G - 1) / total); }
  __device__ int slot(int c, int t) const {
    return 2 * c + (t == dp_tiles + (int)(begin(c) / num_kb) ? 0 : 1);
  }
  __device__ void init(int mode, bool have_scratch) {
    total = 0;
    sk = false;
    dp_tiles = num_tiles;
    G = W;
    if (!have_scratch || mode == 0 || num_kb == 0) return;
    const int grid = W;
    const int waves = num_tiles / grid, rem = num_tiles % grid;
    if (mode == 3) {
      if (rem == 0) return;
      const long long slots = (long long)(waves + 1) * grid;   // whole-tile waves x workers
      const bool poor = 10LL * num_tiles < 6LL * slots, long_k = num_kb >= 128 && 10LL * num_tiles < 9LL * slots;
      if (!poor && !long_k) return;
      mode = 2;
    }
    if (mode == 2) {
      if (rem == 0) return;
      dp_tiles = waves >= 1 ? (waves - 1) * grid : 0;
    } else {
      dp_tiles = 0;
    }
    total = (long long)(num_tiles - dp_tiles) * num_kb;
    sk = total > 0;
    G = (int)(total < (long long)grid ? total : (long long)grid);
  }
};

// Iterates this CTA's segments: (tile, first k-slice, end k-slice).
struct SegIter {
  const Split& sp;
  int tile;            // whole-tile phase
  long long it, end;   // stream-K phase (relative iterations)
  __device__ SegIter(const Split& s) : sp(s) {
    tile = sp.unit0;
    if (sp.sk && sp.wid < sp.G) {
      it = sp.begin(sp.wid);
      end = (long long)(sp.wid + 1) * sp.total / sp.G;
    } else {
      it = end = 0;
    }
  }
  __device__ bool next(int& t, int& k0, int& k1) {
    if (tile < sp.dp_tiles) {
      t = tile;
      k0 = 0;
      k1 = sp.num_kb;
      tile += sp.ustride;
      return true;
    }
    if (it >= end) return false;
    t = sp.dp_tiles + (int)(it / sp.num_kb);
    k0 = (int)(it % sp.num_kb);
    const long long lim = k0 + (end - it);
    k1 = lim < sp.num_kb ? (int)lim : sp.num_kb;
    it += k1 - k0;
    return true;
  }
};

// Store 32 consecutive columns of one output row (bf16 or f32, optional
// accumulate into C, zero rows past the kept count up to the padding).
__device__ __forceinline__ void store32(const TcParams& p, int row, int col, bool row_ok, float* v) {
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

// MODE 0: lone CTAs.
// MODE 2 (BN = 256): the grid is made of 2-CTA clusters; both CTAs of a pair
//           work on the same column tile and on adjacent 128-row tiles, with
//           2-SM MMAs.  Each CTA loads its A tile and half of the B tile into
//           its own shared memory only (32 KB a stage instead of 48), every
//           copy counted on the even CTA's full barrier; the even CTA issues
//           one 256 x 256 MMA over both CTAs' tiles, writing each CTA's 128
//           rows into that CTA's TMEM; its commits reach both CTAs' empty and
//           TMEM-full barriers, and both epilogues release the accumulator on
//           the even CTA's TMEM-empty barrier.  No copy is multicast: each CTA
//           loads only what lands in its own shared memory.
template <int BN, bool A_MN, bool B_MN, int MODE>
__global__ void __launch_bounds__(kTcThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, TcParams p) {
  using Cfg = TcCfg<BN>;
  static_assert(MODE == 0 || MODE == 2, "lone CTAs or 2-SM pairs");
  constexpr bool PAIR = MODE == 2, TWO = MODE == 2;
  static_assert(!TWO || BN == 256, "2-SM tiles are 256 x 256");
  constexpr uint32_t kStageBytes = TWO ? kTwoStageBytes : Cfg::kStageBytes;
  constexpr int S = TWO ? kTwoStages : Cfg::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * kStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S), tfull0 = smem_u32(bars + 2 * S),
                 tempty0 = smem_u32(bars + 2 * S + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(tfull0 + 8 * a, 1);
      mbar_init(tempty0 + 8 * a, TWO ? 256 : 128);
    }
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmA)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmB)) : "memory");
  }
  if (warp == 1) {
    if (TWO) tmem_alloc_pair(smem_u32(tmem_slot), Cfg::kTmemCols);
    else tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
  }
  fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();   // the peer's barriers exist before any copy or commit reaches them
  fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Everything above may run before the kernel ahead in the stream has
  // completed (programmatic dependent launch); the kept count, the operands
  // and the output are read or written only after it has.
  grid_dep_wait();
  int M = p.M, K = p.K;
  if (p.dyn) {
    int nk = *p.n_kept;
    nk = nk < 0 ? 0 : nk;
    if (p.dyn == 1) M = min(M, nk);
    else K = min(K, nk);
  }
  const int rank = PAIR ? static_cast<int>(cluster_ctarank()) : 0;
  Split sp;
  sp.m_tiles = (M + BM - 1) / BM;
  sp.m_units = PAIR ? (sp.m_tiles + 1) / 2 : sp.m_tiles;
  sp.num_tiles = sp.m_units * ((p.N + BN - 1) / BN);
  sp.num_kb = (K + BK - 1) / BK;
  sp.W = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
  sp.wid = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  sp.unit0 = sp.wid;
  sp.ustride = sp.W;
  sp.init(p.split_mode, p.partial != nullptr);
  // partial tile of worker w for tile t: this CTA's 128 rows, stored as
  // [BN / 4][BM][4] f32 so that a warp's 32 rows touch 512 contiguous bytes
  constexpr int R = PAIR ? 2 : 1;
  auto part_at = [&](int w, int t) -> float* {
    return p.partial + ((long long)sp.slot(w, t) * R + rank) * (BM * BN);
  };
  // tile t -> this CTA's output origin
  auto origin = [&](int t, int& m0, int& n0) {
    const int mu = t % sp.m_units;
    m0 = (PAIR ? 2 * mu + rank : mu) * BM;
    n0 = (t / sp.m_units) * BN;
  };

  if (sp.num_kb == 0) {
    // empty reduction (nothing kept): the output is zero
    if (warp >= 2) {
      const int q = warp & 3;
      for (int t = sp.unit0; t < sp.num_tiles; t += sp.ustride) {
        int m0, n0;
        origin(t, m0, n0);
        const int row = m0 + q * 32 + lane;
        const bool row_ok = row < M;
        if (!(row_ok || (p.zero_pad && row < padded_rows(M, p.c_rows)))) continue;
        for (int c = 0; c < BN; c += 32) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0.f;
          store32(p, row, n0 + c, row_ok, v);
        }
      }
    }
  } else if (warp == 0) {
    {
      // ---------------- TMA producer: the converged warp waits, one elected lane issues ----------------
      const bool leader = elect_one();
      auto wait = [&](uint32_t bar, uint32_t parity, unsigned site) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.st, site)) != 0;
      };
      auto aborted = [&]() { return __any_sync(0xffffffffu, *abort_flag != 0); };
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0, armed_parity = 0;   // stages with copies issued, and the phase parity armed
      SegIter si(sp);
      int t, k0, k1;
      while (si.next(t, k0, k1) && !aborted()) {
        int m0, n0;
        origin(t, m0, n0);
        bool ok = true;
        for (int kb = k0; kb < k1; ++kb) {
          if (!wait(empty0 + 8 * stage, phase ^ 1u, 1)) { ok = false; break; }
          const uint32_t fb = full0 + 8 * stage;
          armed |= 1u << stage;
          armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
          const uint32_t sa = smem_u32(smem + stage * kStageBytes), sb = sa + Cfg::kABytes;
          const int kx = kb * BK;
          if (TWO) {
            // both CTAs' copies are counted on the even CTA's full barrier
            if (leader) {
              if (rank == 0) mbar_expect_tx(fb, 2 * kStageBytes);
              const uint32_t lb = map_to_rank(fb, 0);
              if (!A_MN) {
                tma_load_2d_pair(sa, &tmA, lb, kx, m0);
              } else {
                tma_load_2d_pair(sa, &tmA, lb, m0, kx);
                tma_load_2d_pair(sa + 8192, &tmA, lb, m0 + 64, kx);
              }
              if (!B_MN) {
                tma_load_2d_pair(sb, &tmB, lb, kx, n0 + rank * (BN / 2));
              } else {
#pragma unroll
                for (int j = 0; j < BN / 128; ++j)
                  tma_load_2d_pair(sb + 8192 * j, &tmB, lb, n0 + rank * (BN / 2) + 64 * j, kx);
              }
            }
            __syncwarp();
            if (++stage == S) { stage = 0; phase ^= 1u; }
            continue;
          }
          if (leader) {
            mbar_expect_tx(fb, kStageBytes);
            if (!A_MN) {
              tma_load_2d(sa, &tmA, fb, kx, m0);
            } else {
              tma_load_2d(sa, &tmA, fb, m0, kx);
              tma_load_2d(sa + 8192, &tmA, fb, m0 + 64, kx);
            }
            if (!B_MN) {
              tma_load_2d(sb, &tmB, fb, kx, n0);
            } else {
#pragma unroll
              for (int j = 0; j < BN / 64; ++j) tma_load_2d(sb + 8192 * j, &tmB, fb, n0 + 64 * j, kx);
            }
          }
          __syncwarp();
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
      }
      // this CTA's last operands are on their way: the next kernel in the
      // stream may be scheduled (it waits for this grid before reading)
      if (PAIR && !aborted()) {
        // both MMAs release every stage (their commits land in this CTA's
        // empty barriers) before this CTA may leave the cluster
        for (int i = 0; i < S; ++i) {
          if (!wait(empty0 + 8 * stage, phase ^ 1u, 5)) break;
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
      }
      if (aborted() && leader) {
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
    if (!TWO || rank == 0) {
      // ---------------- MMA issuer (the even CTA of a pair in 2-SM mode) ----------------
      // The converged warp waits; one elected lane issues the MMAs and commits.
      const bool leader = elect_one();
      auto wait = [&](uint32_t bar, uint32_t parity, unsigned site) {
        return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.st, site)) != 0;
      };
      constexpr uint32_t idesc = TWO ? idesc_bf16(2 * BM, BN, A_MN, B_MN) : make_idesc<BN, A_MN, B_MN>();
      int stage = 0;
      uint32_t phase = 0;
      int seg = 0;
      SegIter si(sp);
      int t, k0, k1;
      while (si.next(t, k0, k1) && !__any_sync(0xffffffffu, *abort_flag != 0)) {
        const int acc = seg & 1;
        const uint32_t aph = (seg >> 1) & 1;
        if (!wait(tempty0 + 8 * acc, aph ^ 1u, 2)) break;
        fence_after();
        const uint32_t d = tmem_base + acc * BN;
        bool ok = true;
        for (int kb = k0; kb < k1; ++kb) {
          if (!wait(full0 + 8 * stage, phase, 3)) { ok = false; break; }
          fence_after();
          if (leader) {
            const uint32_t sa = smem_u32(smem + stage * kStageBytes), sb = sa + Cfg::kABytes;
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              const uint64_t ad = A_MN ? sdesc(sa + kk * 2048, 8192, 1024) : sdesc(sa + kk * 32, 16, 1024);
              const uint64_t bd = B_MN ? sdesc(sb + kk * 2048, 8192, 1024) : sdesc(sb + kk * 32, 16, 1024);
              if (TWO) mma_bf16_pair(d, ad, bd, idesc, (kb > k0) || (kk > 0));
              else mma_bf16(d, ad, bd, idesc, (kb > k0) || (kk > 0));
            }
            if (TWO) mma_commit_pair_mc(empty0 + 8 * stage, 3);
            else mma_commit(empty0 + 8 * stage);
          }
          __syncwarp();
          if (++stage == S) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (leader) {
          if (TWO) mma_commit_pair_mc(tfull0 + 8 * acc, 3);
          else mma_commit(tfull0 + 8 * acc);
        }
        __syncwarp();
        ++seg;
      }
    }
  } else {
    // ---------------- epilogue (warps 2..5) ----------------
    // the accumulator is handed back to the MMA issuer: in 2-SM mode on the
    // even CTA's barrier, which counts both CTAs' epilogue threads
    auto release_acc = [&](int acc) {
      if (TWO) mbar_arrive_cluster(map_to_rank(tempty0 + 8 * acc, 0));
      else mbar_arrive(tempty0 + 8 * acc);
    };
    // Timeout-only waits: the group synchronises with a named barrier, so all
    // 128 threads leave together.
    volatile int no_abort = 0;
    const int q = warp & 3;   // TMEM lane quadrant this warp may access
    const int et = threadIdx.x - 64;
    int seg = 0;
    SegIter si(sp);
    int t, k0, k1;
    while (si.next(t, k0, k1)) {
      const int acc = seg & 1;
      const uint32_t aph = (seg >> 1) & 1;
      if (!mbar_wait(tfull0 + 8 * acc, aph, &no_abort, p.st, 4)) break;
      fence_after();
      int m0, n0;
      origin(t, m0, n0);
      const int rl = q * 32 + lane;
      const int row = m0 + rl;
      const bool row_ok = row < M;
      const bool row_zero = !row_ok && p.zero_pad && row < padded_rows(M, p.c_rows);
      const uint32_t tcol = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      if (k0 == 0 && k1 == sp.num_kb) {
        // whole tile: straight to the output
        for (int c = 0; c < BN; c += 32) {
          float v[32];
          tmem_ld32(tcol + c, v);
          if (!(row_ok || row_zero)) continue;
          if (row_zero) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
          }
          store32(p, row, n0 + c, row_ok, v);
        }
        fence_before();
        release_acc(acc);
      } else {
        // part of a tile: park it, and finish the tile if this CTA is the last
        float* mine = part_at(sp.wid, t);
        for (int c = 0; c < BN; c += 32) {
          float v[32];
          tmem_ld32(tcol + c, v);
#pragma unroll
          for (int i = 0; i < 32; i += 4)
            __stcg(reinterpret_cast<float4*>(mine + ((long long)((c + i) >> 2) * BM + rl) * 4),
                   make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]));
        }
        fence_before();
        release_acc(acc);
        __threadfence();
        named_bar(1, 128);
        const long long x0 = (long long)(t - sp.dp_tiles) * sp.num_kb;
        const int c_first = sp.owner(x0), c_last = sp.owner(x0 + sp.num_kb - 1);
        if (et == 0) {
          int* ctr = p.counters + (long long)t * R + rank;
          const int old = atomicAdd(ctr, 1);
          const int last = old == c_last - c_first;
          if (last) *ctr = 0;
          *last_flag = last;
        }
        named_bar(1, 128);
        if (*last_flag && (row_ok || row_zero)) {
          __threadfence();
          for (int c = 0; c < BN; c += 32) {
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.f;
            for (int cc = c_first; cc <= c_last; ++cc) {
              const float* src = part_at(cc, t);
#pragma unroll
              for (int i = 0; i < 32; i += 4) {
                const float4 w = __ldcg(reinterpret_cast<const float4*>(src + ((long long)((c + i) >> 2) * BM + rl) * 4));
                v[i] += w.x; v[i + 1] += w.y; v[i + 2] += w.z; v[i + 3] += w.w;
              }
            }
            if (row_zero) {
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = 0.f;
            }
            store32(p, row, n0 + c, row_ok, v);
          }
        }
        named_bar(1, 128);   // last_flag is reused by the next segment
      }
      ++seg;
    }
  }
  fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();
  if (warp == 1) {
    fence_after();
    if (TWO) tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
    else tmem_dealloc(tmem_base, Cfg::kTmemCols);
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

bool make_map(CUtensorMap* m, const void* base, long long inner, long long rows, long long ld, int box_rows) {
  return make_tensor_map(m, base, false, inner, rows, ld, 64, box_rows);
}

template <int BN, bool A_MN, bool B_MN, int MODE>
cudaError_t launch_variant(const Ctx& c, const TcGemm& g, const CUtensorMap& ma, const CUtensorMap& mb,
                           const TcParams& p) {
  constexpr bool PAIR = MODE == 2;
  constexpr size_t kSmemBytes = MODE == 2 ? kTwoSmem : TcCfg<BN>::kSmem;
  auto kern = tc_gemm_kernel<BN, A_MN, B_MN, MODE>;
  // Per-device set-up, the first time each device uses this variant: the
  // shared-memory opt-in (a function attribute), and for the pair variant
  // how many 2-CTA clusters fit on the GPU at once (a persistent grid larger
  // than that would run its last clusters in a second wave).
  static int max_pairs[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  const bool cache = dev >= 0 && dev < 64;
  int pairs_fit = cache ? max_pairs[dev] : 0;
  if (pairs_fit == 0) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(kSmemBytes));
    if (e != cudaSuccess) return e;
    pairs_fit = c.num_sms / 2;
    if (PAIR) {
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.gridDim = dim3(2 * pairs_fit);
      cfg.blockDim = dim3(kTcThreads);
      cfg.dynamicSmemBytes = kSmemBytes;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      if (e != cudaSuccess) return e;
      if (n < 1) return cudaErrorNotSupported;
      pairs_fit = n < pairs_fit ? n : pairs_fit;
    }
    if (cache) max_pairs[dev] = pairs_fit;
  }
  const long long m_tiles = (g.M + BM - 1) / BM, n_tiles = (g.N + BN - 1) / BN;
  if (PAIR) {
    const long long units = (m_tiles + 1) / 2 * n_tiles;
    const int pairs = p.partial ? pairs_fit   // stream-K: every pair takes a share
                                : static_cast<int>(units < pairs_fit ? (units < 1 ? 1 : units) : pairs_fit);
    return launched(launch_k(c, c.pdl, kern, dim3(2 * pairs), dim3(kTcThreads), kSmemBytes, 2, ma, mb, p));
  }
  const long long tiles = m_tiles * n_tiles;
  int grid;
  if (p.partial) {
    grid = c.num_sms < kSkMaxCtas ? c.num_sms : kSkMaxCtas;   // stream-K: one CTA per SM
  } else {
    grid = static_cast<int>(tiles < c.num_sms ? tiles : c.num_sms);
  }
  if (grid < 1) grid = 1;
  return launched(launch_k(c, c.pdl, kern, dim3(grid), dim3(kTcThreads), kSmemBytes, 1, ma, mb, p));
}

}  // namespace

bool make_tensor_map(CUtensorMap* m, const void* base, bool f32, long long inner, long long rows, long long ld,
                     int box_inner, int box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  const int esz = f32 ? 4 : 2;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esz};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_inner), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

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
  // dX: both K-major; dW: both MN-major; the forward's Y = X W: A K-major, B MN-major
  if (g.a_mn_major && !g.b_mn_major) return cudaErrorNotSupported;
  // Work split (launches given stream-K scratch): the auto rule of Split --
  // whole tiles unless they would fill the waves below 60% (90% on a
  // reduction of 128+ k-slices), then a stream-K tail, decided on the device
  // from the real tile count; long static reductions are stream-K throughout.
  // COLLIDER_GEMM_STREAMK=0/1/2/3 forces whole tiles / stream-K / hybrid / auto.
  static const int split_env = [] {
    const char* e = getenv("COLLIDER_GEMM_STREAMK");
    return e ? atoi(e) : -1;
  }();
  // 2-SM pairs for every launch of 256-wide tiles; 128-wide tiles run as
  // lone CTAs.  COLLIDER_GEMM_PAIR=0 forces lone CTAs everywhere.
  static const int pair_env = [] {
    const char* e = getenv("COLLIDER_GEMM_PAIR");
    return e ? atoi(e) : -1;
  }();
  // (A long static reduction -- the dX of the MLP up-projection, 176
  // k-slices -- also runs as pairs with a stream-K tail: as lone CTAs cut
  // evenly by stream-K it read half the DRAM bytes but took 168 against 163 us.)
  const bool pair = pair_env != 0 && bn == 256;
  const int mode = pair ? 2 : 0;
  // counters the stream-K fix-up needs: one per tile, and per CTA of a pair
  const long long m_tiles = (g.M + BM - 1) / BM, n_tiles = (g.N + bn - 1) / bn;
  const long long max_ctrs = (pair ? 2 * ((m_tiles + 1) / 2) : m_tiles) * n_tiles;
  const int split = split_env >= 0 ? split_env : 3;
  const bool sk = split != 0 && g.partial && g.counters && max_ctrs <= g.counter_cap;
  CUtensorMap ma, mb;
  // A: K-major [M rows, K] or MN-major [K rows, M]; B: K-major [N rows, K]
  // (half the tile's rows per box for a pair) or MN-major [K rows, N]
  bool ok = g.a_mn_major ? make_map(&ma, g.A, g.M, g.a_rows, g.lda, 64)
                         : make_map(&ma, g.A, g.K, g.a_rows, g.lda, BM);
  ok = ok && (g.b_mn_major ? make_map(&mb, g.B, g.N, g.b_rows, g.ldb, 64)
                           : make_map(&mb, g.B, g.K, g.b_rows, g.ldb, pair ? bn / 2 : bn));
  if (!ok) return cudaErrorInvalidValue;
  TcParams p{g.M, g.N, g.K, g.dyn, g.n_kept, g.C, g.ldc, g.c_bf16, g.accumulate, g.zero_pad,
             g.c_rows > 0 ? g.c_rows : g.M, sk ? g.partial : nullptr, sk ? g.counters : nullptr,
             split, c.st};
  prof_begin(c, "tc_gemm", g.M, g.N, g.K, g.dyn);
  cudaError_t e;
  const int key = (bn == 256 ? 100 : 0) + (g.a_mn_major ? 10 : (g.b_mn_major ? 20 : 0)) + mode;
  switch (key) {
    case 0: e = launch_variant<128, false, false, 0>(c, g, ma, mb, p); break;
    case 10: e = launch_variant<128, true, true, 0>(c, g, ma, mb, p); break;
    case 20: e = launch_variant<128, false, true, 0>(c, g, ma, mb, p); break;
    case 100: e = launch_variant<256, false, false, 0>(c, g, ma, mb, p); break;
    case 102: e = launch_variant<256, false, false, 2>(c, g, ma, mb, p); break;
    case 110: e = launch_variant<256, true, true, 0>(c, g, ma, mb, p); break;
    case 120: e = launch_variant<256, false, true, 0>(c, g, ma, mb, p); break;
    case 122: e = launch_variant<256, false, true, 2>(c, g, ma, mb, p); break;
    case 112: e = launch_variant<256, true, true, 2>(c, g, ma, mb, p); break;
    default: e = cudaErrorNotSupported; break;
  }
  prof_end(c);
  count_launch();
  return e;
}

}  // namespace collider

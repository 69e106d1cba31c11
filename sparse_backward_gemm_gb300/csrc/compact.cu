// Keep-mask compaction: the ascending list of kept tokens that every
// dimension-reduced dense GEMM of the filtered backward runs over (Collider,
// abstract).  Warp ballots + popcounts give each thread's offset; no atomics,
// so the list is bit-exact and deterministic.
#include "internal.h"

namespace collider {

namespace {

constexpr int kThreads = 1024;          // one block of 32 warps
constexpr int kTokPerThread = 16;       // one 16-byte mask load per thread
constexpr int kChunk = kThreads * kTokPerThread;  // tokens per block pass

// 16 mask bytes starting at `start` -> bit i set if token start+i is kept.
__device__ __forceinline__ uint32_t load_bits(const uint8_t* mask, long long start, long long M) {
  uint32_t bits = 0;
  if (start + kTokPerThread <= M && ((reinterpret_cast<uintptr_t>(mask + start) & 15) == 0)) {
    uint4 v = *reinterpret_cast<const uint4*>(mask + start);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
      for (int b = 0; b < 4; ++b)
        if ((w[j] >> (8 * b)) & 0xffu) bits |= 1u << (4 * j + b);
  } else {
    for (int i = 0; i < kTokPerThread; ++i)
      if (start + i < M && mask[start + i] != 0) bits |= 1u << i;
  }
  return bits;
}

// Exclusive block scan of one int per thread (kThreads threads).  Returns the
// exclusive prefix; *total gets the block sum.  `ws` holds 32 ints.
__device__ __forceinline__ int block_excl_scan(int v, int* ws, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) ws[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = ws[lane];
    int s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s += y;
    }
    ws[lane] = s - w;          // exclusive prefix of warp totals
    if (lane == 31) ws[32] = s;
  }
  __syncthreads();
  int r = ws[warp] + x - v;
  *total = ws[32];
  __syncthreads();
  return r;
}

// Writes the indices of the kept tokens in `bits` (16 tokens from `start`)
// at idx[off...], and cu_kept[b] for every sequence start inside the span.
__device__ __forceinline__ void emit(uint32_t bits, long long start, int off, int B, int T,
                                     int32_t* idx, int32_t* cu_kept, long long M) {
  // sequence starts b*T inside [start, start+16)
  long long b = (start + T - 1) / T;
  for (; b < B && b * (long long)T < start + kTokPerThread && b * (long long)T < M; ++b) {
    int within = (int)(b * (long long)T - start);
    cu_kept[b] = off + __popc(bits & ((1u << within) - 1u));
  }
  int o = off;
  while (bits) {
    int i = __ffs(bits) - 1;
    idx[o++] = (int32_t)(start + i);
    bits &= bits - 1;
  }
}

// Whole mask in one block: loops over kChunk-token passes.
__global__ void __launch_bounds__(kThreads) compact_one_block(const uint8_t* __restrict__ mask, int B,
                                                              int T, int32_t* __restrict__ idx,
                                                              int32_t* __restrict__ cu_kept,
                                                              int32_t* __restrict__ n_kept) {
  __shared__ int ws[33];
  const long long M = (long long)B * T;
  int carry = 0;
  for (long long base = 0; base < M; base += kChunk) {
    long long start = base + (long long)threadIdx.x * kTokPerThread;
    uint32_t bits = (start < M) ? load_bits(mask, start, M) : 0u;
    int total;
    int off = carry + block_excl_scan(__popc(bits), ws, &total);
    if (start < M) emit(bits, start, off, B, T, idx, cu_kept, M);
    carry += total;
  }
  if (threadIdx.x == 0) {
    cu_kept[B] = carry;
    n_kept[0] = carry;
  }
}

// Multi-block path, pass 1: kept count per kChunk-token chunk.
__global__ void __launch_bounds__(kThreads) compact_count(const uint8_t* __restrict__ mask, long long M,
                                                          int* __restrict__ counts) {
  __shared__ int ws[33];
  long long start = (long long)blockIdx.x * kChunk + (long long)threadIdx.x * kTokPerThread;
  uint32_t bits = (start < M) ? load_bits(mask, start, M) : 0u;
  int total;
  block_excl_scan(__popc(bits), ws, &total);
  if (threadIdx.x == 0) counts[blockIdx.x] = total;
}

// Pass 2 (one block): exclusive scan of the chunk counts, in place.
__global__ void __launch_bounds__(kThreads) compact_scan(int* __restrict__ counts, int nchunks, int B,
                                                         int32_t* __restrict__ cu_kept,
                                                         int32_t* __restrict__ n_kept) {
  __shared__ int ws[33];
  int carry = 0;
  for (int base = 0; base < nchunks; base += kThreads) {
    int i = base + threadIdx.x;
    int v = (i < nchunks) ? counts[i] : 0;
    int total;
    int e = block_excl_scan(v, ws, &total);
    if (i < nchunks) counts[i] = carry + e;
    carry += total;
  }
  if (threadIdx.x == 0) {
    cu_kept[B] = carry;
    n_kept[0] = carry;
  }
}

// Pass 3: each chunk writes its kept indices at its scanned offset.
__global__ void __launch_bounds__(kThreads) compact_write(const uint8_t* __restrict__ mask, int B, int T,
                                                          const int* __restrict__ offsets,
                                                          int32_t* __restrict__ idx,
                                                          int32_t* __restrict__ cu_kept) {
  __shared__ int ws[33];
  const long long M = (long long)B * T;
  long long start = (long long)blockIdx.x * kChunk + (long long)threadIdx.x * kTokPerThread;
  uint32_t bits = (start < M) ? load_bits(mask, start, M) : 0u;
  int total;
  int off = offsets[blockIdx.x] + block_excl_scan(__popc(bits), ws, &total);
  if (start < M) emit(bits, start, off, B, T, idx, cu_kept, M);
}

// ---------------------------------------------------------------------------
// Token filter decision from scores (Collider Fig. 2b: the loss of the
// filtered tokens is dropped): per sequence the n lowest scores are filtered,
// equal scores lower position first, NaN above every number.  Keys
// (ordered score bits << 32 | position) are unique, so the n-th smallest key
// X splits the sequence exactly: filtered iff key <= X.  X is found by a radix
// select, 8 bits per pass from the top, one block per sequence.
__device__ __forceinline__ uint32_t order_key(float x) {
  if (x != x) return 0xFFFFFFFFu;
  if (x == 0.f) x = 0.f;   // -0.0 ties with +0.0
  const uint32_t u = __float_as_uint(x);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kThreads) select_keep_kernel(const float* __restrict__ scores, int T, int n,
                                                               uint8_t* __restrict__ mask) {
  __shared__ unsigned hist[256];
  __shared__ unsigned long long s_prefix;
  __shared__ unsigned s_k;
  const float* sc = scores + (long long)blockIdx.x * T;
  uint8_t* mk = mask + (long long)blockIdx.x * T;
  if (n <= 0 || n >= T) {
    for (int i = threadIdx.x; i < T; i += blockDim.x) mk[i] = n <= 0 ? 1 : 0;
    return;
  }
  unsigned long long prefix = 0, himask = 0;
  unsigned k = (unsigned)n;   // rank (1-based) of X among the keys sharing `prefix`
  for (int shift = 56; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < T; i += blockDim.x) {
      const unsigned long long key = ((unsigned long long)order_key(sc[i]) << 32) | (unsigned)i;
      if ((key & himask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // warp 0: lane l owns bins 8l..8l+7; find the bin where the running count reaches k
      const int l = threadIdx.x;
      unsigned c[8], tot = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) { c[j] = hist[8 * l + j]; tot += c[j]; }
      unsigned incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
        if (l >= o) incl += y;
      }
      const unsigned excl = incl - tot;
      const unsigned hit = __ballot_sync(0xffffffffu, excl < k && incl >= k);
      if (l == __ffs(hit) - 1) {
        unsigned cum = excl;
        int d = 0;
        for (; d < 7; ++d) {
          if (cum + c[d] >= k) break;
          cum += c[d];
        }
        s_k = k - cum;
        s_prefix = prefix | ((unsigned long long)(8 * l + d) << shift);
      }
    }
    __syncthreads();
    k = s_k;
    prefix = s_prefix;
    himask |= 0xFFull << shift;
    __syncthreads();
  }
  for (int i = threadIdx.x; i < T; i += blockDim.x) {
    const unsigned long long key = ((unsigned long long)order_key(sc[i]) << 32) | (unsigned)i;
    mk[i] = key > prefix ? 1 : 0;
  }
}

}  // namespace

cudaError_t launch_select_keep(const Ctx& c, const float* scores, int B, int T, int n_filter, uint8_t* mask) {
  prof_begin(c, "select_keep");
  select_keep_kernel<<<B, kThreads, 0, c.stream>>>(scores, T, n_filter, mask);
  prof_end(c);
  count_launch();
  return cudaGetLastError();
}

size_t compact_ws_bytes(long long M) {
  if (M <= kCompactOneBlockMax) return 0;
  long long nchunks = (M + kChunk - 1) / kChunk;
  return (size_t)((nchunks * sizeof(int) + 255) & ~255ll);
}

cudaError_t launch_compact(const Ctx& c, const uint8_t* mask, int B, int T, int32_t* idx,
                           int32_t* cu_kept, int32_t* n_kept, void* ws) {
  long long M = (long long)B * T;
  if (M <= kCompactOneBlockMax) {
    compact_one_block<<<1, kThreads, 0, c.stream>>>(mask, B, T, idx, cu_kept, n_kept);
    count_launch();
    return cudaGetLastError();
  }
  int nchunks = (int)((M + kChunk - 1) / kChunk);
  int* counts = static_cast<int*>(ws);
  compact_count<<<nchunks, kThreads, 0, c.stream>>>(mask, M, counts);
  compact_scan<<<1, kThreads, 0, c.stream>>>(counts, nchunks, B, cu_kept, n_kept);
  compact_write<<<nchunks, kThreads, 0, c.stream>>>(mask, B, T, counts, idx, cu_kept);
  count_launch(3);
  return cudaGetLastError();
}

}  // namespace collider

// ===========================================================================
// collider_compact_noalloc: the same compaction for callers that cannot
// allocate device memory (see include/collider.h).  It always takes the
// three-kernel path, with the per-chunk counts in a fixed array of device
// memory that belongs to this library and lives as long as the process.
// ===========================================================================
#include <cstdio>
#include <mutex>

#include "../../include/collider.h"

namespace collider {
namespace {

// One int per 16,384-token chunk: 65,536 chunks cover 2^30 tokens.  256 KB,
// held by every device that loads the library, until the process exits.
constexpr long long kNoAllocMaxChunks = 65536;
constexpr long long kNoAllocMaxTokens = kNoAllocMaxChunks * kChunk;
static __device__ __align__(256) int g_noalloc_counts[kNoAllocMaxChunks];

std::mutex g_noalloc_mu;
int* g_noalloc_addr[64] = {nullptr};   // device address of g_noalloc_counts, per device

collider_status noalloc_fail(collider_status s, const char* m) {
  set_last_error(m);
  return s;
}

collider_status noalloc_cuda_fail(cudaError_t e, const char* where) {
  char buf[256];
  snprintf(buf, sizeof buf, "collider_compact_noalloc: %s: %s", where, cudaGetErrorString(e));
  set_last_error(buf);
  return COLLIDER_ERR_CUDA;
}

}  // namespace
}  // namespace collider

extern "C" collider_status collider_compact_noalloc(const uint8_t* mask, int B, int T, int32_t* idx,
                                                    int32_t* cu_kept, int32_t* n_kept, void* stream) {
  using namespace collider;
  if (!mask || !idx || !cu_kept || !n_kept)
    return noalloc_fail(COLLIDER_ERR_INVALID_ARG, "collider_compact_noalloc: null pointer");
  if (B < 1 || T < 1)
    return noalloc_fail(COLLIDER_ERR_INVALID_ARG, "collider_compact_noalloc: need B >= 1 and T >= 1");
  const long long M = (long long)B * T;
  if (M > kNoAllocMaxTokens)
    return noalloc_fail(COLLIDER_ERR_INVALID_ARG,
                        "collider_compact_noalloc: B*T exceeds its fixed limit of 1073741824 tokens "
                        "(use collider_compact with a workspace)");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return noalloc_cuda_fail(e, "no current CUDA device");
  if (dev < 0 || dev >= 64)
    return noalloc_fail(COLLIDER_ERR_UNSUPPORTED, "collider_compact_noalloc: device ordinal >= 64");
  e = cudaGetLastError();
  if (e != cudaSuccess) return noalloc_cuda_fail(e, "earlier asynchronous CUDA error");
  int* counts = nullptr;
  {
    // first call on this device: look up the device address of the array
    // (host code cannot use the array's name as a device pointer)
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_noalloc_counts);
      if (e != cudaSuccess) return noalloc_cuda_fail(e, "cudaGetSymbolAddress");
      if (!p) return noalloc_fail(COLLIDER_ERR_CUDA, "collider_compact_noalloc: cudaGetSymbolAddress gave null");
      g_noalloc_addr[dev] = static_cast<int*>(p);
    }
    counts = g_noalloc_addr[dev];
  }
  // every entry read below is written by compact_count first, so nothing
  // left over from an earlier call needs clearing
  const int nchunks = (int)((M + kChunk - 1) / kChunk);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  compact_count<<<nchunks, kThreads, 0, s>>>(mask, M, counts);
  compact_scan<<<1, kThreads, 0, s>>>(counts, nchunks, B, cu_kept, n_kept);
  compact_write<<<nchunks, kThreads, 0, s>>>(mask, B, T, counts, idx, cu_kept);
  count_launch(3);
  e = cudaGetLastError();
  if (e != cudaSuccess) return noalloc_cuda_fail(e, "kernel launch");
  return COLLIDER_OK;
}

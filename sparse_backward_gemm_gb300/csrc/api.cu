// C ABI of libcollider: argument checks, status reporting, workspace carving,
// the launch profiler, and the orchestration of the filtered backward of a
// decoder block and of a decoder stack (Collider, arXiv 2502.00340: activations
// and gradients of filtered tokens are dropped in every layer, the attention
// probabilities are filtered, and each GEMM runs dimension-reduced over the
// kept rows).
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/collider.h"
#include "internal.h"
#include "tc_ptx.cuh"

namespace collider {

// ---------------------------------------------------------------------------
// thread-local error message, launch count, profiler
namespace {
thread_local std::string g_msg;
thread_local long long g_launches = 0;

struct ProfRec {
  const char* name;
  long long m, n, k;
  int dyn;
  cudaEvent_t e0, e1;
  cudaStream_t stream;
};
thread_local bool g_prof_on = false;
thread_local std::vector<ProfRec> g_prof;
thread_local std::vector<cudaEvent_t> g_event_pool;
thread_local size_t g_event_used = 0;
thread_local cudaStream_t g_prof_stream = nullptr;

cudaEvent_t next_event() {
  if (g_event_used == g_event_pool.size()) {
    cudaEvent_t e;
    if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
    g_event_pool.push_back(e);
  }
  return g_event_pool[g_event_used++];
}

collider_status fail(collider_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_msg = buf;
  return s;
}

collider_status cuda_fail(cudaError_t e, const char* where) {
  return fail(COLLIDER_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

// per-device status word and SM count
struct DevInfo {
  DevStatus* st = nullptr;
  int num_sms = 0;
};
std::mutex g_dev_mu;
DevInfo g_dev[64];

collider_status make_ctx(void* stream, Ctx* c) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(COLLIDER_ERR_UNSUPPORTED, "device ordinal %d >= 64", dev);
  // an asynchronous error from earlier work is reported first
  e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, "earlier asynchronous error");
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DevInfo& d = g_dev[dev];
  if (!d.st) {
    void* p = nullptr;
    e = cudaMalloc(&p, 256);
    if (e != cudaSuccess) return cuda_fail(e, "status word allocation");
    e = cudaMemset(p, 0, 256);
    if (e != cudaSuccess) return cuda_fail(e, "status word reset");
    d.st = static_cast<DevStatus*>(p);
    e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "SM count");
  }
  c->stream = static_cast<cudaStream_t>(stream);
  c->st = d.st;
  c->num_sms = d.num_sms;
  return COLLIDER_OK;
}

bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }
size_t up256(size_t b) { return (b + 255) & ~size_t(255); }
long long pad128(long long m) { return (m + 127) & ~127ll; }

// bump allocator over the caller's workspace
struct Carver {
  char* base;
  size_t size;
  size_t used = 0;
  bool dry;  // sizing pass
  template <typename T>
  T* take(size_t count) {
    size_t b = up256(count * sizeof(T));
    T* p = dry ? nullptr : reinterpret_cast<T*>(base + used);
    used += b;
    return p;
  }
};

#define CK(expr)                                      \
  do {                                                \
    cudaError_t _e = (expr);                          \
    if (_e != cudaSuccess) return cuda_fail(_e, #expr); \
  } while (0)

}  // namespace

void count_launch(int n) { g_launches += n; }

bool pdl_allowed() {
  static const bool on = [] {
    const char* e = getenv("COLLIDER_PDL");
    return !(e && e[0] == '0');
  }();
  return on;
}

void set_last_error(const char* msg) { g_msg = msg; }

void prof_begin(const Ctx& c, const char* name, long long m, long long n, long long k, int dyn) {
  if (!g_prof_on) return;
  ProfRec r{name, m, n, k, dyn, next_event(), next_event(), c.stream};
  if (r.e0) cudaEventRecord(r.e0, c.stream);
  g_prof.push_back(r);
  g_prof_stream = c.stream;
}
void prof_end(const Ctx& c) {
  if (!g_prof_on || g_prof.empty()) return;
  if (g_prof.back().e1) cudaEventRecord(g_prof.back().e1, c.stream);
}

}  // namespace collider

using namespace collider;

// ===========================================================================
// status / profiling
// ===========================================================================
extern "C" const char* collider_last_error(void) { return g_msg.c_str(); }

extern "C" long long collider_launch_count(int reset) {
  long long n = g_launches;
  if (reset) g_launches = 0;
  return n;
}

extern "C" collider_status collider_check(void* stream) {
  Ctx c;
  collider_status s = make_ctx(stream, &c);
  if (s != COLLIDER_OK) return s;
  cudaError_t e = cudaStreamSynchronize(c.stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  DevStatus h{};
  e = cudaMemcpy(&h, c.st, sizeof h, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "status read");
  if (h.code == 0) return COLLIDER_OK;
  cudaMemset(c.st, 0, sizeof(DevStatus));
  if (h.code == kErrTimeout)
    return fail(COLLIDER_ERR_TIMEOUT, "a bounded in-kernel wait ran out (site %u, block %u)", h.site, h.block);
  return fail(COLLIDER_ERR_INVALID_ARG, "a kernel skipped an index outside its buffer (site %u, block %u)", h.site,
              h.block);
}

namespace selftest {
// one thread waits on an mbarrier nothing arrives on: the bounded wait runs out
__global__ void wait_kernel(DevStatus* st) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(tc::smem_u32(&bar), 1);
    abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tc::mbar_wait(tc::smem_u32(&bar), 0, &abort_flag, st, 999);
  }
}
}  // namespace selftest

extern "C" collider_status collider_selftest_wait_timeout(void* stream) {
  Ctx c;
  collider_status s = make_ctx(stream, &c);
  if (s != COLLIDER_OK) return s;
  selftest::wait_kernel<<<1, 32, 0, c.stream>>>(c.st);
  count_launch();
  cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? COLLIDER_OK : cuda_fail(e, "self-test wait kernel");
}

// Profiler: record a CUDA event pair around every kernel launch of this host
// thread while enabled.  collider_profile_enable(1) clears earlier records.
extern "C" int collider_profile_enable(int on) {
  g_prof_on = on != 0;
  if (on) {
    g_prof.clear();
    g_event_used = 0;
  }
  return 0;
}

extern "C" int collider_profile_count(void) { return static_cast<int>(g_prof.size()); }

// Record i: kernel name, GEMM extents (0 for other kernels), and elapsed ms.
// Synchronises the recorded events.
extern "C" int collider_profile_get_span(int i, float* start_ms, float* end_ms, int* stream_index) {
  if (i < 0 || i >= static_cast<int>(g_prof.size())) return -1;
  const ProfRec& r = g_prof[i];
  const ProfRec& z = g_prof[0];
  if (start_ms) *start_ms = -1.f;
  if (end_ms) *end_ms = -1.f;
  if (r.e1 && cudaEventSynchronize(r.e1) == cudaSuccess && z.e0) {
    if (start_ms && r.e0) cudaEventElapsedTime(start_ms, z.e0, r.e0);
    if (end_ms) cudaEventElapsedTime(end_ms, z.e0, r.e1);
  }
  if (stream_index) {
    // distinct streams numbered in the order of their first record
    std::vector<cudaStream_t> seen;
    for (int j = 0; j <= i; ++j)
      if (std::find(seen.begin(), seen.end(), g_prof[j].stream) == seen.end()) seen.push_back(g_prof[j].stream);
    *stream_index = static_cast<int>(std::find(seen.begin(), seen.end(), r.stream) - seen.begin());
  }
  return 0;
}

extern "C" int collider_profile_get(int i, const char** name, long long* mnk_dyn, float* ms) {
  if (i < 0 || i >= static_cast<int>(g_prof.size())) return -1;
  const ProfRec& r = g_prof[i];
  if (name) *name = r.name;
  if (mnk_dyn) {
    mnk_dyn[0] = r.m; mnk_dyn[1] = r.n; mnk_dyn[2] = r.k; mnk_dyn[3] = r.dyn;
  }
  if (ms) {
    *ms = -1.f;
    if (r.e0 && r.e1 && cudaEventSynchronize(r.e1) == cudaSuccess) cudaEventElapsedTime(ms, r.e0, r.e1);
  }
  return 0;
}

// ===========================================================================
// token filter decision and a1 compaction
// ===========================================================================
extern "C" collider_status collider_select_keep(const float* scores, int B, int T, int n_filter, uint8_t* mask,
                                                void* stream) {
  if (!scores || !mask) return fail(COLLIDER_ERR_INVALID_ARG, "collider_select_keep: null pointer");
  if (B < 1 || T < 1 || (long long)B * T >= (1ll << 31) || n_filter < 0 || n_filter > T)
    return fail(COLLIDER_ERR_INVALID_ARG, "collider_select_keep: need B, T >= 1, B*T < 2^31, 0 <= n_filter <= T");
  Ctx c;
  collider_status s = make_ctx(stream, &c);
  if (s != COLLIDER_OK) return s;
  CK(launch_select_keep(c, scores, B, T, n_filter, mask));
  return COLLIDER_OK;
}

extern "C" size_t collider_compact_workspace_size(int B, int T) {
  if (B < 1 || T < 1) return 0;
  return compact_ws_bytes((long long)B * T);
}

extern "C" collider_status collider_compact(const uint8_t* mask, int B, int T, int32_t* idx, int32_t* cu_kept,
                                            int32_t* n_kept, void* ws, size_t ws_bytes, void* stream) {
  if (!mask || !idx || !cu_kept || !n_kept) return fail(COLLIDER_ERR_INVALID_ARG, "collider_compact: null pointer");
  if (B < 1 || T < 1 || (long long)B * T >= (1ll << 31))
    return fail(COLLIDER_ERR_INVALID_ARG, "collider_compact: need B, T >= 1 and B*T < 2^31 (B=%d, T=%d)", B, T);
  const size_t need = compact_ws_bytes((long long)B * T);
  if (need && (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255)))
    return fail(COLLIDER_ERR_INVALID_ARG, "collider_compact: needs %zu bytes of 256-aligned workspace", need);
  Ctx c;
  collider_status s = make_ctx(stream, &c);
  if (s != COLLIDER_OK) return s;
  CK(launch_compact(c, mask, B, T, idx, cu_kept, n_kept, ws));
  return COLLIDER_OK;
}

// ===========================================================================
// a2 gather / scatter
// ===========================================================================
extern "C" collider_status collider_gather_rows(const void* src, size_t src_ld_bytes, void* dst,
                                                size_t dst_ld_bytes, size_t row_bytes, int M, const int32_t* idx,
                                                const int32_t* n_kept, void* stream) {
  if (!src || !dst || !idx || !n_kept) return fail(COLLIDER_ERR_INVALID_ARG, "collider_gather_rows: null pointer");
  if (M < 0 || row_bytes == 0 || row_bytes % 16 || src_ld_bytes % 16 || dst_ld_bytes % 16 || !al16(src) ||
      !al16(dst) || row_bytes > src_ld_bytes || row_bytes > dst_ld_bytes || row_bytes > (1u << 30))
    return fail(COLLIDER_ERR_INVALID_ARG, "collider_gather_rows: rows and pointers must be 16-byte multiples");
  Ctx c;
  collider_status s = make_ctx(stream, &c);
  if (s != COLLIDER_OK) return s;
  GatherJob j{static_cast<const char*>(src), static_cast<char*>(dst), (long long)src_ld_bytes,
              (long long)dst_ld_bytes, (int)row_bytes, 0};
  CK(launch_gather(c, &j, 1, M, M, idx, n_kept));
  return COLLIDER_OK;
}

extern "C" collider_status collider_scatter_rows(const void* compact, size_t compact_ld_bytes, void* full,
                                                 size_t full_ld_bytes, size_t row_bytes, int M,
                                                 const int32_t* idx, const int32_t* n_kept, void* stream) {
  if (!compact || !full || !idx || !n_kept)
    return fail(COLLIDER_ERR_INVALID_ARG, "collider_scatter_rows: null pointer");
  if (M < 0 || row_bytes == 0 || row_bytes % 16 || compact_ld_bytes % 16 || full_ld_bytes % 16 || !al16(compact) ||
      !al16(full) || row_bytes > compact_ld_bytes || row_bytes > full_ld_bytes || row_bytes > (1u << 30))
    return fail(COLLIDER_ERR_INVALID_ARG, "collider_scatter_rows: rows and pointers must be 16-byte multiples");
  Ctx c;
  collider_status s = make_ctx(stream, &c);
  if (s != COLLIDER_OK) return s;
  CK(launch_scatter(c, static_cast<const char*>(compact), (long long)compact_ld_bytes, static_cast<char*>(full),
                    (long long)full_ld_bytes, (int)row_bytes, M, idx, n_kept));
  return COLLIDER_OK;
}

// ===========================================================================
// a3/a4 linear backward
// ===========================================================================
namespace {
// stream-K per-tile counters for GEMMs with row extents <= m and columns <= n
long long sk_counter_cap(long long m, long long n) { return ((m + 127) / 128) * ((n + 127) / 128); }

size_t linear_carve(Carver& cv, collider_dtype dt, int M, int K, int N, bool x_full, bool dy_full, bool dx_full,
                    void** xk, void** dyk, void** dxk, float** part) {
  const long long Mp = pad128(M);
  *xk = *dyk = *dxk = nullptr;
  (void)x_full; (void)dy_full;
  if (dt == COLLIDER_BF16) {
    // kept rows of X and dY, zero-padded to 128 rows (also for COMPACT inputs,
    // so the padding rows the reduction reads are exactly zero)
    *xk = cv.take<__nv_bfloat16>((size_t)Mp * K);
    *dyk = cv.take<__nv_bfloat16>((size_t)Mp * N);
    if (dx_full) *dxk = cv.take<__nv_bfloat16>((size_t)Mp * K);
  }
  *part = cv.take<float>(colsum_part_floats(M, N));
  if (dt == COLLIDER_BF16) {
    cv.take<float>(kSkPartialFloats);
    cv.take<int>(sk_counter_cap(std::max<long long>(M, K), std::max(K, N)));
  }
  return cv.used;
}
}  // namespace

extern "C" size_t collider_linear_workspace_size(collider_dtype dtype, int M, int K, int N) {
  if (M < 0 || K < 1 || N < 1) return 0;
  Carver cv{nullptr, 0, 0, true};
  void *a, *b, *d;
  float* p;
  return linear_carve(cv, dtype, M, K, N, true, true, true, &a, &b, &d, &p);
}

extern "C" collider_status collider_linear_bwd(collider_dtype dtype, int M, int K, int N, const void* X,
                                               collider_rows x_rows, const void* W, const void* dY,
                                               collider_rows dy_rows, const int32_t* idx, const int32_t* n_kept,
                                               void* dX, collider_rows dx_rows, float* dW, float* db, void* ws,
                                               size_t ws_bytes, void* stream) {
  if (dtype != COLLIDER_F32 && dtype != COLLIDER_BF16)
    return fail(COLLIDER_ERR_UNSUPPORTED, "collider_linear_bwd: dtype %d", (int)dtype);
  if (M < 0 || K < 1 || N < 1) return fail(COLLIDER_ERR_INVALID_ARG, "collider_linear_bwd: bad sizes");
  if (!idx || !n_kept || !dY) return fail(COLLIDER_ERR_INVALID_ARG, "collider_linear_bwd: null idx/n_kept/dY");
  if (dX && !W) return fail(COLLIDER_ERR_INVALID_ARG, "collider_linear_bwd: dX needs W");
  if (dW && !X) return fail(COLLIDER_ERR_INVALID_ARG, "collider_linear_bwd: dW needs X");
  const bool x_full = x_rows == COLLIDER_ROWS_FULL, dy_full = dy_rows == COLLIDER_ROWS_FULL,
             dx_full = dx_rows == COLLIDER_ROWS_FULL;
  if (dtype == COLLIDER_BF16) {
    if (K % 8 || N % 8) return fail(COLLIDER_ERR_UNSUPPORTED, "collider_linear_bwd: bf16 needs K, N % 8 == 0");
    if (!al16(X) || !al16(W) || !al16(dY) || !al16(dX) || !al16(dW) || !al16(db))
      return fail(COLLIDER_ERR_INVALID_ARG, "collider_linear_bwd: bf16 pointers must be 16-byte aligned");
  } else if (db && (N % 8 || !al16(dY) || !al16(db))) {
    return fail(COLLIDER_ERR_UNSUPPORTED, "collider_linear_bwd: f32 db needs N %% 8 == 0 and 16-byte alignment");
  }
  Carver cv{static_cast<char*>(ws), ws_bytes, 0, false};
  void *xk, *dyk, *dxk;
  float* part;
  Carver dry{nullptr, 0, 0, true};
  void *t0, *t1, *t2;
  float* t3;
  const size_t need = linear_carve(dry, dtype, M, K, N, x_full && dW, dy_full, dx_full && dX, &t0, &t1, &t2, &t3);
  if (need > ws_bytes || (ws && (reinterpret_cast<uintptr_t>(ws) & 255)) || (need && !ws))
    return fail(COLLIDER_ERR_INVALID_ARG, "collider_linear_bwd: needs %zu bytes of 256-aligned workspace", need);
  linear_carve(cv, dtype, M, K, N, x_full && dW, dy_full, dx_full && dX, &xk, &dyk, &dxk, &part);
  Ctx c;
  collider_status s = make_ctx(stream, &c);
  if (s != COLLIDER_OK) return s;
  if (M == 0) return COLLIDER_OK;
  float* sk_partial = nullptr;
  int* sk_counters = nullptr;
  const long long sk_cap = sk_counter_cap(std::max<long long>(M, K), std::max(K, N));
  if (dtype == COLLIDER_BF16) {
    // the stream-K scratch sits at the end of the carve (see linear_carve)
    sk_counters = reinterpret_cast<int*>(static_cast<char*>(ws) + need - up256(sk_cap * sizeof(int)));
    sk_partial = reinterpret_cast<float*>(reinterpret_cast<char*>(sk_counters) - up256(kSkPartialFloats * 4));
    CK(cudaMemsetAsync(sk_counters, 0, sk_cap * sizeof(int), c.stream));
  }

  if (dtype == COLLIDER_F32) {
    const float* Xf = static_cast<const float*>(X);
    const float* Wf = static_cast<const float*>(W);
    const float* dYf = static_cast<const float*>(dY);
    if (dX) {
      // filtered rows of a FULL dX (and padding rows of a COMPACT one) are 0
      CK(cudaMemsetAsync(dX, 0, (size_t)M * K * sizeof(float), c.stream));
      SimtGemm g{};
      g.M = M; g.N = K; g.K = N;
      g.A = dYf; g.lda = N; g.a_trans = 0; g.a_gather = dy_full;
      g.B = Wf; g.ldb = N; g.b_trans = 0; g.b_gather = 0;
      g.C = static_cast<float*>(dX); g.ldc = K; g.c_scatter = dx_full;
      g.idx = idx; g.n_kept = n_kept; g.dyn = 1;
      CK(launch_simt_gemm(c, g));
    }
    if (dW) {
      SimtGemm g{};
      g.M = K; g.N = N; g.K = M;
      g.A = Xf; g.lda = K; g.a_trans = 1; g.a_gather = x_full;
      g.B = dYf; g.ldb = N; g.b_trans = 1; g.b_gather = dy_full;
      g.C = dW; g.ldc = N; g.c_scatter = 0;
      g.idx = idx; g.n_kept = n_kept; g.dyn = 2;
      CK(launch_simt_gemm(c, g));
    }
    if (db) CK(launch_colsum(c, dY, 0, N, M, N, dy_full ? idx : nullptr, n_kept, part, db));
    return COLLIDER_OK;
  }

  // bf16: compact operands (zero-padded to 128 rows), tcgen05 GEMMs
  const __nv_bfloat16* Xk = static_cast<const __nv_bfloat16*>(X);
  const __nv_bfloat16* dYk = static_cast<const __nv_bfloat16*>(dY);
  {
    const GatherJob jx{static_cast<const char*>(X), static_cast<char*>(xk), (long long)K * 2, (long long)K * 2,
                       K * 2, 0};
    const GatherJob jy{static_cast<const char*>(dY), static_cast<char*>(dyk), (long long)N * 2, (long long)N * 2,
                       N * 2, 0};
    if (dW) CK(launch_gather(c, &jx, 1, M, pad128(M), x_full ? idx : nullptr, n_kept));
    CK(launch_gather(c, &jy, 1, M, pad128(M), dy_full ? idx : nullptr, n_kept));
    if (dW) Xk = static_cast<const __nv_bfloat16*>(xk);
    dYk = static_cast<const __nv_bfloat16*>(dyk);
  }
  if (dX) {
    TcGemm g{};
    g.M = M; g.N = K; g.K = N;
    g.A = dYk; g.lda = N; g.a_mn_major = 0; g.a_rows = M;
    g.B = W; g.ldb = N; g.b_mn_major = 0; g.b_rows = K;
    g.C = dx_full ? dxk : dX; g.ldc = K; g.c_bf16 = 1; g.zero_pad = 1; g.c_rows = dx_full ? pad128(M) : M;
    g.n_kept = n_kept; g.dyn = 1;
    g.partial = sk_partial; g.counters = sk_counters; g.counter_cap = sk_cap;
    CK(launch_tc_gemm(c, g));
    if (dx_full) CK(launch_scatter(c, static_cast<const char*>(dxk), (long long)K * 2, static_cast<char*>(dX),
                                   (long long)K * 2, K * 2, M, idx, n_kept));
  }
  if (dW) {
    TcGemm g{};
    g.M = K; g.N = N; g.K = M;
    g.A = Xk; g.lda = K; g.a_mn_major = 1; g.a_rows = M;
    g.B = dYk; g.ldb = N; g.b_mn_major = 1; g.b_rows = M;
    g.C = dW; g.ldc = N; g.c_bf16 = 0;
    g.n_kept = n_kept; g.dyn = 2;
    g.partial = sk_partial; g.counters = sk_counters; g.counter_cap = sk_cap;
    CK(launch_tc_gemm(c, g));
  }
  if (db) CK(launch_colsum(c, dYk, 1, N, M, N, nullptr, n_kept, part, db));
  return COLLIDER_OK;
}

// ===========================================================================
// a7/a8 attention backward
// ===========================================================================
namespace {
struct AttnScratch {
  float* dq_acc;
  float* dk_acc;
  float* dv_acc;
  float* Dvec;
  float* lse2;
  float2* rope;
  int* order;   // work-item ticket + the dQ accumulation turn of every (sequence, head, query block)
};
void attn_carve(Carver& cv, int B, int T, int H, int Hkv, int dh, AttnScratch* a) {
  const size_t M = (size_t)B * T;
  a->dq_acc = cv.take<float>(M * H * dh);
  a->dk_acc = cv.take<float>(M * Hkv * dh);
  a->dv_acc = cv.take<float>(M * Hkv * dh);
  a->Dvec = cv.take<float>(M * H);
  a->lse2 = cv.take<float>(M * H);
  a->rope = cv.take<float2>((size_t)T * (dh / 2));
  a->order = cv.take<int>(attn_order_ints(B, T, H));
}
}  // namespace

extern "C" size_t collider_attn_workspace_size(int B, int T, int H, int Hkv, int dh) {
  if (B < 1 || T < 1 || H < 1 || Hkv < 1 || dh < 1) return 0;
  Carver cv{nullptr, 0, 0, true};
  AttnScratch a;
  attn_carve(cv, B, T, H, Hkv, dh, &a);
  const size_t Mp = pad128((long long)B * T);
  cv.take<__nv_bfloat16>(Mp * H * dh * 2);          // compact Q, dO (FULL inputs)
  cv.take<__nv_bfloat16>(Mp * Hkv * dh * 2);        // compact K, V
  cv.take<__nv_bfloat16>(Mp * (H + 2 * Hkv) * dh);  // compact dQ, dK, dV (FULL outputs)
  return cv.used;
}

extern "C" collider_status collider_attn_bwd(int B, int T, int H, int Hkv, int dh, int causal, float scale,
                                             int rotary_dim, float rope_base, const void* Q, const void* K,
                                             const void* V, const void* O, const void* dO, int q_ld, int kv_ld,
                                             int do_ld, collider_rows in_rows, const float* lse,
                                             const int32_t* idx, const int32_t* cu_kept, const int32_t* n_kept,
                                             void* dQ, void* dK, void* dV, collider_rows out_rows, void* ws,
                                             size_t ws_bytes, void* stream) {
  (void)O;
  if (!Q || !K || !V || !dO || !lse || !idx || !cu_kept || !n_kept || !dQ || !dK || !dV)
    return fail(COLLIDER_ERR_INVALID_ARG, "collider_attn_bwd: null pointer");
  if (B < 1 || T < 1 || H < 1 || Hkv < 1 || H % Hkv || (long long)B * T >= (1ll << 31))
    return fail(COLLIDER_ERR_INVALID_ARG, "collider_attn_bwd: bad B/T/H/Hkv");
  if (dh != 64 && dh != 128) return fail(COLLIDER_ERR_UNSUPPORTED, "collider_attn_bwd: dh must be 64 or 128");
  if (rotary_dim < 0 || rotary_dim > dh || rotary_dim % 16)
    return fail(COLLIDER_ERR_UNSUPPORTED, "collider_attn_bwd: rotary_dim must be a multiple of 16 <= dh");
  if (q_ld < H * dh || kv_ld < Hkv * dh || do_ld < H * dh || q_ld % 8 || kv_ld % 8 || do_ld % 8)
    return fail(COLLIDER_ERR_INVALID_ARG, "collider_attn_bwd: row strides too small or not multiples of 8");
  if (!al16(Q) || !al16(K) || !al16(V) || !al16(dO) || !al16(dQ) || !al16(dK) || !al16(dV))
    return fail(COLLIDER_ERR_INVALID_ARG, "collider_attn_bwd: pointers must be 16-byte aligned");
  const size_t need = collider_attn_workspace_size(B, T, H, Hkv, dh);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255))
    return fail(COLLIDER_ERR_INVALID_ARG, "collider_attn_bwd: needs %zu bytes of 256-aligned workspace", need);
  Ctx c;
  collider_status s = make_ctx(stream, &c);
  if (s != COLLIDER_OK) return s;
  const int M = B * T;
  const long long Mp = pad128(M);
  Carver cv{static_cast<char*>(ws), ws_bytes, 0, false};
  AttnScratch sc;
  attn_carve(cv, B, T, H, Hkv, dh, &sc);
  auto* cq = cv.take<__nv_bfloat16>((size_t)Mp * H * dh);
  auto* cdo = cv.take<__nv_bfloat16>((size_t)Mp * H * dh);
  auto* ck = cv.take<__nv_bfloat16>((size_t)Mp * Hkv * dh);
  auto* cvv = cv.take<__nv_bfloat16>((size_t)Mp * Hkv * dh);
  auto* cdq = cv.take<__nv_bfloat16>((size_t)Mp * H * dh);
  auto* cdk = cv.take<__nv_bfloat16>((size_t)Mp * Hkv * dh);
  auto* cdv = cv.take<__nv_bfloat16>((size_t)Mp * Hkv * dh);

  AttnArgs a{};
  a.B = B; a.T = T; a.H = H; a.Hkv = Hkv; a.dh = dh; a.causal = causal; a.scale = scale;
  a.rotary_dim = rotary_dim; a.rope_base = rope_base;
  a.lse = lse; a.idx = idx; a.cu_kept = cu_kept; a.n_kept = n_kept;
  a.dq_acc = sc.dq_acc; a.Dvec = sc.Dvec; a.lse_k = sc.lse2; a.rope = sc.rope; a.M = M;
  a.dk_acc = sc.dk_acc; a.dv_acc = sc.dv_acc; a.order = sc.order;
  a.in_cap = in_rows == COLLIDER_ROWS_FULL ? Mp : M;
  a.cap = out_rows == COLLIDER_ROWS_FULL ? Mp : M;
  if (in_rows == COLLIDER_ROWS_FULL) {
    GatherJob j[4] = {
        {static_cast<const char*>(Q), reinterpret_cast<char*>(cq), (long long)q_ld * 2, (long long)H * dh * 2,
         H * dh * 2, 0},
        {static_cast<const char*>(dO), reinterpret_cast<char*>(cdo), (long long)do_ld * 2, (long long)H * dh * 2,
         H * dh * 2, 0},
        {static_cast<const char*>(K), reinterpret_cast<char*>(ck), (long long)kv_ld * 2, (long long)Hkv * dh * 2,
         Hkv * dh * 2, 0},
        {static_cast<const char*>(V), reinterpret_cast<char*>(cvv), (long long)kv_ld * 2, (long long)Hkv * dh * 2,
         Hkv * dh * 2, 0}};
    CK(launch_gather(c, j, 4, M, Mp, idx, n_kept));
    a.q = cq; a.dO = cdo; a.k = ck; a.v = cvv;
    a.q_ld = (long long)H * dh; a.do_ld = (long long)H * dh; a.kv_ld = (long long)Hkv * dh;
  } else {
    a.q = static_cast<const __nv_bfloat16*>(Q); a.k = static_cast<const __nv_bfloat16*>(K);
    a.v = static_cast<const __nv_bfloat16*>(V); a.dO = static_cast<const __nv_bfloat16*>(dO);
    a.q_ld = q_ld; a.kv_ld = kv_ld; a.do_ld = do_ld;
  }
  const bool out_full = out_rows == COLLIDER_ROWS_FULL;
  if (out_full) {
    a.dq = cdq; a.dk = cdk; a.dv = cdv;
    a.dq_ld = (long long)H * dh; a.dkv_ld = (long long)Hkv * dh;
  } else {
    // COMPACT outputs use the input strides: dQ with q_ld, dK and dV with kv_ld
    a.dq = static_cast<__nv_bfloat16*>(dQ); a.dk = static_cast<__nv_bfloat16*>(dK);
    a.dv = static_cast<__nv_bfloat16*>(dV);
    a.dq_ld = q_ld; a.dkv_ld = kv_ld;
  }
  CK(launch_attn_bwd(c, a));
  if (out_full) {
    CK(launch_scatter(c, reinterpret_cast<const char*>(cdq), (long long)H * dh * 2, static_cast<char*>(dQ),
                      (long long)q_ld * 2, H * dh * 2, M, idx, n_kept));
    CK(launch_scatter(c, reinterpret_cast<const char*>(cdk), (long long)Hkv * dh * 2, static_cast<char*>(dK),
                      (long long)kv_ld * 2, Hkv * dh * 2, M, idx, n_kept));
    CK(launch_scatter(c, reinterpret_cast<const char*>(cdv), (long long)Hkv * dh * 2, static_cast<char*>(dV),
                      (long long)kv_ld * 2, Hkv * dh * 2, M, idx, n_kept));
  }
  return COLLIDER_OK;
}

// ===========================================================================
// whole block
// ===========================================================================
namespace {

struct LayerBufs {
  __nv_bfloat16 *dout_k, *s_k, *b_k, *o_k, *a_k, *qkv_k;  // gathered (s_k holds gelu(f1) for phi)
  __nv_bfloat16 *ds_k, *dgu_k, *dh_k, *do_k, *dqkv_k;
  float *db_k, *da_k;
  float* norm_part;
  float* norm_part2;     // the middle norm's partials (reduced on the side stream)
  float* col_part;
  float* sk_partial;     // stream-K scratch of the input-gradient chain's GEMMs
  int* sk_counters;
  long long sk_cap;
  AttnScratch at;
  int32_t *id_idx, *id_cu, *id_nk;   // the identity index of a dense (every token kept) call
};

collider_status check_desc(const collider_layer_desc* d) {
  if (!d) return fail(COLLIDER_ERR_INVALID_ARG, "null layer desc");
  if (d->arch != COLLIDER_ARCH_LLAMA && d->arch != COLLIDER_ARCH_PHI)
    return fail(COLLIDER_ERR_UNSUPPORTED, "arch %d", d->arch);
  if (d->B < 1 || d->T < 1 || (long long)d->B * d->T >= (1ll << 31))
    return fail(COLLIDER_ERR_INVALID_ARG, "bad B/T");
  if (d->H < 1 || d->Hkv < 1 || d->H % d->Hkv) return fail(COLLIDER_ERR_INVALID_ARG, "bad head counts");
  if (d->dh != 64 && d->dh != 128) return fail(COLLIDER_ERR_UNSUPPORTED, "head dim %d", d->dh);
  if (d->D % 64 || d->F % 64 || d->D > 4096)
    return fail(COLLIDER_ERR_UNSUPPORTED, "D and F must be multiples of 64, D <= 4096");
  if (d->rotary_dim < 0 || d->rotary_dim > d->dh || d->rotary_dim % 16)
    return fail(COLLIDER_ERR_UNSUPPORTED, "rotary_dim must be a multiple of 16 <= dh");
  const bool llama = d->arch == COLLIDER_ARCH_LLAMA;
  if (llama && (d->norm != COLLIDER_NORM_RMS || d->act != COLLIDER_ACT_SWIGLU))
    return fail(COLLIDER_ERR_UNSUPPORTED, "llama blocks use RMSNorm + SwiGLU");
  if (!llama && (d->norm != COLLIDER_NORM_LAYER || d->act != COLLIDER_ACT_GELU_TANH))
    return fail(COLLIDER_ERR_UNSUPPORTED, "phi blocks use LayerNorm + GELU-tanh");
  return COLLIDER_OK;
}

void layer_carve(Carver& cv, const collider_layer_desc* d, LayerBufs* L) {
  const size_t Mp = pad128((long long)d->B * d->T);
  const size_t D = d->D, F = d->F, Hd = (size_t)d->H * d->dh, Nqkv = (size_t)(d->H + 2 * d->Hkv) * d->dh;
  const bool llama = d->arch == COLLIDER_ARCH_LLAMA;
  const size_t Nup = llama ? 2 * F : F;
  L->dout_k = cv.take<__nv_bfloat16>(Mp * D);
  L->s_k = cv.take<__nv_bfloat16>(Mp * F);
  L->b_k = llama ? cv.take<__nv_bfloat16>(Mp * D) : nullptr;
  L->o_k = cv.take<__nv_bfloat16>(Mp * Hd);
  L->a_k = cv.take<__nv_bfloat16>(Mp * D);
  L->qkv_k = cv.take<__nv_bfloat16>(Mp * Nqkv);
  L->ds_k = cv.take<__nv_bfloat16>(Mp * F);
  L->dgu_k = cv.take<__nv_bfloat16>(Mp * Nup);
  L->dh_k = llama ? cv.take<__nv_bfloat16>(Mp * D) : nullptr;
  L->do_k = cv.take<__nv_bfloat16>(Mp * Hd);
  L->dqkv_k = cv.take<__nv_bfloat16>(Mp * Nqkv);
  L->db_k = llama ? cv.take<float>(Mp * D) : nullptr;
  L->da_k = cv.take<float>(Mp * D);
  L->norm_part = cv.take<float>(norm_part_floats((int)Mp, (int)D));
  L->norm_part2 = llama ? cv.take<float>(norm_part_floats((int)Mp, (int)D)) : nullptr;
  size_t cp = colsum_part_floats((int)Mp, (int)std::max(Nqkv, std::max(Nup, D)));
  L->col_part = cv.take<float>(cp);
  attn_carve(cv, d->B, d->T, d->H, d->Hkv, d->dh, &L->at);
  L->sk_partial = cv.take<float>(kSkPartialFloats);
  const long long mmax = std::max<long long>((long long)Mp, std::max(D, F));
  L->sk_cap = sk_counter_cap(mmax, std::max<long long>(std::max(Nqkv, Nup), std::max(D, F)));
  L->sk_counters = cv.take<int>(L->sk_cap);
  L->id_idx = cv.take<int32_t>((size_t)d->B * d->T);
  L->id_cu = cv.take<int32_t>((size_t)d->B + 1);
  L->id_nk = cv.take<int32_t>(1);
}

// The weight-gradient GEMMs of a block depend on nothing the block computes
// after their inputs, so they run on a second stream (one per host thread and
// device), forked from and joined back into the caller's stream with events:
// they fill the SMs the input-gradient chain leaves idle (GEMM tail waves,
// attention, row kernels).  The input-gradient chain itself runs on a
// high-priority stream (forked from the caller's stream at the start of the
// block, joined back at the end), so when CTAs of both wait for SMs the
// chain's go first.  No host synchronisation.
struct Side {
  cudaStream_t s = nullptr;    // weight gradients, default priority
  cudaStream_t hi = nullptr;   // input-gradient chain, highest priority
  cudaEvent_t ev[12] = {};
};
thread_local Side g_side[64];

// COLLIDER_SIDE_STREAM=0 keeps every launch on the caller's stream (used to
// time kernels one at a time); read at every call.
bool side_enabled() {
  const char* e = getenv("COLLIDER_SIDE_STREAM");
  return !(e && e[0] == '0');
}

collider_status side_ctx(const Ctx& c, Ctx* c2, Side** sd) {
  if (!side_enabled()) {
    *c2 = c;
    *sd = nullptr;
    return COLLIDER_OK;
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  Side& S = g_side[dev & 63];
  if (!S.s) {
    int least = 0, greatest = 0;
    e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
    if (e != cudaSuccess) return cuda_fail(e, "stream priority range");
    e = cudaStreamCreateWithPriority(&S.hi, cudaStreamNonBlocking, greatest);
    if (e != cudaSuccess) return cuda_fail(e, "high-priority stream");
    e = cudaStreamCreateWithFlags(&S.s, cudaStreamNonBlocking);
    if (e != cudaSuccess) return cuda_fail(e, "side stream");
    for (auto& ev : S.ev) {
      e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
      if (e != cudaSuccess) return cuda_fail(e, "side stream event");
    }
  }
  *c2 = c;
  c2->stream = S.s;
  *sd = &S;
  return COLLIDER_OK;
}
// the high-priority stream waits for the caller's stream (event slot 8), and
// the caller's stream waits for it at the end (slot 9)
cudaError_t fork_hi(cudaStream_t caller, Side* S) {
  cudaError_t e = cudaEventRecord(S->ev[8], caller);
  return e == cudaSuccess ? cudaStreamWaitEvent(S->hi, S->ev[8], 0) : e;
}
cudaError_t join_hi(cudaStream_t caller, Side* S) {
  cudaError_t e = cudaEventRecord(S->ev[9], S->hi);
  return e == cudaSuccess ? cudaStreamWaitEvent(caller, S->ev[9], 0) : e;
}
// side stream waits for everything enqueued on the caller's stream so far
cudaError_t fork_side(const Ctx& c, Side* S, int k) {
  if (!S) return cudaSuccess;
  cudaError_t e = cudaEventRecord(S->ev[k], c.stream);
  return e == cudaSuccess ? cudaStreamWaitEvent(S->s, S->ev[k], 0) : e;
}
// caller's stream waits for everything enqueued on the side stream so far
cudaError_t join_side(const Ctx& c, Side* S, int k) {
  if (!S) return cudaSuccess;
  cudaError_t e = cudaEventRecord(S->ev[k], S->s);
  return e == cudaSuccess ? cudaStreamWaitEvent(c.stream, S->ev[k], 0) : e;
}

// stream-K scratch shared by the input-gradient chain's GEMMs of one call
// (they run in stream order)
thread_local float* g_sk_partial = nullptr;
thread_local int* g_sk_counters = nullptr;
thread_local long long g_sk_cap = 0;

// C (bf16 or f32, COMPACT [Mk, N]) = A_k [Mk, K] . W^T with W stored [N, K]
cudaError_t gemm_dx(const Ctx& c, int M, int N, int K, const void* A, const void* W, void* C, int c_bf16,
                    int accumulate, const int32_t* n_kept, long long a_rows = -1) {
  TcGemm g{};
  g.partial = g_sk_partial; g.counters = g_sk_counters; g.counter_cap = g_sk_cap;
  g.M = M; g.N = N; g.K = K;
  g.A = A; g.lda = K; g.a_mn_major = 0; g.a_rows = a_rows > 0 ? a_rows : pad128(M);
  g.B = W; g.ldb = K; g.b_mn_major = 0; g.b_rows = N;
  g.C = C; g.ldc = N; g.c_bf16 = c_bf16; g.accumulate = accumulate; g.zero_pad = 1;
  g.c_rows = pad128(M);
  g.n_kept = n_kept; g.dyn = 1;
  return launch_tc_gemm(c, g);
}

// dW [Kin, Nout] f32 = X_k^T dY_k, X_k [Mk, Kin], dY_k [Mk, Nout] (both COMPACT, zero-padded,
// or -- a dense call -- the caller's M rows: rows = M, the TMA fills past them with zeros)
// (runs on the side stream, concurrently with the input-gradient chain, as
// whole tiles: there a tail wave leaves SMs to the chain's kernels, while
// stream-K would hold every SM to the end -- measured: the block step was
// slower with it)
cudaError_t gemm_dw(const Ctx& c, int M, int Kin, int Nout, const void* Xk, long long ldx, const void* dYk,
                    long long ldy, float* dW, const int32_t* n_kept, long long rows = -1) {
  TcGemm g{};
  g.M = Kin; g.N = Nout; g.K = M;
  g.A = Xk; g.lda = ldx; g.a_mn_major = 1; g.a_rows = rows > 0 ? rows : pad128(M);
  g.B = dYk; g.ldb = ldy; g.b_mn_major = 1; g.b_rows = rows > 0 ? rows : pad128(M);
  g.C = dW; g.ldc = Nout; g.c_bf16 = 0;
  g.n_kept = n_kept; g.dyn = 2;
  return launch_tc_gemm(c, g);
}

// dense: every token is kept (idx, cu_kept, n_kept are the identity index the
// caller made with launch_identity_index into L.id_*): the saved rows and dOut
// are read where they are, nothing is gathered, and dx is written in place.
collider_status layer_bwd_impl(const Ctx& c_in, const collider_layer_desc* d, const collider_layer_weights* w,
                               const collider_layer_saved* sv, const void* dOut, bool dout_full,
                               const int32_t* idx, const int32_t* cu_kept, const int32_t* n_kept,
                               const collider_layer_grads* g, bool dx_full, LayerBufs& L, bool dense = false) {
  // c: the context of the input-gradient chain (the high-priority stream when
  // the side stream is on, else the caller's)
  Ctx c = c_in;
  Ctx cs;
  Side* side = nullptr;
  {
    collider_status st = side_ctx(c_in, &cs, &side);
    if (st != COLLIDER_OK) return st;
  }
  if (side) {
    CK(fork_hi(c_in.stream, side));
    c.stream = side->hi;
  }
  const int M = d->B * d->T;
  const int D = d->D, F = d->F, H = d->H, Hkv = d->Hkv, dh = d->dh;
  const int Hd = H * dh, Nqkv = (H + 2 * Hkv) * dh;
  const bool llama = d->arch == COLLIDER_ARCH_LLAMA;
  const int Nup = llama ? 2 * F : F;
  // (the stream-K counters were zeroed by the entry point; kernels leave them zero)
  g_sk_partial = L.sk_partial;
  g_sk_counters = L.sk_counters;
  g_sk_cap = L.sk_cap;

  // row extent of the GEMM / attention operands: COMPACT buffers are padded
  // to whole 128-row tiles; a dense call reads the caller's M rows in place
  const long long in_rows = dense ? (long long)M : pad128(M);
  using bfp = __nv_bfloat16*;
  if (dense) {
    L.dout_k = bfp(dOut);
    L.b_k = llama ? bfp(sv->b) : nullptr;
    L.o_k = bfp(sv->o);
    L.a_k = bfp(sv->a);
    L.qkv_k = bfp(sv->qkv);
    if (llama) L.s_k = bfp(sv->s);
  }
  // the attention's arguments (its preparation runs ahead on the side stream)
  AttnArgs attn{};
  attn.B = d->B; attn.T = d->T; attn.H = H; attn.Hkv = Hkv; attn.dh = dh; attn.causal = 1;
  attn.scale = 1.0f / sqrtf((float)dh);
  attn.rotary_dim = d->rotary_dim; attn.rope_base = d->rope_base;
  attn.q = L.qkv_k; attn.k = L.qkv_k + Hd; attn.v = L.qkv_k + Hd + Hkv * dh; attn.dO = L.do_k;
  attn.q_ld = Nqkv; attn.kv_ld = Nqkv; attn.do_ld = Hd;
  attn.lse = sv->lse; attn.idx = idx; attn.cu_kept = cu_kept; attn.n_kept = n_kept;
  attn.dq = L.dqkv_k; attn.dk = L.dqkv_k + Hd; attn.dv = L.dqkv_k + Hd + Hkv * dh;
  attn.dq_ld = Nqkv; attn.dkv_ld = Nqkv;
  attn.dq_acc = L.at.dq_acc; attn.Dvec = L.at.Dvec; attn.lse_k = L.at.lse2; attn.rope = L.at.rope; attn.M = M;
  attn.dk_acc = L.at.dk_acc; attn.dv_acc = L.at.dv_acc; attn.order = L.at.order; attn.in_cap = in_rows;
  attn.cap = pad128(M);

  // 1. gather the kept rows of dOut and of the saved GEMM operands.  The
  // input-gradient chain starts from dOut alone: qkv is first needed by the
  // attention, and s, b, o and a feed only the weight-gradient GEMMs, so
  // these are gathered on the side stream, beside the chain (qkv first; the
  // chain waits for it before the attention).
  if (!dense) {
    GatherJob j{static_cast<const char*>(dOut), reinterpret_cast<char*>(L.dout_k), (long long)D * 2,
                (long long)D * 2, D * 2, 0};
    // a COMPACT dOut is copied with its zero padding
    CK(launch_gather(c, &j, 1, M, pad128(M), dout_full ? idx : nullptr, n_kept));
    // from here on each of the chain's kernels follows a kernel of this
    // library, so it is launched with programmatic stream serialisation
    c.pdl = pdl_allowed();
  }
  CK(fork_side(c, side, 0));   // the side stream starts once dOut's kept rows exist
  if (!dense) {
    GatherJob j{static_cast<const char*>(sv->qkv), reinterpret_cast<char*>(L.qkv_k), (long long)Nqkv * 2,
                (long long)Nqkv * 2, Nqkv * 2, 0};
    CK(launch_gather(cs, &j, 1, M, pad128(M), idx, n_kept));
  }
  if (side) {
    AttnArgs prep = attn;
    prep.stage = 1;
    CK(launch_attn_bwd(cs, prep));
    CK(cudaEventRecord(side->ev[6], cs.stream));
  }
  if (!dense) {
    // FULL dx: its filtered rows are zero; the norm backward at the end of
    // the chain writes the kept rows in place
    if (dx_full)
      CK(launch_scatter(cs, nullptr, 0, static_cast<char*>(g->dx), (long long)D * 2, D * 2, M, idx, n_kept));
  }
  {
    GatherJob j[4];
    int n = 0;
    if (llama) {
      // (a saved set without s or b: the SwiGLU and norm2 backward recompute them below)
      if (!dense && sv->s)
        j[n++] = GatherJob{static_cast<const char*>(sv->s), reinterpret_cast<char*>(L.s_k), (long long)F * 2,
                           (long long)F * 2, F * 2, 0};
      if (!dense && sv->b)
        j[n++] = GatherJob{static_cast<const char*>(sv->b), reinterpret_cast<char*>(L.b_k), (long long)D * 2,
                           (long long)D * 2, D * 2, 0};
    } else {
      // gelu(f1) of the kept rows (of every row for a dense call: then not a gather)
      j[n++] = GatherJob{static_cast<const char*>(sv->up), reinterpret_cast<char*>(L.s_k), (long long)F * 2,
                         (long long)F * 2, F * 2, 1};
    }
    if (!dense) {
      j[n++] = GatherJob{static_cast<const char*>(sv->o), reinterpret_cast<char*>(L.o_k), (long long)Hd * 2,
                         (long long)Hd * 2, Hd * 2, 0};
      if (sv->a) {
        j[n++] = GatherJob{static_cast<const char*>(sv->a), reinterpret_cast<char*>(L.a_k), (long long)D * 2,
                           (long long)D * 2, D * 2, 0};
      } else {   // RMSNorm: a = norm1(x), recomputed from x, rstd1 and norm1_w
        j[n++] = GatherJob{static_cast<const char*>(sv->x), reinterpret_cast<char*>(L.a_k), (long long)D * 2,
                           (long long)D * 2, D * 2, 2, sv->rstd1, static_cast<const __nv_bfloat16*>(w->norm1_w)};
      }
    }
    if (n) CK(launch_gather(cs, j, n, M, pad128(M), dense ? nullptr : idx, n_kept));
  }

  // 2. MLP
  const __nv_bfloat16* dres = L.dout_k;   // gradient flowing along the residual into the attention half
  if (llama) {
    // s_k and b_k come from the gathers above, or are recomputed by the
    // SwiGLU backward and the norm2 row pass (saved set without s, b); the
    // weight-gradient GEMMs that read them wait for those kernels then
    const bool s_re = !dense && !sv->s, b_re = !dense && !sv->b;
    if (!s_re) CK(gemm_dw(cs, M, F, D, L.s_k, F, L.dout_k, D, g->dw_down, n_kept, in_rows));   // dW_down = s^T dOut
    CK(gemm_dx(c, M, F, D, L.dout_k, w->w_down, L.ds_k, 1, 0, n_kept, in_rows));      // ds = dOut W_down^T
    c.pdl = pdl_allowed();
    CK(launch_swiglu_bwd(c, L.ds_k, 1, F, static_cast<const __nv_bfloat16*>(sv->up), L.dgu_k, M, pad128(M), idx,
                         n_kept, s_re ? L.s_k : nullptr));
    CK(fork_side(c, side, 1));
    if (s_re) CK(gemm_dw(cs, M, F, D, L.s_k, F, L.dout_k, D, g->dw_down, n_kept, in_rows));
    if (!b_re) CK(gemm_dw(cs, M, D, Nup, L.b_k, D, L.dgu_k, Nup, g->dw_up, n_kept, in_rows));  // dW_up = b^T dgu
    CK(gemm_dx(c, M, D, Nup, L.dgu_k, w->w_up, L.db_k, 0, 0, n_kept));                // db = dgu W_up^T
    NormBwdArgs nb{};
    nb.layer_norm = 0; nb.M = M; nb.D = D;
    nb.dy1 = L.db_k; nb.res = L.dout_k; nb.res_ld = D;
    nb.x = static_cast<const __nv_bfloat16*>(sv->h); nb.rstd = sv->rstd2;
    nb.gamma = static_cast<const __nv_bfloat16*>(w->norm2_w);
    nb.out = L.dh_k; nb.cap = pad128(M); nb.dgamma = g->dnorm2_w; nb.part = L.norm_part2; nb.idx = idx; nb.n_kept = n_kept;
    nb.xn_out = b_re ? L.b_k : nullptr;   // b = norm2(h), recomputed
    // the column pass needs only what the row pass reads, so it is forked
    // before it and the two run side by side
    CK(fork_side(c, side, 7));
    CK(launch_norm_rows(c, nb));                                                         // dh = dOut + norm2'
    CK(launch_norm_cols(cs, nb));                                                        // dnorm2_w, beside the chain
    if (b_re) {
      CK(fork_side(c, side, 11));
      CK(gemm_dw(cs, M, D, Nup, L.b_k, D, L.dgu_k, Nup, g->dw_up, n_kept, in_rows));
    }
    dres = L.dh_k;
  } else {
    CK(gemm_dw(cs, M, F, D, L.s_k, F, L.dout_k, D, g->dw_down, n_kept, in_rows));     // dW2 = gelu(f1)^T dOut
    CK(gemm_dx(c, M, F, D, L.dout_k, w->w_down, L.ds_k, 1, 0, n_kept, in_rows));      // df2 = dOut W2^T
    c.pdl = pdl_allowed();
    if (d->mlp_bias && g->db_down)
      CK(launch_colsum(c, L.dout_k, 1, D, M, D, nullptr, n_kept, L.col_part, g->db_down));
    CK(launch_gelu_bwd(c, L.ds_k, 1, F, static_cast<const __nv_bfloat16*>(sv->up), L.dgu_k, M, pad128(M), idx,
                       n_kept));
    CK(fork_side(c, side, 1));
    CK(gemm_dw(cs, M, D, F, L.a_k, D, L.dgu_k, F, g->dw_up, n_kept, in_rows));        // dW1 = a^T df1
    if (d->mlp_bias && g->db_up)
      CK(launch_colsum(c, L.dgu_k, 1, F, M, F, nullptr, n_kept, L.col_part, g->db_up));
    CK(gemm_dx(c, M, D, F, L.dgu_k, w->w_up, L.da_k, 0, 0, n_kept));                  // da = df1 W1^T
  }

  // 3. attention output projection
  CK(fork_side(c, side, 2));
  CK(gemm_dw(cs, M, Hd, D, L.o_k, Hd, dres, D, g->dw_o, n_kept, in_rows));            // dW_o = o^T dh
  CK(gemm_dx(c, M, Hd, D, dres, w->w_o, L.do_k, 1, 0, n_kept, in_rows));              // do = dh W_o^T
  if (d->out_bias && g->db_o) CK(launch_colsum(c, dres, 1, D, M, D, nullptr, n_kept, L.col_part, g->db_o));

  // 4. filtered attention backward (+ RoPE backward) straight into dqkv_k
  {
    Ctx ca = c;
    if (side) {
      CK(cudaStreamWaitEvent(c.stream, side->ev[6], 0));   // qkv's kept rows, the attention's preparation
      attn.stage = 2;
      ca.pdl = false;   // its first kernel follows the wait, not a kernel
    }
    CK(launch_attn_bwd(ca, attn));
  }

  // 5. QKV projection
  CK(fork_side(c, side, 3));
  CK(gemm_dw(cs, M, D, Nqkv, L.a_k, D, L.dqkv_k, Nqkv, g->dw_qkv, n_kept, in_rows)); // dW_qkv = a^T dqkv
  if (d->qkv_bias && g->db_qkv)
    CK(launch_colsum(cs, L.dqkv_k, 1, Nqkv, M, Nqkv, nullptr, n_kept, L.col_part, g->db_qkv));
  CK(gemm_dx(c, M, D, Nqkv, L.dqkv_k, w->w_qkv, L.da_k, 0, llama ? 0 : 1, n_kept));  // da (+)= dqkv W_qkv^T

  // 6. input norm backward + residual, its rows written where they belong
  // (FULL dx: at idx, the filtered rows zeroed on the side stream above;
  // COMPACT dx, or a dense call, whose COMPACT rows are the FULL rows: in order)
  {
    NormBwdArgs nb{};
    nb.layer_norm = llama ? 0 : 1; nb.M = M; nb.D = D;
    nb.dy1 = L.da_k; nb.res = dres; nb.res_ld = D;
    nb.x = static_cast<const __nv_bfloat16*>(sv->x); nb.mean = sv->mean1; nb.rstd = sv->rstd1;
    nb.gamma = static_cast<const __nv_bfloat16*>(w->norm1_w);
    nb.out = static_cast<__nv_bfloat16*>(g->dx); nb.cap = M; nb.out_full = (dx_full && !dense) ? 1 : 0;
    nb.dgamma = g->dnorm1_w; nb.dbeta = g->dnorm1_b; nb.part = L.norm_part;
    nb.idx = idx; nb.n_kept = n_kept;
    CK(fork_side(c, side, 10));   // (the column pass needs only what the row pass reads)
    CK(launch_norm_rows(c, nb));
    CK(launch_norm_cols(cs, nb));   // dnorm1_w (dnorm1_b), beside the chain
  }
  CK(join_side(c, side, 4));   // the weight gradients are done when the chain is
  if (side) CK(join_hi(c_in.stream, side));
  return COLLIDER_OK;
}

collider_status check_layer_ptrs(const collider_layer_desc* d, const collider_layer_weights* w,
                                 const collider_layer_saved* sv, const collider_layer_grads* g, bool need_dx) {
  if (!w || !sv || !g) return fail(COLLIDER_ERR_INVALID_ARG, "null weights/saved/grads struct");
  const bool llama = d->arch == COLLIDER_ARCH_LLAMA;
  const void* req[] = {w->norm1_w, w->w_qkv, w->w_o, w->w_up, w->w_down, sv->x, sv->rstd1, sv->qkv,
                       sv->o, sv->lse, sv->up, g->dnorm1_w, g->dw_qkv, g->dw_o, g->dw_up, g->dw_down};
  for (const void* p : req)
    if (!p) return fail(COLLIDER_ERR_INVALID_ARG, "a required weight/saved/gradient pointer is null");
  if (need_dx && !g->dx) return fail(COLLIDER_ERR_INVALID_ARG, "grads->dx is null");
  // (llama: a, b and s may be NULL -- recomputed -- except in a dense call, checked there)
  if (llama && (!w->norm2_w || !sv->h || !sv->rstd2 || !g->dnorm2_w))
    return fail(COLLIDER_ERR_INVALID_ARG, "llama block needs norm2_w, h, rstd2 and dnorm2_w");
  if (!llama && (!sv->a || !sv->mean1 || !g->dnorm1_b))
    return fail(COLLIDER_ERR_INVALID_ARG, "phi block needs a, mean1 and dnorm1_b");
  const void* al[] = {w->norm1_w, w->w_qkv, w->w_o, w->w_up, w->w_down, w->norm2_w, sv->x, sv->a, sv->qkv,
                      sv->o, sv->h, sv->b, sv->up, sv->s, g->dx, g->dw_qkv, g->dw_o, g->dw_up, g->dw_down,
                      g->dnorm1_w, g->dnorm1_b, g->dnorm2_w, g->db_qkv, g->db_o, g->db_up, g->db_down};
  for (const void* p : al)
    if (!al16(p)) return fail(COLLIDER_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  return COLLIDER_OK;
}

// Where the saved set and dOut live: device or managed memory, or pinned host
// memory that the device addresses at the same pointer (unified addressing).
// The filtered backward reads those inputs only with plain loads, at the kept
// rows (through idx), so from host memory only the kept rows cross the host
// link; the dense call hands whole tensors to TMA and needs device memory.
// Anything else (pageable host memory) is refused rather than read.  The
// weights (TMA operands) and the gradients must be device or managed memory.
collider_status check_input_memory(const collider_layer_weights* w, const collider_layer_saved* sv,
                                   const void* dOut, const collider_layer_grads* g, bool dense) {
  const void* ps[] = {sv->x, sv->a, sv->mean1, sv->rstd1, sv->qkv, sv->o, sv->lse, sv->h, sv->b,
                      sv->rstd2, sv->up, sv->s, dOut,
                      // from here on: device or managed memory only
                      w->norm1_w, w->w_qkv, w->w_o, w->norm2_w, w->w_up, w->w_down,
                      g->dx, g->dnorm1_w, g->dnorm1_b, g->dw_qkv, g->db_qkv, g->dw_o, g->db_o, g->dnorm2_w,
                      g->dw_up, g->db_up, g->dw_down, g->db_down};
  constexpr int kHostOk = 13;   // the saved set and dOut
  for (int i = 0; i < static_cast<int>(sizeof(ps) / sizeof(ps[0])); ++i) {
    const void* p = ps[i];
    if (!p) continue;
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
      cudaGetLastError();
      return fail(COLLIDER_ERR_INVALID_ARG, "collider_layer_bwd: a pointer the CUDA runtime does not know");
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) continue;
    if (i < kHostOk && a.type == cudaMemoryTypeHost && a.devicePointer == p) {
      if (dense)
        return fail(COLLIDER_ERR_INVALID_ARG, "collider_layer_bwd: the dense call needs its inputs in device memory");
      continue;
    }
    return fail(COLLIDER_ERR_INVALID_ARG,
                i < kHostOk ? "collider_layer_bwd: inputs must be device memory or pinned host memory the device "
                              "can address"
                            : "collider_layer_bwd: weights and gradients must be device memory");
  }
  return COLLIDER_OK;
}

}  // namespace

extern "C" size_t collider_layer_workspace_size(const collider_layer_desc* d) {
  if (check_desc(d) != COLLIDER_OK) return 0;
  Carver cv{nullptr, 0, 0, true};
  LayerBufs L;
  layer_carve(cv, d, &L);
  return cv.used;
}

extern "C" collider_status collider_layer_bwd(const collider_layer_desc* d, const collider_layer_weights* w,
                                              const collider_layer_saved* sv, const void* dOut,
                                              collider_rows dout_rows, const int32_t* idx, const int32_t* cu_kept,
                                              const int32_t* n_kept, const collider_layer_grads* g,
                                              collider_rows dx_rows, void* ws, size_t ws_bytes, void* stream) {
  collider_status s = check_desc(d);
  if (s != COLLIDER_OK) return s;
  const bool dense = !idx && !cu_kept && !n_kept;   // every token kept: the unfiltered dense backward
  if (!dOut || !al16(dOut) || (!dense && (!idx || !cu_kept || !n_kept)))
    return fail(COLLIDER_ERR_INVALID_ARG,
                "collider_layer_bwd: null or misaligned dOut, or only some of idx/cu_kept/n_kept given");
  s = check_layer_ptrs(d, w, sv, g, true);
  if (s != COLLIDER_OK) return s;
  if (dense && d->arch == COLLIDER_ARCH_LLAMA && (!sv->a || !sv->b || !sv->s))
    return fail(COLLIDER_ERR_INVALID_ARG, "collider_layer_bwd: the dense call reads a, b and s in place: none may be NULL");
  const size_t need = collider_layer_workspace_size(d);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255))
    return fail(COLLIDER_ERR_INVALID_ARG, "collider_layer_bwd: needs %zu bytes of 256-aligned workspace", need);
  Ctx c;
  s = make_ctx(stream, &c);
  if (s != COLLIDER_OK) return s;
  s = check_input_memory(w, sv, dOut, g, dense);
  if (s != COLLIDER_OK) return s;
  Carver cv{static_cast<char*>(ws), ws_bytes, 0, false};
  LayerBufs L;
  layer_carve(cv, d, &L);
  // stream-K counters start at zero (every GEMM leaves them zero); zeroed here,
  // on the caller's stream, before any work of this call is forked off it
  CK(cudaMemsetAsync(L.sk_counters, 0, L.sk_cap * sizeof(int), c.stream));
  if (dense) {
    CK(launch_identity_index(c, d->B, d->T, L.id_idx, L.id_cu, L.id_nk));
    return layer_bwd_impl(c, d, w, sv, dOut, true, L.id_idx, L.id_cu, L.id_nk, g, true, L, true);
  }
  return layer_bwd_impl(c, d, w, sv, dOut, dout_rows == COLLIDER_ROWS_FULL, idx, cu_kept, n_kept, g,
                        dx_rows == COLLIDER_ROWS_FULL, L);
}

// ===========================================================================
// dense forward of one block
// ===========================================================================
namespace {

struct FwdBufs {
  float *qkv_acc, *attn_acc, *up_acc, *mlp_acc;   // f32 projection outputs [M, N]
  __nv_bfloat16* act;   // PHI: gelu(f1) [M, F]
  float* lse2;          // [H, M]
  float2* rope;         // [T, rotary_dim / 2]
  int32_t* cu;          // [B + 1]
};

void fwd_carve(Carver& cv, const collider_layer_desc* d, FwdBufs* f) {
  const size_t M = (size_t)d->B * d->T;
  const size_t D = d->D, F = d->F, Nqkv = (size_t)(d->H + 2 * d->Hkv) * d->dh;
  const bool llama = d->arch == COLLIDER_ARCH_LLAMA;
  f->qkv_acc = cv.take<float>(M * Nqkv);
  f->attn_acc = cv.take<float>(M * D);
  f->up_acc = llama ? nullptr : cv.take<float>(M * F);   // LLAMA's GEMM writes the saved bf16 up itself
  f->mlp_acc = cv.take<float>(M * D);
  f->act = llama ? nullptr : cv.take<__nv_bfloat16>(M * F);
  f->lse2 = cv.take<float>(M * d->H);
  f->rope = cv.take<float2>((size_t)d->T * (d->rotary_dim > 0 ? d->rotary_dim / 2 : 1));
  f->cu = cv.take<int32_t>((size_t)d->B + 1);
}

// C [M, N] = A [M, K] . W with W stored [K, N] (the MN-major B operand); C is
// f32, or bf16 (rounded once, in the epilogue) when c_bf16
cudaError_t gemm_fwd(const Ctx& c, int M, int K, int N, const void* A, const void* W, void* C, int c_bf16 = 0) {
  TcGemm g{};
  g.M = M; g.N = N; g.K = K;
  g.A = A; g.lda = K; g.a_mn_major = 0; g.a_rows = M;
  g.B = W; g.ldb = N; g.b_mn_major = 1; g.b_rows = K;
  g.C = C; g.ldc = N; g.c_bf16 = c_bf16; g.c_rows = M;
  return launch_tc_gemm(c, g);
}

collider_status layer_fwd_impl(const Ctx& c, const collider_layer_desc* d, const collider_layer_params* w,
                               const void* x_, void* y_, const collider_layer_acts* ac, FwdBufs& F) {
  using bf = __nv_bfloat16;
  const int M = d->B * d->T;
  const int D = d->D, Ff = d->F, H = d->H, Hkv = d->Hkv, dh = d->dh;
  const int Hd = H * dh, Nqkv = (H + 2 * Hkv) * dh;
  const bool llama = d->arch == COLLIDER_ARCH_LLAMA;
  const bf* x = static_cast<const bf*>(x_);
  auto B16 = [](const void* p) { return static_cast<const bf*>(p); };
  const bf* b_qkv = d->qkv_bias ? B16(w->b_qkv) : nullptr;
  const bf* b_o = d->out_bias ? B16(w->b_o) : nullptr;
  const bf* b_up = (!llama && d->mlp_bias) ? B16(w->b_up) : nullptr;
  const bf* b_down = (!llama && d->mlp_bias) ? B16(w->b_down) : nullptr;
  bf* a = static_cast<bf*>(ac->a);
  bf* qkv = static_cast<bf*>(ac->qkv);
  bf* o = static_cast<bf*>(ac->o);

  // 1. input norm
  NormFwdArgs n1{};
  n1.layer_norm = llama ? 0 : 1; n1.M = M; n1.D = D; n1.eps = d->eps; n1.x = x;
  n1.gamma = B16(w->norm1_w); n1.beta = llama ? nullptr : B16(w->norm1_b);
  n1.out = a; n1.mean = llama ? nullptr : ac->mean1; n1.rstd = ac->rstd1;
  CK(launch_norm_fwd(c, n1));
  // 2. QKV projection, bias and RoPE (without a bias the GEMM rounds to bf16 itself)
  const int qkv16 = b_qkv ? 0 : 1;
  CK(gemm_fwd(c, M, D, Nqkv, a, w->w_qkv, F.qkv_acc, qkv16));
  const int rot_half = d->rotary_dim / 2;
  CK(launch_rope_table(c, d->T, rot_half, d->rope_base, F.rope));
  CK(launch_qkv_rope_fwd(c, M, Nqkv, H + Hkv, dh, rot_half, d->T, F.qkv_acc, qkv16, b_qkv, F.rope, qkv));
  // 3. causal attention over every sequence
  CK(launch_iota_cu(c, d->B, d->T, F.cu));
  {
    AttnFwdArgs at{};
    at.B = d->B; at.T = d->T; at.H = H; at.Hkv = Hkv; at.dh = dh; at.scale = 1.0f / sqrtf((float)dh);
    at.q = qkv; at.k = qkv + Hd; at.v = qkv + Hd + Hkv * dh; at.q_ld = Nqkv; at.kv_ld = Nqkv;
    at.o = o; at.o_ld = Hd; at.lse = ac->lse; at.lse2 = F.lse2; at.cu = F.cu; at.M = M;
    CK(launch_attn_fwd(c, at));
  }
  // 4. output projection, then the MLP
  CK(gemm_fwd(c, M, Hd, D, o, w->w_o, F.attn_acc));
  bf* y = static_cast<bf*>(y_);
  if (llama) {
    NormFwdArgs n2{};
    n2.layer_norm = 0; n2.M = M; n2.D = D; n2.eps = d->eps; n2.x = x;
    n2.add = F.attn_acc; n2.add_ld = D; n2.add_bias = b_o; n2.sum_out = static_cast<bf*>(ac->h);
    n2.gamma = B16(w->norm2_w); n2.out = static_cast<bf*>(ac->b); n2.rstd = ac->rstd2;
    CK(launch_norm_fwd(c, n2));                                                    // h = x + attn, b = norm2(h)
    CK(gemm_fwd(c, M, D, 2 * Ff, ac->b, w->w_up, ac->up, 1));                       // [g | u] = b W_up (bf16)
    CK(launch_swiglu_fwd(c, M, Ff, static_cast<const bf*>(ac->up), static_cast<bf*>(ac->s)));
    CK(gemm_fwd(c, M, Ff, D, ac->s, w->w_down, F.mlp_acc));                         // s W_down
    CK(launch_residual_out(c, M, D, static_cast<const bf*>(ac->h), F.mlp_acc, nullptr, nullptr, nullptr, y));
  } else {
    CK(gemm_fwd(c, M, D, Ff, a, w->w_up, F.up_acc));                                // f1 = a W1 (+ b1)
    CK(launch_act_fwd(c, 1, M, Ff, F.up_acc, b_up, static_cast<bf*>(ac->up), F.act));
    CK(gemm_fwd(c, M, Ff, D, F.act, w->w_down, F.mlp_acc));                         // gelu(f1) W2
    CK(launch_residual_out(c, M, D, x, F.attn_acc, b_o, F.mlp_acc, b_down, y));
  }
  return COLLIDER_OK;
}

collider_status check_fwd_ptrs(const collider_layer_desc* d, const collider_layer_params* w, const void* x,
                               const void* y, const collider_layer_acts* ac) {
  if (!w || !ac || !x || !y) return fail(COLLIDER_ERR_INVALID_ARG, "null params/acts/x/y");
  if (x == y) return fail(COLLIDER_ERR_INVALID_ARG, "y must not alias x (x is part of the saved set)");
  const bool llama = d->arch == COLLIDER_ARCH_LLAMA;
  const void* req[] = {w->norm1_w, w->w_qkv, w->w_o, w->w_up, w->w_down, ac->a, ac->rstd1, ac->qkv, ac->o,
                       ac->lse, ac->up};
  for (const void* p : req)
    if (!p) return fail(COLLIDER_ERR_INVALID_ARG, "a required parameter or saved-set pointer is null");
  if (llama && (!w->norm2_w || !ac->h || !ac->b || !ac->rstd2 || !ac->s))
    return fail(COLLIDER_ERR_INVALID_ARG, "llama block needs norm2_w, h, b, rstd2 and s");
  if (!llama && (!w->norm1_b || !ac->mean1))
    return fail(COLLIDER_ERR_INVALID_ARG, "phi block needs norm1_b and mean1");
  if ((d->qkv_bias && !w->b_qkv) || (d->out_bias && !w->b_o) || (!llama && d->mlp_bias && (!w->b_up || !w->b_down)))
    return fail(COLLIDER_ERR_INVALID_ARG, "a bias the desc asks for is null");
  const void* al[] = {x, y, w->norm1_w, w->norm1_b, w->w_qkv, w->b_qkv, w->w_o, w->b_o, w->norm2_w, w->w_up,
                      w->b_up, w->w_down, w->b_down, ac->a, ac->qkv, ac->o, ac->h, ac->b, ac->up, ac->s};
  for (const void* p : al)
    if (!al16(p)) return fail(COLLIDER_ERR_INVALID_ARG, "pointers must be 16-byte aligned");
  return COLLIDER_OK;
}

}  // namespace

extern "C" size_t collider_layer_fwd_workspace_size(const collider_layer_desc* d) {
  if (check_desc(d) != COLLIDER_OK) return 0;
  Carver cv{nullptr, 0, 0, true};
  FwdBufs f;
  fwd_carve(cv, d, &f);
  return cv.used;
}

extern "C" collider_status collider_layer_fwd(const collider_layer_desc* d, const collider_layer_params* w,
                                              const void* x, void* y, const collider_layer_acts* acts, void* ws,
                                              size_t ws_bytes, void* stream) {
  collider_status s = check_desc(d);
  if (s != COLLIDER_OK) return s;
  s = check_fwd_ptrs(d, w, x, y, acts);
  if (s != COLLIDER_OK) return s;
  const size_t need = collider_layer_fwd_workspace_size(d);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255))
    return fail(COLLIDER_ERR_INVALID_ARG, "collider_layer_fwd: needs %zu bytes of 256-aligned workspace", need);
  Ctx c;
  s = make_ctx(stream, &c);
  if (s != COLLIDER_OK) return s;
  Carver cv{static_cast<char*>(ws), ws_bytes, 0, false};
  FwdBufs f;
  fwd_carve(cv, d, &f);
  return layer_fwd_impl(c, d, w, x, y, acts, f);
}

// ===========================================================================
// whole stack
// ===========================================================================
namespace {
struct StackBufs {
  __nv_bfloat16 *dz_k, *y_k, *dy_k, *dxa, *dxb;
  float* dyf_k;
  float* part;
};
void stack_carve(Carver& cv, const collider_layer_desc* d, int V, StackBufs* S) {
  const size_t Mp = pad128((long long)d->B * d->T);
  S->dz_k = cv.take<__nv_bfloat16>(Mp * V);
  S->y_k = cv.take<__nv_bfloat16>(Mp * d->D);
  S->dyf_k = cv.take<float>(Mp * d->D);
  S->dy_k = nullptr;
  S->dxa = cv.take<__nv_bfloat16>(Mp * d->D);
  S->dxb = cv.take<__nv_bfloat16>(Mp * d->D);
  S->part = cv.take<float>(norm_part_floats((int)Mp, d->D));
}
}  // namespace

extern "C" size_t collider_stack_workspace_size(const collider_layer_desc* d, int L, int V) {
  if (check_desc(d) != COLLIDER_OK || L < 1 || V < 8) return 0;
  Carver cv{nullptr, 0, 0, true};
  StackBufs S;
  stack_carve(cv, d, V, &S);
  LayerBufs LB;
  layer_carve(cv, d, &LB);
  return cv.used;
}

extern "C" collider_status collider_stack_bwd(const collider_layer_desc* d, int nL, int V,
                                              const collider_layer_weights* w, const collider_layer_saved* sv,
                                              const void* logits, const int32_t* targets, const int32_t* ids,
                                              const void* y, const void* xL, const float* rstdf, const void* normf_w,
                                              const void* w_lm, const int32_t* idx, const int32_t* cu_kept,
                                              const int32_t* n_kept, const collider_layer_grads* grads,
                                              float* dnormf_w, float* dw_lm, float* dE, void* ws, size_t ws_bytes,
                                              void* stream) {
  collider_status s = check_desc(d);
  if (s != COLLIDER_OK) return s;
  if (d->arch != COLLIDER_ARCH_LLAMA) return fail(COLLIDER_ERR_UNSUPPORTED, "collider_stack_bwd: llama blocks only");
  if (nL < 1 || V < 8 || V % 8) return fail(COLLIDER_ERR_INVALID_ARG, "collider_stack_bwd: L >= 1, V % 8 == 0");
  if (d->D > 2048) return fail(COLLIDER_ERR_UNSUPPORTED, "collider_stack_bwd: D <= 2048");
  const bool dense = !idx && !cu_kept && !n_kept;   // every token kept: the unfiltered dense backward
  if (!w || !sv || !grads || !logits || !targets || !ids || !y || !xL || !rstdf || !normf_w || !w_lm ||
      (!dense && (!idx || !cu_kept || !n_kept)) || !dnormf_w || !dw_lm || !dE)
    return fail(COLLIDER_ERR_INVALID_ARG, "collider_stack_bwd: null pointer");
  if (!al16(logits) || !al16(y) || !al16(xL) || !al16(normf_w) || !al16(w_lm) || !al16(dnormf_w) || !al16(dw_lm) ||
      !al16(dE))
    return fail(COLLIDER_ERR_INVALID_ARG, "collider_stack_bwd: pointers must be 16-byte aligned");
  for (int l = 0; l < nL; ++l) {
    s = check_layer_ptrs(d, &w[l], &sv[l], &grads[l], false);
    if (s != COLLIDER_OK) return s;
    if (dense && (!sv[l].a || !sv[l].b || !sv[l].s))
      return fail(COLLIDER_ERR_INVALID_ARG, "collider_stack_bwd: the dense call reads a, b and s in place: none may be NULL");
  }
  const size_t need = collider_stack_workspace_size(d, nL, V);
  if (!ws || ws_bytes < need || (reinterpret_cast<uintptr_t>(ws) & 255))
    return fail(COLLIDER_ERR_INVALID_ARG, "collider_stack_bwd: needs %zu bytes of 256-aligned workspace", need);
  Ctx c;
  s = make_ctx(stream, &c);
  if (s != COLLIDER_OK) return s;
  Carver cv{static_cast<char*>(ws), ws_bytes, 0, false};
  StackBufs S;
  stack_carve(cv, d, V, &S);
  LayerBufs LB;
  layer_carve(cv, d, &LB);
  const int M = d->B * d->T, D = d->D;
  g_sk_partial = LB.sk_partial;
  g_sk_counters = LB.sk_counters;
  g_sk_cap = LB.sk_cap;
  CK(cudaMemsetAsync(LB.sk_counters, 0, LB.sk_cap * sizeof(int), c.stream));
  if (dense) {
    CK(launch_identity_index(c, d->B, d->T, LB.id_idx, LB.id_cu, LB.id_nk));
    idx = LB.id_idx;
    cu_kept = LB.id_cu;
    n_kept = LB.id_nk;
  }

  // LM head: dz = (softmax(z) - onehot) / n_kept on kept rows
  CK(launch_ce_bwd(c, static_cast<const __nv_bfloat16*>(logits), targets, V, M, pad128(M), idx, n_kept, S.dz_k));
  const __nv_bfloat16* yk = static_cast<const __nv_bfloat16*>(y);   // a dense call reads y in place
  if (!dense) {
    GatherJob j{static_cast<const char*>(y), reinterpret_cast<char*>(S.y_k), (long long)D * 2, (long long)D * 2,
                D * 2, 0};
    CK(launch_gather(c, &j, 1, M, pad128(M), idx, n_kept));
    yk = S.y_k;
  }
  {
    Ctx cs;
    Side* side = nullptr;
    s = side_ctx(c, &cs, &side);
    if (s != COLLIDER_OK) return s;
    CK(fork_side(c, side, 5));
    CK(gemm_dw(cs, M, D, V, yk, D, S.dz_k, V, dw_lm, n_kept,             // dW_lm = y^T dz (side stream;
               dense ? (long long)M : -1));                                // joined by the last block)
  }
  CK(gemm_dx(c, M, D, V, S.dz_k, w_lm, S.dyf_k, 0, 0, n_kept));           // dy = dz W_lm^T
  {
    NormBwdArgs nb{};
    nb.layer_norm = 0; nb.M = M; nb.D = D;
    nb.dy1 = S.dyf_k; nb.res = nullptr;
    nb.x = static_cast<const __nv_bfloat16*>(xL); nb.rstd = rstdf;
    nb.gamma = static_cast<const __nv_bfloat16*>(normf_w);
    nb.out = S.dxa; nb.cap = pad128(M); nb.dgamma = dnormf_w; nb.part = S.part; nb.idx = idx; nb.n_kept = n_kept;
    CK(launch_norm_bwd(c, nb));
  }
  // blocks, last to first, staying COMPACT between blocks
  __nv_bfloat16* cur = S.dxa;
  __nv_bfloat16* nxt = S.dxb;
  for (int l = nL - 1; l >= 0; --l) {
    collider_layer_grads gl = grads[l];
    gl.dx = nxt;
    s = layer_bwd_impl(c, d, &w[l], &sv[l], cur, false, idx, cu_kept, n_kept, &gl, false, LB, dense);
    if (s != COLLIDER_OK) return s;
    std::swap(cur, nxt);
  }
  // embedding gradient
  CK(cudaMemsetAsync(dE, 0, (size_t)V * D * sizeof(float), c.stream));
  CK(launch_embed_bwd(c, cur, D, D, ids, V, M, idx, n_kept, dE));
  return COLLIDER_OK;
}

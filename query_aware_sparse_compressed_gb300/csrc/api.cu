// C-ABI entry points of libqasc: argument validation, workspace layout and
// kernel launches.  See include/qasc.h for the contract of each call.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "common.cuh"
#include "internal.h"
#include "qasc.h"

#ifdef QASC_NVTX
#include <nvtx3/nvToolsExt.h>
#endif

namespace {

// Built with -DQASC_NVTX, every call that enqueues work is one NVTX range
// named after the entry point (host side: validation and launches), so a
// timeline shows which library call issued which kernels.  Without the flag
// the macro is empty.
#ifdef QASC_NVTX
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};
#define QASC_RANGE(name) const CallRange qasc_call_range_(name)
#else
#define QASC_RANGE(name) static_cast<void>(0)
#endif

thread_local std::string g_last_error;

// Kernels record device-side failures (a bounded wait that ran out) here.
__device__ unsigned int g_device_error_word;

qasc_status fail(qasc_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
qasc_status fail(qasc_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

qasc_status ok() {
  g_last_error.clear();
  return QASC_OK;
}

qasc_status cuda_fail(int rc, const char* where) {
  if (rc < 0) return fail(QASC_ERR_UNSUPPORTED, "%s: configuration not compiled in", where);
  const cudaError_t e = static_cast<cudaError_t>(rc);
  return fail(QASC_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool group_supported(int gq) { return gq == 1 || gq == 2 || gq == 4 || gq == 8; }

qasc_status check_shape(const qasc_shape* s, const char* fn) {
  if (!s) return fail(QASC_ERR_INVALID_ARG, "%s: shape is NULL", fn);
  if (s->d != qasc::kHeadDim || s->d_idx != qasc::kIndexDim)
    return fail(QASC_ERR_UNSUPPORTED, "%s: only d=128, d_idx=32 are compiled in (got d=%d, d_idx=%d)", fn, s->d,
                s->d_idx);
  if (s->B < 1 || s->Hq < 1 || s->Hkv < 1)
    return fail(QASC_ERR_INVALID_ARG, "%s: B, Hq, Hkv must be >= 1 (got %d, %d, %d)", fn, s->B, s->Hq, s->Hkv);
  if (s->Hq % s->Hkv != 0)
    return fail(QASC_ERR_INVALID_ARG, "%s: Hq=%d is not a multiple of Hkv=%d", fn, s->Hq, s->Hkv);
  if (s->Hq > 64) return fail(QASC_ERR_INVALID_ARG, "%s: Hq=%d exceeds 64", fn, s->Hq);
  if (!group_supported(s->Hq / s->Hkv))
    return fail(QASC_ERR_UNSUPPORTED, "%s: group size Hq/Hkv=%d not compiled in (1, 2, 4, 8)", fn,
                s->Hq / s->Hkv);
  if (s->n_cap < 1 || s->n_cap >= (int64_t(1) << 24))
    return fail(QASC_ERR_INVALID_ARG, "%s: n_cap=%lld outside [1, 2^24)", fn, static_cast<long long>(s->n_cap));
  if (s->n < 1 || s->n > s->n_cap)
    return fail(QASC_ERR_INVALID_ARG, "%s: n=%lld outside [1, n_cap=%lld]", fn, static_cast<long long>(s->n),
                static_cast<long long>(s->n_cap));
  if (static_cast<int64_t>(s->B) * s->Hkv > 65535)
    return fail(QASC_ERR_INVALID_ARG, "%s: B*Hkv=%lld exceeds 65535", fn,
                static_cast<long long>(s->B) * s->Hkv);
  if (static_cast<int64_t>(s->B) * s->Hkv * s->n_cap >= (int64_t(1) << 31))
    return fail(QASC_ERR_INVALID_ARG, "%s: B*Hkv*n_cap=%lld rows exceed 2^31", fn,
                static_cast<long long>(s->B) * s->Hkv * s->n_cap);
  return QASC_OK;
}

qasc_status check_ts_params(const qasc_shape* s, const qasc_ts_params* p, const char* fn) {
  if (!p) return fail(QASC_ERR_INVALID_ARG, "%s: params is NULL", fn);
  if (p->sink < 0 || p->local < 0)
    return fail(QASC_ERR_INVALID_ARG, "%s: sink=%d and local=%d must be >= 0", fn, p->sink, p->local);
  if (p->vmin < 1) return fail(QASC_ERR_INVALID_ARG, "%s: vmin=%d must be >= 1", fn, p->vmin);
  const qasc::Regions R = qasc::regions_of(s->n, p->sink, p->local);
  if (p->K < 0 || p->K > R.nc())
    return fail(QASC_ERR_INVALID_ARG, "%s: K=%d outside [0, |C|=%lld]", fn, p->K, static_cast<long long>(R.nc()));
  return QASC_OK;
}

// [start, start + count) within [0, cap), written so that no sum can overflow.
qasc_status check_rows(int64_t start, int64_t count, int64_t cap, const char* what, const char* fn) {
  if (start < 0 || count < 0 || start > cap || count > cap - start)
    return fail(QASC_ERR_INVALID_ARG, "%s: %s start=%lld count=%lld outside [0, n_cap=%lld)", fn, what,
                static_cast<long long>(start), static_cast<long long>(count), static_cast<long long>(cap));
  return QASC_OK;
}

qasc_status check_snap_params(const qasc_shape* s, const qasc_snap_params* p, const char* fn) {
  if (!p) return fail(QASC_ERR_INVALID_ARG, "%s: params is NULL", fn);
  if (p->c < 1) return fail(QASC_ERR_INVALID_ARG, "%s: c=%d must be >= 1", fn, p->c);
  if (p->pool_k < 1 || p->pool_k % 2 == 0)
    return fail(QASC_ERR_INVALID_ARG, "%s: pool_k=%d must be odd and >= 1", fn, p->pool_k);
  if (p->pool_k > 65) return fail(QASC_ERR_UNSUPPORTED, "%s: pool_k=%d exceeds the supported width 65", fn, p->pool_k);
  if (p->window < 1) return fail(QASC_ERR_INVALID_ARG, "%s: window=%d must be >= 1", fn, p->window);
  const int gq = s->Hq / s->Hkv;
  if (p->window > 128 / gq)  // Gq * window > 128, without forming the product
    return fail(QASC_ERR_UNSUPPORTED, "%s: Gq=%d times window=%d exceeds one 128-row tile", fn, gq, p->window);
  return QASC_OK;
}

#define QASC_CHECK(expr)               \
  do {                                 \
    const qasc_status st__ = (expr);   \
    if (st__ != QASC_OK) return st__;  \
  } while (0)

// A size query answers only for arguments its call accepts: otherwise it
// returns 0 and leaves the reason in qasc_last_error().
#define QASC_SIZE_CHECK(expr)              \
  do {                                     \
    if ((expr) != QASC_OK) return 0;       \
  } while (0)

#define QASC_REQUIRE_PTR(ptr, align, fn)                                                              \
  do {                                                                                                \
    if ((ptr) == nullptr) return fail(QASC_ERR_INVALID_ARG, "%s: %s is NULL", fn, #ptr);            \
    if (!aligned((ptr), (align)))                                                                     \
      return fail(QASC_ERR_INVALID_ARG, "%s: %s is not %d-byte aligned", fn, #ptr, int(align));     \
  } while (0)

const qasc::DeviceInfo* need_device(const char* fn, qasc_status* st) {
  const qasc::DeviceInfo* dev = qasc::device_info();
  if (!dev) {
    // Tell a device of another architecture apart from a missing or failing one.
    int d = -1, major = 0, minor = 0;
    const cudaError_t e = cudaGetDevice(&d);
    if (e == cudaSuccess && cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d) == cudaSuccess &&
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d) == cudaSuccess &&
        !(major == 10 && minor == 3)) {
      *st = fail(QASC_ERR_UNSUPPORTED, "%s: device %d is sm_%d%d; the library is built for sm_103a only", fn, d,
                 major, minor);
      return nullptr;
    }
    *st = fail(QASC_ERR_CUDA, "%s: no usable CUDA device (%s)", fn,
               cudaGetErrorString(e != cudaSuccess ? e : cudaGetLastError()));
    return nullptr;
  }
  *st = QASC_OK;
  return dev;
}

}  // namespace

namespace qasc {

const DeviceInfo* device_info() {
  static DeviceInfo infos[64];
  static bool ready[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!ready[dev]) {
    DeviceInfo& d = infos[dev];
    d.device = dev;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess) return nullptr;
    if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) return nullptr;
    if (major != 10 || minor != 3) return nullptr;  // built for sm_103a only
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
    if (cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return nullptr;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error_word) != cudaSuccess) return nullptr;
    d.err_word = static_cast<unsigned*>(p);
    if (configure_score_kernels(d) != cudaSuccess || configure_select_kernels(d) != cudaSuccess ||
        configure_head_select_kernels(d) != cudaSuccess || configure_group_kernels(d) != cudaSuccess ||
        configure_expand_kernels(d) != cudaSuccess ||
        configure_attn_kernels(d) != cudaSuccess || configure_snapkv_kernels(d) != cudaSuccess)
      return nullptr;
    ready[dev] = true;
  }
  return &infos[dev];
}

EncodeTiledFn encode_tiled_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

}  // namespace qasc

extern "C" {

QASC_API int32_t qasc_version(void) { return 100; }  // 0.1.0

QASC_API const char* qasc_status_string(qasc_status status) {
  switch (status) {
    case QASC_OK: return "QASC_OK";
    case QASC_ERR_INVALID_ARG: return "QASC_ERR_INVALID_ARG";
    case QASC_ERR_UNSUPPORTED: return "QASC_ERR_UNSUPPORTED";
    case QASC_ERR_WORKSPACE: return "QASC_ERR_WORKSPACE";
    case QASC_ERR_CUDA: return "QASC_ERR_CUDA";
    case QASC_ERR_TIMEOUT: return "QASC_ERR_TIMEOUT";
    case QASC_ERR_BAD_TABLE: return "QASC_ERR_BAD_TABLE";
    case QASC_ERR_INTERNAL: return "QASC_ERR_INTERNAL";
  }
  return "QASC_ERR_UNKNOWN";
}

QASC_API const char* qasc_last_error(void) { return g_last_error.c_str(); }

QASC_API const char* qasc_last_cuda_error(void) { return g_last_error.c_str(); }

QASC_API qasc_status qasc_device_error(void* stream) {
  static const char* fn = "qasc_device_error";
  qasc_status st;
  if (!need_device(fn, &st)) return st;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  unsigned word = 0;
  e = cudaMemcpyFromSymbol(&word, g_device_error_word, sizeof(word));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  if (word != 0) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_device_error_word, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, fn);
    if (word & qasc::kErrTimeout)
      return fail(QASC_ERR_TIMEOUT, "%s: a device-side wait ran out (error bits 0x%x)", fn, word);
    if (!(word & qasc::kErrBadPage))
      return fail(QASC_ERR_INTERNAL, "%s: a kernel met an index of its own outside its buffer (error bits 0x%x)", fn,
                  word);
    return fail(QASC_ERR_BAD_TABLE, "%s: a block-table entry lies outside the page pool (error bits 0x%x)", fn,
                word);
  }
  return ok();
}

namespace {
// One CTA waits on a barrier that nothing arrives on, with the same bounded
// wait every kernel of the library uses: the wait gives up after limit_ns,
// records the timeout in the device error word and the kernel returns.
__global__ void selftest_wait_kernel(unsigned* err, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    qasc::mbar_init(&bar, 1);
    qasc::fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !qasc::mbar_wait_for(&bar, 0, limit_ns)) qasc::record_error(err, qasc::kErrTimeout);
}
}  // namespace

QASC_API qasc_status qasc_selftest_bounded_wait(int32_t limit_us, void* stream) {
  static const char* fn = "qasc_selftest_bounded_wait";
  QASC_RANGE(fn);
  if (limit_us < 1 || limit_us > 2000000)
    return fail(QASC_ERR_INVALID_ARG, "%s: limit_us=%d must lie in [1, 2000000]", fn, limit_us);
  qasc_status st;
  const qasc::DeviceInfo* dev = need_device(fn, &st);
  if (!dev) return st;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      dev->err_word, static_cast<unsigned long long>(limit_us) * 1000ull);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

QASC_API qasc_status ts_index_append(const qasc_shape* shape, const uint16_t* K, const uint16_t* W, uint16_t* index,
                                     int64_t start, int64_t count, void* stream) {
  static const char* fn = "ts_index_append";
  QASC_RANGE(fn);
  QASC_CHECK(check_shape(shape, fn));
  QASC_CHECK(check_rows(start, count, shape->n_cap, "rows", fn));
  QASC_REQUIRE_PTR(K, 16, fn);
  QASC_REQUIRE_PTR(W, 16, fn);
  QASC_REQUIRE_PTR(index, 16, fn);
  if (count == 0) return ok();
  qasc_status st;
  if (!need_device(fn, &st)) return st;
  const cudaError_t e =
      qasc::launch_index_append(*shape, K, W, index, start, count, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

QASC_API size_t ts_select_workspace_bytes(const qasc_shape* shape, const qasc_ts_params* params) {
  static const char* fn = "ts_select_workspace_bytes";
  QASC_SIZE_CHECK(check_shape(shape, fn));
  QASC_SIZE_CHECK(check_ts_params(shape, params, fn));
  ok();
  return qasc::select_layout(*shape, *params).total;
}

namespace {
// The voting select over a contiguous index (pm == nullptr) or a paged pool.
qasc_status vote_select_call(const char* fn, const qasc_shape* shape, const qasc_ts_params* params,
                             const uint16_t* q, const uint16_t* W, const uint16_t* index, int32_t* sel,
                             void* workspace, size_t ws_bytes, void* stream, const qasc::PageMap* pm) {
  QASC_RANGE(fn);
  QASC_REQUIRE_PTR(q, 16, fn);
  QASC_REQUIRE_PTR(W, 16, fn);
  QASC_REQUIRE_PTR(index, 16, fn);
  if (params->K == 0) return ok();
  QASC_REQUIRE_PTR(sel, 16, fn);
  const qasc::SelectLayout L = qasc::select_layout(*shape, *params);
  if (!workspace || ws_bytes < L.total)
    return fail(QASC_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn, L.total,
                workspace ? ws_bytes : size_t(0));
  QASC_REQUIRE_PTR(workspace, 256, fn);
  qasc_status st;
  const qasc::DeviceInfo* dev = need_device(fn, &st);
  if (!dev) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const qasc::Regions R = qasc::regions_of(shape->n, params->sink, params->local);
  qasc::ScoreOut so;
  so.scores = reinterpret_cast<float*>(ws + L.off_scores);
  so.hist = reinterpret_cast<uint32_t*>(ws + L.off_hist);
  so.nc_pad = L.nc_pad;
  so.max_splits = qasc::score_grid(*shape, qasc::score_span(R, pm != nullptr), dev->num_sms).max_splits;
  if (pm) so.pm = *pm;
  int rc = qasc::launch_scores(*shape, *params, q, W, index, so, *dev, s);
  if (rc != 0) return cuda_fail(rc, fn);
  rc = qasc::launch_select(*shape, *params, L, ws, sel, *dev, s, pm != nullptr);
  if (rc != 0) return cuda_fail(rc, fn);
  return ok();
}
}  // namespace

QASC_API qasc_status ts_score_vote_select(const qasc_shape* shape, const qasc_ts_params* params, const uint16_t* q,
                                          const uint16_t* W, const uint16_t* index, int32_t* sel, void* workspace,
                                          size_t ws_bytes, void* stream) {
  static const char* fn = "ts_score_vote_select";
  QASC_CHECK(check_shape(shape, fn));
  QASC_CHECK(check_ts_params(shape, params, fn));
  return vote_select_call(fn, shape, params, q, W, index, sel, workspace, ws_bytes, stream, nullptr);
}

QASC_API size_t ts_attn_workspace_bytes(const qasc_shape* shape, const qasc_ts_params* params) {
  static const char* fn = "ts_attn_workspace_bytes";
  QASC_SIZE_CHECK(check_shape(shape, fn));
  QASC_SIZE_CHECK(check_ts_params(shape, params, fn));
  ok();
  // Sized for the largest split count any device would use.
  return qasc::attn_layout(*shape, *params, qasc::kMaxSmsForSizing).total;
}

namespace {
qasc_status sparse_attn_call(const char* fn, bool per_kv, const qasc_shape* shape, const qasc_ts_params* params,
                             const uint16_t* q, const uint16_t* K, const uint16_t* V, const int32_t* sel, float* out,
                             float* lse, void* workspace, size_t ws_bytes, void* stream,
                             const int32_t* sel_len = nullptr, const qasc::PageMap* pm = nullptr,
                             const qasc::RingMap* ring = nullptr) {
  QASC_RANGE(fn);
  if (!pm) {
    QASC_CHECK(check_shape(shape, fn));
    QASC_CHECK(check_ts_params(shape, params, fn));
  }
  QASC_REQUIRE_PTR(q, 16, fn);
  QASC_REQUIRE_PTR(K, 16, fn);
  QASC_REQUIRE_PTR(V, 16, fn);
  QASC_REQUIRE_PTR(out, 16, fn);
  if (params->K > 0) QASC_REQUIRE_PTR(sel, 4, fn);
  if (lse && !aligned(lse, 4)) return fail(QASC_ERR_INVALID_ARG, "%s: lse is not 4-byte aligned", fn);
  if (sel_len && !aligned(sel_len, 4)) return fail(QASC_ERR_INVALID_ARG, "%s: sel_len is not 4-byte aligned", fn);
  qasc_status st;
  const qasc::DeviceInfo* dev = need_device(fn, &st);
  if (!dev) return st;
  const qasc::AttnLayout L = qasc::attn_layout(*shape, *params, dev->num_sms);
  if (!workspace || ws_bytes < L.total)
    return fail(QASC_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn, L.total,
                workspace ? ws_bytes : size_t(0));
  QASC_REQUIRE_PTR(workspace, 256, fn);
  const int rc = qasc::launch_sparse_attn(*shape, *params, L, q, K, V, sel, out, lse,
                                          static_cast<uint8_t*>(workspace), *dev, static_cast<cudaStream_t>(stream),
                                          per_kv, params->K > 0 ? sel_len : nullptr, pm, ring);
  if (rc != 0) return cuda_fail(rc, fn);
  return ok();
}
}  // namespace

QASC_API qasc_status ts_sparse_attn(const qasc_shape* shape, const qasc_ts_params* params, const uint16_t* q,
                                    const uint16_t* K, const uint16_t* V, const int32_t* sel, float* out, float* lse,
                                    void* workspace, size_t ws_bytes, void* stream) {
  return sparse_attn_call("ts_sparse_attn", false, shape, params, q, K, V, sel, out, lse, workspace, ws_bytes,
                          stream);
}

QASC_API qasc_status ts_sparse_attn_per_head(const qasc_shape* shape, const qasc_ts_params* params,
                                             const uint16_t* q, const uint16_t* K, const uint16_t* V,
                                             const int32_t* sel, float* out, float* lse, void* workspace,
                                             size_t ws_bytes, void* stream) {
  return sparse_attn_call("ts_sparse_attn_per_head", true, shape, params, q, K, V, sel, out, lse, workspace,
                          ws_bytes, stream);
}

QASC_API qasc_status ts_sparse_attn_ex(const qasc_shape* shape, const qasc_ts_params* params, const uint16_t* q,
                                       const uint16_t* K, const uint16_t* V, const int32_t* sel,
                                       const int32_t* sel_len, int32_t sel_per_kv_head, float* out, float* lse,
                                       void* workspace, size_t ws_bytes, void* stream) {
  return sparse_attn_call("ts_sparse_attn_ex", sel_per_kv_head != 0, shape, params, q, K, V, sel, out, lse,
                          workspace, ws_bytes, stream, sel_len);
}

// ---------------------------------------------------------------- paged cache
namespace {
qasc_status check_paged(const qasc_shape* shape, const qasc_paged_cache* cache, const char* fn, qasc::PageMap* m) {
  QASC_CHECK(check_shape(shape, fn));
  if (!cache) return fail(QASC_ERR_INVALID_ARG, "%s: cache is NULL", fn);
  const int64_t P = cache->page_tokens;
  if (P < 64 || P > 65536 || (P & (P - 1)) != 0)
    return fail(QASC_ERR_INVALID_ARG, "%s: page_tokens=%lld must be a power of two in [64, 65536]", fn,
                static_cast<long long>(P));
  if (cache->pages_per_seq < 1 || cache->num_pages < 1)
    return fail(QASC_ERR_INVALID_ARG, "%s: pages_per_seq=%d and num_pages=%lld must be >= 1", fn,
                cache->pages_per_seq, static_cast<long long>(cache->num_pages));
  if (shape->n_cap != static_cast<int64_t>(cache->pages_per_seq) * P)
    return fail(QASC_ERR_INVALID_ARG, "%s: n_cap=%lld must equal pages_per_seq * page_tokens = %lld", fn,
                static_cast<long long>(shape->n_cap), static_cast<long long>(cache->pages_per_seq * P));
  const int64_t rows_per_page = static_cast<int64_t>(shape->Hkv) * P;  // <= 64 * 2^16
  if (cache->num_pages > (int64_t(1) << 31) / rows_per_page || cache->num_pages * rows_per_page >= (int64_t(1) << 31))
    return fail(QASC_ERR_INVALID_ARG, "%s: num_pages=%lld times Hkv*page_tokens=%lld rows reaches 2^31", fn,
                static_cast<long long>(cache->num_pages), static_cast<long long>(rows_per_page));
  QASC_REQUIRE_PTR(cache->block_table, 4, fn);
  m->table = cache->block_table;
  m->pages_per_seq = cache->pages_per_seq;
  m->num_pages = cache->num_pages;
  int sh = 0;
  while ((int64_t(1) << sh) < P) ++sh;
  m->page_shift = sh;
  return QASC_OK;
}

qasc_status check_ring(const qasc_local_ring* ring, int64_t min_slots, const char* fn, qasc::RingMap* r) {
  if (!ring) return fail(QASC_ERR_INVALID_ARG, "%s: ring is NULL", fn);
  QASC_REQUIRE_PTR(ring->K, 16, fn);
  QASC_REQUIRE_PTR(ring->V, 16, fn);
  if (ring->ring_tokens < 1 || ring->ring_tokens > (1 << 24) || ring->ring_tokens < min_slots)
    return fail(QASC_ERR_INVALID_ARG, "%s: ring_tokens=%d must lie in [max(1, %lld), 2^24]", fn, ring->ring_tokens,
                static_cast<long long>(min_slots));
  r->K = ring->K;
  r->V = ring->V;
  r->R = ring->ring_tokens;
  return QASC_OK;
}
}  // namespace

QASC_API qasc_status ts_index_append_paged(const qasc_shape* shape, const qasc_paged_cache* cache,
                                           const uint16_t* K_pool, const uint16_t* W, uint16_t* index_pool,
                                           int64_t start, int64_t count, void* stream) {
  static const char* fn = "ts_index_append_paged";
  QASC_RANGE(fn);
  qasc::PageMap pm;
  QASC_CHECK(check_paged(shape, cache, fn, &pm));
  QASC_CHECK(check_rows(start, count, shape->n_cap, "tokens", fn));
  QASC_REQUIRE_PTR(K_pool, 16, fn);
  QASC_REQUIRE_PTR(W, 16, fn);
  QASC_REQUIRE_PTR(index_pool, 16, fn);
  if (count == 0) return ok();
  qasc_status st;
  const qasc::DeviceInfo* dev = need_device(fn, &st);
  if (!dev) return st;
  const cudaError_t e = qasc::launch_index_append_paged(*shape, pm, K_pool, W, index_pool, start, count,
                                                        dev->err_word, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

QASC_API qasc_status ts_score_vote_select_paged(const qasc_shape* shape, const qasc_ts_params* params,
                                                const qasc_paged_cache* cache, const uint16_t* q, const uint16_t* W,
                                                const uint16_t* index_pool, int32_t* sel, void* workspace,
                                                size_t ws_bytes, void* stream) {
  static const char* fn = "ts_score_vote_select_paged";
  qasc::PageMap pm;
  QASC_CHECK(check_paged(shape, cache, fn, &pm));
  QASC_CHECK(check_ts_params(shape, params, fn));
  return vote_select_call(fn, shape, params, q, W, index_pool, sel, workspace, ws_bytes, stream, &pm);
}

QASC_API qasc_status ts_sparse_attn_paged(const qasc_shape* shape, const qasc_ts_params* params,
                                          const qasc_paged_cache* cache, const qasc_local_ring* ring,
                                          const uint16_t* q, const uint16_t* K_pool, const uint16_t* V_pool,
                                          const int32_t* sel, const int32_t* sel_len, int32_t sel_per_kv_head,
                                          float* out, float* lse, void* workspace, size_t ws_bytes, void* stream) {
  static const char* fn = "ts_sparse_attn_paged";
  qasc::PageMap pm;
  QASC_CHECK(check_paged(shape, cache, fn, &pm));
  QASC_CHECK(check_ts_params(shape, params, fn));
  qasc::RingMap rm;
  if (ring) QASC_CHECK(check_ring(ring, params->local, fn, &rm));
  return sparse_attn_call(fn, sel_per_kv_head != 0, shape, params, q, K_pool, V_pool, sel, out, lse, workspace,
                          ws_bytes, stream, sel_len, &pm, ring ? &rm : nullptr);
}

QASC_API qasc_status ts_ring_flush(const qasc_shape* shape, const qasc_paged_cache* cache,
                                   const qasc_local_ring* ring, const uint16_t* W, uint16_t* K_pool,
                                   uint16_t* V_pool, uint16_t* index_pool, int64_t start, int64_t count,
                                   void* stream) {
  static const char* fn = "ts_ring_flush";
  QASC_RANGE(fn);
  qasc::PageMap pm;
  QASC_CHECK(check_paged(shape, cache, fn, &pm));
  qasc::RingMap rm;
  QASC_CHECK(check_ring(ring, count, fn, &rm));
  QASC_CHECK(check_rows(start, count, shape->n_cap, "tokens", fn));
  QASC_REQUIRE_PTR(W, 16, fn);
  QASC_REQUIRE_PTR(K_pool, 16, fn);
  QASC_REQUIRE_PTR(V_pool, 16, fn);
  QASC_REQUIRE_PTR(index_pool, 16, fn);
  if (count == 0) return ok();
  qasc_status st;
  const qasc::DeviceInfo* dev = need_device(fn, &st);
  if (!dev) return st;
  const cudaError_t e = qasc::launch_ring_flush(*shape, pm, rm, W, K_pool, V_pool, index_pool, start, count,
                                                dev->err_word, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, fn);
  return ok();
}

namespace {
qasc_status check_expand_rows(int32_t rows, const char* fn) {
  if (rows < 1 || rows > 65535) return fail(QASC_ERR_INVALID_ARG, "%s: rows=%d must lie in [1, 65535]", fn, rows);
  return QASC_OK;
}

qasc_status check_radius(int32_t radius, const char* fn) {
  if (radius < 0 || radius > (1 << 20))
    return fail(QASC_ERR_INVALID_ARG, "%s: radius=%d must lie in [0, 2^20]", fn, radius);
  return QASC_OK;
}

int64_t expand_capacity(const qasc_shape& s, const qasc_ts_params& p, int32_t radius) {
  const qasc::Regions R = qasc::regions_of(s.n, p.sink, p.local);
  const int64_t grown = (2 * static_cast<int64_t>(radius) + 1) * p.K;
  return grown < R.nc() ? grown : R.nc();
}
}  // namespace

QASC_API int32_t ts_expand_capacity(const qasc_shape* shape, const qasc_ts_params* params, int32_t radius) {
  static const char* fn = "ts_expand_capacity";
  QASC_SIZE_CHECK(check_shape(shape, fn));
  QASC_SIZE_CHECK(check_ts_params(shape, params, fn));
  QASC_SIZE_CHECK(check_radius(radius, fn));
  ok();
  return static_cast<int32_t>(expand_capacity(*shape, *params, radius));
}

QASC_API size_t ts_expand_workspace_bytes(const qasc_shape* shape, const qasc_ts_params* params, int32_t rows) {
  static const char* fn = "ts_expand_workspace_bytes";
  QASC_SIZE_CHECK(check_shape(shape, fn));
  QASC_SIZE_CHECK(check_ts_params(shape, params, fn));
  QASC_SIZE_CHECK(check_expand_rows(rows, fn));
  ok();
  return qasc::expand_workspace_bytes(*shape, *params, rows);
}

QASC_API qasc_status ts_expand_neighbors(const qasc_shape* shape, const qasc_ts_params* params, int32_t rows,
                                         const int32_t* sel, int32_t radius, int32_t* sel_out, int32_t cap,
                                         int32_t* len, void* workspace, size_t ws_bytes, void* stream) {
  static const char* fn = "ts_expand_neighbors";
  QASC_RANGE(fn);
  QASC_CHECK(check_shape(shape, fn));
  QASC_CHECK(check_ts_params(shape, params, fn));
  QASC_CHECK(check_expand_rows(rows, fn));
  QASC_CHECK(check_radius(radius, fn));
  const int64_t need = expand_capacity(*shape, *params, radius);
  if (cap < 1 || cap < need)
    return fail(QASC_ERR_INVALID_ARG, "%s: cap=%d, at least max(1, %lld) needed", fn, cap,
                static_cast<long long>(need));
  if (params->K > 0) QASC_REQUIRE_PTR(sel, 4, fn);
  QASC_REQUIRE_PTR(sel_out, 4, fn);
  QASC_REQUIRE_PTR(len, 4, fn);
  const size_t need_ws = qasc::expand_workspace_bytes(*shape, *params, rows);
  if (!workspace || ws_bytes < need_ws)
    return fail(QASC_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn, need_ws,
                workspace ? ws_bytes : size_t(0));
  QASC_REQUIRE_PTR(workspace, 256, fn);
  qasc_status st;
  if (!need_device(fn, &st)) return st;
  const int rc = qasc::launch_expand(*shape, *params, rows, sel, radius, sel_out, cap, len, workspace,
                                     static_cast<cudaStream_t>(stream));
  if (rc != 0) return cuda_fail(rc, fn);
  return ok();
}

QASC_API size_t ts_head_select_workspace_bytes(const qasc_shape* shape, const qasc_ts_params* params) {
  static const char* fn = "ts_head_select_workspace_bytes";
  QASC_SIZE_CHECK(check_shape(shape, fn));
  QASC_SIZE_CHECK(check_ts_params(shape, params, fn));
  ok();
  return qasc::head_select_layout(*shape, *params).total;
}

namespace {
// The per-KV-head select over a contiguous index (pm == nullptr) or a paged pool.
qasc_status head_select_call(const char* fn, const qasc_shape* shape, const qasc_ts_params* params,
                             const uint16_t* q, const uint16_t* W, const uint16_t* index, int32_t* sel,
                             void* workspace, size_t ws_bytes, void* stream, const qasc::PageMap* pm) {
  QASC_RANGE(fn);
  QASC_REQUIRE_PTR(q, 16, fn);
  QASC_REQUIRE_PTR(W, 16, fn);
  QASC_REQUIRE_PTR(index, 16, fn);
  if (params->K == 0) return ok();
  QASC_REQUIRE_PTR(sel, 16, fn);
  const qasc::HeadSelLayout L = qasc::head_select_layout(*shape, *params);
  if (!workspace || ws_bytes < L.total)
    return fail(QASC_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn, L.total,
                workspace ? ws_bytes : size_t(0));
  QASC_REQUIRE_PTR(workspace, 256, fn);
  qasc_status st;
  const qasc::DeviceInfo* dev = need_device(fn, &st);
  if (!dev) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const qasc::Regions R = qasc::regions_of(shape->n, params->sink, params->local);
  qasc::GroupScoreArgs ga;
  ga.qp = reinterpret_cast<float*>(ws + L.off_qp);
  ga.gsum = reinterpret_cast<float*>(ws + L.off_gsum);
  ga.range = reinterpret_cast<uint2*>(ws + L.off_range);
  ga.nc_pad = L.nc_pad;
  if (pm) ga.pm = *pm;
  int rc = qasc::launch_group_scores(*shape, *params, q, W, index, ga, *dev, s);
  if (rc != 0) return cuda_fail(rc, fn);
  rc = qasc::launch_head_topc(*shape, *params, L, ws, qasc::group_score_blocks(R, pm != nullptr), sel, *dev, s);
  if (rc != 0) return cuda_fail(rc, fn);
  return ok();
}
}  // namespace

QASC_API qasc_status ts_score_select_per_head(const qasc_shape* shape, const qasc_ts_params* params,
                                              const uint16_t* q, const uint16_t* W, const uint16_t* index,
                                              int32_t* sel, void* workspace, size_t ws_bytes, void* stream) {
  static const char* fn = "ts_score_select_per_head";
  QASC_CHECK(check_shape(shape, fn));
  QASC_CHECK(check_ts_params(shape, params, fn));
  return head_select_call(fn, shape, params, q, W, index, sel, workspace, ws_bytes, stream, nullptr);
}

QASC_API qasc_status ts_score_select_per_head_paged(const qasc_shape* shape, const qasc_ts_params* params,
                                                    const qasc_paged_cache* cache, const uint16_t* q,
                                                    const uint16_t* W, const uint16_t* index_pool, int32_t* sel,
                                                    void* workspace, size_t ws_bytes, void* stream) {
  static const char* fn = "ts_score_select_per_head_paged";
  qasc::PageMap pm;
  QASC_CHECK(check_paged(shape, cache, fn, &pm));
  QASC_CHECK(check_ts_params(shape, params, fn));
  return head_select_call(fn, shape, params, q, W, index_pool, sel, workspace, ws_bytes, stream, &pm);
}

namespace {
// Every token attended: all n are "sink", nothing is selected or local.
qasc_ts_params dense_params(const qasc_shape& s) {
  qasc_ts_params p;
  p.K = 0;
  p.sink = static_cast<int32_t>(s.n);
  p.local = 0;
  p.vmin = 1;
  return p;
}
}  // namespace

QASC_API size_t ts_dense_attn_workspace_bytes(const qasc_shape* shape) {
  QASC_SIZE_CHECK(check_shape(shape, "ts_dense_attn_workspace_bytes"));
  ok();
  const qasc_ts_params p = dense_params(*shape);
  return qasc::attn_layout(*shape, p, qasc::kMaxSmsForSizing).total;
}

QASC_API qasc_status ts_dense_attn(const qasc_shape* shape, const uint16_t* q, const uint16_t* K, const uint16_t* V,
                                   float* out, float* lse, void* workspace, size_t ws_bytes, void* stream) {
  static const char* fn = "ts_dense_attn";
  QASC_RANGE(fn);
  QASC_CHECK(check_shape(shape, fn));
  if (shape->n < 1) return fail(QASC_ERR_INVALID_ARG, "%s: n=%lld must be >= 1", fn, static_cast<long long>(shape->n));
  QASC_REQUIRE_PTR(q, 16, fn);
  QASC_REQUIRE_PTR(K, 16, fn);
  QASC_REQUIRE_PTR(V, 16, fn);
  QASC_REQUIRE_PTR(out, 16, fn);
  if (lse && !aligned(lse, 4)) return fail(QASC_ERR_INVALID_ARG, "%s: lse is not 4-byte aligned", fn);
  qasc_status st;
  const qasc::DeviceInfo* dev = need_device(fn, &st);
  if (!dev) return st;
  const qasc_ts_params p = dense_params(*shape);
  const qasc::AttnLayout L = qasc::attn_layout(*shape, p, dev->num_sms);
  if (!workspace || ws_bytes < L.total)
    return fail(QASC_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn, L.total,
                workspace ? ws_bytes : size_t(0));
  QASC_REQUIRE_PTR(workspace, 256, fn);
  const int rc = qasc::launch_sparse_attn(*shape, p, L, q, K, V, nullptr, out, lse, static_cast<uint8_t*>(workspace),
                                          *dev, static_cast<cudaStream_t>(stream));
  if (rc != 0) return cuda_fail(rc, fn);
  return ok();
}

QASC_API qasc_status ts_sparse_attn_noalloc(const qasc_shape* shape, const qasc_ts_params* params,
                                            const uint16_t* q, const uint16_t* K, const uint16_t* V,
                                            const int32_t* sel, float* out, float* lse, void* stream) {
  static const char* fn = "ts_sparse_attn_noalloc";
  QASC_RANGE(fn);
  QASC_CHECK(check_shape(shape, fn));
  QASC_CHECK(check_ts_params(shape, params, fn));
  QASC_REQUIRE_PTR(q, 16, fn);
  QASC_REQUIRE_PTR(K, 16, fn);
  QASC_REQUIRE_PTR(V, 16, fn);
  QASC_REQUIRE_PTR(out, 16, fn);
  if (params->K > 0) QASC_REQUIRE_PTR(sel, 4, fn);
  if (lse && !aligned(lse, 4)) return fail(QASC_ERR_INVALID_ARG, "%s: lse is not 4-byte aligned", fn);
  qasc_status st;
  const qasc::DeviceInfo* dev = need_device(fn, &st);
  if (!dev) return st;
  const qasc::AttnLayout L = qasc::attn_layout(*shape, *params, dev->num_sms);
  const size_t cap = qasc::sparse_attn_noalloc_capacity();
  if (L.total > cap)
    return fail(QASC_ERR_WORKSPACE,
                "%s: this shape needs %zu bytes of split-K scratch but the built-in area holds %zu; "
                "use ts_sparse_attn with a workspace",
                fn, L.total, cap);
  const int rc = qasc::launch_sparse_attn_noalloc(*shape, *params, L, q, K, V, sel, out, lse, *dev,
                                                  static_cast<cudaStream_t>(stream));
  if (rc != 0) return cuda_fail(rc, fn);
  return ok();
}

QASC_API size_t snapkv_workspace_bytes(const qasc_shape* shape, const qasc_snap_params* params) {
  static const char* fn = "snapkv_workspace_bytes";
  QASC_SIZE_CHECK(check_shape(shape, fn));
  QASC_SIZE_CHECK(check_snap_params(shape, params, fn));
  ok();
  return qasc::snap_layout(*shape, *params).total;
}

QASC_API qasc_status snapkv_compress(const qasc_shape* shape, const qasc_snap_params* params, const uint16_t* q_obs,
                                     const uint16_t* K, const uint16_t* V, int32_t* idx, uint16_t* K_out,
                                     uint16_t* V_out, void* workspace, size_t ws_bytes, void* stream) {
  static const char* fn = "snapkv_compress";
  QASC_RANGE(fn);
  QASC_CHECK(check_shape(shape, fn));
  QASC_CHECK(check_snap_params(shape, params, fn));
  QASC_REQUIRE_PTR(q_obs, 16, fn);
  QASC_REQUIRE_PTR(K, 16, fn);
  QASC_REQUIRE_PTR(V, 16, fn);
  QASC_REQUIRE_PTR(idx, 16, fn);
  QASC_REQUIRE_PTR(K_out, 16, fn);
  QASC_REQUIRE_PTR(V_out, 16, fn);
  const qasc::SnapLayout L = qasc::snap_layout(*shape, *params);
  if (!workspace || ws_bytes < L.total)
    return fail(QASC_ERR_WORKSPACE, "%s: workspace of %zu bytes needed, %zu given", fn, L.total,
                workspace ? ws_bytes : size_t(0));
  QASC_REQUIRE_PTR(workspace, 256, fn);
  qasc_status st;
  const qasc::DeviceInfo* dev = need_device(fn, &st);
  if (!dev) return st;
  const int rc = qasc::launch_snapkv(*shape, *params, L, q_obs, K, V, idx, K_out, V_out,
                                     static_cast<uint8_t*>(workspace), *dev, static_cast<cudaStream_t>(stream));
  if (rc != 0) return cuda_fail(rc, fn);
  return ok();
}

}  // extern "C"

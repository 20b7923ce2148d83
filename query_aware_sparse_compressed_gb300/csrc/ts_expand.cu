// Neighbour expansion of selected token sets.
//
// TokenButler page, section "Optimierungen": the selected tokens are expanded
// to their spatial neighbours (with a prediction interval, one selection
// serves several decode steps); SnapKV page, section "Top-k Selection と
// Cluster-based Retention": S_final = union over the selected j of
// {j - k, ..., j + k}.  Here: the union of [j - r, j + r] over each row's
// selected tokens, clipped to the candidates C (the sink and local tokens are
// attended anyway), emitted ascending.  Its size varies per row, so the rows
// have a fixed capacity and a length; ts_sparse_attn_ex attends to the
// entries in use.
//
// Two kernels over (row, chunk of kExChunk candidates) CTAs.  expand_count
// builds the chunk's part of the union as a bitmap in shared memory and stores
// it with its population count; expand_write places the chunk's members at
// the offset the earlier chunks' counts give.  The selected tokens that reach
// a chunk are found with a block-wide lower bound of the ascending row; each
// covers [j - r, j + r] cut short where the next token's interval begins, so
// the bitmap work is O(entries + chunk words) whatever the radius.  The length
// is the sum of the counts; the unused capacity repeats the last member,
// min(c1 - 1, j* + r) for the last token j* with j* - r < c1.
#include "common.cuh"
#include "internal.h"

namespace qasc {
namespace {

constexpr int kExChunk = 4096;               // candidates per CTA
constexpr int kExWords = kExChunk / 32;      // bitmap words per chunk
constexpr int kExThreads = kExWords;         // one word per thread

struct ExArgs {
  const int32_t* sel;   // [rows][K] ascending
  int32_t* out;         // [rows][cap]
  int32_t* len;         // [rows]
  uint32_t* words;      // [rows][nchunks][kExWords] bitmaps
  uint32_t* counts;     // [rows][nchunks]
  int32_t* last;        // [rows] last member of the union (when not empty)
  int K, radius, c0, nc, cap, nchunks;
};

__device__ __forceinline__ int64_t i64min(int64_t x, int64_t y) { return x < y ? x : y; }
__device__ __forceinline__ int64_t i64max(int64_t x, int64_t y) { return x > y ? x : y; }

// First indices of the ascending row with row[i] >= v0 and >= v1 (K if
// none), found by the whole block: each round probes kExThreads evenly spaced
// entries of the open range of each search, which shrinks it by that factor.
// Every thread takes the same branch (the counts are block-wide).  A row that
// is not ascending still gives indices in [0, K].
__device__ int2 block_lower_bounds(const int32_t* row, int K, int v0, int v1) {
  int lo[2] = {0, 0}, hi[2] = {K, K};
  const int v[2] = {v0, v1};
  while (hi[0] > lo[0] || hi[1] > lo[1]) {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const int span = hi[q] - lo[q];
      const int st = span > 0 ? (span + kExThreads - 1) / kExThreads : 1;
      const int np = span > 0 ? (span + st - 1) / st : 0;         // probes lo + t st, t < np
      const bool pr = static_cast<int>(threadIdx.x) < np && __ldg(row + lo[q] + threadIdx.x * st) < v[q];
      const int c = __syncthreads_count(pr);
      if (span > 0) {
        const int base = lo[q];
        if (c > 0) lo[q] = base + (c - 1) * st + 1;
        if (c < np) hi[q] = base + c * st;
      }
    }
  }
  return make_int2(lo[0], lo[1]);
}

// grid (nchunks, rows)
__global__ void __launch_bounds__(kExThreads) expand_count_kernel(const ExArgs a) {
  __shared__ uint32_t bm[kExWords];
  __shared__ uint32_t wsum[kExThreads / 32];
  const int ch = blockIdx.x, row = blockIdx.y, tid = threadIdx.x;
  const int p0 = ch * kExChunk;                    // chunk = candidates c0 + [p0, p1)
  const int p1 = min(a.nc, p0 + kExChunk);
  bm[tid] = 0;
  pdl_wait();
  const int32_t* s = a.sel + static_cast<int64_t>(row) * a.K;
  // tokens whose interval reaches the chunk: j + r >= c0 + p0 and j - r < c0 + p1
  const int2 rg = block_lower_bounds(s, a.K, a.c0 + p0 - a.radius, a.c0 + p1 + a.radius);
  for (int e = rg.x + tid; e < rg.y; e += kExThreads) {
    const int64_t j = __ldg(s + e);
    int64_t top = j + a.radius;
    if (e + 1 < a.K) top = min(top, static_cast<int64_t>(__ldg(s + e + 1)) - a.radius - 1);
    const int lo = static_cast<int>(i64max(a.c0 + p0, j - a.radius) - (a.c0 + p0));
    const int hi = static_cast<int>(i64min(a.c0 + p1 - 1, top) - (a.c0 + p0));
    if (lo > hi) continue;
    for (int w = lo >> 5; w <= (hi >> 5); ++w) {
      uint32_t m = ~0u;
      const int b0 = w * 32;
      if (lo > b0) m &= ~0u << (lo - b0);
      if (hi < b0 + 31) m &= ~0u >> (b0 + 31 - hi);
      atomicOr(&bm[w], m);
    }
  }
  __syncthreads();
  const int64_t cell = static_cast<int64_t>(row) * a.nchunks + ch;
  const uint32_t word = bm[tid];
  a.words[cell * kExWords + tid] = word;
  const uint32_t r = __reduce_add_sync(0xffffffffu, static_cast<uint32_t>(__popc(word)));
  if ((tid & 31) == 0) wsum[tid >> 5] = r;
  __syncthreads();
  if (tid == 0) {
    uint32_t t = 0;
    for (int w = 0; w < kExThreads / 32; ++w) t += wsum[w];
    a.counts[cell] = t;
    // the last chunk's upper bound is the first token with j - r >= c1
    if (ch == a.nchunks - 1)
      a.last[row] = rg.y > 0 ? static_cast<int32_t>(i64min(a.c0 + a.nc - 1,
                                                                  static_cast<int64_t>(__ldg(s + rg.y - 1)) + a.radius))
                             : a.c0;
  }
  pdl_trigger();
}

// grid (nchunks, rows)
__global__ void __launch_bounds__(kExThreads) expand_write_kernel(const ExArgs a) {
  __shared__ uint32_t wsum[kExThreads / 32];
  __shared__ uint32_t base_total[2];
  const int ch = blockIdx.x, row = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();
  const int64_t cell = static_cast<int64_t>(row) * a.nchunks + ch;
  if (warp == 0) {   // offset of this chunk and the row's total
    const uint32_t* cnt = a.counts + static_cast<int64_t>(row) * a.nchunks;
    uint32_t before = 0, total = 0;
    for (int i = lane; i < a.nchunks; i += 32) {
      const uint32_t v = __ldcg(cnt + i);
      total += v;
      before += i < ch ? v : 0u;
    }
    before = __reduce_add_sync(0xffffffffu, before);
    total = __reduce_add_sync(0xffffffffu, total);
    if (lane == 0) {
      base_total[0] = before;
      base_total[1] = total;
    }
  }
  const uint32_t word = __ldcg(a.words + cell * kExWords + tid);
  const uint32_t c = __popc(word);
  uint32_t inc = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += t;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  uint32_t pos = base_total[0] + inc - c;
  for (int w = 0; w < warp; ++w) pos += wsum[w];
  int32_t* o = a.out + static_cast<int64_t>(row) * a.cap;
  const int first = a.c0 + ch * kExChunk + 32 * tid;
  uint32_t m = word;
  while (m) {
    const int bit = __ffs(m) - 1;
    m &= m - 1;
    if (pos < static_cast<uint32_t>(a.cap)) o[pos] = first + bit;
    ++pos;
  }
  // the length, and the unused capacity (shared out among the row's CTAs)
  const int used = static_cast<int>(min(base_total[1], static_cast<uint32_t>(a.cap)));
  if (ch == 0 && tid == 0) a.len[row] = used;
  const int32_t fill = used > 0 ? __ldcg(a.last + row) : a.c0;
  for (int64_t i = used + static_cast<int64_t>(ch) * kExThreads + tid; i < a.cap;
       i += static_cast<int64_t>(a.nchunks) * kExThreads)
    o[i] = fill;
  pdl_trigger();
}

struct ExLayout {
  int nchunks;
  size_t off_counts, off_last, total;
};

ExLayout expand_layout(const qasc_shape& s, const qasc_ts_params& p, int rows) {
  const Regions R = regions_of(s.n, p.sink, p.local);
  ExLayout L;
  L.nchunks = static_cast<int>((R.nc() + kExChunk - 1) / kExChunk);
  if (L.nchunks < 1) L.nchunks = 1;
  const size_t cells = static_cast<size_t>(rows) * L.nchunks;
  L.off_counts = align_up(cells * kExWords * sizeof(uint32_t), 256);
  L.off_last = L.off_counts + align_up(cells * sizeof(uint32_t), 256);
  L.total = L.off_last + align_up(static_cast<size_t>(rows) * sizeof(int32_t), 256);
  return L;
}

}  // namespace

cudaError_t configure_expand_kernels(const DeviceInfo&) { return cudaSuccess; }

size_t expand_workspace_bytes(const qasc_shape& s, const qasc_ts_params& p, int rows) {
  return expand_layout(s, p, rows).total;
}

int launch_expand(const qasc_shape& s, const qasc_ts_params& p, int rows, const int32_t* sel, int radius,
                  int32_t* out, int cap, int32_t* len, void* ws, cudaStream_t stream) {
  const Regions R = regions_of(s.n, p.sink, p.local);
  const ExLayout L = expand_layout(s, p, rows);
  char* w = static_cast<char*>(ws);
  ExArgs a;
  a.sel = sel;
  a.out = out;
  a.len = len;
  a.words = reinterpret_cast<uint32_t*>(w);
  a.counts = reinterpret_cast<uint32_t*>(w + L.off_counts);
  a.last = reinterpret_cast<int32_t*>(w + L.off_last);
  a.K = p.K;
  a.radius = radius;
  a.c0 = static_cast<int>(R.c0);
  a.nc = static_cast<int>(R.nc());
  a.cap = cap;
  a.nchunks = L.nchunks;
  const dim3 grid(static_cast<unsigned>(a.nchunks), static_cast<unsigned>(rows));
  cudaError_t e = launch_dependent(expand_count_kernel, grid, dim3(kExThreads), 0, stream, 1, a);
  if (e != cudaSuccess) return e;
  return launch_dependent(expand_write_kernel, grid, dim3(kExThreads), 0, stream, 1, a);
}

}  // namespace qasc

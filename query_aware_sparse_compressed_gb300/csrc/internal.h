// Host-side interfaces between the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "qasc.h"

namespace qasc {

// Launches `kernel` as a programmatic dependent of the preceding kernel in
// the stream (see pdl_wait / pdl_trigger), optionally as clusters of
// `cluster` CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             unsigned cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  unsigned n = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

constexpr int kHeadDim = 128;
constexpr int kIndexDim = 32;
// Workspace queries made without a device size split-K scratch for this many
// SMs, an upper bound for any device the library runs on.
constexpr int kMaxSmsForSizing = 256;

// Token regions of a cache of n tokens (TokenSelect page, table of
// always-included tokens): sink [0, sink_end), candidates C [c0, c1),
// local [local_start, n).
struct Regions {
  int64_t sink_end, c0, c1, local_start;
  int64_t nc() const { return c1 - c0; }
};

// Where the rows of token t of (b, g) live.  Contiguous (table == nullptr):
// row (b Hkv + g) n_cap + t of a [B][Hkv][n_cap] cache.  Paged: row
// (page Hkv + g) P + t mod P of a [num_pages][Hkv][P] pool, page =
// table[b][t / P] (P = 2^page_shift).
struct PageMap {
  const int32_t* table = nullptr;   // [B][pages_per_seq]
  int64_t pages_per_seq = 0, num_pages = 0;
  int page_shift = 0;
};

// Circular local buffer: K and V rows of token t of (b, g) at slot t mod R
// of [B][Hkv][R][d] (K == nullptr: none).
struct RingMap {
  const uint16_t* K = nullptr;
  const uint16_t* V = nullptr;
  int64_t R = 0;
};

#ifdef __CUDACC__
// Row of token t of (b, g) under m, or -1 when its block-table entry lies
// outside the pool.
__device__ __forceinline__ int64_t cache_row(const PageMap& m, int b, int g, int Hkv, int64_t n_cap, int64_t t) {
  if (m.table == nullptr) return (static_cast<int64_t>(b) * Hkv + g) * n_cap + t;
  const int32_t page = __ldg(m.table + b * m.pages_per_seq + (t >> m.page_shift));
  if (page < 0 || page >= m.num_pages) return -1;
  return ((static_cast<int64_t>(page) * Hkv + g) << m.page_shift) + (t & ((int64_t(1) << m.page_shift) - 1));
}
#endif

inline Regions regions_of(int64_t n, int32_t sink, int32_t local) {
  Regions r;
  r.sink_end = n < sink ? n : sink;
  r.c0 = sink;
  r.c1 = n - local > r.c0 ? n - local : r.c0;
  r.local_start = n - local > r.sink_end ? n - local : r.sink_end;
  return r;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace of ts_score_vote_select.
struct SelectLayout {
  int64_t nc = 0, nc_pad = 0;
  size_t off_scores = 0, off_theta = 0, off_keys = 0, off_hist = 0, off_vhist = 0, total = 0;
  int hist_splits = 0;   // partial-histogram slots per (b, g), sized for kMaxSmsForSizing
};
SelectLayout select_layout(const qasc_shape& s, const qasc_ts_params& p);

// Workspace of ts_sparse_attn.
struct AttnLayout {
  int64_t t_len = 0;       // |T| = sink + K + local tokens attended
  int splits = 1;          // split-K pieces per (b, g)
  int64_t per_split = 0;   // T positions per split
  size_t off_part = 0, total = 0;
};
AttnLayout attn_layout(const qasc_shape& s, const qasc_ts_params& p, int num_sms);

// Per-device facts the launchers need.
struct DeviceInfo {
  int device = 0;
  int num_sms = 0;
  int max_smem_optin = 0;
  unsigned* err_word = nullptr;   // device address of the error word
  int cut_clusters16 = 0;         // co-resident 16-CTA clusters of the top-K cutoff (0: not schedulable)
  int topc_clusters[3] = {0, 0, 0};  // co-resident top-c clusters of 8, 4 and 2 CTAs
};
const DeviceInfo* device_info();  // current device; nullptr on CUDA failure

// One-time per-device kernel attributes (dynamic shared memory limits), run
// by device_info() so that no attribute call happens while a stream is being
// captured into a graph.
cudaError_t configure_score_kernels(const DeviceInfo& dev);
cudaError_t configure_select_kernels(DeviceInfo& dev);
cudaError_t configure_attn_kernels(const DeviceInfo& dev);
cudaError_t configure_snapkv_kernels(DeviceInfo& dev);

// cuTensorMapEncodeTiled resolved through the runtime (no libcuda link).
using EncodeTiledFn = int (*)(void* tmap, int dtype, unsigned rank, void* gaddr, const uint64_t* gdim,
                              const uint64_t* gstride, const unsigned* box, const unsigned* estride, int interleave,
                              int swizzle, int l2promo, int oobfill);
EncodeTiledFn encode_tiled_fn();

// Workspace of snapkv_compress.
struct SnapLayout {
  int64_t c_out = 0;      // kept entries per KV head: min(c, n)
  int parts = 1;          // key-range pieces per (b, g)
  size_t off_stats = 0, off_score = 0, off_pool = 0, off_phist = 0, off_khist = 0, total = 0;
};
SnapLayout snap_layout(const qasc_shape& s, const qasc_snap_params& p);

int launch_snapkv(const qasc_shape& s, const qasc_snap_params& p, const SnapLayout& L, const uint16_t* q_obs,
                  const uint16_t* K, const uint16_t* V, int32_t* idx, uint16_t* K_out, uint16_t* V_out, uint8_t* ws,
                  const DeviceInfo& dev, cudaStream_t stream);

cudaError_t launch_index_append(const qasc_shape& s, const uint16_t* K, const uint16_t* W, uint16_t* index,
                                int64_t start, int64_t count, cudaStream_t stream);
// The same over a paged pool (K and index rows through pm).
cudaError_t launch_index_append_paged(const qasc_shape& s, const PageMap& pm, const uint16_t* K, const uint16_t* W,
                                      uint16_t* index, int64_t start, int64_t count, unsigned* err,
                                      cudaStream_t stream);
// Tokens [start, start + count) from the ring into their pages: K and V rows
// copied, index rows written.
cudaError_t launch_ring_flush(const qasc_shape& s, const PageMap& pm, const RingMap& ring, const uint16_t* W,
                              uint16_t* K_pool, uint16_t* V_pool, uint16_t* index, int64_t start, int64_t count,
                              unsigned* err, cudaStream_t stream);

// Geometry of the persistent scoring grid (one CTA per SM over 256-token
// tiles) and of the per-(b, g) partial histograms it writes.
struct ScoreGrid {
  int tiles_per_bg = 0, total = 0, grid = 1, max_splits = 1, hist_bits = 12;
};
// span = tokens the score tiles of one (b, g) cover: score_span().
ScoreGrid score_grid(const qasc_shape& s, int64_t span, int num_sms);
// The candidates for the contiguous cache; tokens [0, c1) for a paged pool
// (its tiles start at token 0 so that they split at page boundaries).
inline int64_t score_span(const Regions& R, bool paged) { return paged ? R.c1 : R.nc(); }

struct ScoreOut {
  float* scores;        // [B][Hq][nc_pad]
  uint32_t* hist;       // [B*Hkv][max_splits][GQ][2^hist_bits] partial histograms
  int64_t nc_pad;
  int max_splits;
  PageMap pm;           // index rows of a paged pool (pm.table != nullptr)
};

// Scores for all (b, h, i in C); returns a CUDA error or a negative value
// for an unsupported configuration.
int launch_scores(const qasc_shape& s, const qasc_ts_params& p, const uint16_t* q, const uint16_t* W,
                  const uint16_t* index, const ScoreOut& o, const DeviceInfo& dev, cudaStream_t stream);

// paged: the scores were computed over a paged pool (tiles from token 0).
int launch_select(const qasc_shape& s, const qasc_ts_params& p, const SelectLayout& L, uint8_t* ws, int32_t* sel,
                  const DeviceInfo& dev, cudaStream_t stream, bool paged = false);

// Per-KV-head selection (no voting): each (b, g) keeps the K candidates
// with the largest group-summed score, ascending in sel [B][Hkv][K].  A q'
// pass and the group scoring pass (ts_group.cu) write the group sums and the
// key range of every 512-token block; the top-c kernel selects.
constexpr int kGroupBlock = 512;
struct HeadSelLayout {
  int64_t nc = 0, nc_pad = 0;
  int parts = 0;             // range partials per (b, g) row (blocks, sized for either blocking)
  size_t off_qp = 0, off_gsum = 0, off_range = 0, total = 0;
};
HeadSelLayout head_select_layout(const qasc_shape& s, const qasc_ts_params& p);

struct GroupScoreArgs {
  float* qp = nullptr;       // [B*Hq][32] q'_h / sqrt(d'), written by the q' pass
  float* gsum = nullptr;     // [B*Hkv][nc_pad] group sums
  uint2* range = nullptr;    // [B*Hkv][blocks] {min, max} order-preserving key per block
  int64_t nc_pad = 0;
  PageMap pm;                // index rows of a paged pool (pm.table != nullptr)
};
// 512-token blocks of one (b, g): of the candidates (contiguous cache), of
// tokens [0, c1) for a paged pool (its blocks start at token 0).
int group_score_blocks(const Regions& R, bool paged);
// The q' pass, then the group scoring pass.
int launch_group_scores(const qasc_shape& s, const qasc_ts_params& p, const uint16_t* q, const uint16_t* W,
                        const uint16_t* index, const GroupScoreArgs& a, const DeviceInfo& dev, cudaStream_t stream);
cudaError_t configure_group_kernels(const DeviceInfo& dev);
int launch_head_topc(const qasc_shape& s, const qasc_ts_params& p, const HeadSelLayout& L, uint8_t* ws, int parts,
                     int32_t* sel, const DeviceInfo& dev, cudaStream_t stream);
cudaError_t configure_head_select_kernels(DeviceInfo& dev);

// sel holds one list of K per sequence ([B][K]), or one per KV head
// ([B][Hkv][K]) when sel_per_kv; sel_len, when given, holds the entries in
// use of each list ([B] or [B][Hkv]); the others are masked.
int launch_sparse_attn(const qasc_shape& s, const qasc_ts_params& p, const AttnLayout& L, const uint16_t* q,
                       const uint16_t* K, const uint16_t* V, const int32_t* sel, float* out, float* lse,
                       uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream, bool sel_per_kv = false,
                       const int32_t* sel_len = nullptr, const PageMap* pm = nullptr,
                       const RingMap* ring = nullptr);

// Neighbour expansion: rows of K ascending candidates in, the ascending union
// of their +-radius neighbourhoods within C out ([rows][cap], the first
// len[row] entries in use, the rest repeating the last).
size_t expand_workspace_bytes(const qasc_shape& s, const qasc_ts_params& p, int rows);
int launch_expand(const qasc_shape& s, const qasc_ts_params& p, int rows, const int32_t* sel, int radius,
                  int32_t* out, int cap, int32_t* len, void* ws, cudaStream_t stream);
cudaError_t configure_expand_kernels(const DeviceInfo& dev);

// ts_sparse_attn with its split-K scratch in a fixed area built into the
// library (see ts_attn.cu); the caller checks L.total against the capacity.
size_t sparse_attn_noalloc_capacity();
int launch_sparse_attn_noalloc(const qasc_shape& s, const qasc_ts_params& p, const AttnLayout& L, const uint16_t* q,
                               const uint16_t* K, const uint16_t* V, const int32_t* sel, float* out, float* lse,
                               const DeviceInfo& dev, cudaStream_t stream);

}  // namespace qasc

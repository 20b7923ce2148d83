// Per-KV-head token selection: the TokenSelect variant without voting.
//
// TokenSelect page, section "Ablation" (table アブレーション): "w/o Voting"
// replaces the vote by an independent selection per head.  Reading, for GQA:
// each KV head g keeps its own set S_g of K candidates, ranked by the sum of
// its query heads' index scores (Score_h of section "Query-Key Dot Product
// Index" summed over the Gq heads of the group; with Gq = 1 this is the
// head's own score), ties to the lower token index, emitted ascending.  The
// sink and local tokens stay outside the budget, as on the voting path, and
// every query head of the group attends to sink + S_g + local.
//
// Kernels: the scoring grid of ts_score.cu writes Score_h for every
// candidate; group_sum_kernel adds each group's heads and records the key
// range of each of its CTAs; topc_kernel (topc.cuh) selects each row's K
// largest on an 8-CTA cluster.
#include "common.cuh"
#include "internal.h"

namespace qasc {
namespace {

namespace cg = cooperative_groups;

#include "topc.cuh"

constexpr int kGsThreads = 256;
constexpr int kGsTok = 4 * kGsThreads;   // candidates per CTA (four per thread)

// grid (ceil(nc / kGsTok), B * Hkv): gs[b][g][j] = sum over the group's
// heads (in head order) of Score_h(c0 + j), four consecutive candidates per
// thread (one float4 per head).  This is the last reader of the scores:
// after reading, the warp's lanes drop its 512-byte run of every head of the
// group from L2, so the dead scratch is never written back.  Each CTA writes
// the smallest and largest order-preserving key of its sums.
__global__ void __launch_bounds__(kGsThreads) group_sum_kernel(const float* __restrict__ scores,
                                                               float* __restrict__ gs, uint2* __restrict__ range,
                                                               int Hq, int Hkv, int nc, int64_t nc_pad) {
  __shared__ uint32_t wmin[kGsThreads / 32], wmax[kGsThreads / 32];
  const int bg = blockIdx.y;
  const int b = bg / Hkv, g = bg - b * Hkv;
  const int gq = Hq / Hkv;
  const int i4 = blockIdx.x * kGsThreads + threadIdx.x;
  const int j0 = 4 * i4;
  const int lane = threadIdx.x & 31;
  pdl_wait();
  const float* src = scores + (static_cast<int64_t>(b) * Hq + static_cast<int64_t>(g) * gq) * nc_pad;
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  if (j0 < nc) {
    const float4* s4 = reinterpret_cast<const float4*>(src) + i4;
    const int64_t hstride = nc_pad / 4;
    float4 acc = __ldcg(s4);
    for (int hh = 1; hh < gq; ++hh) {
      const float4 v = __ldcg(s4 + hh * hstride);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    reinterpret_cast<float4*>(gs + static_cast<int64_t>(bg) * nc_pad)[i4] = acc;
    const float a4[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (j0 + u < nc) {
        const uint32_t key = ord_key(a4[u]);
        kmin = min(kmin, key);
        kmax = max(kmax, key);
      }
  }
  __syncwarp();
  // the warp's 128 candidates = up to four 128-byte lines per head; a line
  // that starts at nc_pad (a multiple of 64 floats) belongs to the next head
  const int w0 = j0 - 4 * lane;
  if (w0 < nc)
    for (int t = lane; t < gq * 4; t += 32) {
      const int64_t x = w0 + 32 * (t & 3);
      if (x < nc_pad) discard_l2_line(src + static_cast<int64_t>(t >> 2) * nc_pad + x);
    }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (lane == 0) {
    wmin[threadIdx.x >> 5] = kmin;
    wmax[threadIdx.x >> 5] = kmax;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < kGsThreads / 32; ++w) {
      kmin = min(kmin, wmin[w]);
      kmax = max(kmax, wmax[w]);
    }
    range[static_cast<int64_t>(bg) * gridDim.x + blockIdx.x] = make_uint2(kmin, kmax);
  }
  pdl_trigger();
}

}  // namespace

cudaError_t configure_head_select_kernels(const DeviceInfo&) { return configure_topc(); }

HeadSelLayout head_select_layout(const qasc_shape& s, const qasc_ts_params& p) {
  HeadSelLayout L;
  const Regions R = regions_of(s.n, p.sink, p.local);
  L.nc = R.nc();
  L.nc_pad = static_cast<int64_t>(align_up(static_cast<size_t>(L.nc > 0 ? L.nc : 1), 64));
  L.parts = static_cast<int>((L.nc + kGsTok - 1) / kGsTok);
  const size_t bh = static_cast<size_t>(s.B) * s.Hq, bg = static_cast<size_t>(s.B) * s.Hkv;
  // partial histograms of the scoring pass for either tiling (contiguous or paged)
  ScoreGrid sg = score_grid(s, score_span(R, false), kMaxSmsForSizing);
  const ScoreGrid sgp = score_grid(s, score_span(R, true), kMaxSmsForSizing);
  if (sgp.max_splits > sg.max_splits) sg.max_splits = sgp.max_splits;
  size_t off = 0;
  L.off_scores = off;
  off = align_up(off + bh * L.nc_pad * sizeof(float), 256);
  L.off_hist = off;
  off = align_up(off + bg * sg.max_splits * (s.Hq / s.Hkv) * (size_t(1) << sg.hist_bits) * sizeof(uint32_t), 256);
  L.off_gsum = off;
  off = align_up(off + bg * L.nc_pad * sizeof(float), 256);
  L.off_range = off;
  off = align_up(off + bg * (L.parts > 0 ? L.parts : 1) * sizeof(uint2), 256);
  L.total = off;
  return L;
}

int launch_head_select(const qasc_shape& s, const qasc_ts_params& p, const HeadSelLayout& L, uint8_t* ws,
                       int32_t* sel, const DeviceInfo& dev, cudaStream_t stream) {
  const Regions R = regions_of(s.n, p.sink, p.local);
  const int nc = static_cast<int>(L.nc);
  float* scores = reinterpret_cast<float*>(ws + L.off_scores);
  float* gs = reinterpret_cast<float*>(ws + L.off_gsum);
  uint2* range = reinterpret_cast<uint2*>(ws + L.off_range);
  const unsigned bg = static_cast<unsigned>(s.B * s.Hkv);
  cudaError_t e = launch_dependent(group_sum_kernel, dim3(static_cast<unsigned>(L.parts), bg), dim3(kGsThreads), 0,
                                   stream, 1, static_cast<const float*>(scores), gs, range, s.Hq, s.Hkv, nc,
                                   L.nc_pad);
  if (e != cudaSuccess) return e;
  return launch_topc(gs, reinterpret_cast<const uint32_t*>(range), L.parts, sel, static_cast<int>(bg),
                     static_cast<int64_t>(nc), L.nc_pad, p.K, static_cast<int>(R.c0), dev.num_sms, stream);
}

}  // namespace qasc

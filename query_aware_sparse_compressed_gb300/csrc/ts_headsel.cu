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

// grid (ceil(nc / kGsThreads), B * Hkv): gs[b][g][j] = sum over the group's
// heads (in head order) of Score_h(c0 + j).  This is the last reader of the
// scores: after reading, the warp's lanes drop its 128-byte line of every
// head of the group from L2, so the dead scratch is never written back.
// Each CTA writes the smallest and largest order-preserving key of its sums.
__global__ void __launch_bounds__(kGsThreads) group_sum_kernel(const float* __restrict__ scores,
                                                               float* __restrict__ gs, uint2* __restrict__ range,
                                                               int Hq, int Hkv, int nc, int64_t nc_pad) {
  __shared__ uint32_t wmin[kGsThreads / 32], wmax[kGsThreads / 32];
  const int bg = blockIdx.y;
  const int b = bg / Hkv, g = bg - b * Hkv;
  const int gq = Hq / Hkv;
  const int j = blockIdx.x * kGsThreads + threadIdx.x;
  const int lane = threadIdx.x & 31;
  pdl_wait();
  const float* src = scores + (static_cast<int64_t>(b) * Hq + static_cast<int64_t>(g) * gq) * nc_pad;
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  if (j < nc) {
    float s = 0.0f;
    for (int hh = 0; hh < gq; ++hh) s += __ldcg(src + hh * nc_pad + j);
    gs[static_cast<int64_t>(bg) * nc_pad + j] = s;
    kmin = kmax = ord_key(s);
  }
  __syncwarp();
  const int w0 = j - lane;   // first candidate of the warp: a 128-byte line per head
  if (w0 < nc)
    for (int hh = lane; hh < gq; hh += 32) discard_l2_line(src + hh * nc_pad + w0);
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

cudaError_t configure_head_select_kernels(const DeviceInfo&) {
  return cudaFuncSetAttribute(topc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(sizeof(TopcShared)));
}

HeadSelLayout head_select_layout(const qasc_shape& s, const qasc_ts_params& p) {
  HeadSelLayout L;
  const Regions R = regions_of(s.n, p.sink, p.local);
  L.nc = R.nc();
  L.nc_pad = static_cast<int64_t>(align_up(static_cast<size_t>(L.nc > 0 ? L.nc : 1), 64));
  L.parts = static_cast<int>((L.nc + kGsThreads - 1) / kGsThreads);
  const size_t bh = static_cast<size_t>(s.B) * s.Hq, bg = static_cast<size_t>(s.B) * s.Hkv;
  const ScoreGrid sg = score_grid(s, L.nc, kMaxSmsForSizing);
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
                       int32_t* sel, const DeviceInfo&, cudaStream_t stream) {
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
  const int slice = ((nc + kPcCS - 1) / kPcCS + kPcKPT - 1) / kPcKPT * kPcKPT;
  return launch_dependent(topc_kernel, dim3(bg * kPcCS), dim3(kPcThreads), sizeof(TopcShared), stream, 1,
                          static_cast<const float*>(gs), reinterpret_cast<const uint32_t*>(range), L.parts, sel,
                          static_cast<int64_t>(nc), L.nc_pad, p.K, slice, static_cast<int>(R.c0));
}

}  // namespace qasc

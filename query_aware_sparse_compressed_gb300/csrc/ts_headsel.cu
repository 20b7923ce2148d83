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
// Kernels: the scoring pass in group mode (ts_score.cu) writes each
// candidate's group-summed score and the key range of every 512-token block;
// topc_kernel (topc.cuh) selects each row's K largest on a thread-block
// cluster.
#include "common.cuh"
#include "internal.h"

namespace qasc {
namespace {

namespace cg = cooperative_groups;

#include "topc.cuh"

}  // namespace

cudaError_t configure_head_select_kernels(DeviceInfo& dev) { return configure_topc(dev.topc_clusters); }

HeadSelLayout head_select_layout(const qasc_shape& s, const qasc_ts_params& p) {
  HeadSelLayout L;
  const Regions R = regions_of(s.n, p.sink, p.local);
  L.nc = R.nc();
  L.nc_pad = static_cast<int64_t>(align_up(static_cast<size_t>(L.nc > 0 ? L.nc : 1), 64));
  // range partials for either blocking (contiguous candidates or a paged pool from token 0)
  const int64_t span = R.c1 > L.nc ? R.c1 : L.nc;
  L.parts = static_cast<int>((span + kGroupBlock - 1) / kGroupBlock);
  if (L.parts < 1) L.parts = 1;
  const size_t bh = static_cast<size_t>(s.B) * s.Hq, bg = static_cast<size_t>(s.B) * s.Hkv;
  size_t off = 0;
  L.off_qp = off;
  off = align_up(off + bh * kIndexDim * sizeof(float), 256);
  L.off_gsum = off;
  off = align_up(off + bg * L.nc_pad * sizeof(float), 256);
  L.off_range = off;
  off = align_up(off + bg * static_cast<size_t>(L.parts) * sizeof(uint2), 256);
  L.total = off;
  return L;
}

int launch_head_topc(const qasc_shape& s, const qasc_ts_params& p, const HeadSelLayout& L, uint8_t* ws, int parts,
                     int32_t* sel, const DeviceInfo& dev, cudaStream_t stream) {
  const Regions R = regions_of(s.n, p.sink, p.local);
  const float* gs = reinterpret_cast<const float*>(ws + L.off_gsum);
  const uint2* range = reinterpret_cast<const uint2*>(ws + L.off_range);
  return launch_topc(gs, reinterpret_cast<const uint32_t*>(range), parts, nullptr, sel, s.B * s.Hkv,
                     static_cast<int64_t>(L.nc), L.nc_pad, p.K, static_cast<int>(R.c0), dev.topc_clusters, stream);
}

}  // namespace qasc

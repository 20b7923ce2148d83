// Per-head index scores for every candidate token.
//
// TokenSelect page, section "Query-Key Dot Product Index", equation Score_h:
//   Score_h(i) = q'_h . k_index(i) / sqrt(d'),  q'_h = W_{g(h)}^T q_h (fp32).
//
// This is the dominant HBM stream of the select step: every candidate's
// 64-byte index row is read once.  A persistent grid (one CTA per SM) walks
// contiguous runs of 256-token tiles (16 KB, contiguous in memory); one
// producer lane streams each tile with a single bulk copy into an 8-deep ring
// of shared-memory stages, and eight consumer warps (up to four heads per
// thread) turn rows into scores with packed fp32 FMAs (f32x2).  A thread reads its 64-byte row as four 16-byte
// chunks in a rotated order ((row / 2) mod 4 first), which makes every
// 8-thread phase of a 128-bit shared load hit 8 distinct bank groups; the
// rotation is folded into the order of the thread's q' registers.
//
// q'_h for every (b, h) is formed first by qproj_kernel (one CTA per (b, g),
// lane j of head h forms column j) into the workspace; consumers load their
// heads' q' with independent 16-byte loads at each change of (b, g).
#include "common.cuh"
#include "internal.h"

namespace qasc {
namespace {

constexpr int kTileTok = 256;                 // tokens per stage
constexpr int kTileBytes = kTileTok * kDIdx * 2;
constexpr int kStages = 8;
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;
constexpr float kInvSqrtDIdx = 0.17677669529663688f;  // 1 / sqrt(32)

// The CTA of a persistent grid of G CTAs over `total` items (CTA c takes
// [c total / G, (c+1) total / G)) that holds item x.
__host__ __device__ __forceinline__ int first_cta(int64_t x, int64_t total, int G) {
  int64_t c = ((x + 1) * G + total - 1) / total - 1;
  return static_cast<int>(c < 0 ? 0 : (c >= G ? G - 1 : c));
}

template <int GQ>
struct Split {
  static constexpr int HPT = GQ < 4 ? GQ : 4;   // heads per thread
  static constexpr int TPT = GQ / HPT;          // threads per token row
};

// First radix digit of the per-head threshold search (see ts_select.cu):
// the top hist_bits(GQ) bits of the order-preserving score key.
__host__ __device__ constexpr int hist_bits(int gq) { return gq <= 4 ? 12 : 11; }

template <int GQ>
struct ScoreSmem {
  uint8_t tile[kStages][kTileBytes];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint32_t hist[GQ][1 << hist_bits(GQ)];
};

// grid B * Hkv, block 32 * GQ: q'[b, h, :] = W_g^T q[b, h, :] / sqrt(d'), fp32.
template <int GQ>
__global__ void __launch_bounds__(32 * GQ) qproj_kernel(const uint16_t* __restrict__ q,
                                                       const uint16_t* __restrict__ W, float* __restrict__ qp,
                                                       int Hq, int Hkv) {
  __shared__ float qs[GQ][kD];
  __shared__ __align__(16) uint16_t ws[kD * kDIdx];
  const int bg = blockIdx.x, b = bg / Hkv, g = bg - b * Hkv;
  // stage W_g (8 KB) and the queries with independent 16-byte loads
  const uint4* w4 = reinterpret_cast<const uint4*>(W + static_cast<int64_t>(g) * kD * kDIdx);
  for (int i = threadIdx.x; i < kD * kDIdx / 8; i += 32 * GQ) reinterpret_cast<uint4*>(ws)[i] = __ldg(w4 + i);
  const uint16_t* qb = q + (static_cast<int64_t>(b) * Hq + g * GQ) * kD;
  for (int i = threadIdx.x; i < GQ * kD; i += 32 * GQ) qs[i / kD][i % kD] = bf_to_f(qb[i]);
  __syncthreads();
  const int hh = threadIdx.x >> 5, j = threadIdx.x & 31;
  float acc = 0.0f;
#pragma unroll 16
  for (int e = 0; e < kD; ++e) acc = fmaf(qs[hh][e], bf_to_f(ws[e * kDIdx + j]), acc);
  qp[(static_cast<int64_t>(b) * Hq + g * GQ + hh) * kDIdx + j] = acc * kInvSqrtDIdx;
}

template <int GQ>
__global__ void __launch_bounds__(kThreads, 1) score_kernel(const uint16_t* __restrict__ index,
                                                           const float* __restrict__ qp,
                                                           float* __restrict__ scores,
                                                           uint32_t* __restrict__ hist_part, int Hq, int Hkv,
                                                           int64_t n_cap, int c0, int nc, int64_t nc_pad,
                                                           int tiles_per_bg, int total_tiles, int max_splits,
                                                           unsigned* err) {
  using Sp = Split<GQ>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  ScoreSmem<GQ>& S = *reinterpret_cast<ScoreSmem<GQ>*>(smem_raw);
  constexpr int kNB = 1 << hist_bits(GQ);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int it0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * total_tiles / G);
  const int it1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * total_tiles / G);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kConsumerWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---- producer: one lane issues one bulk copy per tile
    if (lane == 0) {
      const uint64_t pol = policy_evict_first();
      for (int it = it0; it < it1; ++it) {
        const int k = it - it0;
        const int slot = k % kStages;
        const uint32_t ph = (k / kStages) & 1u;
        if (!mbar_wait(&S.empty[slot], ph ^ 1u)) {
          record_error(err, kErrTimeout);
          break;
        }
        const int bg = it / tiles_per_bg;
        const int t = it - bg * tiles_per_bg;
        const int rows = min(kTileTok, nc - t * kTileTok);
        const uint32_t bytes = static_cast<uint32_t>(rows) * kDIdx * 2;
        const uint16_t* src = index + (static_cast<int64_t>(bg) * n_cap + c0 + static_cast<int64_t>(t) * kTileTok) * kDIdx;
        mbar_arrive_expect_tx(&S.full[slot], bytes);
        bulk_g2s_hint(&S.tile[slot][0], src, bytes, &S.full[slot], pol);
      }
    }
    return;
  }

  // ---- consumers
  const int hs = tid % Sp::TPT;   // which HPT-head slice of the group
  const int r0 = tid / Sp::TPT;   // first row handled in a tile
  constexpr int kRowStep = kConsumers / Sp::TPT;
  const int rot = (r0 >> 1) & 3;  // chunk rotation (same for every row of this thread)
  float2 qr[Sp::HPT][kDIdx / 2];
  int cur_bg = -1;
  int b = 0, g = 0;
  bool dead = false;   // a bounded wait ran out: skip work but keep every barrier

  for (int i = tid; i < GQ * kNB; i += kConsumers) (&S.hist[0][0])[i] = 0;
  named_bar_sync(1, kConsumers);

  // Writes this CTA's histograms of (b, g) to its partial slot and clears them.
  auto flush = [&](int fbg) {
    named_bar_sync(1, kConsumers);
    const int split = static_cast<int>(blockIdx.x) - first_cta(static_cast<int64_t>(fbg) * tiles_per_bg,
                                                                 total_tiles, G);
    uint4* dst = reinterpret_cast<uint4*>(hist_part + (static_cast<int64_t>(fbg) * max_splits + split) * GQ * kNB);
    uint4* src = reinterpret_cast<uint4*>(&S.hist[0][0]);
    for (int i = tid; i < GQ * kNB / 4; i += kConsumers) {
      dst[i] = src[i];
      src[i] = make_uint4(0, 0, 0, 0);
    }
    named_bar_sync(1, kConsumers);
  };

  for (int it = it0; it < it1; ++it) {
    const int k = it - it0;
    const int slot = k % kStages;
    const uint32_t ph = (k / kStages) & 1u;
    const int bg = it / tiles_per_bg;
    const int t = it - bg * tiles_per_bg;
    if (bg != cur_bg) {
      if (cur_bg >= 0) flush(cur_bg);
      b = bg / Hkv;
      g = bg - b * Hkv;
      // this thread's heads, in the rotated chunk order: step p covers chunk (p + rot) mod 4
      const float* qh0 = qp + (static_cast<int64_t>(b) * Hq + g * GQ + hs * Sp::HPT) * kDIdx;
#pragma unroll
      for (int hh = 0; hh < Sp::HPT; ++hh) {
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int c = (p + rot) & 3;
          const float4 lo = __ldcg(reinterpret_cast<const float4*>(qh0 + hh * kDIdx + 8 * c));
          const float4 hi = __ldcg(reinterpret_cast<const float4*>(qh0 + hh * kDIdx + 8 * c + 4));
          qr[hh][4 * p + 0] = make_float2(lo.x, lo.y);
          qr[hh][4 * p + 1] = make_float2(lo.z, lo.w);
          qr[hh][4 * p + 2] = make_float2(hi.x, hi.y);
          qr[hh][4 * p + 3] = make_float2(hi.z, hi.w);
        }
      }
      cur_bg = bg;
    }
    if (!dead) {
      const bool ok = mbar_wait(&S.full[slot], ph);
      if (!__all_sync(0xffffffffu, ok)) {
        record_error(err, kErrTimeout);
        dead = true;
      }
    }
    if (!dead) {
      const uint8_t* st = S.tile[slot];
      float* out_base = scores + (static_cast<int64_t>(b) * Hq + g * GQ + hs * Sp::HPT) * nc_pad;
#pragma unroll 1
      for (int r = r0; r < kTileTok; r += kRowStep) {
        const int tok = t * kTileTok + r;
        if (tok >= nc) break;
        float2 acc[Sp::HPT];
#pragma unroll
        for (int hh = 0; hh < Sp::HPT; ++hh) acc[hh] = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int c = (p + rot) & 3;
          const uint4 v = *reinterpret_cast<const uint4*>(st + r * 64 + c * 16);
          const float2 x0 = bf2_to_f2(v.x), x1 = bf2_to_f2(v.y), x2 = bf2_to_f2(v.z), x3 = bf2_to_f2(v.w);
#pragma unroll
          for (int hh = 0; hh < Sp::HPT; ++hh) {
            acc[hh] = ffma2(qr[hh][4 * p + 0], x0, acc[hh]);
            acc[hh] = ffma2(qr[hh][4 * p + 1], x1, acc[hh]);
            acc[hh] = ffma2(qr[hh][4 * p + 2], x2, acc[hh]);
            acc[hh] = ffma2(qr[hh][4 * p + 3], x3, acc[hh]);
          }
        }
#pragma unroll
        for (int hh = 0; hh < Sp::HPT; ++hh) {
          const float sc = acc[hh].x + acc[hh].y;
          out_base[hh * nc_pad + tok] = sc;
          atomicAdd(&S.hist[hs * Sp::HPT + hh][ord_key(sc) >> (32 - hist_bits(GQ))], 1u);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[slot]);
  }
  if (cur_bg >= 0) flush(cur_bg);
}

template <int GQ>
int launch_gq(const qasc_shape& s, const Regions& R, const uint16_t* index, const uint16_t* q, const uint16_t* W,
              const ScoreOut& o, const DeviceInfo& dev, cudaStream_t stream) {
  qproj_kernel<GQ><<<s.B * s.Hkv, 32 * GQ, 0, stream>>>(q, W, o.qp, s.Hq, s.Hkv);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const ScoreGrid sg = score_grid(s, R.nc(), dev.num_sms);
  score_kernel<GQ><<<sg.grid, kThreads, sizeof(ScoreSmem<GQ>), stream>>>(
      index, o.qp, o.scores, o.hist, s.Hq, s.Hkv, s.n_cap, static_cast<int>(R.c0), static_cast<int>(R.nc()),
      o.nc_pad, sg.tiles_per_bg, sg.total, o.max_splits, dev.err_word);
  return cudaGetLastError();
}

template <int GQ>
cudaError_t configure_gq() {
  return cudaFuncSetAttribute(score_kernel<GQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(sizeof(ScoreSmem<GQ>)));
}

}  // namespace

cudaError_t configure_score_kernels(const DeviceInfo&) {
  cudaError_t e;
  if ((e = configure_gq<1>()) != cudaSuccess) return e;
  if ((e = configure_gq<2>()) != cudaSuccess) return e;
  if ((e = configure_gq<4>()) != cudaSuccess) return e;
  return configure_gq<8>();
}

ScoreGrid score_grid(const qasc_shape& s, int64_t nc, int num_sms) {
  ScoreGrid g;
  g.tiles_per_bg = static_cast<int>((nc + kTileTok - 1) / kTileTok);
  g.total = g.tiles_per_bg * s.B * s.Hkv;
  g.grid = g.total < num_sms ? g.total : num_sms;
  if (g.grid < 1) g.grid = 1;
  // CTAs covering one (b, g): each holds at least floor(total / grid) tiles.
  const int per = g.total / g.grid;
  g.max_splits = (g.tiles_per_bg - 1) / (per > 0 ? per : 1) + 2;
  g.hist_bits = hist_bits(s.Hq / s.Hkv);
  return g;
}

int launch_scores(const qasc_shape& s, const qasc_ts_params& p, const uint16_t* q, const uint16_t* W,
                  const uint16_t* index, const ScoreOut& o, const DeviceInfo& dev, cudaStream_t stream) {
  const Regions R = regions_of(s.n, p.sink, p.local);
  if (R.nc() <= 0) return 0;
  switch (s.Hq / s.Hkv) {
    case 1: return launch_gq<1>(s, R, index, q, W, o, dev, stream);
    case 2: return launch_gq<2>(s, R, index, q, W, o, dev, stream);
    case 4: return launch_gq<4>(s, R, index, q, W, o, dev, stream);
    case 8: return launch_gq<8>(s, R, index, q, W, o, dev, stream);
    default: return -1;
  }
}

}  // namespace qasc

// Per-head index scores for every candidate token.
//
// TokenSelect page, section "Query-Key Dot Product Index", equation Score_h:
//   Score_h(i) = q'_h . k_index(i) / sqrt(d'),  q'_h = W_{g(h)}^T q_h (fp32).
//
// This is the dominant HBM stream of the select step: every candidate's
// 64-byte index row is read once.  A persistent grid (one CTA per SM) walks
// contiguous runs of 256-token tiles (16 KB, contiguous in memory); one
// producer lane streams each tile with a single bulk copy into a 4-deep ring
// of shared-memory stages, and eight consumer warps turn rows into scores with
// packed fp32 FMAs (f32x2).  A thread reads its 64-byte row as four 16-byte
// chunks in a rotated order ((row / 2) mod 4 first), which makes every
// 8-thread phase of a 128-bit shared load hit 8 distinct bank groups; the
// rotation is folded into the order of the thread's q' registers.
//
// q'_h is computed per warp at each change of (b, g): the warp stages W_g
// (8 KB) and the group's query rows in its own shared-memory scratch with
// independent 16-byte loads, then lane j forms column j of q'.
#include "common.cuh"
#include "internal.h"

namespace qasc {
namespace {

constexpr int kTileTok = 256;                 // tokens per stage
constexpr int kTileBytes = kTileTok * kDIdx * 2;
constexpr int kStages = 4;
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = 32 * kConsumerWarps;
constexpr int kThreads = kConsumers + 32;
constexpr float kInvSqrtDIdx = 0.17677669529663688f;  // 1 / sqrt(32)

template <int GQ>
struct Split {
  static constexpr int HPT = GQ < 4 ? GQ : 4;   // heads per thread
  static constexpr int TPT = GQ / HPT;          // threads per token row
};

template <int GQ>
struct WarpScratch {
  uint16_t w[kD * kDIdx];      // W_g, row-major [e][j]
  uint16_t q[GQ][kD];          // query rows of the group
  float qp[GQ][kDIdx];         // q'_h, scaled by 1/sqrt(d')
};

template <int GQ>
struct ScoreSmem {
  uint8_t tile[kStages][kTileBytes];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  WarpScratch<GQ> ws[kConsumerWarps];
};

template <int GQ>
__global__ void __launch_bounds__(kThreads, 1) score_kernel(const uint16_t* __restrict__ index,
                                                           const uint16_t* __restrict__ q,
                                                           const uint16_t* __restrict__ W,
                                                           float* __restrict__ scores, int Hq, int Hkv,
                                                           int64_t n_cap, int c0, int nc, int64_t nc_pad,
                                                           int tiles_per_bg, int total_tiles, unsigned* err) {
  using Sp = Split<GQ>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  ScoreSmem<GQ>& S = *reinterpret_cast<ScoreSmem<GQ>*>(smem_raw);

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
  WarpScratch<GQ>& X = S.ws[warp];
  float2 qr[Sp::HPT][kDIdx / 2];
  int cur_bg = -1;
  int b = 0, g = 0;

  for (int it = it0; it < it1; ++it) {
    const int k = it - it0;
    const int slot = k % kStages;
    const uint32_t ph = (k / kStages) & 1u;
    const int bg = it / tiles_per_bg;
    const int t = it - bg * tiles_per_bg;
    if (bg != cur_bg) {
      b = bg / Hkv;
      g = bg - b * Hkv;
      // stage W_g and the group's queries (independent 16-byte loads)
      const uint4* wsrc = reinterpret_cast<const uint4*>(W + static_cast<int64_t>(g) * kD * kDIdx);
      uint4* wdst = reinterpret_cast<uint4*>(X.w);
#pragma unroll
      for (int i = 0; i < kD * kDIdx / 8 / 32; ++i) wdst[lane + 32 * i] = __ldg(wsrc + lane + 32 * i);
      const uint4* qsrc = reinterpret_cast<const uint4*>(q + (static_cast<int64_t>(b) * Hq + g * GQ) * kD);
      uint4* qdst = reinterpret_cast<uint4*>(&X.q[0][0]);
      for (int i = lane; i < GQ * kD / 8; i += 32) qdst[i] = __ldg(qsrc + i);
      __syncwarp();
      float acc[GQ];
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) acc[hh] = 0.0f;
#pragma unroll 4
      for (int e = 0; e < kD; ++e) {
        const float w = bf_to_f(X.w[e * kDIdx + lane]);
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) acc[hh] = fmaf(bf_to_f(X.q[hh][e]), w, acc[hh]);
      }
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) X.qp[hh][lane] = acc[hh] * kInvSqrtDIdx;
      __syncwarp();
      // registers in the rotated chunk order: step p covers chunk (p + rot) mod 4
#pragma unroll
      for (int hh = 0; hh < Sp::HPT; ++hh) {
        const float* qh = X.qp[hs * Sp::HPT + hh];
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          const int c = (p + rot) & 3;
#pragma unroll
          for (int j = 0; j < 4; ++j) qr[hh][4 * p + j] = make_float2(qh[8 * c + 2 * j], qh[8 * c + 2 * j + 1]);
        }
      }
      __syncwarp();
      cur_bg = bg;
    }
    const bool ok = mbar_wait(&S.full[slot], ph);
    if (!__all_sync(0xffffffffu, ok)) {
      record_error(err, kErrTimeout);
      return;
    }
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
      for (int hh = 0; hh < Sp::HPT; ++hh) out_base[hh * nc_pad + tok] = acc[hh].x + acc[hh].y;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[slot]);
  }
}

template <int GQ>
int launch_gq(const qasc_shape& s, const Regions& R, const uint16_t* index, const uint16_t* q, const uint16_t* W,
              float* scores, int64_t nc_pad, const DeviceInfo& dev, cudaStream_t stream) {
  const int tiles_per_bg = static_cast<int>((R.nc() + kTileTok - 1) / kTileTok);
  const int total = tiles_per_bg * s.B * s.Hkv;
  const int grid = total < dev.num_sms ? total : dev.num_sms;
  score_kernel<GQ><<<grid, kThreads, sizeof(ScoreSmem<GQ>), stream>>>(
      index, q, W, scores, s.Hq, s.Hkv, s.n_cap, static_cast<int>(R.c0), static_cast<int>(R.nc()), nc_pad,
      tiles_per_bg, total, dev.err_word);
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

int launch_scores(const qasc_shape& s, const qasc_ts_params& p, const uint16_t* q, const uint16_t* W,
                  const uint16_t* index, float* scores, int64_t nc_pad, const DeviceInfo& dev, cudaStream_t stream) {
  const Regions R = regions_of(s.n, p.sink, p.local);
  if (R.nc() <= 0) return 0;
  switch (s.Hq / s.Hkv) {
    case 1: return launch_gq<1>(s, R, index, q, W, scores, nc_pad, dev, stream);
    case 2: return launch_gq<2>(s, R, index, q, W, scores, nc_pad, dev, stream);
    case 4: return launch_gq<4>(s, R, index, q, W, scores, nc_pad, dev, stream);
    case 8: return launch_gq<8>(s, R, index, q, W, scores, nc_pad, dev, stream);
    default: return -1;
  }
}

}  // namespace qasc

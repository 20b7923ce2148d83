// Per-head index scores for every candidate token.
//
// TokenSelect page, section "Query-Key Dot Product Index", equation Score_h:
//   Score_h(i) = q'_h . k_index(i) / sqrt(d'),  q'_h = W_{g(h)}^T q_h (fp32).
//
// This is the dominant HBM stream of the decode step: every candidate's 64-byte
// index row is read once.  A persistent grid (one CTA per SM) walks contiguous
// runs of 256-token tiles; one producer warp streams tiles into a 4-deep ring
// of shared-memory stages with 3-D TMA copies (64-byte swizzle so that a thread
// reading one 64-byte row hits every bank once per 8-thread phase), and eight
// consumer warps turn each row into scores with packed fp32 FMAs (f32x2).
// With GQ query heads per KV head, a token row is shared by GQ/HPT threads,
// each holding HPT heads' projected queries in registers.
#include <cuda.h>

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

__host__ __device__ constexpr size_t score_smem_bytes(int gq) {
  return 1024 /*alignment slack*/ + static_cast<size_t>(kStages) * kTileBytes + 2 * kStages * sizeof(uint64_t) +
         static_cast<size_t>(kConsumerWarps) * gq * kDIdx * sizeof(float);
}

template <int GQ>
__global__ void __launch_bounds__(kThreads, 1) score_kernel(const __grid_constant__ CUtensorMap tmap,
                                                           const uint16_t* __restrict__ q,
                                                           const uint16_t* __restrict__ W,
                                                           float* __restrict__ scores, int Hq, int Hkv, int c0,
                                                           int nc, int64_t nc_pad, int tiles_per_bg,
                                                           int total_tiles, unsigned* err) {
  using S = Split<GQ>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stage = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(stage + kStages * kTileBytes);
  uint64_t* empty = full + kStages;
  float* qp_s = reinterpret_cast<float*>(empty + kStages);  // [warp][GQ][32]

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int it0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * total_tiles / G);
  const int it1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * total_tiles / G);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ---- producer: one lane issues the tile copies
    if (lane == 0) {
      prefetch_tensormap(&tmap);
      const uint64_t pol = policy_evict_first();
      for (int it = it0; it < it1; ++it) {
        const int k = it - it0;
        const int slot = k % kStages;
        const uint32_t ph = (k / kStages) & 1u;
        if (!mbar_wait(&empty[slot], ph ^ 1u)) {
          record_error(err, kErrTimeout);
          break;
        }
        const int bg = it / tiles_per_bg;
        const int t = it - bg * tiles_per_bg;
        mbar_arrive_expect_tx(&full[slot], kTileBytes);
        asm volatile(
            "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
            "[%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(stage + slot * kTileBytes)),
            "l"(&tmap), "r"(0), "r"(c0 + t * kTileTok), "r"(bg), "r"(smem_u32(&full[slot])), "l"(pol)
            : "memory");
      }
    }
    return;
  }

  // ---- consumers
  const int hs = tid % S::TPT;   // which HPT-head slice of the group
  const int r0 = tid / S::TPT;   // first row handled in a tile
  constexpr int kRowStep = kConsumers / S::TPT;
  float2 qr[S::HPT][kDIdx / 2];
  int cur_bg = -1;
  int b = 0, g = 0;

  for (int it = it0; it < it1; ++it) {
    const int k = it - it0;
    const int slot = k % kStages;
    const uint32_t ph = (k / kStages) & 1u;
    const int bg = it / tiles_per_bg;
    const int t = it - bg * tiles_per_bg;
    if (bg != cur_bg) {
      // q'_h = W_g^T q_h for the GQ heads of this KV head, computed by each
      // warp into its own scratch row (lane j owns column j), scaled by
      // 1/sqrt(d').  Same arithmetic in every warp, so identical values.
      b = bg / Hkv;
      g = bg - b * Hkv;
      float* qw = qp_s + warp * GQ * kDIdx;
      const uint16_t* wcol = W + static_cast<int64_t>(g) * kD * kDIdx + lane;
      for (int hh = 0; hh < GQ; ++hh) {
        const uint16_t* qrow = q + (static_cast<int64_t>(b) * Hq + g * GQ + hh) * kD;
        float acc = 0.0f;
#pragma unroll 8
        for (int e = 0; e < kD; ++e) acc = fmaf(bf_to_f(__ldg(qrow + e)), bf_to_f(__ldg(wcol + e * kDIdx)), acc);
        qw[hh * kDIdx + lane] = acc * kInvSqrtDIdx;
      }
      __syncwarp();
#pragma unroll
      for (int hh = 0; hh < S::HPT; ++hh)
#pragma unroll
        for (int p = 0; p < kDIdx / 2; ++p)
          qr[hh][p] = make_float2(qw[(hs * S::HPT + hh) * kDIdx + 2 * p], qw[(hs * S::HPT + hh) * kDIdx + 2 * p + 1]);
      __syncwarp();
      cur_bg = bg;
    }
    const bool ok = mbar_wait(&full[slot], ph);
    if (!__all_sync(0xffffffffu, ok)) {
      record_error(err, kErrTimeout);
      return;
    }
    const uint8_t* st = stage + slot * kTileBytes;
    float* out_base = scores + (static_cast<int64_t>(b) * Hq + g * GQ + hs * S::HPT) * nc_pad;
#pragma unroll 1
    for (int r = r0; r < kTileTok; r += kRowStep) {
      const int swz = (r >> 1) & 3;
      const int tok = t * kTileTok + r;
      float2 acc[S::HPT];
#pragma unroll
      for (int hh = 0; hh < S::HPT; ++hh) acc[hh] = make_float2(0.0f, 0.0f);
      // One 16-byte chunk (8 index values) at a time keeps few values live.
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const uint4 c = *reinterpret_cast<const uint4*>(st + r * 64 + ((p ^ swz) << 4));
        const float2 x0 = bf2_to_f2(c.x), x1 = bf2_to_f2(c.y), x2 = bf2_to_f2(c.z), x3 = bf2_to_f2(c.w);
#pragma unroll
        for (int hh = 0; hh < S::HPT; ++hh) {
          acc[hh] = ffma2(qr[hh][4 * p + 0], x0, acc[hh]);
          acc[hh] = ffma2(qr[hh][4 * p + 1], x1, acc[hh]);
          acc[hh] = ffma2(qr[hh][4 * p + 2], x2, acc[hh]);
          acc[hh] = ffma2(qr[hh][4 * p + 3], x3, acc[hh]);
        }
      }
      if (tok < nc) {
#pragma unroll
        for (int hh = 0; hh < S::HPT; ++hh) out_base[hh * nc_pad + tok] = acc[hh].x + acc[hh].y;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
  }
}

template <int GQ>
int launch_gq(const CUtensorMap& tmap, const qasc_shape& s, const Regions& R, const uint16_t* q, const uint16_t* W,
              float* scores, int64_t nc_pad, const DeviceInfo& dev, cudaStream_t stream) {
  const int tiles_per_bg = static_cast<int>((R.nc() + kTileTok - 1) / kTileTok);
  const int total = tiles_per_bg * s.B * s.Hkv;
  const int grid = total < dev.num_sms ? total : dev.num_sms;
  const size_t smem = score_smem_bytes(GQ);
  cudaError_t e = cudaFuncSetAttribute(score_kernel<GQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  score_kernel<GQ><<<grid, kThreads, smem, stream>>>(tmap, q, W, scores, s.Hq, s.Hkv, static_cast<int>(R.c0),
                                                    static_cast<int>(R.nc()), nc_pad, tiles_per_bg, total,
                                                    dev.err_word);
  return cudaGetLastError();
}

}  // namespace

int launch_scores(const qasc_shape& s, const qasc_ts_params& p, const uint16_t* q, const uint16_t* W,
                  const uint16_t* index, float* scores, int64_t nc_pad, const DeviceInfo& dev, cudaStream_t stream) {
  const Regions R = regions_of(s.n, p.sink, p.local);
  if (R.nc() <= 0) return 0;
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cudaErrorNotSupported;
  // The index viewed as a 3-D tensor [B*Hkv][n_cap][32] of bf16; a box is one
  // 256-row tile of one (b, g).  Rows past n_cap read as zero.
  alignas(64) CUtensorMap tmap;
  const uint64_t gdim[3] = {static_cast<uint64_t>(kDIdx), static_cast<uint64_t>(s.n_cap),
                            static_cast<uint64_t>(s.B) * s.Hkv};
  const uint64_t gstride[2] = {kDIdx * 2ull, static_cast<uint64_t>(s.n_cap) * kDIdx * 2ull};
  const unsigned box[3] = {kDIdx, kTileTok, 1};
  const unsigned estr[3] = {1, 1, 1};
  int rc = enc(&tmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(index), gdim, gstride, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (rc != 0) return cudaErrorInvalidValue;
  const int gq = s.Hq / s.Hkv;
  switch (gq) {
    case 1: return launch_gq<1>(tmap, s, R, q, W, scores, nc_pad, dev, stream);
    case 2: return launch_gq<2>(tmap, s, R, q, W, scores, nc_pad, dev, stream);
    case 4: return launch_gq<4>(tmap, s, R, q, W, scores, nc_pad, dev, stream);
    case 8: return launch_gq<8>(tmap, s, R, q, W, scores, nc_pad, dev, stream);
    case 16: return launch_gq<16>(tmap, s, R, q, W, scores, nc_pad, dev, stream);
    default: return -1;
  }
}

}  // namespace qasc

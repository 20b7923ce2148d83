// Per-head index scores for every candidate token.
//
// TokenSelect page, section "Query-Key Dot Product Index", equation Score_h:
//   Score_h(i) = q'_h . k_index(i) / sqrt(d'),  q'_h = W_{g(h)}^T q_h (fp32).
//
// This is the dominant HBM stream of the select step: every candidate's
// 64-byte index row is read once.  The dot products of one (b, g) form a
// small dense contraction, [256 tokens x 32] x [32 x Gq], which runs on the
// tcgen05 tensor cores so that the CUDA cores only store scores and count
// histograms:
//   - The B operand of a (b, g) segment: q'_h / sqrt(d') in fp32, split into
//     three bf16 parts hi + mid + lo (each the round-to-nearest-even of what
//     the earlier parts leave; their sum equals the fp32 value to ~2^-24
//     relative), as row part * Gq + head of an N-row tile (N = 16, or 32 for
//     Gq = 8; zero padded) of 32 bf16 in the 64-byte-swizzled K-major layout.
//     The epilogue warps build it in shared memory (W_g and the queries
//     staged there first): the CTA's first two segments' operands before the
//     first tile, each later one while the segment two back is flushed.
//   - The kernel is persistent (one CTA per SM over contiguous runs of
//     512-token tiles).  A TMA warp loads each 32 KB index tile (2-D tensor
//     map, 64-byte swizzle, two 256-row boxes) into a 4-stage ring; one MMA
//     thread issues eight
//     M=128 x N x K=16 MMAs per tile (four 128-token quarters x two K steps,
//     interleaved so that the four accumulation chains overlap) into TMEM;
//     eight epilogue warps (two per TMEM lane quarter) read two tokens' 3 Gq
//     partial scores per thread, add the parts (lo + mid first), store the
//     scores and count the first radix digit of each head's threshold search
//     in shared histograms, flushed per (b, g) segment.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace qasc {
namespace {

constexpr int kTileTok = 512;                 // tokens per stage
constexpr int kTileBytes = kTileTok * kDIdx * 2;
constexpr int kBoxRows = 256;                 // rows per TMA box (two boxes per stage; paged: min(P, 256))
constexpr int kSub = kTileTok / 128;          // 128-token MMA tiles per stage
constexpr int kStages = 4;
constexpr int kAccStages = 4;                 // TMEM accumulators (one stage each)
constexpr int kEpiWarps = 8;
constexpr int kEpi = 32 * kEpiWarps;
constexpr int kThreads = kEpi + 64;           // TMA warp, MMA warp, epilogue warps
constexpr int kParts = 3;                     // q' = hi + mid + lo
constexpr int kBStride = 2048;                // bytes per (b, g) of the B operand buffer
// MMA N: the 3 Gq rows of (part, head), padded to a multiple of 16.
__host__ __device__ constexpr int mma_n(int gq) { return gq <= 4 ? 16 : 32; }
__host__ __device__ constexpr int tmem_cols(int gq) { return kAccStages * kSub * mma_n(gq); }
constexpr float kInvSqrtDIdx = 0.17677669529663688f;  // 1 / sqrt(32)

// The CTA of a persistent grid of G CTAs over `total` items (CTA c takes
// [c total / G, (c+1) total / G)) that holds item x.
__host__ __device__ __forceinline__ int first_cta(int64_t x, int64_t total, int G) {
  int64_t c = ((x + 1) * G + total - 1) / total - 1;
  return static_cast<int>(c < 0 ? 0 : (c >= G ? G - 1 : c));
}

// First radix digit of the per-head threshold search (see ts_select.cu):
// the top hist_bits(GQ) bits of the order-preserving score key.
__host__ __device__ constexpr int hist_bits(int gq) { return gq <= 4 ? 12 : 11; }

template <int GQ>
struct ScoreSmem {
  uint8_t tile[kStages][kTileBytes];          // 1024-byte aligned (swizzle atoms)
  uint8_t bq[2][kBStride];                    // B operand of two segments
  uint32_t hist[GQ][1 << hist_bits(GQ)];
  alignas(16) uint16_t wst[kD * kDIdx];       // W_g of the operand being built
  float qst[GQ][kD];                          // its queries
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t bfull[2];
  uint64_t bempty[2];
  uint64_t acc_full[kAccStages];
  uint64_t acc_empty[kAccStages];
  uint32_t tmem_base;
};

// Round to nearest even bf16 (finite inputs).
__device__ __forceinline__ uint32_t bf16_rne_bits(float x) {
  uint32_t u = __float_as_uint(x);
  u += 0x7fffu + ((u >> 16) & 1u);
  return u >> 16;
}

// Byte offset of element (n, k) of an N x 32 bf16 K-major tile stored with
// the 64-byte swizzle (16-byte chunk c of row n at chunk c ^ ((n / 2) mod 4)).
__device__ __forceinline__ int sw64_offset(int n, int k) {
  return n * 64 + ((((k >> 3) ^ (n >> 1)) & 3) << 4) + (k & 7) * 2;
}

// The epilogue threads (etid = 0..kEpi-1) build segment bg's B operand in
// slot `slot` and publish it on bfull[slot].
template <int GQ>
__device__ void build_b(ScoreSmem<GQ>& S, const uint16_t* __restrict__ q, const uint16_t* __restrict__ W, int bg,
                        int Hq, int Hkv, int slot, int etid) {
  constexpr int kTPO = 8 / GQ;                 // threads per output (32 GQ outputs, 256 threads)
  const int b = bg / Hkv, g = bg - b * Hkv;
  const uint4* w4 = reinterpret_cast<const uint4*>(W + static_cast<int64_t>(g) * kD * kDIdx);
  for (int i = etid; i < kD * kDIdx / 8; i += kEpi) reinterpret_cast<uint4*>(S.wst)[i] = __ldg(w4 + i);
  const uint16_t* qsrc = q + (static_cast<int64_t>(b) * Hq + g * GQ) * kD;
  for (int i = etid; i < GQ * kD; i += kEpi) S.qst[i / kD][i % kD] = bf_to_f(qsrc[i]);
  named_bar_sync(2, kEpi);
  const int o = etid / kTPO, part = etid % kTPO;
  const int hh = o / kDIdx, j = o % kDIdx;
  constexpr int kSpan = kD / kTPO;
  float acc = 0.0f;
#pragma unroll 8
  for (int e = part * kSpan; e < (part + 1) * kSpan; ++e) acc = fmaf(S.qst[hh][e], bf_to_f(S.wst[e * kDIdx + j]), acc);
#pragma unroll
  for (int off = kTPO / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (part == 0) {
    const float x = acc * kInvSqrtDIdx;
    const uint32_t hi = bf16_rne_bits(x);
    const float r1 = x - __uint_as_float(hi << 16);
    const uint32_t mid = bf16_rne_bits(r1);
    const float r2 = r1 - __uint_as_float(mid << 16);
    const uint32_t lo = bf16_rne_bits(r2);
    uint8_t* dst = S.bq[slot];
    *reinterpret_cast<uint16_t*>(dst + sw64_offset(hh, j)) = static_cast<uint16_t>(hi);
    *reinterpret_cast<uint16_t*>(dst + sw64_offset(GQ + hh, j)) = static_cast<uint16_t>(mid);
    *reinterpret_cast<uint16_t*>(dst + sw64_offset(2 * GQ + hh, j)) = static_cast<uint16_t>(lo);
  }
  fence_async_smem();
  named_bar_sync(2, kEpi);
  if (etid == 0) mbar_arrive(&S.bfull[slot]);
}

// Where the index tiles come from.  Contiguous (table == nullptr): tile t of
// (b, g) holds candidates [c0 + 512 t, ...) of the [B][Hkv][n_cap] rows, in
// two 256-row boxes.  Paged: tiles start at token 0 (tile t holds tokens
// [512 t, 512 t + 512), so every box of box_rows = min(P, 256) rows lies in
// one page); rows below c0 are skipped, and boxes wholly at or above c1 are
// not loaded.
struct IdxSrc {
  const int32_t* table;      // [B][pages_per_seq], or nullptr
  int64_t pages_per_seq, num_pages;
  int page_shift, box_rows, box_shift;   // box_rows = 2^box_shift
  int pos_shift;             // token of tile row 0 minus the candidate position of tile row 0 (paged: c0)
  int c1;
};

template <int GQ>
__global__ void __launch_bounds__(kThreads, 1) score_kernel(const __grid_constant__ CUtensorMap tmap_idx,
                                                           const IdxSrc src,
                                                           const uint16_t* __restrict__ q,
                                                           const uint16_t* __restrict__ W,
                                                           float* __restrict__ scores,
                                                           uint32_t* __restrict__ hist_part, int Hq, int Hkv,
                                                           int64_t n_cap, int c0, int nc, int64_t nc_pad,
                                                           int tiles_per_bg, int total_tiles, int max_splits,
                                                           unsigned* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  ScoreSmem<GQ>& S = *reinterpret_cast<ScoreSmem<GQ>*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  constexpr int kNB = 1 << hist_bits(GQ);
  constexpr int kShift = 32 - hist_bits(GQ);
  constexpr int kN = mma_n(GQ);

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  const int it0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * total_tiles / G);
  const int it1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * total_tiles / G);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.bfull[i], 1);
      mbar_init(&S.bempty[i], 1);
    }
    for (int i = 0; i < kAccStages; ++i) {
      mbar_init(&S.acc_full[i], 1);
      mbar_init(&S.acc_empty[i], kEpiWarps);
    }
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&S.tmem_base, tmem_cols(GQ));
  if (warp >= 2) {
    for (int i = tid - 64; i < GQ * kNB; i += kEpi) (&S.hist[0][0])[i] = 0;
    // operand padding rows 3 GQ .. N-1 stay zero
    for (int i = tid - 64; i < 2 * (kN - kParts * GQ) * kDIdx; i += kEpi) {
      const int sl = i / ((kN - kParts * GQ) * kDIdx), r = i % ((kN - kParts * GQ) * kDIdx);
      *reinterpret_cast<uint16_t*>(S.bq[sl] + sw64_offset(kParts * GQ + r / kDIdx, r % kDIdx)) = 0;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  // While the preceding kernel drains: warm L2 with this CTA's first ring of
  // index tiles (contiguous cache) and the projection and queries of its
  // first two segments.
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmap_idx);
    if (src.table == nullptr)
      for (int it = it0; it < it1 && it < it0 + kStages; ++it) {
        const int bg = it / tiles_per_bg, t = it - (it / tiles_per_bg) * tiles_per_bg;
        const int row = static_cast<int>(static_cast<int64_t>(bg) * n_cap + c0 + static_cast<int64_t>(t) * kTileTok);
#pragma unroll
        for (int bx = 0; bx < kTileTok / kBoxRows; ++bx) tma_prefetch_2d(&tmap_idx, 0, row + bx * kBoxRows);
      }
  } else if (warp >= 2 && it0 < it1) {
    const int etid = tid - 64;
    const int bg0 = it0 / tiles_per_bg;
    const int nseg = (it1 - 1) / tiles_per_bg - bg0 + 1;
    constexpr int kWLines = kD * kDIdx * 2 / 128, kQLines = GQ * kD * 2 / 128;
    for (int i = etid; i < (nseg < 2 ? nseg : 2) * (kWLines + kQLines); i += kEpi) {
      const int sg = i / (kWLines + kQLines), r = i - sg * (kWLines + kQLines);
      const int b = (bg0 + sg) / Hkv, g = (bg0 + sg) - b * Hkv;
      const uint16_t* line = r < kWLines ? W + static_cast<int64_t>(g) * kD * kDIdx + r * 64
                                         : q + (static_cast<int64_t>(b) * Hq + g * GQ) * kD + (r - kWLines) * 64;
      prefetch_l2(line);
    }
  }
  pdl_wait();

  if (warp == 0) {
    // ---- TMA issue: index tiles.  Lane 0 issues; in a paged pool the whole
    // warp reads the block table ahead, one entry per lane for a window of
    // 32 / ppt tiles (ppt = entries per tile), the next window loaded while
    // the current one is used.
    const uint64_t pol = policy_evict_first();
    const bool paged = src.table != nullptr;
    const int ppt = paged ? max(1, kTileTok >> src.page_shift) : 1;
    const int tpw = 32 / ppt;
    auto window_entry = [&](int w) -> int32_t {   // this lane's entry of the window starting at tile w
      const int itl = w + lane / ppt;
      if (!paged || itl >= it1) return 0;
      const int bg_ = itl / tiles_per_bg, t_ = itl - bg_ * tiles_per_bg;
      const int L = t_ * kTileTok + (lane % ppt) * (ppt > 1 ? (1 << src.page_shift) : 0);
      if (L >= src.c1) return 0;   // past c1: never loaded
      return __ldg(src.table + static_cast<int64_t>(bg_ / Hkv) * src.pages_per_seq + (L >> src.page_shift));
    };
    int w0 = it0;
    int32_t cur = window_entry(w0);
    int32_t nxt = window_entry(w0 + tpw);
    int issued = 0;
    for (int it = it0; it < it1; ++it) {
      const int k = it - it0;
      const int bg = it / tiles_per_bg;
      const int t = it - bg * tiles_per_bg;
      const int slot = k % kStages;
      if (paged && it >= w0 + tpw) {   // warp-uniform
        w0 += tpw;
        cur = nxt;
        nxt = window_entry(w0 + tpw);
      }
      int nbox = kTileTok / kBoxRows;
      if (paged) {   // boxes that hold tokens below c1
        const int rem = src.c1 - t * kTileTok;
        nbox = rem >= kTileTok ? (kTileTok >> src.box_shift) : ((rem + src.box_rows - 1) >> src.box_shift);
      }
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&S.empty[slot], ((k / kStages) & 1u) ^ 1u);
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        if (lane == 0) record_error(err, kErrTimeout);
        break;
      }
      if (!paged) {
        if (lane == 0) {
          mbar_arrive_expect_tx(&S.full[slot], kTileBytes);
          const int row = static_cast<int>(static_cast<int64_t>(bg) * n_cap + c0 + static_cast<int64_t>(t) * kTileTok);
#pragma unroll
          for (int bx = 0; bx < kTileTok / kBoxRows; ++bx)
            tma_load_2d_hint(&S.tile[slot][bx * kBoxRows * kDIdx * 2], &tmap_idx, 0, row + bx * kBoxRows,
                             &S.full[slot], pol);
        }
      } else {
        if (lane == 0) mbar_arrive_expect_tx(&S.full[slot], static_cast<uint32_t>(nbox) << (src.box_shift + 6));
        const int g = bg - (bg / Hkv) * Hkv;
        // box bx lies in the tile's page bx (P <= 256: one page per box) or in its only page
        for (int bx = 0; bx < nbox; ++bx) {   // warp-uniform
          int32_t page = __shfl_sync(0xffffffffu, cur, (it - w0) * ppt + (ppt > 1 ? bx : 0));
          if (lane == 0) {
            if (page < 0 || page >= src.num_pages) {
              record_error(err, kErrBadPage);
              page = 0;
            }
            const int L = t * kTileTok + (bx << src.box_shift);
            const int row = static_cast<int>(((static_cast<int64_t>(page) * Hkv + g) << src.page_shift) +
                                             (L & ((1 << src.page_shift) - 1)));
            tma_load_2d_hint(&S.tile[slot][bx << (src.box_shift + 6)], &tmap_idx, 0, row, &S.full[slot], pol);
          }
        }
      }
      issued = k + 1;
      __syncwarp();
    }
    // no copy may land after the CTA has left: wait (bounded) for each
    // slot's last tile (already complete unless a wait ran out elsewhere)
    if (lane == 0)
      for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
        if (!mbar_wait(&S.full[j % kStages], (j / kStages) & 1u)) {
          record_error(err, kErrTimeout);
          break;
        }
  } else if (warp == 1) {
    // ---- MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = mma_idesc(128, kN);
      int seg = -1, cur_bg = -1;
      for (int it = it0; it < it1; ++it) {
        const int k = it - it0;
        const int bg = it / tiles_per_bg;
        if (bg != cur_bg) {
          if (cur_bg >= 0) mma_commit(&S.bempty[seg & 1]);   // the previous segment's B is free once these finish
          ++seg;
          cur_bg = bg;
          if (!mbar_wait(&S.bfull[seg & 1], (seg >> 1) & 1u)) {
            record_error(err, kErrTimeout);
            break;
          }
        }
        const int slot = k % kStages;
        const int ab = k % kAccStages;
        if (!mbar_wait(&S.full[slot], (k / kStages) & 1u) ||
            !mbar_wait(&S.acc_empty[ab], ((k / kAccStages) & 1u) ^ 1u)) {
          record_error(err, kErrTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(&S.tile[slot][0]);
        const uint32_t b0 = smem_u32(&S.bq[seg & 1][0]);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
          for (int sub = 0; sub < kSub; ++sub)
            mma_bf16(tmem + (ab * kSub + sub) * kN, sw64_desc(a0 + sub * 128 * kDIdx * 2 + kk * 32),
                     sw64_desc(b0 + kk * 32), idesc, kk);
        }
        mma_commit(&S.empty[slot]);
        mma_commit(&S.acc_full[ab]);
      }
    }
  } else {
    // ---- epilogue: two tokens per thread per tile (quarters sub and sub + 2)
    const int quarter = warp & 3;
    const int sub = (warp - 2) >> 2;
    const int row = sub * 128 + quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + sub * kN;
    const int etid = tid - 64;
    // scores stay in L2 for the threshold and vote passes (the vote pass
    // drops them afterwards)
    const uint64_t keep = policy_evict_last();
    int cur_bg = -1, b = 0, g = 0;
    bool dead = false;   // a bounded wait ran out: skip work but keep every barrier

    // Writes this CTA's histograms of (b, g) to its partial slot and clears them.
    auto flush = [&](int fbg) {
      named_bar_sync(1, kEpi);
      const int split = static_cast<int>(blockIdx.x) - first_cta(static_cast<int64_t>(fbg) * tiles_per_bg,
                                                                   total_tiles, G);
      uint4* dst = reinterpret_cast<uint4*>(hist_part + (static_cast<int64_t>(fbg) * max_splits + split) * GQ * kNB);
      uint4* src = reinterpret_cast<uint4*>(&S.hist[0][0]);
      for (int i = etid; i < GQ * kNB / 4; i += kEpi) {
        dst[i] = src[i];
        src[i] = make_uint4(0, 0, 0, 0);
      }
      named_bar_sync(1, kEpi);
    };

    // B operands: the first two segments now, segment j + 2 after segment j
    const int bg_first = it0 / tiles_per_bg;
    const int nseg = it1 > it0 ? (it1 - 1) / tiles_per_bg - bg_first + 1 : 0;
    for (int j = 0; j < min(2, nseg); ++j) build_b<GQ>(S, q, W, bg_first + j, Hq, Hkv, j, etid);
    auto next_b = [&](int fbg) {   // after flushing segment fbg
      const int j = fbg - bg_first;
      if (j + 2 >= nseg) return;
      if (etid == 0 && !mbar_wait(&S.bempty[j & 1], (j >> 1) & 1u)) record_error(err, kErrTimeout);
      build_b<GQ>(S, q, W, fbg + 2, Hq, Hkv, j & 1, etid);
    };

    for (int it = it0; it < it1; ++it) {
      const int k = it - it0;
      const int ab = k % kAccStages;
      const int bg = it / tiles_per_bg;
      const int t = it - bg * tiles_per_bg;
      if (bg != cur_bg) {
        if (cur_bg >= 0) {
          flush(cur_bg);
          next_b(cur_bg);
        }
        b = bg / Hkv;
        g = bg - b * Hkv;
        cur_bg = bg;
      }
      if (!dead) {
        const bool ok = mbar_wait(&S.acc_full[ab], (k / kAccStages) & 1u);
        if (!__all_sync(0xffffffffu, ok)) {
          record_error(err, kErrTimeout);
          dead = true;
        }
      }
      if (dead) continue;
      tc_fence_after();
      float v[2][kN];
      tmem_ld_cols<kN>(tl + ab * kSub * kN, v[0]);
      tmem_ld_cols<kN>(tl + ab * kSub * kN + 2 * kN, v[1]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.acc_empty[ab]);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int tok = t * kTileTok + row + u * 256 - src.pos_shift;
        if (tok >= 0 && tok < nc) {
          float* out = scores + (static_cast<int64_t>(b) * Hq + g * GQ) * nc_pad + tok;
#pragma unroll
          for (int hh = 0; hh < GQ; ++hh) {
            const float sc = (v[u][2 * GQ + hh] + v[u][GQ + hh]) + v[u][hh];
            st_global_hint(out + hh * nc_pad, sc, keep);
            atomicAdd(&S.hist[hh][ord_key(sc) >> kShift], 1u);
          }
        }
      }
    }
    if (cur_bg >= 0) flush(cur_bg);
  }
  tc_fence_before();
  __syncthreads();
  pdl_trigger();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols(GQ));
  }
}

// Tensor map over the index as rows of 32 bf16 (64 bytes), box_rows-row
// boxes, 64-byte swizzle.
int encode_index_map(CUtensorMap* m, const uint16_t* index, uint64_t rows, unsigned box_rows, EncodeTiledFn enc) {
  const uint64_t gdim[2] = {static_cast<uint64_t>(kDIdx), rows};
  const uint64_t gstride[1] = {static_cast<uint64_t>(kDIdx) * 2};
  const unsigned box[2] = {static_cast<unsigned>(kDIdx), box_rows};
  const unsigned estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(index), gdim, gstride, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <int GQ>
int launch_gq(const qasc_shape& s, const Regions& R, const uint16_t* index, const uint16_t* q, const uint16_t* W,
              const ScoreOut& o, const DeviceInfo& dev, cudaStream_t stream) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cudaErrorNotSupported;
  alignas(64) CUtensorMap tmap;
  IdxSrc src = {};
  const bool paged = o.pm.table != nullptr;
  uint64_t rows = static_cast<uint64_t>(s.B) * s.Hkv * s.n_cap;
  unsigned box_rows = kBoxRows;
  if (paged) {
    src.table = o.pm.table;
    src.pages_per_seq = o.pm.pages_per_seq;
    src.num_pages = o.pm.num_pages;
    src.page_shift = o.pm.page_shift;
    box_rows = (1u << o.pm.page_shift) < kBoxRows ? (1u << o.pm.page_shift) : kBoxRows;
    src.box_rows = static_cast<int>(box_rows);
    src.box_shift = 0;
    while ((1u << src.box_shift) < box_rows) ++src.box_shift;
    src.pos_shift = static_cast<int>(R.c0);
    src.c1 = static_cast<int>(R.c1);
    rows = static_cast<uint64_t>(o.pm.num_pages) * s.Hkv << o.pm.page_shift;
  }
  if (encode_index_map(&tmap, index, rows, box_rows, enc) != 0) return cudaErrorInvalidValue;
  const ScoreGrid sg = score_grid(s, score_span(R, paged), dev.num_sms);
  return launch_dependent(score_kernel<GQ>, dim3(sg.grid), dim3(kThreads), sizeof(ScoreSmem<GQ>) + 1024, stream, 1,
                          tmap, src, q, W, o.scores, o.hist, s.Hq, s.Hkv, s.n_cap,
                          static_cast<int>(R.c0), static_cast<int>(R.nc()), o.nc_pad, sg.tiles_per_bg, sg.total,
                          o.max_splits, dev.err_word);
}

template <int GQ>
cudaError_t configure_gq() {
  return cudaFuncSetAttribute(score_kernel<GQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(sizeof(ScoreSmem<GQ>) + 1024));
}

}  // namespace

cudaError_t configure_score_kernels(const DeviceInfo&) {
  cudaError_t e;
  if ((e = configure_gq<1>()) != cudaSuccess) return e;
  if ((e = configure_gq<2>()) != cudaSuccess) return e;
  if ((e = configure_gq<4>()) != cudaSuccess) return e;
  return configure_gq<8>();
}

ScoreGrid score_grid(const qasc_shape& s, int64_t span, int num_sms) {
  ScoreGrid g;
  g.tiles_per_bg = static_cast<int>((span + kTileTok - 1) / kTileTok);
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

// snapkv_compress: observation-window attention scores, pooled, top-c per KV
// head, gathered into a compact cache.
//
// SnapKV page, section "Attention Score計算とPooling": A = softmax(Q_obs K^T /
// sqrt(d_k)) per head and its mean over the window rows; section "Top-k
// SelectionとCluster-based Retention": the c highest; section "アルゴリズム":
// average pooling (kernel k, padding k/2, stride 1), top-k of min(c, n), sort,
// gather.  Grouped-query reading: the mean runs over the Gq heads of a KV
// group too, so one group's Gq * w window rows (128 for Gq = 4, w = 32) form
// one 128-row tensor-core tile.
//
// Two passes over the keys, both on tcgen05 tensor cores (bf16 operands in
// 128B-swizzled shared memory loaded by TMA, fp32 accumulators in TMEM):
//   pass 1: D = Q K_tile^T (rows in TMEM lanes): per-row online max and sum
//           of exp, written as per-CTA partial statistics;
//   pass 2: D = K_tile Q^T (keys in TMEM lanes): each thread owns one key
//           and sums exp(x - m_r) / (R l_r) over its 32-row column slice;
//           the four slices of a key are added in slice order through
//           shared memory into the window/group mean a_j.
// A CTA is one warp of TMA issue, one warp of MMA issue (which also owns the
// TMEM allocation) and sixteen epilogue warps (four per TMEM lane quarter); a
// 5-stage ring of key tiles and two TMEM accumulators keep loads, MMAs and
// epilogues overlapped.  Each pass is one launch over every KV head (a grid
// of key-range parts per (b, g), one CTA per SM); pass 2 walks each CTA's
// tiles from the end, where pass 1 finished, so that it starts on the keys
// most likely still in L2.  (Grouping the KV heads so that a group's keys
// fit in half of L2, one launch pair per group, measured slower: 170 against
// 140 us per layer at B2, n = 65536, with four groups.)
// Then: pool_kernel (3-tap mean, zero padded), topc_kernel (radix select of
// the c-th largest pooled score per KV head, ties to the lower index, and an
// ordered compaction of the kept indices) and gather_kernel (bit copies of
// the kept K and V rows).
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace qasc {
namespace {

namespace cg = cooperative_groups;

constexpr int kTileKeys = 128;                 // keys per tile
constexpr int kRowsTile = 128;                 // query rows per group tile
constexpr int kBoxBytes = 128 * 128;           // 64 bf16 columns x 128 rows
constexpr int kTileBytes = 2 * kBoxBytes;      // full d = 128
constexpr int kKStages = 5;
constexpr int kEpiWarps = 16;                  // four per TMEM lane quarter, 32 columns each
constexpr int kSlices = kEpiWarps / 4;         // column slices of the 128-column accumulator
constexpr int kSliceCols = 128 / kSlices;
constexpr int kThreadsP = 64 + 32 * kEpiWarps;  // TMA warp, MMA warp, epilogue warps
constexpr int kTmemCols = 256;                 // two 128-column accumulators
// log2(e) / sqrt(128)
constexpr float kLogitScale = 1.4426950408889634f * 0.08838834764831845f;

struct SnapSmem {
  uint8_t q[kTileBytes];
  uint8_t k[kKStages][kTileBytes];
  uint64_t full[kKStages];
  uint64_t empty[kKStages];
  uint64_t qbar;
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint32_t tmem_base;
  alignas(16) float rowm[kRowsTile];
  float part_m[kSlices - 1][kRowsTile];   // column slices 1.. of each row (pass 1)
  float part_l[kSlices - 1][kRowsTile];
  float red[2][kSlices][kTileKeys];       // pass 2: each slice's partial mean of a tile's keys
};

// 2^x on the special-function unit (relative error ~2^-22, flushes subnormals).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct PassArgs {
  int Hq, Hkv, Gq, w, R;
  int64_t n, n_cap;
  int base_parts, extra, pstride;   // key-range parts: base_parts per (b, g), one more for the first `extra`
  int ntiles, bgs;
  int64_t n_pad;
  float* stats;       // [B*Hkv][pstride][128][2]  (max in log2 units, sum)
  float* a;           // [B*Hkv][n_pad]: the window/group mean of every key
  uint32_t* hist;     // [B*Hkv][4096] the pooled keys' histogram, zeroed by pass 1
  int64_t hist_words;
  unsigned* err;
};

// PASS 1: per-row statistics.  PASS 2: per-key window/group mean.
template <int PASS>
__global__ void __launch_bounds__(kThreadsP, 1)
    snap_pass_kernel(const PassArgs a, const __grid_constant__ CUtensorMap tmap_q,
                     const __grid_constant__ CUtensorMap tmap_k) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  SnapSmem& S = *reinterpret_cast<SnapSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // (b, g) and part of this CTA: the first `extra` (b, g) have one part more
  const int x = static_cast<int>(blockIdx.x), big = a.extra * (a.base_parts + 1);
  const int bgl = x < big ? x / (a.base_parts + 1) : a.extra + (x - big) / a.base_parts;
  const int nparts = a.base_parts + (bgl < a.extra ? 1 : 0);
  const int part = x < big ? x - bgl * (a.base_parts + 1) : (x - big) - (bgl - a.extra) * a.base_parts;
  const int bg = bgl;
  const int b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int t_begin = static_cast<int>(static_cast<int64_t>(part) * a.ntiles / nparts);
  const int t_end = static_cast<int>(static_cast<int64_t>(part + 1) * a.ntiles / nparts);
  const int ntl = t_end - t_begin;
  // pass 2 walks its tiles from the end, where pass 1 finished: those keys
  // are the ones most likely still in L2
  auto tile_of = [&](int i) { return PASS == 2 ? t_end - 1 - i : t_begin + i; };

  if (tid == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    mbar_init(&S.qbar, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.acc_full[i], 1);
      mbar_init(&S.acc_empty[i], kEpiWarps);
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, kTmemCols);
  }
  pdl_wait();   // the statistics (pass 2) and the operands may come from earlier kernels
  if (PASS == 1)   // the pooling step adds into this histogram; the previous call's reader is done
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + tid; i < a.hist_words;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
      a.hist[i] = 0u;
  if (PASS == 2 && warp >= 2 && warp < 6) {
    // Global row statistics from every part's partials.
    const int r = tid - 64;
    float m = -INFINITY, l = 0.0f;
    if (r < a.R) {
      const float* st = a.stats + (static_cast<int64_t>(bg) * a.pstride) * kRowsTile * 2 + r * 2;
      for (int p = 0; p < nparts; ++p) m = fmaxf(m, st[static_cast<int64_t>(p) * kRowsTile * 2]);
      for (int p = 0; p < nparts; ++p) {
        const float mp = st[static_cast<int64_t>(p) * kRowsTile * 2];
        if (mp != -INFINITY) l += st[static_cast<int64_t>(p) * kRowsTile * 2 + 1] * ex2(mp - m);
      }
    }
    // exp2(x - m_r) / (R l_r) = exp2(x - (m_r + log2(R l_r))): one offset
    // per row; padding rows get +inf, i.e. exp2(-inf) = 0
    S.rowm[r] = r < a.R ? m + log2f(static_cast<float>(a.R) * l) : INFINITY;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  bool dead = false;

  if (warp == 0) {
    // ---- TMA issue
    if (lane == 0) {
      prefetch_tensormap(&tmap_q);
      prefetch_tensormap(&tmap_k);
      const int qrow = (b * a.Hq + g * a.Gq) * a.w;
      mbar_arrive_expect_tx(&S.qbar, kTileBytes);
      tma_load_2d(&S.q[0], &tmap_q, 0, qrow, &S.qbar);
      tma_load_2d(&S.q[kBoxBytes], &tmap_q, 64, qrow, &S.qbar);
      const int64_t krow0 = static_cast<int64_t>(bg) * a.n_cap;
      int issued = 0;
      for (int i = 0; i < ntl; ++i) {
        const int slot = i % kKStages;
        const uint32_t ph = (i / kKStages) & 1u;
        if (!mbar_wait(&S.empty[slot], ph ^ 1u)) {
          record_error(a.err, kErrTimeout);
          break;
        }
        const int krow = static_cast<int>(krow0 + static_cast<int64_t>(tile_of(i)) * kTileKeys);
        mbar_arrive_expect_tx(&S.full[slot], kTileBytes);
        tma_load_2d(&S.k[slot][0], &tmap_k, 0, krow, &S.full[slot]);
        tma_load_2d(&S.k[slot][kBoxBytes], &tmap_k, 64, krow, &S.full[slot]);
        issued = i + 1;
      }
      // no copy may land after the CTA has left: wait (bounded) for the
      // queries and each slot's last tile (already complete unless a wait
      // ran out elsewhere)
      if (!mbar_wait(&S.qbar, 0)) record_error(a.err, kErrTimeout);
      for (int j = issued > kKStages ? issued - kKStages : 0; j < issued; ++j)
        if (!mbar_wait(&S.full[j % kKStages], (j / kKStages) & 1u)) {
          record_error(a.err, kErrTimeout);
          break;
        }
    }
  } else if (warp == 1) {
    // ---- MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = mma_idesc(128, 128);
      if (!mbar_wait(&S.qbar, 0)) {
        record_error(a.err, kErrTimeout);
        dead = true;
      }
      const uint32_t qaddr = smem_u32(&S.q[0]);
      for (int i = 0; i < ntl && !dead; ++i) {
        const int slot = i % kKStages;
        const int ab = i & 1;
        if (!mbar_wait(&S.full[slot], (i / kKStages) & 1u) || !mbar_wait(&S.acc_empty[ab], ((i >> 1) & 1u) ^ 1u)) {
          record_error(a.err, kErrTimeout);
          dead = true;
          break;
        }
        tc_fence_after();
        const uint32_t kaddr = smem_u32(&S.k[slot][0]);
        const uint32_t aaddr = PASS == 1 ? qaddr : kaddr;
        const uint32_t baddr = PASS == 1 ? kaddr : qaddr;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
          mma_bf16(tmem + ab * 128, sw128_desc(aaddr + off), sw128_desc(baddr + off), idesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(&S.empty[slot]);
        mma_commit(&S.acc_full[ab]);
      }
    }
    __syncwarp();
  } else {
    // ---- epilogue: TMEM lane quarter (warp % 4), column slice (warp - 2) / 4;
    // eight independent chains per thread keep the exp2 unit busy
    const int quarter = warp & 3;
    const int slice = (warp - 2) >> 2;
    const int lrow = 32 * quarter + lane;     // TMEM lane of this thread
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * quarter) << 16) + kSliceCols * slice;
    float m = -INFINITY, l = 0.0f;
    for (int i = 0; i < ntl; ++i) {
      const int ab = i & 1;
      bool ok = !dead && mbar_wait(&S.acc_full[ab], (i >> 1) & 1u);
      if (!__all_sync(0xffffffffu, ok)) {
        if (!dead) record_error(a.err, kErrTimeout);
        dead = true;
        if (PASS == 1) break;
        // pass 2: no work, but every per-tile barrier of its lane quarter
        named_bar_sync(2 + quarter, 32 * kSlices);
        continue;
      }
      tc_fence_after();
      const int64_t key0 = static_cast<int64_t>(tile_of(i)) * kTileKeys;
      float v[kSliceCols];
      tmem_ld_cols<kSliceCols>(tlane + ab * 128, v);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.acc_empty[ab]);   // the accumulator is in registers now
      if (PASS == 1) {
        // this thread is query row lrow; its columns are keys kSliceCols*slice + [0, kSliceCols).
        // The maximum is taken on the raw logits (the scale is positive) and
        // the scale folds into one FMA per exp2 argument; only a (b, g)'s last
        // tile has columns past n, masked to -inf.
        const int valid = static_cast<int>(min(static_cast<int64_t>(kTileKeys), a.n - key0)) - kSliceCols * slice;
        if (valid < kSliceCols) {
#pragma unroll
          for (int j = 0; j < kSliceCols; ++j)
            if (j >= valid) v[j] = -INFINITY;
        }
        float t8[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) t8[j] = v[j];
#pragma unroll
        for (int j = 8; j < kSliceCols; ++j) t8[j & 7] = fmaxf(t8[j & 7], v[j]);
        const float tm = fmaxf(fmaxf(fmaxf(t8[0], t8[1]), fmaxf(t8[2], t8[3])),
                               fmaxf(fmaxf(t8[4], t8[5]), fmaxf(t8[6], t8[7])));
        const float m_new = fmaxf(m, tm * kLogitScale);
        if (m_new != -INFINITY) {
          float s8[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) s8[j] = 0.0f;
#pragma unroll
          for (int j = 0; j < kSliceCols; ++j) s8[j & 7] += ex2(fmaf(v[j], kLogitScale, -m_new));
          l = (m == -INFINITY ? 0.0f : l * ex2(m - m_new)) +
              (((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7])));
          m = m_new;
        }
      } else {
        // this thread is key key0 + lrow; its columns are rows kSliceCols*slice + [0, kSliceCols)
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
#pragma unroll
        for (int r4 = 0; r4 < kSliceCols / 4; ++r4) {
          const int r = kSliceCols * slice + 4 * r4;
          const float4 mr = *reinterpret_cast<const float4*>(&S.rowm[r]);
          float* ac = acc + 4 * (r4 & 1);
          ac[0] += ex2(fmaf(v[4 * r4 + 0], kLogitScale, -mr.x));
          ac[1] += ex2(fmaf(v[4 * r4 + 1], kLogitScale, -mr.y));
          ac[2] += ex2(fmaf(v[4 * r4 + 2], kLogitScale, -mr.z));
          ac[3] += ex2(fmaf(v[4 * r4 + 3], kLogitScale, -mr.w));
        }
        // the four column slices of each key summed in slice order through
        // shared memory; the four warps of a lane quarter (the same keys)
        // meet at their own barrier.  Double-buffered by accumulator: a
        // buffer is reused two tiles later, after those warps have passed
        // the next barrier.
        S.red[ab][slice][lrow] = ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
        named_bar_sync(2 + quarter, 32 * kSlices);   // the four warps of this lane quarter
        const int64_t key = key0 + lrow;
        if (slice == 0 && key < a.n) {
          float sum = S.red[ab][0][lrow];
#pragma unroll
          for (int q = 1; q < kSlices; ++q) sum += S.red[ab][q][lrow];
          a.a[static_cast<int64_t>(bg) * a.n_pad + key] = sum;
        }
      }
    }
    if (PASS == 1) {
      // merge the column slices of each row in slice order, then write the
      // CTA's partial
      if (slice > 0) {
        S.part_m[slice - 1][lrow] = m;
        S.part_l[slice - 1][lrow] = l;
      }
      named_bar_sync(1, 32 * kEpiWarps);
      if (slice == 0 && lrow < a.R) {
        float mm = m, ll = l;
#pragma unroll
        for (int q = 0; q < kSlices - 1; ++q) {
          const float m2 = S.part_m[q][lrow], l2 = S.part_l[q][lrow];
          const float mx = fmaxf(mm, m2);
          ll = (mm == -INFINITY ? 0.0f : ll * ex2(mm - mx)) + (m2 == -INFINITY ? 0.0f : l2 * ex2(m2 - mx));
          mm = mx;
        }
        float* st = a.stats + ((static_cast<int64_t>(bg) * a.pstride + part) * kRowsTile + lrow) * 2;
        st[0] = mm;
        st[1] = ll;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  pdl_trigger();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ pooling
// p_j = (a_{j-r} + ... + a_{j+r}) / k with zeros outside [0, n), k = 2r + 1;
// a_j is the window/group mean written by pass 2.  grid
// (ceil(n / 1024), B * Hkv), block 256, four consecutive keys per thread: a
// CTA stages the means of its keys and of the r keys on either side in
// shared memory once, then each thread adds its windows.  For the top-c
// select each CTA adds its keys' top-12-bit histogram (shared, then one
// global add per bin in use) into its row's histogram, which pass 1 zeroed,
// and writes the smallest and largest order-preserving key of its scores.
constexpr int kPoolThreads = 256;
constexpr int kPoolKeys = 4 * kPoolThreads;
constexpr int kPoolMaxR = 32;   // pool_k <= 65
constexpr int kHistBins = 4096;

__global__ void __launch_bounds__(kPoolThreads) pool_kernel(const float* __restrict__ a, float* __restrict__ p,
                                                            uint2* __restrict__ prange, uint32_t* __restrict__ hist,
                                                            int64_t n, int64_t n_pad, int pool_k) {
  __shared__ float as[kPoolKeys + 2 * kPoolMaxR];
  __shared__ uint32_t hs[kHistBins];
  __shared__ uint32_t wmin[kPoolThreads / 32], wmax[kPoolThreads / 32];
  const int bg = blockIdx.y;
  const int r = pool_k / 2;
  const int64_t jb = static_cast<int64_t>(blockIdx.x) * kPoolKeys;
  for (int i = threadIdx.x; i < kHistBins; i += kPoolThreads) hs[i] = 0u;
  pdl_wait();
  const float* a0 = a + static_cast<int64_t>(bg) * n_pad;
  for (int t = threadIdx.x; t < kPoolKeys + 2 * r; t += kPoolThreads) {
    const int64_t i = jb - r + t;
    as[t] = i >= 0 && i < n ? __ldcg(a0 + i) : 0.0f;
  }
  __syncthreads();
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  float pv[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int o = 4 * threadIdx.x + u;
    float sum = 0.0f;
    for (int t = 0; t <= 2 * r; ++t) sum += as[o + t];
    pv[u] = sum / static_cast<float>(pool_k);
    if (jb + o < n) {
      const uint32_t key = ord_key(pv[u]);
      kmin = min(kmin, key);
      kmax = max(kmax, key);
      atomicAdd(&hs[key >> 20], 1u);
    }
  }
  float* prow = p + static_cast<int64_t>(bg) * n_pad + jb + 4 * threadIdx.x;
  if (jb + 4 * threadIdx.x + 4 <= n) {
    *reinterpret_cast<float4*>(prow) = make_float4(pv[0], pv[1], pv[2], pv[3]);
  } else {
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (jb + 4 * threadIdx.x + u < n) prow[u] = pv[u];
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if ((threadIdx.x & 31) == 0) {
    wmin[threadIdx.x >> 5] = kmin;
    wmax[threadIdx.x >> 5] = kmax;
  }
  __syncthreads();
  uint32_t* hrow = hist + static_cast<int64_t>(bg) * kHistBins;
  for (int i = threadIdx.x; i < kHistBins; i += kPoolThreads)
    if (hs[i] != 0u) atomicAdd(hrow + i, hs[i]);
  if (threadIdx.x == 0) {
    for (int w = 1; w < kPoolThreads / 32; ++w) {
      kmin = min(kmin, wmin[w]);
      kmax = max(kmax, wmax[w]);
    }
    prange[static_cast<int64_t>(bg) * gridDim.x + blockIdx.x] = make_uint2(kmin, kmax);
  }
  pdl_trigger();
}

#include "topc.cuh"

// -------------------------------------------------------------- row gather
// grid (ceil(c / 32), B * Hkv), block 256: a warp copies the K and V rows
// (256 bytes each, one half-warp per row) of four kept tokens, all four
// loads of a thread in flight before its stores.  An index outside [0, n)
// (which the top-c select never produces) copies zeros and is flagged.
constexpr int kGatherTok = 4;   // tokens per warp

__global__ void gather_kernel(const uint16_t* __restrict__ K, const uint16_t* __restrict__ V,
                              const int32_t* __restrict__ idx, uint16_t* __restrict__ K_out,
                              uint16_t* __restrict__ V_out, int64_t n, int64_t n_cap, int c_out, unsigned* err) {
  const int bg = blockIdx.y;
  const int t0 = (blockIdx.x * 8 + (threadIdx.x >> 5)) * kGatherTok;
  pdl_wait();
  if (t0 >= c_out) return;
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4, l16 = lane & 15;
  const uint16_t* src_base = half ? V : K;
  uint16_t* dst_base = half ? V_out : K_out;
  const int32_t* id = idx + static_cast<int64_t>(bg) * c_out;
  uint4 v[kGatherTok];
#pragma unroll
  for (int u = 0; u < kGatherTok; ++u) {
    v[u] = make_uint4(0u, 0u, 0u, 0u);
    if (t0 + u < c_out) {
      const int32_t ix = __ldg(id + t0 + u);
      if (ix >= 0 && ix < n) {
        v[u] = __ldcs(reinterpret_cast<const uint4*>(src_base + (static_cast<int64_t>(bg) * n_cap + ix) * kD) + l16);
      } else if (l16 == 0) {   // the top-c select never hands out such an index: flag it, copy zeros
        record_error(err, kErrInternal);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kGatherTok; ++u)
    if (t0 + u < c_out) {
      const int64_t dst_row = static_cast<int64_t>(bg) * c_out + t0 + u;
      __stcs(reinterpret_cast<uint4*>(dst_base + dst_row * kD) + l16, v[u]);
    }
}

int encode_2d(CUtensorMap* m, const uint16_t* base, uint64_t rows, EncodeTiledFn enc) {
  const uint64_t gdim[2] = {static_cast<uint64_t>(kD), rows};
  const uint64_t gstride[1] = {static_cast<uint64_t>(kD) * 2};
  const unsigned box[2] = {64, 128};
  const unsigned estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(base), gdim, gstride, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

}  // namespace

SnapLayout snap_layout(const qasc_shape& s, const qasc_snap_params& p) {
  SnapLayout L;
  L.c_out = p.c < s.n ? p.c : s.n;
  const int64_t bgs = static_cast<int64_t>(s.B) * s.Hkv;
  const int64_t n_pad = static_cast<int64_t>(align_up(static_cast<size_t>(s.n), 64));
  // Partial statistics are sized for the most parts any device would use.
  L.parts = kMaxSmsForSizing;
  size_t off = 0;
  L.off_stats = off;
  off = align_up(off + static_cast<size_t>(bgs) * L.parts * kRowsTile * 2 * sizeof(float), 256);
  L.off_score = off;
  off = align_up(off + static_cast<size_t>(bgs) * n_pad * sizeof(float), 256);
  L.off_pool = off;
  off = align_up(off + static_cast<size_t>(bgs) * n_pad * sizeof(float), 256);
  L.off_phist = off;
  off = align_up(off + static_cast<size_t>(bgs) * ((s.n + kPoolKeys - 1) / kPoolKeys) * sizeof(uint2), 256);
  L.off_khist = off;
  off = align_up(off + static_cast<size_t>(bgs) * kHistBins * sizeof(uint32_t), 256);
  L.total = off;
  return L;
}

cudaError_t configure_snapkv_kernels(DeviceInfo& dev) {
  const int smem = static_cast<int>(sizeof(SnapSmem) + 1024);
  cudaError_t e = cudaFuncSetAttribute(snap_pass_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(snap_pass_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return configure_topc(dev.topc_clusters);
}

int launch_snapkv(const qasc_shape& s, const qasc_snap_params& p, const SnapLayout& L, const uint16_t* q_obs,
                  const uint16_t* K, const uint16_t* V, int32_t* idx, uint16_t* K_out, uint16_t* V_out, uint8_t* ws,
                  const DeviceInfo& dev, cudaStream_t stream) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cudaErrorNotSupported;
  const int gq = s.Hq / s.Hkv;
  alignas(64) CUtensorMap tq, tk;
  if (encode_2d(&tq, q_obs, static_cast<uint64_t>(s.B) * s.Hq * p.window, enc) != 0 ||
      encode_2d(&tk, K, static_cast<uint64_t>(s.B) * s.Hkv * s.n_cap, enc) != 0)
    return cudaErrorInvalidValue;
  cudaError_t e;
  const int64_t bgs = static_cast<int64_t>(s.B) * s.Hkv;
  const int64_t n_pad = static_cast<int64_t>(align_up(static_cast<size_t>(s.n), 64));
  const int ntiles = static_cast<int>((s.n + kTileKeys - 1) / kTileKeys);
  // key-range parts per (b, g): one CTA per SM over all KV heads, the SMs
  // left over by an even split going to the first (b, g) as one part more
  int base_parts = static_cast<int>(dev.num_sms / bgs), extra = static_cast<int>(dev.num_sms % bgs);
  if (base_parts < 1) {
    base_parts = 1;
    extra = 0;
  }
  if (base_parts >= ntiles) {
    base_parts = ntiles;
    extra = 0;
  }
  if (base_parts + 1 > L.parts) {
    base_parts = L.parts - 1;
    extra = 0;
  }
  PassArgs a;
  a.Hq = s.Hq;
  a.Hkv = s.Hkv;
  a.Gq = gq;
  a.w = p.window;
  a.R = gq * p.window;
  a.n = s.n;
  a.n_cap = s.n_cap;
  a.base_parts = base_parts;
  a.extra = extra;
  a.pstride = base_parts + (extra > 0 ? 1 : 0);
  a.ntiles = ntiles;
  a.n_pad = n_pad;
  a.bgs = static_cast<int>(bgs);
  a.stats = reinterpret_cast<float*>(ws + L.off_stats);
  a.a = reinterpret_cast<float*>(ws + L.off_score);
  a.hist = reinterpret_cast<uint32_t*>(ws + L.off_khist);
  a.hist_words = bgs * kHistBins;
  a.err = dev.err_word;
  const size_t smem = sizeof(SnapSmem) + 1024;
  const dim3 grid(static_cast<unsigned>(bgs * base_parts + extra));
  if ((e = launch_dependent(snap_pass_kernel<1>, grid, dim3(kThreadsP), smem, stream, 1, a, tq, tk)) != cudaSuccess)
    return e;
  if ((e = launch_dependent(snap_pass_kernel<2>, grid, dim3(kThreadsP), smem, stream, 1, a, tq, tk)) != cudaSuccess)
    return e;
  float* pool = reinterpret_cast<float*>(ws + L.off_pool);
  uint2* prange = reinterpret_cast<uint2*>(ws + L.off_phist);
  const int pparts = static_cast<int>((s.n + kPoolKeys - 1) / kPoolKeys);
  if ((e = launch_dependent(pool_kernel, dim3(static_cast<unsigned>(pparts), static_cast<unsigned>(bgs)),
                            dim3(kPoolThreads), 0, stream, 1, static_cast<const float*>(a.a), pool, prange, a.hist,
                            s.n, n_pad, p.pool_k)) != cudaSuccess)
    return e;
  const int c_out = static_cast<int>(L.c_out);
  if ((e = launch_topc(pool, reinterpret_cast<const uint32_t*>(prange), pparts, a.hist, idx, static_cast<int>(bgs),
                       s.n, n_pad, c_out, 0, dev.topc_clusters, stream)) != cudaSuccess)
    return e;
  return launch_dependent(gather_kernel,
                          dim3(static_cast<unsigned>((c_out + 8 * kGatherTok - 1) / (8 * kGatherTok)),
                               static_cast<unsigned>(bgs)),
                          dim3(256), 0, stream, 1, K, V, static_cast<const int32_t*>(idx), K_out, V_out, s.n,
                          s.n_cap, c_out, dev.err_word);
}

}  // namespace qasc

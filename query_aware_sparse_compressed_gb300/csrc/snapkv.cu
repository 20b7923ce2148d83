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
//           and sums exp(x - m_r) / (R l_r) over the 128 row columns, which
//           is the window/group mean a_j with no cross-lane reduction.
// A CTA is one warp of TMA issue, one warp of MMA issue (which also owns the
// TMEM allocation) and four epilogue warps (one per TMEM lane quarter); a
// 4-stage ring of key tiles and two TMEM accumulators keep loads, MMAs and
// epilogues overlapped.  KV heads are processed in groups whose keys fit in
// L2, so pass 2 re-reads its tiles from L2.
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

constexpr int kTileKeys = 128;                 // keys per tile
constexpr int kRowsTile = 128;                 // query rows per group tile
constexpr int kBoxBytes = 128 * 128;           // 64 bf16 columns x 128 rows
constexpr int kTileBytes = 2 * kBoxBytes;      // full d = 128
constexpr int kKStages = 4;
constexpr int kThreadsP = 320;                 // TMA warp, MMA warp, 8 epilogue warps
constexpr int kEpiWarps = 8;                   // two per TMEM lane quarter, 64 columns each
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
  alignas(16) float rowinv[kRowsTile];
  float half_m[kRowsTile];
  float half_l[kRowsTile];
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
  int bg0, parts, ntiles, bgs;
  int64_t n_pad;
  float* stats;       // [B*Hkv][parts][128][2]  (max in log2 units, sum)
  float* a;           // [2][B*Hkv][n_pad]: the two column halves' partial means
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
  const int bgl = blockIdx.x / a.parts, part = blockIdx.x - bgl * a.parts;
  const int bg = a.bg0 + bgl;
  const int b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int t_begin = static_cast<int>(static_cast<int64_t>(part) * a.ntiles / a.parts);
  const int t_end = static_cast<int>(static_cast<int64_t>(part + 1) * a.ntiles / a.parts);
  const int ntl = t_end - t_begin;

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
  if (PASS == 2 && warp >= 2 && warp < 6) {
    // Global row statistics from every part's partials.
    const int r = tid - 64;
    float m = -INFINITY, l = 0.0f;
    if (r < a.R) {
      const float* st = a.stats + (static_cast<int64_t>(bg) * a.parts) * kRowsTile * 2 + r * 2;
      for (int p = 0; p < a.parts; ++p) m = fmaxf(m, st[static_cast<int64_t>(p) * kRowsTile * 2]);
      for (int p = 0; p < a.parts; ++p) {
        const float mp = st[static_cast<int64_t>(p) * kRowsTile * 2];
        if (mp != -INFINITY) l += st[static_cast<int64_t>(p) * kRowsTile * 2 + 1] * ex2(mp - m);
      }
    }
    // padding rows contribute exp2(-inf) * 0 = 0
    S.rowm[r] = r < a.R ? m : INFINITY;
    S.rowinv[r] = r < a.R ? 1.0f / (static_cast<float>(a.R) * l) : 0.0f;
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
      for (int i = 0; i < ntl; ++i) {
        const int slot = i % kKStages;
        const uint32_t ph = (i / kKStages) & 1u;
        if (!mbar_wait(&S.empty[slot], ph ^ 1u)) {
          record_error(a.err, kErrTimeout);
          break;
        }
        const int krow = static_cast<int>(krow0 + static_cast<int64_t>(t_begin + i) * kTileKeys);
        mbar_arrive_expect_tx(&S.full[slot], kTileBytes);
        tma_load_2d(&S.k[slot][0], &tmap_k, 0, krow, &S.full[slot]);
        tma_load_2d(&S.k[slot][kBoxBytes], &tmap_k, 64, krow, &S.full[slot]);
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
    // ---- epilogue: TMEM lane quarter (warp % 4), column half (warp - 2) / 4
    const int quarter = warp & 3;
    const int chalf = (warp - 2) >> 2;
    const int lrow = 32 * quarter + lane;     // TMEM lane of this thread
    const uint32_t tlane = tmem + (static_cast<uint32_t>(32 * quarter) << 16) + 64 * chalf;
    float m = -INFINITY, l = 0.0f;
    for (int i = 0; i < ntl; ++i) {
      const int ab = i & 1;
      bool ok = !dead && mbar_wait(&S.acc_full[ab], (i >> 1) & 1u);
      if (!__all_sync(0xffffffffu, ok)) {
        if (!dead) record_error(a.err, kErrTimeout);
        dead = true;
        break;
      }
      tc_fence_after();
      const int64_t key0 = static_cast<int64_t>(t_begin + i) * kTileKeys;
      float v[64];
      tmem_ld64(tlane + ab * 128, v);
      if (PASS == 1) {
        // this thread is query row lrow; its columns are keys 64*chalf + [0, 64)
        const int valid = static_cast<int>(min(static_cast<int64_t>(kTileKeys), a.n - key0)) - 64 * chalf;
        float t4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          v[j] = j < valid ? v[j] * kLogitScale : -INFINITY;
          t4[j & 3] = fmaxf(t4[j & 3], v[j]);
        }
        const float m_new = fmaxf(m, fmaxf(fmaxf(t4[0], t4[1]), fmaxf(t4[2], t4[3])));
        if (m_new != -INFINITY) {
          float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
          for (int j = 0; j < 64; ++j) s4[j & 3] += ex2(v[j] - m_new);
          l = (m == -INFINITY ? 0.0f : l * ex2(m - m_new)) + ((s4[0] + s4[1]) + (s4[2] + s4[3]));
          m = m_new;
        }
      } else {
        // this thread is key key0 + lrow; its columns are rows 64*chalf + [0, 64)
        float acc4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int r4 = 0; r4 < 16; ++r4) {
          const int r = 64 * chalf + 4 * r4;
          const float4 mr = *reinterpret_cast<const float4*>(&S.rowm[r]);
          const float4 ir = *reinterpret_cast<const float4*>(&S.rowinv[r]);
          acc4[0] = fmaf(ex2(fmaf(v[4 * r4 + 0], kLogitScale, -mr.x)), ir.x, acc4[0]);
          acc4[1] = fmaf(ex2(fmaf(v[4 * r4 + 1], kLogitScale, -mr.y)), ir.y, acc4[1]);
          acc4[2] = fmaf(ex2(fmaf(v[4 * r4 + 2], kLogitScale, -mr.z)), ir.z, acc4[2]);
          acc4[3] = fmaf(ex2(fmaf(v[4 * r4 + 3], kLogitScale, -mr.w)), ir.w, acc4[3]);
        }
        const int64_t key = key0 + lrow;
        if (key < a.n)
          a.a[(static_cast<int64_t>(chalf) * a.bgs + bg) * a.n_pad + key] = (acc4[0] + acc4[1]) + (acc4[2] + acc4[3]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.acc_empty[ab]);
    }
    if (PASS == 1) {
      // merge the two column halves of each row, then write the CTA's partial
      if (chalf == 1) {
        S.half_m[lrow] = m;
        S.half_l[lrow] = l;
      }
      named_bar_sync(1, 32 * kEpiWarps);
      if (chalf == 0 && lrow < a.R) {
        const float m2 = S.half_m[lrow], l2 = S.half_l[lrow];
        const float mm = fmaxf(m, m2);
        const float ll = (m == -INFINITY ? 0.0f : l * ex2(m - mm)) + (m2 == -INFINITY ? 0.0f : l2 * ex2(m2 - mm));
        float* st = a.stats + ((static_cast<int64_t>(bg) * a.parts + part) * kRowsTile + lrow) * 2;
        st[0] = mm;
        st[1] = ll;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------------ pooling
// p_j = (a_{j-r} + ... + a_{j+r}) / k with zeros outside [0, n), k = 2r + 1;
// a_j is the sum of the two column halves written by pass 2.
__global__ void pool_kernel(const float* __restrict__ a, float* __restrict__ p, int64_t n, int64_t n_pad,
                            int64_t half_stride, int pool_k) {
  const int bg = blockIdx.y;
  const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (j >= n) return;
  const float* a0 = a + static_cast<int64_t>(bg) * n_pad;
  const float* a1 = a0 + half_stride;
  const int r = pool_k / 2;
  float s = 0.0f;
  for (int t = -r; t <= r; ++t) {
    const int64_t i = j + t;
    if (i >= 0 && i < n) s += __ldcg(a0 + i) + __ldcg(a1 + i);
  }
  p[static_cast<int64_t>(bg) * n_pad + j] = s / static_cast<float>(pool_k);
}

// -------------------------------------------------------------- top-c select
// One CTA per (b, g): radix select of the c-th largest pooled score (digits
// of 12, 12 and 8 bits; keys of the winning first digit are gathered into
// shared memory), then an ordered compaction: every score above the cutoff,
// plus the lowest-index ties, written ascending.
constexpr int kSThreads = 1024;
constexpr int kSWarps = kSThreads / 32;
constexpr int kSBins = 4096;
constexpr int kSCap = 8192;

struct TopcShared {
  uint32_t hist[kSBins];
  uint32_t cand[kSCap];
  uint32_t ncand;
  uint32_t wsum[kSWarps];
  uint32_t wtie[kSWarps];
  int res[2];
};

__device__ void s_find_crossing(const uint32_t* cnt, int nbins, uint32_t k, TopcShared& S) {
  const int per = nbins >= kSThreads ? nbins / kSThreads : 1;
  const int b0 = threadIdx.x * per;
  uint32_t local = 0;
  if (b0 < nbins)
    for (int i = 0; i < per; ++i) local += cnt[b0 + i];
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  uint32_t sfx = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_down_sync(0xffffffffu, sfx, o);
    if (l + o < 32) sfx += t;
  }
  if (l == 0) S.wsum[w] = sfx;
  __syncthreads();
  uint32_t above = sfx - local;
  for (int i = w + 1; i < kSWarps; ++i) above += S.wsum[i];
  if (b0 < nbins && above < k && k <= above + local) {
    uint32_t acc = above;
    for (int i = per - 1; i >= 0; --i) {
      const uint32_t c = cnt[b0 + i];
      if (acc + c >= k) {
        S.res[0] = b0 + i;
        S.res[1] = static_cast<int>(acc);
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

// Calls f(i, ord_key(p_i)) for every index of the row, four float4 loads in
// flight per thread (rows are padded to a multiple of 64 floats).
template <class F>
__device__ __forceinline__ void for_each_pkey(const float* pb, int nn, F&& f) {
  const float4* p4 = reinterpret_cast<const float4*>(pb);
  const int n4 = (nn + 3) / 4;
  int i4 = threadIdx.x;
  for (; i4 + 3 * kSThreads < n4; i4 += 4 * kSThreads) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldcg(p4 + i4 + u * kSThreads);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int base = 4 * (i4 + u * kSThreads);
      if (base + 0 < nn) f(base + 0, ord_key(v[u].x));
      if (base + 1 < nn) f(base + 1, ord_key(v[u].y));
      if (base + 2 < nn) f(base + 2, ord_key(v[u].z));
      if (base + 3 < nn) f(base + 3, ord_key(v[u].w));
    }
  }
  for (; i4 < n4; i4 += kSThreads) {
    const float4 v = __ldcg(p4 + i4);
    const int base = 4 * i4;
    if (base + 0 < nn) f(base + 0, ord_key(v.x));
    if (base + 1 < nn) f(base + 1, ord_key(v.y));
    if (base + 2 < nn) f(base + 2, ord_key(v.z));
    if (base + 3 < nn) f(base + 3, ord_key(v.w));
  }
}

__global__ void __launch_bounds__(kSThreads, 1) topc_kernel(const float* __restrict__ p, int32_t* __restrict__ idx,
                                                          int64_t n, int64_t n_pad, int c_out) {
  extern __shared__ __align__(16) uint8_t dyn[];
  TopcShared& S = *reinterpret_cast<TopcShared*>(dyn);
  const int bg = blockIdx.x;
  const float* pb = p + static_cast<int64_t>(bg) * n_pad;
  const int nn = static_cast<int>(n);
  const int kShift[3] = {20, 8, 0};
  const int kBits[3] = {12, 12, 8};
  uint32_t prefix = 0, pmask = 0, k = static_cast<uint32_t>(c_out);
  bool in_smem = false;
#pragma unroll 1
  for (int lv = 0; lv < 3; ++lv) {
    const int shift = kShift[lv];
    const int nb = 1 << kBits[lv];
    const uint32_t dmask = static_cast<uint32_t>(nb - 1);
    for (int i = threadIdx.x; i < nb; i += kSThreads) S.hist[i] = 0;
    __syncthreads();
    if (in_smem) {
      const int m = static_cast<int>(S.ncand);
      for (int i = threadIdx.x; i < m; i += kSThreads) {
        const uint32_t key = S.cand[i];
        if ((key & pmask) == prefix) atomicAdd(&S.hist[(key >> shift) & dmask], 1u);
      }
    } else {
      for_each_pkey(pb, nn, [&](int, uint32_t key) {
        if ((key & pmask) == prefix) atomicAdd(&S.hist[(key >> shift) & dmask], 1u);
      });
    }
    __syncthreads();
    s_find_crossing(S.hist, nb, k, S);
    const uint32_t digit = static_cast<uint32_t>(S.res[0]);
    k -= static_cast<uint32_t>(S.res[1]);
    const uint32_t inbin = S.hist[digit];
    prefix |= digit << shift;
    pmask |= dmask << shift;
    __syncthreads();
    if (!in_smem && lv < 2 && inbin <= kSCap) {
      if (threadIdx.x == 0) S.ncand = 0;
      __syncthreads();
      for_each_pkey(pb, nn, [&](int, uint32_t key) {
        if ((key & pmask) == prefix) S.cand[atomicAdd(&S.ncand, 1u)] = key;
      });
      __syncthreads();
      in_smem = true;
    }
  }
  // prefix is now the c-th largest key; k ties (key == prefix) are taken.
  const uint32_t cut = prefix, t_take = k;
  // Ordered compaction: warp w owns a contiguous run walked 32 indices at a
  // time (coalesced), ballots give in-order ranks.
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int run = ((nn + kSWarps - 1) / kSWarps + 31) & ~31;
  const int w0 = min(nn, warp * run), w1 = min(nn, w0 + run);
  uint32_t n_strict = 0, n_tie = 0;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < w1 ? ord_key(__ldcg(pb + i)) : 0u;
    n_strict += __popc(__ballot_sync(0xffffffffu, i < w1 && key > cut));
    n_tie += __popc(__ballot_sync(0xffffffffu, i < w1 && key == cut));
  }
  if (lane == 0) {
    S.wsum[warp] = n_strict;
    S.wtie[warp] = n_tie;
  }
  __syncthreads();
  uint32_t strict_before = 0, tie_before = 0;
  for (int i = 0; i < warp; ++i) {
    strict_before += S.wsum[i];
    tie_before += S.wtie[i];
  }
  int32_t* out = idx + static_cast<int64_t>(bg) * c_out;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const uint32_t key = i < w1 ? ord_key(__ldcg(pb + i)) : 0u;
    const bool strict = i < w1 && key > cut;
    const bool tie = i < w1 && key == cut;
    const uint32_t tb = __ballot_sync(0xffffffffu, tie);
    const uint32_t sb = __ballot_sync(0xffffffffu, strict);
    const uint32_t my_tie = tie_before + __popc(tb & lanemask_lt());
    const bool take = strict || (tie && my_tie < t_take);
    const uint32_t pos = strict_before + __popc(sb & lanemask_lt()) + min(my_tie, t_take);
    if (take && pos < static_cast<uint32_t>(c_out)) out[pos] = i;
    strict_before += __popc(sb);
    tie_before += __popc(tb);
  }
}

// -------------------------------------------------------------- row gather
// grid (ceil(c / 8), B * Hkv), block 256: a half-warp copies one 256-byte row.
__global__ void gather_kernel(const uint16_t* __restrict__ K, const uint16_t* __restrict__ V,
                              const int32_t* __restrict__ idx, uint16_t* __restrict__ K_out,
                              uint16_t* __restrict__ V_out, int64_t n_cap, int c_out) {
  const int bg = blockIdx.y;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= c_out) return;
  const int lane = threadIdx.x & 31;
  const int64_t src_row = static_cast<int64_t>(bg) * n_cap + idx[static_cast<int64_t>(bg) * c_out + t];
  const int64_t dst_row = static_cast<int64_t>(bg) * c_out + t;
  const int half = lane >> 4, l16 = lane & 15;
  const uint4* src = reinterpret_cast<const uint4*>((half ? V : K) + src_row * kD) + l16;
  uint4* dst = reinterpret_cast<uint4*>((half ? V_out : K_out) + dst_row * kD) + l16;
  *dst = __ldcs(src);
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

// KV heads per pass-pair: as many as keep their keys within ~half of L2.
int bgs_per_group(const qasc_shape& s, int l2_bytes) {
  const int64_t per_bg = s.n * kD * 2;
  int64_t g = (static_cast<int64_t>(l2_bytes) / 2) / (per_bg > 0 ? per_bg : 1);
  if (g < 1) g = 1;
  const int64_t total = static_cast<int64_t>(s.B) * s.Hkv;
  return static_cast<int>(g < total ? g : total);
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
  off = align_up(off + 2 * static_cast<size_t>(bgs) * n_pad * sizeof(float), 256);
  L.off_pool = off;
  off = align_up(off + static_cast<size_t>(bgs) * n_pad * sizeof(float), 256);
  L.total = off;
  return L;
}

cudaError_t configure_snapkv_kernels(const DeviceInfo&) {
  const int smem = static_cast<int>(sizeof(SnapSmem) + 1024);
  cudaError_t e = cudaFuncSetAttribute(snap_pass_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(snap_pass_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(topc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(sizeof(TopcShared)));
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
  int l2 = 0;
  cudaError_t e = cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev.device);
  if (e != cudaSuccess) return e;
  const int64_t bgs = static_cast<int64_t>(s.B) * s.Hkv;
  const int64_t n_pad = static_cast<int64_t>(align_up(static_cast<size_t>(s.n), 64));
  const int ntiles = static_cast<int>((s.n + kTileKeys - 1) / kTileKeys);
  const int per_group = bgs_per_group(s, l2);
  int parts = dev.num_sms / per_group;
  if (parts < 1) parts = 1;
  if (parts > ntiles) parts = ntiles;
  if (parts > L.parts) parts = L.parts;
  PassArgs a;
  a.Hq = s.Hq;
  a.Hkv = s.Hkv;
  a.Gq = gq;
  a.w = p.window;
  a.R = gq * p.window;
  a.n = s.n;
  a.n_cap = s.n_cap;
  a.parts = parts;
  a.ntiles = ntiles;
  a.n_pad = n_pad;
  a.bgs = static_cast<int>(bgs);
  a.stats = reinterpret_cast<float*>(ws + L.off_stats);
  a.a = reinterpret_cast<float*>(ws + L.off_score);
  a.err = dev.err_word;
  const size_t smem = sizeof(SnapSmem) + 1024;
  for (int64_t g0 = 0; g0 < bgs; g0 += per_group) {
    const int nbg = static_cast<int>(bgs - g0 < per_group ? bgs - g0 : per_group);
    a.bg0 = static_cast<int>(g0);
    snap_pass_kernel<1><<<nbg * parts, kThreadsP, smem, stream>>>(a, tq, tk);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    snap_pass_kernel<2><<<nbg * parts, kThreadsP, smem, stream>>>(a, tq, tk);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  float* pool = reinterpret_cast<float*>(ws + L.off_pool);
  pool_kernel<<<dim3(static_cast<unsigned>((s.n + 255) / 256), static_cast<unsigned>(bgs)), 256, 0, stream>>>(
      a.a, pool, s.n, n_pad, bgs * n_pad, p.pool_k);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const int c_out = static_cast<int>(L.c_out);
  topc_kernel<<<static_cast<unsigned>(bgs), kSThreads, sizeof(TopcShared), stream>>>(pool, idx, s.n, n_pad, c_out);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  gather_kernel<<<dim3(static_cast<unsigned>((c_out + 7) / 8), static_cast<unsigned>(bgs)), 256, 0, stream>>>(
      K, V, idx, K_out, V_out, s.n_cap, c_out);
  return cudaGetLastError();
}

}  // namespace qasc

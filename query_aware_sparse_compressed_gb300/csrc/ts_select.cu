// Per-head thresholds, votes and the top-K token set.
//
// TokenSelect page, section "Voting Mechanism": Vote(i) = sum_h 1[Score_h(i) >
// theta_h]; section "Token-Level Selection と Sparse Attention": S = top-K of
// the candidates with Vote(i) >= V_min.  theta_h is head h's K-th largest
// score over C; candidates are ranked by (Vote desc, sum_h Score_h desc,
// index asc) and S is emitted in ascending token order.
//
// Three kernels:
//   theta_kernel   one 8-CTA cluster per (b, h): exact K-th largest score.
//   vote_kernel    one thread per (b, i): Vote(i) and the head sum, packed as
//                  a 64-bit key  vote << 32 | ord(sum).
//   cutoff_kernel  one 8-CTA cluster per b: exact K-th largest composite key,
//                  then an ordered (ballot/prefix) compaction of S.
//
// K-th largest without a sort.  A pass histograms the values inside the
// current window [lo, hi] into 2048 bins with a monotone map (linear in value;
// linear in the order-preserving integer key if the value span is not a finite
// float).  Because the map is monotone, the bin holding the K-th largest is
// exact; the window shrinks to that bin's value range and k drops by the
// count above it.  Once that bin holds at most kCap values they are gathered
// into rank 0's shared memory and finished there by the same procedure.  The
// per-CTA histograms are summed through distributed shared memory: CTA r owns
// bins [256 r, 256 r + 256) of the reduction.  All synchronisation is the
// hardware cluster barrier.
#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace qasc {
namespace {

constexpr int kCS = 8;                 // CTAs per cluster
constexpr int kNB = 2048;              // histogram bins
constexpr int kSeg = kNB / kCS;        // bins reduced by one CTA
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kCap = 4096;             // candidates finished inside rank 0
constexpr int kMaxVoteBins = 65;       // votes 0..64
// Binning shrinks the window by ~2048x per pass (integer-key binning from
// pass 8 on ends within 3 more), so this cap is never reached on valid input;
// it only guarantees termination.
constexpr int kMaxPasses = 24;

// ------------------------------------------------------------- binning
struct Binner {
  float lo, scale;
  uint32_t klo;
  uint64_t kspan;
  bool keyspace;
};

__device__ __forceinline__ Binner make_binner(float lo, float hi, int pass) {
  Binner B;
  B.lo = lo;
  B.klo = ord_key(lo);
  B.kspan = static_cast<uint64_t>(ord_key(hi)) - B.klo + 1ull;
  const float span = hi - lo;
  B.scale = static_cast<float>(kNB) / span;
  B.keyspace = !(isfinite(span) && span > 0.0f && isfinite(B.scale)) || pass >= 8;
  return B;
}

__device__ __forceinline__ int bin_of(float x, const Binner& B) {
  if (!B.keyspace) {
    const int b = static_cast<int>((x - B.lo) * B.scale);
    return b < kNB - 1 ? b : kNB - 1;
  }
  const uint64_t k = static_cast<uint64_t>(ord_key(x) - B.klo);
  return static_cast<int>((k * kNB) / B.kspan);
}

__device__ __forceinline__ bool in_window(float x, float lo, float hi) { return x >= lo && x <= hi; }

// ------------------------------------------------------ block reductions
struct Scratch {
  float f[kWarps];
  float f2[kWarps];
  uint32_t u[kWarps];
  uint32_t u2[kWarps];
  int res[4];
  float resf[2];
};

__device__ __forceinline__ void block_minmax(float& lo, float& hi, Scratch& sc) {
  lo = warp_min(lo);
  hi = warp_max(hi);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    sc.f[w] = lo;
    sc.f2[w] = hi;
  }
  __syncthreads();
  lo = sc.f[0];
  hi = sc.f2[0];
#pragma unroll
  for (int i = 1; i < kWarps; ++i) {
    lo = fminf(lo, sc.f[i]);
    hi = fmaxf(hi, sc.f2[i]);
  }
  __syncthreads();
}

__device__ __forceinline__ uint32_t block_sum(uint32_t v, Scratch& sc) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) sc.u[w] = v;
  __syncthreads();
  uint32_t t = 0;
#pragma unroll
  for (int i = 0; i < kWarps; ++i) t += sc.u[i];
  __syncthreads();
  return t;
}

// Sum over threads with a higher index than the caller (suffix, exclusive).
__device__ __forceinline__ uint32_t block_suffix_excl(uint32_t v, Scratch& sc) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  uint32_t s = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_down_sync(0xffffffffu, s, o);
    if (l + o < 32) s += t;
  }
  if (l == 0) sc.u2[w] = s;  // warp total
  __syncthreads();
  uint32_t above = 0;
  for (int i = w + 1; i < kWarps; ++i) above += sc.u2[i];
  __syncthreads();
  return above + (s - v);
}

// Finds the bin holding the k-th largest (1-based) of the counts cnt[0, nbins)
// (larger bin = larger values).  Thread t owns bins [t * per, t * per + per).
// Result in sc.res = {bin, count above it, count in it}; valid if k <= total.
__device__ void find_crossing(const uint32_t* cnt, int nbins, uint32_t k, Scratch& sc) {
  const int per = nbins >= kThreads ? nbins / kThreads : 1;
  const int b0 = threadIdx.x * per;
  uint32_t local = 0;
  if (b0 < nbins)
    for (int i = 0; i < per; ++i) local += cnt[b0 + i];
  const uint32_t above = block_suffix_excl(local, sc);
  if (b0 < nbins && above < k && k <= above + local) {
    uint32_t acc = above;
    for (int i = per - 1; i >= 0; --i) {
      const uint32_t c = cnt[b0 + i];
      if (acc + c >= k) {
        sc.res[0] = b0 + i;
        sc.res[1] = static_cast<int>(acc);
        sc.res[2] = static_cast<int>(c);
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

// Exact k-th largest (1-based) of v[0, m) held in this CTA's shared memory,
// by repeated monotone binning.  hist is kNB counters of scratch.  Returns the
// value and, in *n_greater, how many of the m values are strictly larger.
__device__ float block_kth_largest(const float* v, int m, uint32_t k, uint32_t* hist, Scratch& sc,
                                   uint32_t* n_greater) {
  float lo = INFINITY, hi = -INFINITY;
  for (int i = threadIdx.x; i < m; i += kThreads) {
    lo = fminf(lo, v[i]);
    hi = fmaxf(hi, v[i]);
  }
  block_minmax(lo, hi, sc);
  uint32_t above_total = 0;
  for (int pass = 0;; ++pass) {
    if (!(lo < hi) || pass >= kMaxPasses) break;  // window holds one distinct value
    const Binner B = make_binner(lo, hi, pass);
    for (int i = threadIdx.x; i < kNB; i += kThreads) hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < m; i += kThreads) {
      const float x = v[i];
      if (in_window(x, lo, hi)) atomicAdd(&hist[bin_of(x, B)], 1u);
    }
    __syncthreads();
    find_crossing(hist, kNB, k, sc);
    const int bstar = sc.res[0];
    k -= static_cast<uint32_t>(sc.res[1]);
    above_total += static_cast<uint32_t>(sc.res[1]);
    __syncthreads();
    float nlo = INFINITY, nhi = -INFINITY;
    for (int i = threadIdx.x; i < m; i += kThreads) {
      const float x = v[i];
      if (in_window(x, lo, hi) && bin_of(x, B) == bstar) {
        nlo = fminf(nlo, x);
        nhi = fmaxf(nhi, x);
      }
    }
    block_minmax(nlo, nhi, sc);
    lo = nlo;
    hi = nhi;
  }
  // All remaining window values equal lo; those above the window were counted.
  *n_greater = above_total;
  return lo;
}

// Shared-memory layout common to both cluster kernels (static part).
struct ClusterShared {
  uint32_t hist[kNB];
  uint32_t tot[kSeg];
  uint32_t seg_tot[kCS];
  int res[4];            // {bin, above, count, -}: written by the owning CTA
  float mm[2][2];        // per-pass window exchange (double-buffered)
  float cand[kCap];
  uint32_t cand_count;
  uint32_t vote_hist[kMaxVoteBins];
  uint32_t cta_cnt[kCS][2];
  float bcast_f[2];
  int bcast_i[4];
  Scratch sc;
};

// One cluster-wide histogram pass: returns {bstar, above, count} in every CTA.
template <class Src>
__device__ void cluster_hist_pass(cg::cluster_group& cl, ClusterShared& S, const Src& src, int m, float lo, float hi,
                                  const Binner& B, uint32_t k) {
  const int rank = static_cast<int>(cl.block_rank());
  for (int i = threadIdx.x; i < kNB; i += kThreads) S.hist[i] = 0;
  __syncthreads();
  for (int i = threadIdx.x; i < m; i += kThreads) {
    float x;
    if (src.get(i, x) && in_window(x, lo, hi)) atomicAdd(&S.hist[bin_of(x, B)], 1u);
  }
  __syncthreads();
  cl.sync();
  // Distributed reduction: this CTA sums its 256-bin segment across the cluster.
  uint32_t seg = 0;
  if (threadIdx.x < kSeg) {
    uint32_t t = 0;
#pragma unroll
    for (int c = 0; c < kCS; ++c) t += cl.map_shared_rank(S.hist, c)[rank * kSeg + threadIdx.x];
    S.tot[threadIdx.x] = t;
    seg = t;
  }
  seg = block_sum(seg, S.sc);
  if (threadIdx.x < kCS) cl.map_shared_rank(S.seg_tot, threadIdx.x)[rank] = seg;
  cl.sync();
  // Which segment holds the k-th largest?  Every CTA computes the same answer.
  uint32_t above = 0;
  int rstar = 0;
  for (int r = kCS - 1; r >= 0; --r) {
    if (above + S.seg_tot[r] >= k) {
      rstar = r;
      break;
    }
    above += S.seg_tot[r];
  }
  if (rank == rstar) {
    find_crossing(S.tot, kSeg, k - above, S.sc);
    if (threadIdx.x < kCS) {
      int* dst = cl.map_shared_rank(S.res, threadIdx.x);
      dst[0] = rstar * kSeg + S.sc.res[0];
      dst[1] = static_cast<int>(above) + S.sc.res[1];
      dst[2] = S.sc.res[2];
    }
  }
  cl.sync();
}

// Cluster-wide min/max of the values in [lo, hi] whose bin is bstar.
template <class Src>
__device__ void cluster_bin_range(cg::cluster_group& cl, ClusterShared& S, const Src& src, int m, float lo, float hi,
                                  const Binner& B, int bstar, int parity, float& nlo, float& nhi) {
  float a = INFINITY, z = -INFINITY;
  for (int i = threadIdx.x; i < m; i += kThreads) {
    float x;
    if (src.get(i, x) && in_window(x, lo, hi) && bin_of(x, B) == bstar) {
      a = fminf(a, x);
      z = fmaxf(z, x);
    }
  }
  block_minmax(a, z, S.sc);
  if (threadIdx.x == 0) {
    S.mm[parity][0] = a;
    S.mm[parity][1] = z;
  }
  cl.sync();
  a = INFINITY;
  z = -INFINITY;
  for (int c = 0; c < kCS; ++c) {
    const float* r = cl.map_shared_rank(&S.mm[parity][0], c);
    a = fminf(a, r[0]);
    z = fmaxf(z, r[1]);
  }
  nlo = a;
  nhi = z;
}

// Shared cluster routine: the k-th largest value among this cluster's
// elements that `src` admits.  Returns (in rank 0) the value and the number
// of admitted elements strictly above it.  `lo`/`hi` are the admitted range.
// Callers must pass one more cluster barrier before their CTAs exit: the
// early-out paths return right after reading peers' shared memory.
template <class Src>
__device__ bool cluster_kth_largest(cg::cluster_group& cl, ClusterShared& S, const Src& src, int m, float lo, float hi,
                                    uint32_t k, float* value, uint32_t* n_greater) {
  const int rank = static_cast<int>(cl.block_rank());
  uint32_t above_total = 0;
  for (int pass = 0;; ++pass) {
    if (!(lo < hi) || pass >= kMaxPasses) {
      *value = lo;
      *n_greater = above_total;
      return rank == 0;
    }
    const Binner B = make_binner(lo, hi, pass);
    cluster_hist_pass(cl, S, src, m, lo, hi, B, k);
    const int bstar = S.res[0];
    const uint32_t above = static_cast<uint32_t>(S.res[1]);
    const uint32_t inbin = static_cast<uint32_t>(S.res[2]);
    k -= above;
    above_total += above;
    if (inbin <= kCap) {
      // Gather the bin's values into rank 0 and finish there.
      uint32_t* cnt0 = cl.map_shared_rank(&S.cand_count, 0);
      float* cand0 = cl.map_shared_rank(S.cand, 0);
      for (int i = threadIdx.x; i < m; i += kThreads) {
        float x;
        if (src.get(i, x) && in_window(x, lo, hi) && bin_of(x, B) == bstar) {
          const uint32_t pos = atomicAdd(cnt0, 1u);
          cand0[pos] = x;
        }
      }
      cl.sync();
      if (rank != 0) return false;
      uint32_t ng = 0;
      *value = block_kth_largest(S.cand, static_cast<int>(S.cand_count), k, S.hist, S.sc, &ng);
      *n_greater = above_total + ng;
      return true;
    }
    float nlo, nhi;
    cluster_bin_range(cl, S, src, m, lo, hi, B, bstar, pass & 1, nlo, nhi);
    lo = nlo;
    hi = nhi;
  }
}

// ------------------------------------------------------------ theta kernel
// One CTA per (b, h).  Radix select on order-preserving 32-bit keys in three
// digit levels: each level histograms the keys that match the digits fixed
// so far and picks the digit holding the K-th largest.  The first level's
// histogram (top 12 bits; 11 for 8-head groups) is built by the scoring grid
// as it writes the scores, so this kernel only sums those partials; the keys
// of the winning first digit (~1-4 % of |C|) are then gathered from L2 into
// shared memory in one pass and the remaining levels run there.
constexpr int kTThreads = 1024;
constexpr int kTWarps = kTThreads / 32;
constexpr int kTBins = 8192;   // >= every level's bin count
constexpr int kTCap = 8192;

struct ThetaShared {
  uint32_t hist[kTBins];
  uint32_t cand[kTCap];
  uint32_t ncand;
  uint32_t wsum[kTWarps];
  int res[3];
};

// Bin holding the k-th largest of cnt[0, nbins); res = {bin, count above}.
__device__ void t_find_crossing(const uint32_t* cnt, int nbins, uint32_t k, ThetaShared& S) {
  const int per = nbins >= kTThreads ? nbins / kTThreads : 1;
  const int b0 = threadIdx.x * per;
  uint32_t local = 0;
  if (b0 < nbins)
    for (int i = 0; i < per; ++i) local += cnt[b0 + i];
  // suffix (exclusive) sum over threads
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
  for (int i = w + 1; i < kTWarps; ++i) above += S.wsum[i];
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

// Calls f(ord_key(x)) for every score x of the row, four float4 loads in
// flight per thread.
template <class F>
__device__ __forceinline__ void for_each_key(const float4* src4, int n4, int nc, F&& f) {
  int i4 = threadIdx.x;
  for (; i4 + 3 * kTThreads < n4; i4 += 4 * kTThreads) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldcg(src4 + i4 + u * kTThreads);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int base = 4 * (i4 + u * kTThreads);
      if (base + 0 < nc) f(ord_key(v[u].x));
      if (base + 1 < nc) f(ord_key(v[u].y));
      if (base + 2 < nc) f(ord_key(v[u].z));
      if (base + 3 < nc) f(ord_key(v[u].w));
    }
  }
  for (; i4 < n4; i4 += kTThreads) {
    const float4 v = __ldcg(src4 + i4);
    const int base = 4 * i4;
    if (base + 0 < nc) f(ord_key(v.x));
    if (base + 1 < nc) f(ord_key(v.y));
    if (base + 2 < nc) f(ord_key(v.z));
    if (base + 3 < nc) f(ord_key(v.w));
  }
}

// The CTA of a persistent grid of G CTAs over `total` items that holds item x
// (same partition as the scoring grid).
__device__ __forceinline__ int grid_cta_of(int64_t x, int64_t total, int G) {
  int64_t c = ((x + 1) * G + total - 1) / total - 1;
  return static_cast<int>(c < 0 ? 0 : (c >= G ? G - 1 : c));
}

struct ThetaArgs {
  const float* scores;
  const uint32_t* hist_part;   // first-digit histograms written by the scoring grid
  float* theta;
  int nc;
  int64_t nc_pad;
  uint32_t K;
  int Hq, Hkv;
  int tiles_per_bg, total_tiles, score_grid, max_splits, bits0;
};

__global__ void __launch_bounds__(kTThreads, 1) theta_kernel(const ThetaArgs a) {
  extern __shared__ __align__(16) uint8_t dyn[];
  ThetaShared& S = *reinterpret_cast<ThetaShared*>(dyn);
  const int bh = blockIdx.x;
  const int b = bh / a.Hq, h = bh - b * a.Hq;
  const int gq = a.Hq / a.Hkv;
  const int g = h / gq, hh = h - g * gq;
  const int bg = b * a.Hkv + g;
  const float4* src4 = reinterpret_cast<const float4*>(a.scores + static_cast<int64_t>(bh) * a.nc_pad);
  const int n4 = (a.nc + 3) / 4;
  const int nc = a.nc;

  // Level 0: the first digit's histogram, summed over the scoring CTAs that
  // covered (b, g).
  const int nb0 = 1 << a.bits0;
  const int64_t t0 = static_cast<int64_t>(bg) * a.tiles_per_bg;
  const int c_first = grid_cta_of(t0, a.total_tiles, a.score_grid);
  const int nsp = grid_cta_of(t0 + a.tiles_per_bg - 1, a.total_tiles, a.score_grid) - c_first + 1;
  const uint32_t* hp = a.hist_part + (static_cast<int64_t>(bg) * a.max_splits * gq + hh) * nb0;
  for (int bin = threadIdx.x; bin < nb0; bin += kTThreads) {
    uint32_t sum = 0;
#pragma unroll 4
    for (int sp = 0; sp < nsp; ++sp) sum += __ldcg(hp + static_cast<int64_t>(sp) * gq * nb0 + bin);
    S.hist[bin] = sum;
  }
  __syncthreads();
  uint32_t k = a.K;
  t_find_crossing(S.hist, nb0, k, S);
  uint32_t digit = static_cast<uint32_t>(S.res[0]);
  k -= static_cast<uint32_t>(S.res[1]);
  uint32_t inbin = S.hist[digit];
  const int shift0 = 32 - a.bits0;
  uint32_t prefix = digit << shift0;
  uint32_t pmask = static_cast<uint32_t>(nb0 - 1) << shift0;
  bool in_smem = false;
  __syncthreads();
  if (inbin <= kTCap) {
    if (threadIdx.x == 0) S.ncand = 0;
    __syncthreads();
    for_each_key(src4, n4, nc, [&](uint32_t key) {
      if ((key & pmask) == prefix) S.cand[atomicAdd(&S.ncand, 1u)] = key;
    });
    __syncthreads();
    in_smem = true;
  }
  // Levels 1 and 2: the remaining (24 - bits0) + 8 bits.
  const int kShift[2] = {8, 0};
  const int kBits[2] = {24 - a.bits0, 8};
#pragma unroll 1
  for (int lv = 0; lv < 2; ++lv) {
    const int shift = kShift[lv];
    const int nb = 1 << kBits[lv];
    const uint32_t dmask = static_cast<uint32_t>(nb - 1);
    for (int i = threadIdx.x; i < nb; i += kTThreads) S.hist[i] = 0;
    __syncthreads();
    if (in_smem) {
      const int m = static_cast<int>(S.ncand);
      for (int i = threadIdx.x; i < m; i += kTThreads) {
        const uint32_t key = S.cand[i];
        if ((key & pmask) == prefix) atomicAdd(&S.hist[(key >> shift) & dmask], 1u);
      }
    } else {
      for_each_key(src4, n4, nc, [&](uint32_t key) {
        if ((key & pmask) == prefix) atomicAdd(&S.hist[(key >> shift) & dmask], 1u);
      });
    }
    __syncthreads();
    t_find_crossing(S.hist, nb, k, S);
    digit = static_cast<uint32_t>(S.res[0]);
    k -= static_cast<uint32_t>(S.res[1]);
    inbin = S.hist[digit];
    prefix |= digit << shift;
    pmask |= dmask << shift;
    __syncthreads();
    if (!in_smem && lv == 0 && inbin <= kTCap) {
      if (threadIdx.x == 0) S.ncand = 0;
      __syncthreads();
      for_each_key(src4, n4, nc, [&](uint32_t key) {
        if ((key & pmask) == prefix) S.cand[atomicAdd(&S.ncand, 1u)] = key;
      });
      __syncthreads();
      in_smem = true;
    }
  }
  if (threadIdx.x == 0) a.theta[bh] = ord_val(prefix);
}

// ------------------------------------------------------------- vote kernel
// grid (ceil(nc / 1024), B), block 256: four consecutive candidates per thread
// (one float4 of scores per head; all head loads independent).  This is the
// last reader of the scores: each warp then drops its 512-byte run of every
// head's scores from L2, so the dead scratch is never written back to HBM.
__global__ void __launch_bounds__(256) vote_kernel(const float* __restrict__ scores,
                                                   const float* __restrict__ theta, uint64_t* __restrict__ keys,
                                                   int Hq, int nc, int64_t nc_pad) {
  __shared__ float th[64];
  const int b = blockIdx.y;
  if (threadIdx.x < Hq) th[threadIdx.x] = theta[b * Hq + threadIdx.x];
  __syncthreads();
  const int i4 = blockIdx.x * 256 + threadIdx.x;
  const float* sb = scores + static_cast<int64_t>(b) * Hq * nc_pad;
  if (4 * i4 < nc) {
    const float4* s = reinterpret_cast<const float4*>(sb) + i4;
    const int64_t hstride = nc_pad / 4;
    uint32_t v0 = 0, v1 = 0, v2 = 0, v3 = 0;
    float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
#pragma unroll 8
    for (int h = 0; h < Hq; ++h) {
      const float4 x = __ldcg(s + h * hstride);
      const float t = th[h];
      v0 += x.x > t;
      v1 += x.y > t;
      v2 += x.z > t;
      v3 += x.w > t;
      s0 += x.x;
      s1 += x.y;
      s2 += x.z;
      s3 += x.w;
    }
    uint64_t* out = keys + static_cast<int64_t>(b) * nc_pad + 4 * i4;
    const uint64_t k0 = (static_cast<uint64_t>(v0) << 32) | ord_key(s0);
    const uint64_t k1 = (static_cast<uint64_t>(v1) << 32) | ord_key(s1);
    const uint64_t k2 = (static_cast<uint64_t>(v2) << 32) | ord_key(s2);
    const uint64_t k3 = (static_cast<uint64_t>(v3) << 32) | ord_key(s3);
    reinterpret_cast<ulonglong2*>(out)[0] = make_ulonglong2(k0, k1);
    reinterpret_cast<ulonglong2*>(out)[1] = make_ulonglong2(k2, k3);
  }
  __syncwarp();
  // the warp's 128 candidates = up to four 128-byte lines per head; a line
  // that starts at nc_pad (a multiple of 64 floats) belongs to the next head
  const int w0 = 4 * (i4 & ~31);
  if (w0 < nc) {
    const int lane = threadIdx.x & 31;
    for (int j = lane; j < Hq * 4; j += 32) {
      const int64_t x = w0 + 32 * (j & 3);
      if (x < nc_pad) discard_l2_line(sb + static_cast<int64_t>(j >> 2) * nc_pad + x);
    }
  }
}

// ----------------------------------------------------------- cutoff kernel
// Admits the head sums of tokens whose vote equals `vstar`.
struct SumOfVoteSrc {
  const uint64_t* p;
  uint32_t vstar;
  __device__ __forceinline__ bool get(int i, float& x) const {
    const uint64_t key = p[i];
    x = ord_val(static_cast<uint32_t>(key));
    return static_cast<uint32_t>(key >> 32) == vstar;
  }
};

__global__ void __cluster_dims__(kCS, 1, 1) __launch_bounds__(kThreads, 1)
    cutoff_kernel(const uint64_t* __restrict__ keys, int32_t* __restrict__ sel, int nc, int64_t nc_pad, int slice,
                  int cache_slice, uint32_t K, int c0, int Hq) {
  extern __shared__ __align__(16) uint8_t dyn[];
  __shared__ ClusterShared S;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = static_cast<int>(cl.block_rank());
  const int b = blockIdx.x / kCS;
  const int i0 = rank * slice;
  const int m = max(0, min(nc - i0, slice));
  const uint64_t* g = keys + static_cast<int64_t>(b) * nc_pad + i0;
  const uint64_t* v = g;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) S.cand_count = 0;
  for (int i = threadIdx.x; i < kMaxVoteBins; i += kThreads) S.vote_hist[i] = 0;
  __syncthreads();

  // Cache the slice (independent 16-byte loads, four in flight per thread),
  // then build the vote histogram from it with warp-aggregated atomics.
  uint64_t* c = reinterpret_cast<uint64_t*>(dyn);
  if (cache_slice) {
    const int m2 = m / 2;   // slice starts are multiples of 4 keys, so 16-byte aligned
    const ulonglong2* g2 = reinterpret_cast<const ulonglong2*>(g);
    ulonglong2* c2 = reinterpret_cast<ulonglong2*>(c);
    int i = threadIdx.x;
    for (; i + 3 * kThreads < m2; i += 4 * kThreads) {
      ulonglong2 t[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) t[u] = __ldcg(g2 + i + u * kThreads);
#pragma unroll
      for (int u = 0; u < 4; ++u) c2[i + u * kThreads] = t[u];
    }
    for (; i < m2; i += kThreads) c2[i] = __ldcg(g2 + i);
    if ((m & 1) && threadIdx.x == 0) c[m - 1] = g[m - 1];
    __syncthreads();
    v = c;
  }
  const int mpad = (m + 31) & ~31;
  for (int i = threadIdx.x; i < mpad; i += kThreads) {
    const bool valid = i < m;
    const uint64_t key = valid ? v[i] : 0ull;
    const uint32_t vote = valid ? static_cast<uint32_t>(key >> 32) : 0xffffffffu;
    const uint32_t peers = __match_any_sync(0xffffffffu, vote);
    if (valid && (__ffs(peers) - 1) == lane) atomicAdd(&S.vote_hist[vote], __popc(peers));
  }
  __syncthreads();
  cl.sync();

  // Cutoff vote V*: #(vote > V*) < K <= #(vote >= V*).
  if (warp == 0) {
    uint32_t tot[3] = {0, 0, 0};
    for (int j = 0; j < 3; ++j) {
      const int vv = lane + 32 * j;
      if (vv <= Hq)
        for (int r = 0; r < kCS; ++r) tot[j] += cl.map_shared_rank(S.vote_hist, r)[vv];
    }
    for (int j = 0; j < 3; ++j) {
      const int vv = lane + 32 * j;
      if (vv <= Hq) S.tot[vv] = tot[j];
    }
    __syncwarp();
    if (lane == 0) {
      uint32_t above = 0;
      int vstar = 0;
      for (int vv = Hq; vv >= 0; --vv) {
        if (above + S.tot[vv] >= K) {
          vstar = vv;
          break;
        }
        above += S.tot[vv];
      }
      S.bcast_i[0] = vstar;
      S.bcast_i[1] = static_cast<int>(above);
    }
  }
  __syncthreads();
  const uint32_t vstar = static_cast<uint32_t>(S.bcast_i[0]);
  const uint32_t above_v = static_cast<uint32_t>(S.bcast_i[1]);
  const SumOfVoteSrc src{v, vstar};

  // Range of the head sums among vote == V* (cluster-wide).
  float lo = INFINITY, hi = -INFINITY;
  for (int i = threadIdx.x; i < m; i += kThreads) {
    float x;
    if (src.get(i, x)) {
      lo = fminf(lo, x);
      hi = fmaxf(hi, x);
    }
  }
  block_minmax(lo, hi, S.sc);
  if (threadIdx.x == 0) {
    S.bcast_f[0] = lo;
    S.bcast_f[1] = hi;
  }
  cl.sync();
  lo = INFINITY;
  hi = -INFINITY;
  for (int r = 0; r < kCS; ++r) {
    const float* p = cl.map_shared_rank(S.bcast_f, r);
    lo = fminf(lo, p[0]);
    hi = fmaxf(hi, p[1]);
  }
  cl.sync();  // every CTA has read bcast_f before it is rewritten below

  float sstar;
  uint32_t ng;
  const uint32_t kv = K - above_v;
  if (cluster_kth_largest(cl, S, src, m, lo, hi, kv, &sstar, &ng)) {
    // Rank 0 broadcasts the cutoff: (V*, sigma*, ties to take).
    if (threadIdx.x < kCS) {
      int* di = cl.map_shared_rank(S.bcast_i, threadIdx.x);
      float* df = cl.map_shared_rank(S.bcast_f, threadIdx.x);
      di[2] = static_cast<int>(kv - ng);
      df[0] = sstar;
    }
  }
  cl.sync();
  const uint32_t t_take = static_cast<uint32_t>(S.bcast_i[2]);
  const uint32_t skey = ord_key(S.bcast_f[0]);
  const uint64_t cut = (static_cast<uint64_t>(vstar) << 32) | skey;

  // Ordered compaction.  Warp w owns a contiguous run of the slice, walked
  // 32 elements at a time; ballots give in-order ranks.
  const int run = ((m + kWarps - 1) / kWarps + 31) & ~31;
  const int w0 = min(m, warp * run), w1 = min(m, w0 + run);
  uint32_t n_strict = 0, n_tie = 0;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const uint64_t key = i < w1 ? v[i] : 0ull;
    const bool strict = i < w1 && key > cut;
    const bool tie = i < w1 && key == cut;
    n_strict += __popc(__ballot_sync(0xffffffffu, strict));
    n_tie += __popc(__ballot_sync(0xffffffffu, tie));
  }
  if (lane == 0) {
    S.sc.u[warp] = n_strict;
    S.sc.u2[warp] = n_tie;
  }
  __syncthreads();
  uint32_t strict_before = 0, tie_before = 0, cta_strict = 0, cta_tie = 0;
  for (int w = 0; w < kWarps; ++w) {
    if (w < warp) {
      strict_before += S.sc.u[w];
      tie_before += S.sc.u2[w];
    }
    cta_strict += S.sc.u[w];
    cta_tie += S.sc.u2[w];
  }
  if (threadIdx.x < kCS) {
    uint32_t* d = cl.map_shared_rank(&S.cta_cnt[0][0], threadIdx.x);
    d[2 * rank + 0] = cta_strict;
    d[2 * rank + 1] = cta_tie;
  }
  cl.sync();
  for (int r = 0; r < rank; ++r) {
    strict_before += S.cta_cnt[r][0];
    tie_before += S.cta_cnt[r][1];
  }
  int32_t* out = sel + static_cast<int64_t>(b) * K;
  for (int base = w0; base < w1; base += 32) {
    const int i = base + lane;
    const uint64_t key = i < w1 ? v[i] : 0ull;
    const bool strict = i < w1 && key > cut;
    const bool tie = i < w1 && key == cut;
    const uint32_t tb = __ballot_sync(0xffffffffu, tie);
    const uint32_t my_tie_rank = tie_before + __popc(tb & lanemask_lt());
    const bool take = strict || (tie && my_tie_rank < t_take);
    const uint32_t sb = __ballot_sync(0xffffffffu, strict);
    const uint32_t s_before = strict_before + __popc(sb & lanemask_lt());
    const uint32_t ties_taken_before = min(my_tie_rank, t_take);
    const uint32_t pos = s_before + ties_taken_before;
    if (take && pos < K) out[pos] = c0 + i0 + i;
    strict_before += __popc(sb);
    tie_before += __popc(tb);
  }
}

size_t slice_room(const DeviceInfo& dev) {
  return static_cast<size_t>(dev.max_smem_optin) - sizeof(ClusterShared) - 1024;
}

}  // namespace

cudaError_t configure_select_kernels(const DeviceInfo& dev) {
  const int room = static_cast<int>(slice_room(dev));
  cudaError_t e = cudaFuncSetAttribute(theta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sizeof(ThetaShared)));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(cutoff_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, room);
}

SelectLayout select_layout(const qasc_shape& s, const qasc_ts_params& p) {
  SelectLayout L;
  const Regions R = regions_of(s.n, p.sink, p.local);
  L.nc = R.nc();
  L.nc_pad = static_cast<int64_t>(align_up(static_cast<size_t>(L.nc > 0 ? L.nc : 1), 64));
  size_t off = 0;
  L.off_scores = off;
  off = align_up(off + static_cast<size_t>(s.B) * s.Hq * L.nc_pad * sizeof(float), 256);
  L.off_theta = off;
  off = align_up(off + static_cast<size_t>(s.B) * s.Hq * sizeof(float), 256);
  L.off_keys = off;
  off = align_up(off + static_cast<size_t>(s.B) * L.nc_pad * sizeof(uint64_t), 256);
  L.off_qp = off;
  off = align_up(off + static_cast<size_t>(s.B) * s.Hkv * kQbBytesPerBg, 256);
  const ScoreGrid sg = score_grid(s, L.nc, kMaxSmsForSizing);
  L.hist_splits = sg.max_splits;
  L.off_hist = off;
  off = align_up(off + static_cast<size_t>(s.B) * s.Hkv * sg.max_splits * (s.Hq / s.Hkv) *
                           (size_t(1) << sg.hist_bits) * sizeof(uint32_t),
                 256);
  L.total = off;
  return L;
}

int launch_select(const qasc_shape& s, const qasc_ts_params& p, const SelectLayout& L, uint8_t* ws, int32_t* sel,
                  const DeviceInfo& dev, cudaStream_t stream) {
  float* scores = reinterpret_cast<float*>(ws + L.off_scores);
  float* theta = reinterpret_cast<float*>(ws + L.off_theta);
  uint64_t* keys = reinterpret_cast<uint64_t*>(ws + L.off_keys);
  const int nc = static_cast<int>(L.nc);
  const Regions R = regions_of(s.n, p.sink, p.local);
  const uint32_t K = static_cast<uint32_t>(p.K);
  const int slice = ((nc + kCS - 1) / kCS + 3) & ~3;
  // Shared memory left for caching a slice after the static part.
  const size_t room = slice_room(dev);
  cudaError_t e;

  {
    const ScoreGrid sg = score_grid(s, L.nc, dev.num_sms);
    ThetaArgs ta;
    ta.scores = scores;
    ta.hist_part = reinterpret_cast<const uint32_t*>(ws + L.off_hist);
    ta.theta = theta;
    ta.nc = nc;
    ta.nc_pad = L.nc_pad;
    ta.K = K;
    ta.Hq = s.Hq;
    ta.Hkv = s.Hkv;
    ta.tiles_per_bg = sg.tiles_per_bg;
    ta.total_tiles = sg.total;
    ta.score_grid = sg.grid;
    ta.max_splits = sg.max_splits;
    ta.bits0 = sg.hist_bits;
    theta_kernel<<<s.B * s.Hq, kTThreads, sizeof(ThetaShared), stream>>>(ta);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    dim3 grid(static_cast<unsigned>((nc + 1023) / 1024), static_cast<unsigned>(s.B));
    vote_kernel<<<grid, 256, 0, stream>>>(scores, theta, keys, s.Hq, nc, L.nc_pad);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    const size_t bytes = static_cast<size_t>(slice) * sizeof(uint64_t);
    const int cache = bytes <= room ? 1 : 0;
    const size_t dyn = cache ? bytes : 0;
    cutoff_kernel<<<s.B * kCS, kThreads, dyn, stream>>>(keys, sel, nc, L.nc_pad, slice, cache, K,
                                                        static_cast<int>(R.c0), s.Hq);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return 0;
}

}  // namespace qasc

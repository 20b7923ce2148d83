// Per-head thresholds, votes and the top-K token set.
//
// TokenSelect page, section "Voting Mechanism": Vote(i) = sum_h 1[Score_h(i) >
// theta_h]; section "Token-Level Selection と Sparse Attention": S = top-K of
// the candidates with Vote(i) >= V_min.  theta_h is head h's K-th largest
// score over C; candidates are ranked by (Vote desc, sum_h Score_h desc,
// index asc) and S is emitted in ascending token order.
//
// Three kernels, all exact selection without sorting (radix select on
// order-preserving integer keys):
//   theta_kernel   one CTA per (b, h): K-th largest score.
//   vote_kernel    Vote(i) and the head sum of every candidate, packed as a
//                  64-bit key  vote << 32 | ord(sum), plus each sequence's
//                  histogram of votes.
//   cutoff_kernel  one cluster per b: the K-th largest composite key, then an
//                  ordered compaction of S.
#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace qasc {
namespace {

constexpr int kMaxVoteBins = 65;       // votes 0..64

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
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
  // totals of the warps above this one: a suffix scan of the 32 warp totals
  uint32_t wsfx = S.wsum[l];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_down_sync(0xffffffffu, wsfx, o);
    if (l + o < 32) wsfx += t;
  }
  const uint32_t warps_above = __shfl_sync(0xffffffffu, wsfx, (w + 1) & 31);
  const uint32_t above = sfx - local + (w + 1 < kTWarps ? warps_above : 0u);
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

// Appends the key of every score whose key matches the fixed digits
// ((key & pmask) == prefix) to S.cand: eight float4 loads in flight per
// thread, then one shared atomic per warp reserves the warp's slots.  The
// order-preserving key is increasing on each sign, so the matching keys are
// one contiguous range of float bit patterns (of x + 0, which maps -0 to +0
// as ord_key does): each score costs an add, a subtract and one unsigned
// compare, and only matches are turned into keys.
__device__ __forceinline__ void gather_matches(const float4* src4, int n4, int nc, uint32_t pmask, uint32_t prefix,
                                               ThetaShared& S) {
  constexpr int U = 8;
  const int lane = threadIdx.x & 31;
  const uint32_t k1 = prefix | ~pmask;                                   // keys [prefix, k1]
  const uint32_t lo = (prefix & 0x80000000u) ? (prefix ^ 0x80000000u)   // positive: bits = key ^ 2^31
                                             : ~k1;                      // negative: bits = ~key
  const uint32_t span = k1 - prefix;
  const int n4_full = nc >> 2;   // float4s made only of candidates
  for (int base4 = 0; base4 < n4; base4 += U * kTThreads) {
    float4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i4 = base4 + u * kTThreads + static_cast<int>(threadIdx.x);
      v[u] = i4 < n4 ? __ldcg(src4 + i4) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    }
    const bool full = base4 + U * kTThreads <= n4_full;   // block-uniform
    uint32_t hit = 0;   // bit 4u + c: component c of load u matches
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = 4 * (base4 + u * kTThreads + static_cast<int>(threadIdx.x));
      const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        bool m = __float_as_uint(__fadd_rn(x[c], 0.0f)) - lo <= span;
        if (!full) m = m && i + c < nc;
        if (m) hit |= 1u << (4 * u + c);
      }
    }
    const uint32_t cnt = __popc(hit);
    const uint32_t inc = warp_incl_scan(cnt);
    uint32_t pos = 0;
    if (lane == 31 && inc > 0) pos = atomicAdd(&S.ncand, inc);
    pos = __shfl_sync(0xffffffffu, pos, 31) + inc - cnt;
    if (hit) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const uint32_t nib = (hit >> (4 * u)) & 0xfu;
        if (nib) {
          if (nib & 1u) S.cand[pos++] = ord_key(v[u].x);
          if (nib & 2u) S.cand[pos++] = ord_key(v[u].y);
          if (nib & 4u) S.cand[pos++] = ord_key(v[u].z);
          if (nib & 8u) S.cand[pos++] = ord_key(v[u].w);
        }
      }
    }
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
  uint32_t* vhist;             // [B][65] vote histograms, zeroed here
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
  pdl_wait();
  // the vote kernel accumulates each sequence's vote histogram from zero
  if (h == 0 && threadIdx.x < kMaxVoteBins) a.vhist[b * kMaxVoteBins + threadIdx.x] = 0;
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
  // four bins per thread, eight partial slots' loads in flight
  const int64_t qstride = static_cast<int64_t>(gq) * nb0 / 4;
  for (int qd = threadIdx.x; qd < nb0 / 4; qd += kTThreads) {
    const uint4* p = reinterpret_cast<const uint4*>(hp) + qd;
    uint4 acc = make_uint4(0, 0, 0, 0);
    for (int sp0 = 0; sp0 < nsp; sp0 += 8) {
      uint4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = sp0 + u < nsp ? __ldcg(p + (sp0 + u) * qstride) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        acc.x += v[u].x;
        acc.y += v[u].y;
        acc.z += v[u].z;
        acc.w += v[u].w;
      }
    }
    reinterpret_cast<uint4*>(S.hist)[qd] = acc;
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
    gather_matches(src4, n4, nc, pmask, prefix, S);
    __syncthreads();
    in_smem = true;
  }
  // Levels 1 and 2: the remaining (24 - bits0) + 8 bits.
#pragma unroll 1
  for (int lv = 0; lv < 2; ++lv) {
    const int shift = lv == 0 ? 8 : 0;
    const int nb = 1 << (lv == 0 ? 24 - a.bits0 : 8);
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
      gather_matches(src4, n4, nc, pmask, prefix, S);
      __syncthreads();
      in_smem = true;
    }
  }
  if (threadIdx.x == 0) a.theta[bh] = ord_val(prefix);
  pdl_trigger();
}

// ------------------------------------------------------------- vote kernel
// grid (ceil(nc / 1024), B), block 256: four consecutive candidates per thread
// (one float4 of scores per head; all head loads independent), and the
// sequence's histogram of votes (shared, then one global add per bin).  This
// is the last reader of the scores: each warp then drops its 512-byte run of
// every head's scores from L2, so the dead scratch is never written back.
__global__ void __launch_bounds__(256) vote_kernel(const float* __restrict__ scores,
                                                   const float* __restrict__ theta, uint64_t* __restrict__ keys,
                                                   uint32_t* __restrict__ vhist, int Hq, int nc, int64_t nc_pad) {
  __shared__ float th[64];
  __shared__ uint32_t vh[kMaxVoteBins];
  const int b = blockIdx.y;
  pdl_wait();
  if (threadIdx.x < Hq) th[threadIdx.x] = theta[b * Hq + threadIdx.x];
  if (threadIdx.x < kMaxVoteBins) vh[threadIdx.x] = 0;
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
    atomicAdd(&vh[v0], 1u);
    if (4 * i4 + 1 < nc) atomicAdd(&vh[v1], 1u);
    if (4 * i4 + 2 < nc) atomicAdd(&vh[v2], 1u);
    if (4 * i4 + 3 < nc) atomicAdd(&vh[v3], 1u);
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
  __syncthreads();
  if (threadIdx.x <= Hq && vh[threadIdx.x] != 0) atomicAdd(vhist + b * kMaxVoteBins + threadIdx.x, vh[threadIdx.x]);
  pdl_trigger();
}

// ----------------------------------------------------------- cutoff kernel
// One cluster of CS CTAs (1024 threads each) per sequence b; CTA r owns a
// contiguous slice of the candidates, 8 consecutive keys per thread per
// chunk (the first chunk stays in registers).
//  1. V* from the vote histogram: #(vote > V*) < K <= #(vote >= V*), and
//     kv = K - #(vote > V*).
//  2. sigma*: the kv-th largest ord(sum) among the tokens with vote == V*, by
//     radix select on its 32 bits in digits of 12, 12 and 8 bits.  A cluster
//     level histograms the keys that match the digits fixed so far; the CTA
//     histograms are summed through distributed shared memory (CTA r owns
//     1/CS of the bins) and the owner of the crossing bin broadcasts it.  As
//     soon as the matching keys number at most kCutCap they are gathered into
//     rank 0, which runs the remaining digits alone.
//  3. Ordered compaction: a token is taken if its key exceeds the cut key
//     (V*, sigma*), or equals it and is among the first kv - #greater such
//     tokens in index order; its slot in S is the number of taken tokens
//     before it (block scans, CTA offsets through distributed shared memory).
constexpr int kCutThreads = 1024;
constexpr int kCutWarps = kCutThreads / 32;
constexpr int kCutKPT = 8;
constexpr int kCutChunk = kCutThreads * kCutKPT;
constexpr int kCutBins = 4096;
constexpr int kCutCap = 8192;
// digit levels of the 32-bit ord(sum): bits [31:20], [19:8], [7:0]
__device__ __forceinline__ int cut_shift(int level) { return level == 0 ? 20 : (level == 1 ? 8 : 0); }
__device__ __forceinline__ int cut_bits(int level) { return level == 2 ? 8 : 12; }

template <int CS>
struct CutShared {
  uint32_t hist[kCutBins];
  uint32_t tot[kCutBins / CS];   // this CTA's reduced segment of the bins
  uint32_t cand[kCutCap];        // rank 0: gathered low key words
  uint32_t seg_tot[CS];
  uint32_t cta_cnt[CS][2];
  uint32_t ws[2][kCutWarps];
  uint32_t scan_tot[2];
  uint32_t cand_count;
  int res[3];                    // level result {digit, count above, count in digit}
  uint32_t cut[2];               // {sigma*, ties to take}
  int vstar;
  uint32_t above_v;
};

// This CTA's slice of one sequence's keys.
struct CutKeys {
  const uint64_t* g;   // slice start (64-byte aligned)
  int m;               // keys in the slice
  int nchunks;
  uint64_t r[kCutKPT]; // chunk 0

  __device__ __forceinline__ void load(int c, uint64_t (&k)[kCutKPT]) const {
    const int i0 = c * kCutChunk + static_cast<int>(threadIdx.x) * kCutKPT;
    if (i0 + kCutKPT <= m) {
      const ulonglong2* p = reinterpret_cast<const ulonglong2*>(g + i0);
#pragma unroll
      for (int j = 0; j < kCutKPT / 2; ++j) {
        const ulonglong2 v = __ldcg(p + j);
        k[2 * j] = v.x;
        k[2 * j + 1] = v.y;
      }
    } else {
#pragma unroll
      for (int j = 0; j < kCutKPT; ++j) k[j] = i0 + j < m ? __ldcg(g + i0 + j) : 0ull;
    }
  }
  // f(slice index, key) for every key of this thread, in index order.
  template <class F>
  __device__ __forceinline__ void visit(F&& f) const {
    for (int c = 0; c < nchunks; ++c) {
      uint64_t t[kCutKPT];
      if (c > 0) load(c, t);
      const int i0 = c * kCutChunk + static_cast<int>(threadIdx.x) * kCutKPT;
#pragma unroll
      for (int j = 0; j < kCutKPT; ++j)
        if (i0 + j < m) f(i0 + j, c == 0 ? r[j] : t[j]);
    }
  }
};

// Block-wide exclusive scans of two counters; also returns their totals.
template <int CS>
__device__ __forceinline__ void block_excl2(CutShared<CS>& S, uint32_t a, uint32_t b, uint32_t& ea, uint32_t& eb,
                                            uint32_t& ta, uint32_t& tb) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint32_t ia = warp_incl_scan(a), ib = warp_incl_scan(b);
  if (lane == 31) {
    S.ws[0][w] = ia;
    S.ws[1][w] = ib;
  }
  __syncthreads();
  if (w == 0) {
    const uint32_t xa = S.ws[0][lane], xb = S.ws[1][lane];
    const uint32_t sa = warp_incl_scan(xa), sb = warp_incl_scan(xb);
    __syncwarp();
    S.ws[0][lane] = sa - xa;
    S.ws[1][lane] = sb - xb;
    if (lane == 31) {
      S.scan_tot[0] = sa;
      S.scan_tot[1] = sb;
    }
  }
  __syncthreads();
  ea = S.ws[0][w] + ia - a;
  eb = S.ws[1][w] + ib - b;
  ta = S.scan_tot[0];
  tb = S.scan_tot[1];
  __syncthreads();
}

// Bin of cnt[0, nb) holding the k-th largest (1-based; larger bin = larger
// keys), found by one warp.  The lane that finds it calls out(bin, above, in).
template <class Out>
__device__ __forceinline__ void warp_find_kth(const uint32_t* cnt, int nb, uint32_t k, Out&& out) {
  const int lane = threadIdx.x & 31;
  const int per = (nb + 31) / 32;
  const int hi = nb - lane * per;            // lane 0 owns the top bins
  const int lo = hi - per > 0 ? hi - per : 0;
  uint32_t s = 0;
  for (int i = lo; i < hi; ++i) s += cnt[i];
  const uint32_t inc = warp_incl_scan(s);
  const bool mine = inc - s < k && k <= inc;
  if (mine) {
    uint32_t acc = inc - s;
    for (int i = hi - 1; i >= lo; --i) {
      const uint32_t c = cnt[i];
      if (acc + c >= k) {
        out(i, acc, c);
        break;
      }
      acc += c;
    }
  }
}

// Same over 4096 bins with the whole block (4 bins per thread).
template <int CS>
__device__ __forceinline__ void block_find_kth(CutShared<CS>& S, const uint32_t* cnt, int nb, uint32_t k) {
  const int per = nb / kCutThreads > 0 ? nb / kCutThreads : 1;
  const int t = static_cast<int>(threadIdx.x);
  const int hi = nb - t * per;
  const int lo = hi - per > 0 ? hi - per : 0;
  uint32_t s = 0;
  for (int i = lo; i < hi; ++i) s += cnt[i];
  uint32_t e, e2, tot, tot2;
  block_excl2(S, s, 0u, e, e2, tot, tot2);
  if (e < k && k <= e + s) {
    uint32_t acc = e;
    for (int i = hi - 1; i >= lo; --i) {
      const uint32_t c = cnt[i];
      if (acc + c >= k) {
        S.res[0] = i;
        S.res[1] = static_cast<int>(acc);
        S.res[2] = static_cast<int>(c);
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

template <int CS>
__global__ void __launch_bounds__(kCutThreads, 1)
    cutoff_kernel(const uint64_t* __restrict__ keys, const uint32_t* __restrict__ vhist, int32_t* __restrict__ sel,
                  int nc, int64_t nc_pad, int slice, uint32_t K, int c0, int Hq) {
  extern __shared__ __align__(16) uint8_t dyn[];
  CutShared<CS>& S = *reinterpret_cast<CutShared<CS>*>(dyn);
  cg::cluster_group cl = cg::this_cluster();
  const int rank = static_cast<int>(cl.block_rank());
  const int b = blockIdx.x / CS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i0 = rank * slice;
  pdl_wait();

  CutKeys ks;
  ks.g = keys + static_cast<int64_t>(b) * nc_pad + i0;
  ks.m = max(0, min(nc - i0, slice));
  ks.nchunks = (ks.m + kCutChunk - 1) / kCutChunk;
  if (ks.nchunks > 0) ks.load(0, ks.r);
  if (tid == 0) S.cand_count = 0;

  // 1. V* from the vote histogram (every CTA; no exchange needed): the bins
  // are staged in shared memory by as many threads, then one thread walks
  // them from the top
  if (tid < kMaxVoteBins) S.hist[tid] = tid <= Hq ? __ldcg(vhist + b * kMaxVoteBins + tid) : 0u;
  __syncthreads();
  if (warp == 0)
    warp_find_kth(S.hist, Hq + 1, K, [&](int v, uint32_t above, uint32_t) {
      S.vstar = v;
      S.above_v = above;
    });
  __syncthreads();
  const uint32_t vstar = static_cast<uint32_t>(S.vstar);
  uint32_t k = K - S.above_v;     // rank of the cut among vote == V*, from the top
  uint32_t ng = S.above_v;        // keys known to be strictly above the cut
  uint32_t prefix = 0, pmask = 0;
  int level = 0;
  bool gathered = false;

  // 2. cluster digit levels until the matching keys fit in rank 0
  for (; level < 3; ++level) {
    const int shift = cut_shift(level), nb = 1 << cut_bits(level);
    const uint32_t dmask = static_cast<uint32_t>(nb - 1);
    for (int i = tid; i < nb; i += kCutThreads) S.hist[i] = 0;
    __syncthreads();
    ks.visit([&](int, uint64_t key) {
      const uint32_t lo = static_cast<uint32_t>(key);
      if (static_cast<uint32_t>(key >> 32) == vstar && (lo & pmask) == prefix) atomicAdd(&S.hist[(lo >> shift) & dmask], 1u);
    });
    cl.sync();
    const int seg = nb / CS;
    uint32_t t = 0;
    if (tid < seg) {
#pragma unroll
      constexpr int kPeers = CS < 8 ? CS : 8;   // peers' loads in flight at a time
      for (int c0 = 0; c0 < CS; c0 += kPeers) {
        uint32_t v[kPeers];
#pragma unroll
        for (int c = 0; c < kPeers; ++c) v[c] = cl.map_shared_rank(S.hist, c0 + c)[rank * seg + tid];
#pragma unroll
        for (int c = 0; c < kPeers; ++c) t += v[c];
      }
      S.tot[tid] = t;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    if (lane == 0) S.ws[0][warp] = t;
    __syncthreads();
    if (tid < CS) {
      uint32_t st = 0;
      for (int w = 0; w < (seg + 31) / 32; ++w) st += S.ws[0][w];
      cl.map_shared_rank(S.seg_tot, tid)[rank] = st;
    }
    cl.sync();
    uint32_t above = 0;
    int rstar = -1;
    for (int r = CS - 1; r >= 0; --r) {
      if (above + S.seg_tot[r] >= k) {
        rstar = r;
        break;
      }
      above += S.seg_tot[r];
    }
    // the owner of the crossing segment finds the bin and broadcasts it (one
    // remote store per CTA: cheaper than every CTA reading the segment)
    if (rank == rstar && warp == 0) {
      warp_find_kth(S.tot, seg, k - above, [&](int bin, uint32_t ab, uint32_t in) {
#pragma unroll 1
        for (int c = 0; c < CS; ++c) {
          int* d = cl.map_shared_rank(S.res, c);
          d[0] = rstar * seg + bin;
          d[1] = static_cast<int>(above + ab);
          d[2] = static_cast<int>(in);
        }
      });
    }
    cl.sync();
    const uint32_t digit = static_cast<uint32_t>(S.res[0]);
    const uint32_t ab = static_cast<uint32_t>(S.res[1]);
    const uint32_t inbin = static_cast<uint32_t>(S.res[2]);
    k -= ab;
    ng += ab;
    prefix |= digit << shift;
    pmask |= dmask << shift;
    if (level == 2) break;                 // sigma* fully known
    if (inbin <= kCutCap) {
      // gather the matching keys' low words into rank 0 (one remote atomic per warp)
      uint32_t* cnt0 = cl.map_shared_rank(&S.cand_count, 0);
      uint32_t* cand0 = cl.map_shared_rank(S.cand, 0);
      for (int c = 0; c < ks.nchunks; ++c) {
        uint64_t tt[kCutKPT];
        if (c > 0) ks.load(c, tt);
        const int ib = c * kCutChunk + tid * kCutKPT;
        uint32_t mine = 0;
#pragma unroll
        for (int j = 0; j < kCutKPT; ++j) {
          const uint64_t key = c == 0 ? ks.r[j] : tt[j];
          mine += (ib + j < ks.m && static_cast<uint32_t>(key >> 32) == vstar &&
                   (static_cast<uint32_t>(key) & pmask) == prefix);
        }
        const uint32_t inc = warp_incl_scan(mine);
        const uint32_t wt = __shfl_sync(0xffffffffu, inc, 31);
        uint32_t base = 0;
        if (lane == 31 && wt > 0) base = atomicAdd(cnt0, wt);
        base = __shfl_sync(0xffffffffu, base, 31) + inc - mine;
        if (mine) {
#pragma unroll
          for (int j = 0; j < kCutKPT; ++j) {
            const uint64_t key = c == 0 ? ks.r[j] : tt[j];
            if (ib + j < ks.m && static_cast<uint32_t>(key >> 32) == vstar &&
                (static_cast<uint32_t>(key) & pmask) == prefix)
              cand0[base++] = static_cast<uint32_t>(key);
          }
        }
      }
      cl.sync();
      gathered = true;
      ++level;
      break;
    }
  }

  // rank 0 finishes the remaining digits on the gathered words: digits of at
  // most 8 bits, each histogram searched by one warp (few words, so small
  // histograms and few block barriers beat wide digits)
  if (gathered) {
    if (rank == 0) {
      const int m = static_cast<int>(S.cand_count);
      for (int top = cut_shift(level - 1); top > 0;) {
        const int bits = top >= 8 ? 8 : top;
        const int shift = top - bits, nb = 1 << bits;
        const uint32_t dmask = static_cast<uint32_t>(nb - 1);
        if (tid < nb) S.hist[tid] = 0;
        __syncthreads();
        for (int i = tid; i < m; i += kCutThreads) {
          const uint32_t x = S.cand[i];
          if ((x & pmask) == prefix) atomicAdd(&S.hist[(x >> shift) & dmask], 1u);
        }
        __syncthreads();
        if (warp == 0)
          warp_find_kth(S.hist, nb, k, [&](int bin, uint32_t above, uint32_t) {
            S.res[0] = bin;
            S.res[1] = static_cast<int>(above);
          });
        __syncthreads();
        k -= static_cast<uint32_t>(S.res[1]);
        ng += static_cast<uint32_t>(S.res[1]);
        prefix |= static_cast<uint32_t>(S.res[0]) << shift;
        pmask |= dmask << shift;
        top = shift;
      }
      if (tid < CS) {
        uint32_t* d = cl.map_shared_rank(S.cut, tid);
        d[0] = prefix;
        d[1] = k;
      }
    }
    cl.sync();
  } else if (tid == 0) {
    S.cut[0] = prefix;
    S.cut[1] = k;
  }
  __syncthreads();
  const uint64_t cut = (static_cast<uint64_t>(vstar) << 32) | S.cut[0];
  const uint32_t t_take = S.cut[1];

  // 3. ordered compaction
  uint32_t n_strict = 0, n_tie = 0;
  ks.visit([&](int, uint64_t key) {
    n_strict += key > cut;
    n_tie += key == cut;
  });
  uint32_t e0, e1, cta_strict, cta_tie;
  block_excl2(S, n_strict, n_tie, e0, e1, cta_strict, cta_tie);
  if (tid < CS) {
    uint32_t* d = cl.map_shared_rank(&S.cta_cnt[0][0], tid);
    d[2 * rank + 0] = cta_strict;
    d[2 * rank + 1] = cta_tie;
  }
  cl.sync();
  uint32_t strict_base = 0, tie_base = 0;
  for (int r = 0; r < rank; ++r) {
    strict_base += S.cta_cnt[r][0];
    tie_base += S.cta_cnt[r][1];
  }
  int32_t* out = sel + static_cast<int64_t>(b) * K;
  for (int c = 0; c < ks.nchunks; ++c) {
    uint64_t tt[kCutKPT];
    if (c > 0) ks.load(c, tt);
    const int ib = c * kCutChunk + tid * kCutKPT;
    uint32_t cs = 0, ct = 0;
#pragma unroll
    for (int j = 0; j < kCutKPT; ++j) {
      const uint64_t key = c == 0 ? ks.r[j] : tt[j];
      const bool v = ib + j < ks.m;
      cs += v && key > cut;
      ct += v && key == cut;
    }
    uint32_t es = e0, et = e1, ts = 0, tt2 = 0;   // one chunk: the counts' scan already gave the offsets
    if (ks.nchunks > 1) block_excl2(S, cs, ct, es, et, ts, tt2);
    uint32_t sb = strict_base + es, tb = tie_base + et;
#pragma unroll
    for (int j = 0; j < kCutKPT; ++j) {
      const uint64_t key = c == 0 ? ks.r[j] : tt[j];
      if (ib + j >= ks.m) break;
      const bool strict = key > cut, tie = key == cut;
      if (strict || (tie && tb < t_take)) {
        const uint32_t pos = sb + min(tb, t_take);
        if (pos < K) out[pos] = c0 + i0 + ib + j;
      }
      sb += strict;
      tb += tie;
    }
    strict_base += ts;
    tie_base += tt2;
  }
  // no cluster sync here: every access to a peer's shared memory happened
  // before the counts' cluster sync, which every CTA has passed
  pdl_trigger();
}

template <int CS>
cudaError_t launch_cutoff(const uint64_t* keys, const uint32_t* vhist, int32_t* sel, int B, int nc, int64_t nc_pad,
                          uint32_t K, int c0, int Hq, cudaStream_t stream) {
  const int slice = ((nc + CS - 1) / CS + kCutKPT - 1) / kCutKPT * kCutKPT;
  return launch_dependent(cutoff_kernel<CS>, dim3(static_cast<unsigned>(B * CS)), dim3(kCutThreads),
                          sizeof(CutShared<CS>), stream, CS, keys, static_cast<const uint32_t*>(vhist), sel, nc,
                          nc_pad, slice, K, c0, Hq);
}

template <int CS>
cudaError_t configure_cutoff(int* clusters) {
  cudaError_t e = cudaFuncSetAttribute(cutoff_kernel<CS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sizeof(CutShared<CS>)));
  if (e != cudaSuccess) return e;
  if (CS > 8) {
    e = cudaFuncSetAttribute(cutoff_kernel<CS>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CS);
  cfg.blockDim = dim3(kCutThreads);
  cfg.dynamicSmemBytes = sizeof(CutShared<CS>);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(clusters, cutoff_kernel<CS>, &cfg);
}

}  // namespace

cudaError_t configure_select_kernels(DeviceInfo& dev) {
  cudaError_t e = cudaFuncSetAttribute(theta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sizeof(ThetaShared)));
  if (e != cudaSuccess) return e;
  int n8 = 0, n16 = 0;
  if ((e = configure_cutoff<8>(&n8)) != cudaSuccess) return e;
  if (n8 < 1) return cudaErrorNotSupported;
  // 16-CTA clusters where the device schedules them; 8 otherwise
  // clusters of 16 where the device schedules them; launch_select uses them
  // while every sequence's cluster is resident at once
  dev.cut_clusters16 = configure_cutoff<16>(&n16) == cudaSuccess ? n16 : 0;
  cudaGetLastError();
  return cudaSuccess;
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
  // partial histograms for either tiling (contiguous cache or paged pool)
  ScoreGrid sg = score_grid(s, score_span(R, false), kMaxSmsForSizing);
  const ScoreGrid sgp = score_grid(s, score_span(R, true), kMaxSmsForSizing);
  if (sgp.max_splits > sg.max_splits) sg.max_splits = sgp.max_splits;
  L.hist_splits = sg.max_splits;
  L.off_hist = off;
  off = align_up(off + static_cast<size_t>(s.B) * s.Hkv * sg.max_splits * (s.Hq / s.Hkv) *
                           (size_t(1) << sg.hist_bits) * sizeof(uint32_t),
                 256);
  L.off_vhist = off;
  off = align_up(off + static_cast<size_t>(s.B) * kMaxVoteBins * sizeof(uint32_t), 256);
  L.total = off;
  return L;
}

int launch_select(const qasc_shape& s, const qasc_ts_params& p, const SelectLayout& L, uint8_t* ws, int32_t* sel,
                  const DeviceInfo& dev, cudaStream_t stream, bool paged) {
  const Regions R = regions_of(s.n, p.sink, p.local);
  float* scores = reinterpret_cast<float*>(ws + L.off_scores);
  float* theta = reinterpret_cast<float*>(ws + L.off_theta);
  uint64_t* keys = reinterpret_cast<uint64_t*>(ws + L.off_keys);
  const int nc = static_cast<int>(L.nc);
  const uint32_t K = static_cast<uint32_t>(p.K);
  uint32_t* vhist = reinterpret_cast<uint32_t*>(ws + L.off_vhist);
  cudaError_t e;

  {
    const ScoreGrid sg = score_grid(s, score_span(R, paged), dev.num_sms);
    ThetaArgs ta;
    ta.scores = scores;
    ta.hist_part = reinterpret_cast<const uint32_t*>(ws + L.off_hist);
    ta.theta = theta;
    ta.vhist = vhist;
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
    e = launch_dependent(theta_kernel, dim3(s.B * s.Hq), dim3(kTThreads), sizeof(ThetaShared), stream, 1, ta);
    if (e != cudaSuccess) return e;
  }
  {
    dim3 grid(static_cast<unsigned>((nc + 1023) / 1024), static_cast<unsigned>(s.B));
    e = launch_dependent(vote_kernel, grid, dim3(256), 0, stream, 1, static_cast<const float*>(scores),
                         static_cast<const float*>(theta), keys, vhist, s.Hq, nc, L.nc_pad);
    if (e != cudaSuccess) return e;
  }
  // clusters of 8 while their CTAs hold their slices in one chunk of keys
  // (fewer peers per exchange: 68.4 against 70.4 us per 64K x B2 select),
  // 16 beyond that while every sequence's cluster is resident at once
  const int chunks = (nc + kCutChunk - 1) / kCutChunk;
  const int c0i = static_cast<int>(R.c0);
  if (chunks <= 8 || s.B > dev.cut_clusters16)
    e = launch_cutoff<8>(keys, vhist, sel, s.B, nc, L.nc_pad, K, c0i, s.Hq, stream);
  else
    e = launch_cutoff<16>(keys, vhist, sel, s.B, nc, L.nc_pad, K, c0i, s.Hq, stream);
  return e;
}

}  // namespace qasc

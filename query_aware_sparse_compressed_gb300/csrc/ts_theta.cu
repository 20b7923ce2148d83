// Per-head thresholds of the voting select.
//
// TokenSelect page, section "Voting Mechanism": each head votes for the
// tokens whose score exceeds a head-specific threshold theta_h; reading:
// theta_h is head h's K-th largest Score_h over the candidates C.
//
// No pass keeps every head's scores.  Two kernels bracket the scoring pass:
//   band_kernel     before it: q'_h / sqrt(d') of every head (the scoring
//                   pass's B operand) and, per head, a band [lo, hi] that
//                   should hold theta_h, read off a stratified sample of the
//                   head's candidates.  The scoring pass then counts each
//                   head's scores above hi (their votes are certain) and
//                   lists the scores inside the band.
//   resolve_kernel  after it, one CTA per (b, h): if the count above hi is
//                   below K and the count plus the list reaches K, theta_h is
//                   the (K - above)-th largest listed score, and the listed
//                   scores above it get their vote bit.  Otherwise (the band
//                   missed theta_h, or the list overflowed its capacity) the
//                   CTA recounts the head exactly from the index: three
//                   radix-digit passes over recomputed scores give theta_h,
//                   and a fourth sets the head's vote bit of every candidate
//                   from the same recomputed scores.
// The band only decides which of the two routes runs; both give theta_h
// exactly and the same votes (up to the order of fp32 roundings in a score).
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace qasc {
namespace {

constexpr float kInvSqrtDIdx = 0.17677669529663688f;  // 1 / sqrt(32)
constexpr int kBins = 4096;                             // 12-bit radix digits

// ------------------------------------------------------------------ helpers
// A 32-bit integer hash (xor-shift / multiply rounds) for sample positions.
__device__ __forceinline__ uint32_t mix32(uint32_t x) {
  x ^= x >> 16;
  x *= 0x7feb352du;
  x ^= x >> 15;
  x *= 0x846ca68bu;
  x ^= x >> 16;
  return x;
}

// Score of one 64-byte index row (32 bf16, as four uint4) against q' (fp32).
__device__ __forceinline__ float row_score(const uint4 (&r)[4], const float* qp) {
  float acc = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w[4] = {r[i].x, r[i].y, r[i].z, r[i].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = bf2_to_f2(w[j]);
      acc = fmaf(f.x, qp[8 * i + 2 * j], acc);
      acc = fmaf(f.y, qp[8 * i + 2 * j + 1], acc);
    }
  }
  return acc;
}

__device__ __forceinline__ void load_row(const uint16_t* index, int64_t row, uint4 (&r)[4]) {
  const uint4* p = reinterpret_cast<const uint4*>(index + row * kDIdx);
#pragma unroll
  for (int i = 0; i < 4; ++i) r[i] = __ldg(p + i);
}

// Bin of hist[0, nb) that holds the k-th largest entry (1-based; a larger
// bin holds larger keys): res[0] = bin, res[1] = entries in higher bins.
// Whole block of NT threads; k must lie in [1, total].
template <int NT>
__device__ void find_kth_bin(const uint32_t* hist, int nb, uint32_t k, uint32_t* wsum, int* res) {
  constexpr int kWarps = NT / 32;
  const int per = nb >= NT ? nb / NT : 1;
  const int b0 = static_cast<int>(threadIdx.x) * per;
  uint32_t local = 0;
  if (b0 < nb)
    for (int i = 0; i < per; ++i) local += hist[b0 + i];
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  uint32_t sfx = local;   // suffix sum within the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_down_sync(0xffffffffu, sfx, o);
    if (l + o < 32) sfx += t;
  }
  if (l == 0) wsum[w] = sfx;
  __syncthreads();
  uint32_t above = sfx - local;
  for (int i = w + 1; i < kWarps; ++i) above += wsum[i];
  if (b0 < nb && above < k && k <= above + local) {
    uint32_t acc = above;
    for (int i = per - 1; i >= 0; --i) {
      const uint32_t c = hist[b0 + i];
      if (acc + c >= k) {
        res[0] = b0 + i;
        res[1] = static_cast<int>(acc);
        break;
      }
      acc += c;
    }
  }
  __syncthreads();
}

// Largest order-preserving key that is a float (above it lie NaN patterns),
// and the smallest.
constexpr uint32_t kKeyPosInf = 0xff800000u;
constexpr uint32_t kKeyNegInf = 0x007fffffu;

// ------------------------------------------------------------- band kernel
// One cluster of kBandCTAs CTAs per (b, g).  Every CTA computes q' of the
// group's heads (rank 0 stores it); CTA r scores samples [r m / C, (r+1) m / C)
// of the group's m = min(|C|, kBandSamples) strata (stratum j covers
// candidates [j |C| / m, (j+1) |C| / m), one position in it picked by a hash)
// and sends head hh's sample key to CTA hh.  CTA hh then reads off two order
// statistics of its head's samples: with p = K / |C| the expected share of
// candidates at or above theta_h, the band runs from the sample ranked
// p m + z sd + 1 from the top (lo) to the one ranked p m - z sd (hi), sd =
// sqrt(m p (1 - p)) the binomial spread of the sample count above theta_h.
// Each rank is located to a 24-bit key prefix (two 12-bit digit levels); hi
// is the largest float of its prefix and lo the smallest, so the band only
// widens by those prefixes.
constexpr int kBandCTAs = 8;
constexpr int kBandThreads = 256;
constexpr int kBandSamples = 4096;
constexpr float kBandZ = 5.0f;

struct BandShared {
  uint32_t keys[kBandSamples];           // this CTA's head: every sample key
  union {
    uint16_t w[kD * kDIdx];              // W_g while q' is formed
    uint32_t hist[kBins];                // then the digit histograms
  } u;
  float q[8][kD];
  float qp[8][kDIdx];
  uint32_t wsum[kBandThreads / 32];
  int res[2];
};

__global__ void __launch_bounds__(kBandThreads) band_kernel(const BandArgs a, int Hq, int Hkv, int64_t n_cap, int c0,
                                                            int nc, uint32_t K, int m) {
  __shared__ __align__(16) BandShared S;
  cg::cluster_group cl = cg::this_cluster();
  const int rank = static_cast<int>(cl.block_rank());
  const int bg = static_cast<int>(blockIdx.x) / kBandCTAs;
  const int b = bg / Hkv, g = bg - (bg / Hkv) * Hkv;
  const int gq = Hq / Hkv;
  const int tid = threadIdx.x;
  pdl_wait();
  // The scoring pass may launch now: it waits for this grid before it reads
  // anything written here.
  pdl_trigger();
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * kBandThreads + tid; i < a.n_zero;
       i += static_cast<int64_t>(gridDim.x) * kBandThreads)
    a.zero[i] = 0u;

  // q'_h = W_g^T q_h / sqrt(d') for the group's heads (fp32)
  const uint4* w4 = reinterpret_cast<const uint4*>(a.W + static_cast<int64_t>(g) * kD * kDIdx);
  for (int i = tid; i < kD * kDIdx / 8; i += kBandThreads) reinterpret_cast<uint4*>(S.u.w)[i] = __ldg(w4 + i);
  const uint16_t* qsrc = a.q + (static_cast<int64_t>(b) * Hq + static_cast<int64_t>(g) * gq) * kD;
  for (int i = tid; i < gq * kD; i += kBandThreads) S.q[i / kD][i % kD] = bf_to_f(qsrc[i]);
  __syncthreads();
  {
    const int tpo = 8 / gq;   // threads per output: gq * 32 outputs over 256 threads
    const int o = tid / tpo, part = tid - (tid / tpo) * tpo;
    const int hh = o / kDIdx, j = o - (o / kDIdx) * kDIdx;
    const int span = kD / tpo;
    float acc = 0.0f;
    for (int e = part * span; e < (part + 1) * span; ++e) acc = fmaf(S.q[hh][e], bf_to_f(S.u.w[e * kDIdx + j]), acc);
    for (int off = tpo / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (part == 0) {
      const float x = acc * kInvSqrtDIdx;
      S.qp[hh][j] = x;
      if (rank == 0) a.qp[(static_cast<int64_t>(b) * Hq + g * gq + hh) * kDIdx + j] = x;
    }
  }
  __syncthreads();
  if (a.mode == 0) return;
  if (a.mode == 2) {
    if (rank == 0 && tid < gq) {
      const int64_t bh = static_cast<int64_t>(b) * Hq + g * gq + tid;
      a.band[bh] = a.band_in[bh];
    }
    return;
  }

  // samples of this CTA's strata, each scored for every head of the group
  const int j0 = rank * m / kBandCTAs, j1 = (rank + 1) * m / kBandCTAs;
  for (int j = j0 + tid; j < j1; j += kBandThreads) {
    const int64_t s0 = static_cast<int64_t>(j) * nc / m, s1 = static_cast<int64_t>(j + 1) * nc / m;
    const uint32_t len = static_cast<uint32_t>(s1 - s0);   // >= 1 since m <= nc
    const uint32_t off = mix32(static_cast<uint32_t>(j) * 0x9e3779b9u ^ (static_cast<uint32_t>(bg) * 0x85ebca6bu +
                                                                         0x68e31da4u)) % len;
    const int64_t row = cache_row(a.pm, b, g, Hkv, n_cap, c0 + s0 + off);
    uint4 r[4];
    if (row >= 0) {
      load_row(a.index, row, r);
    } else {
      record_error(a.err, kErrBadPage);
#pragma unroll
      for (int i = 0; i < 4; ++i) r[i] = make_uint4(0, 0, 0, 0);
    }
    for (int hh = 0; hh < gq; ++hh) cl.map_shared_rank(S.keys, hh)[j] = ord_key(row_score(r, S.qp[hh]));
  }
  cl.sync();   // every sample key has reached its head's CTA; no remote access follows
  if (rank >= gq) return;

  const float p = static_cast<float>(K) / static_cast<float>(nc);
  const float mu = p * static_cast<float>(m);
  const float sd = sqrtf(static_cast<float>(m) * p * (1.0f - p));
  const int r_hi = static_cast<int>(floorf(mu - kBandZ * sd));       // < 1: no upper end
  const int r_lo = static_cast<int>(ceilf(mu + kBandZ * sd)) + 1;    // > m: no lower end
  float lo = -INFINITY, hi = INFINITY;
  for (int i = tid; i < kBins; i += kBandThreads) S.u.hist[i] = 0;
  __syncthreads();
  for (int i = tid; i < m; i += kBandThreads) atomicAdd(&S.u.hist[S.keys[i] >> 20], 1u);
  __syncthreads();
  int top[2] = {-1, -1};
  uint32_t kk[2] = {0, 0};
  const int want[2] = {r_hi, r_lo};
#pragma unroll
  for (int t = 0; t < 2; ++t)
    if (want[t] >= 1 && want[t] <= m) {
      find_kth_bin<kBandThreads>(S.u.hist, kBins, static_cast<uint32_t>(want[t]), S.wsum, S.res);
      top[t] = S.res[0];
      kk[t] = static_cast<uint32_t>(want[t]) - static_cast<uint32_t>(S.res[1]);
      __syncthreads();
    }
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    if (top[t] < 0) continue;
    for (int i = tid; i < kBins; i += kBandThreads) S.u.hist[i] = 0;
    __syncthreads();
    for (int i = tid; i < m; i += kBandThreads) {
      const uint32_t key = S.keys[i];
      if (static_cast<int>(key >> 20) == top[t]) atomicAdd(&S.u.hist[(key >> 8) & 0xfffu], 1u);
    }
    __syncthreads();
    find_kth_bin<kBandThreads>(S.u.hist, kBins, kk[t], S.wsum, S.res);
    const uint32_t pre = (static_cast<uint32_t>(top[t]) << 20) | (static_cast<uint32_t>(S.res[0]) << 8);
    if (t == 0) {
      const uint32_t key = pre | 0xffu;
      hi = key >= kKeyPosInf ? INFINITY : ord_val(key);
    } else {
      lo = pre <= kKeyNegInf ? -INFINITY : ord_val(pre);
    }
    __syncthreads();
  }
  if (tid == 0) a.band[static_cast<int64_t>(b) * Hq + g * gq + rank] = make_float2(lo, hi);
}

// ----------------------------------------------------------- resolve kernel
constexpr int kRThreads = 512;
constexpr int kRCap = 16384;   // band-list entries resolved in shared memory

struct ResolveShared {
  uint32_t keys[kRCap];
  uint32_t hist[kBins];
  int delta[kMaxVoteBins];     // changes to this sequence's vote histogram
  uint32_t wsum[kRThreads / 32];
  uint32_t wmax[kRThreads / 32];
  int res[2];
  float qp[kDIdx];
};

// k-th largest (1-based) of keys[0, m) in shared memory: radix digits of at
// most 12 bits, starting below the keys' common leading bits.
__device__ uint32_t select_kth(const uint32_t* keys, int m, uint32_t k, ResolveShared& S) {
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  for (int i = threadIdx.x; i < m; i += kRThreads) {
    kmin = min(kmin, keys[i]);
    kmax = max(kmax, keys[i]);
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if ((threadIdx.x & 31) == 0) {
    S.wsum[threadIdx.x >> 5] = kmin;
    S.wmax[threadIdx.x >> 5] = kmax;
  }
  __syncthreads();
  for (int w = 0; w < kRThreads / 32; ++w) {
    kmin = min(kmin, S.wsum[w]);
    kmax = max(kmax, S.wmax[w]);
  }
  __syncthreads();
  int top = kmin == kmax ? 0 : 32 - __clz(kmin ^ kmax);   // bits [top, 32) are common
  uint32_t pmask = top >= 32 ? 0u : ~0u << top;
  uint32_t prefix = kmin & pmask;
  while (top > 0) {
    const int bits = top > 12 ? 12 : top;
    const int shift = top - bits, nb = 1 << bits;
    const uint32_t dmask = static_cast<uint32_t>(nb - 1);
    for (int i = threadIdx.x; i < nb; i += kRThreads) S.hist[i] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < m; i += kRThreads) {
      const uint32_t x = keys[i];
      if ((x & pmask) == prefix) atomicAdd(&S.hist[(x >> shift) & dmask], 1u);
    }
    __syncthreads();
    find_kth_bin<kRThreads>(S.hist, nb, k, S.wsum, S.res);
    k -= static_cast<uint32_t>(S.res[1]);
    prefix |= static_cast<uint32_t>(S.res[0]) << shift;
    pmask |= dmask << shift;
    top = shift;
    __syncthreads();
  }
  return prefix;
}

struct RecountArgs {
  int b, g, Hkv, c0, nc;
  int64_t n_cap;
};

// Calls f(i, score) for every candidate i of (b, g), the score recomputed
// from its index row in fp32 (four rows in flight per thread).
template <class F>
__device__ __forceinline__ void for_each_score(const ResolveArgs& a, const RecountArgs& r, const float* qp, F&& f) {
  constexpr int U = 4;
  for (int i0 = threadIdx.x; i0 < r.nc; i0 += U * kRThreads) {
    uint4 v[U][4];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * kRThreads;
      int64_t row = i < r.nc ? cache_row(a.pm, r.b, r.g, r.Hkv, r.n_cap, r.c0 + i) : -1;
      if (i < r.nc && row < 0) record_error(a.err, kErrBadPage);
      if (row >= 0) {
        load_row(a.index, row, v[u]);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) v[u][q] = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int i = i0 + u * kRThreads;
      if (i < r.nc) f(i, row_score(v[u], qp));
    }
  }
}

__global__ void __launch_bounds__(kRThreads, 1) resolve_kernel(const ResolveArgs a, int Hq, int Hkv, int64_t n_cap,
                                                               int c0, int nc, uint32_t K) {
  extern __shared__ __align__(16) uint8_t dyn[];
  ResolveShared& S = *reinterpret_cast<ResolveShared*>(dyn);
  const int bh = blockIdx.x;
  const int b = bh / Hq, h = bh - (bh / Hq) * Hq;
  const int g = h / (Hq / Hkv);
  const int tid = threadIdx.x;
  for (int i = tid; i < kMaxVoteBins; i += kRThreads) S.delta[i] = 0;
  pdl_wait();
  const uint32_t above = __ldcg(a.above + bh);
  const uint32_t cnt = __ldcg(a.lcount + bh);
  const bool listed = cnt <= static_cast<uint32_t>(a.list_cap) && cnt <= static_cast<uint32_t>(kRCap) && above < K &&
                      K - above <= cnt;
  uint64_t* mask = a.mask + static_cast<int64_t>(b) * a.nc_pad;
  const uint64_t bit = 1ull << h;
  float theta;
  if (listed) {
    const uint2* lst = a.list + static_cast<int64_t>(bh) * a.list_cap;
    for (int i = tid; i < static_cast<int>(cnt); i += kRThreads) S.keys[i] = ord_key(__uint_as_float(__ldcg(lst + i).x));
    __syncthreads();
    theta = ord_val(select_kth(S.keys, static_cast<int>(cnt), K - above, S));
    // the listed scores above theta_h vote (none has its bit yet: listed
    // scores lie at or below the band's upper end)
    for (int i = tid; i < static_cast<int>(cnt); i += kRThreads) {
      const uint2 e = __ldcg(lst + i);
      if (__uint_as_float(e.x) > theta) {
        const int v = __popcll(atomicOr(reinterpret_cast<unsigned long long*>(mask + e.y), bit));
        atomicSub(&S.delta[v], 1);
        atomicAdd(&S.delta[v + 1], 1);
      }
    }
  } else {
    // exact recount from the index: theta_h by three digit levels (12, 12
    // and 8 bits) over recomputed scores, then the head's vote bit of every
    // candidate from the same scores
    if (tid < kDIdx) S.qp[tid] = __ldcg(a.qp + static_cast<int64_t>(bh) * kDIdx + tid);
    __syncthreads();
    const RecountArgs r = {b, g, Hkv, c0, nc, n_cap};
    uint32_t prefix = 0, pmask = 0, k = K;
    for (int level = 0; level < 3; ++level) {
      const int shift = level == 0 ? 20 : (level == 1 ? 8 : 0);
      const int nb = level == 2 ? 256 : kBins;
      const uint32_t dmask = static_cast<uint32_t>(nb - 1);
      for (int i = tid; i < nb; i += kRThreads) S.hist[i] = 0;
      __syncthreads();
      for_each_score(a, r, S.qp, [&](int, float s) {
        const uint32_t key = ord_key(s);
        if ((key & pmask) == prefix) atomicAdd(&S.hist[(key >> shift) & dmask], 1u);
      });
      __syncthreads();
      find_kth_bin<kRThreads>(S.hist, nb, k, S.wsum, S.res);
      k -= static_cast<uint32_t>(S.res[1]);
      prefix |= static_cast<uint32_t>(S.res[0]) << shift;
      pmask |= dmask << shift;
      __syncthreads();
    }
    theta = ord_val(prefix);
    for_each_score(a, r, S.qp, [&](int i, float s) {
      const bool want = s > theta;
      const bool have = (__ldcg(mask + i) & bit) != 0;
      if (want != have) {
        const int v = __popcll(atomicXor(reinterpret_cast<unsigned long long*>(mask + i), bit));
        atomicSub(&S.delta[v], 1);
        atomicAdd(&S.delta[want ? v + 1 : v - 1], 1);
      }
    });
  }
  __syncthreads();
  for (int v = tid; v < kMaxVoteBins; v += kRThreads)
    if (S.delta[v] != 0) atomicAdd(a.vhist + b * kMaxVoteBins + v, static_cast<uint32_t>(S.delta[v]));
  if (tid == 0) {
    a.theta[bh] = theta;
    a.flag[bh] = listed ? 0 : 1;
  }
  pdl_trigger();
}

}  // namespace

cudaError_t configure_theta_kernels(const DeviceInfo&) {
  return cudaFuncSetAttribute(resolve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(sizeof(ResolveShared)));
}

int launch_band(const qasc_shape& s, const qasc_ts_params& p, const BandArgs& a, cudaStream_t stream) {
  const Regions R = regions_of(s.n, p.sink, p.local);
  const int nc = static_cast<int>(R.nc());
  const int m = nc < kBandSamples ? nc : kBandSamples;
  const unsigned grid = static_cast<unsigned>(s.B) * s.Hkv * kBandCTAs;
  return launch_dependent(band_kernel, dim3(grid), dim3(kBandThreads), 0, stream, kBandCTAs, a, s.Hq, s.Hkv,
                          s.n_cap, static_cast<int>(R.c0), nc, static_cast<uint32_t>(p.K), m);
}

int launch_resolve(const qasc_shape& s, const qasc_ts_params& p, const ResolveArgs& a, cudaStream_t stream) {
  const Regions R = regions_of(s.n, p.sink, p.local);
  return launch_dependent(resolve_kernel, dim3(static_cast<unsigned>(s.B) * s.Hq), dim3(kRThreads),
                          sizeof(ResolveShared), stream, 1, a, s.Hq, s.Hkv, s.n_cap, static_cast<int>(R.c0),
                          static_cast<int>(R.nc()), static_cast<uint32_t>(p.K));
}

// Entries the band list of one head is sized for: twice the candidates a
// band from the sample is expected to hold, at least 2048, at most |C|.
int64_t band_list_capacity(int64_t nc, int64_t K) {
  if (nc <= 0) return 1;
  const double m = static_cast<double>(nc < kBandSamples ? nc : kBandSamples);
  const double p = static_cast<double>(K) / static_cast<double>(nc);
  const double sd = std::sqrt(m * p * (1.0 - p));
  const double frac = (2.0 * kBandZ * sd + 4.0) / m + 2.0 / 4096.0;
  int64_t cap = static_cast<int64_t>(2.0 * frac * static_cast<double>(nc)) + 1024;
  if (cap < 2048) cap = 2048;
  if (cap > nc) cap = nc;
  return cap;
}

}  // namespace qasc

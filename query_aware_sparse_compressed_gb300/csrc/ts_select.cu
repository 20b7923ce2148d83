// The top-K token set of the voting select.
//
// TokenSelect page, section "Voting Mechanism": Vote(i) = sum_h 1[Score_h(i) >
// theta_h]; section "Token-Level Selection と Sparse Attention": S = top-K of
// the candidates with Vote(i) >= V_min.  Candidates are ranked by (Vote desc,
// sum_h Score_h desc, index asc) and S is emitted in ascending token order.
//
// By the time this kernel runs, the scoring and threshold passes have left
// per candidate a 64-bit vote mask (bit h: Score_h > theta_h) and the sum of
// its head scores, and per sequence the histogram of votes.  The cutoff
// forms each candidate's 64-bit key  popcount(mask) << 32 | ord(sum)  and
// selects exactly, without sorting (radix select on the key's low word among
// the candidates with the cut vote).
#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

namespace qasc {
namespace {

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
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

// This CTA's slice of one sequence's keys, formed from the vote masks and
// head sums.
struct CutKeys {
  const uint64_t* mask;  // slice start (64-byte aligned)
  const float* sig;      // slice start (32-byte aligned)
  int m;                 // keys in the slice
  int nchunks;
  uint64_t r[kCutKPT];   // chunk 0

  __device__ __forceinline__ void load(int c, uint64_t (&k)[kCutKPT]) const {
    const int i0 = c * kCutChunk + static_cast<int>(threadIdx.x) * kCutKPT;
    if (i0 + kCutKPT <= m) {
      const ulonglong2* pm = reinterpret_cast<const ulonglong2*>(mask + i0);
      const float4* ps = reinterpret_cast<const float4*>(sig + i0);
      uint64_t mv[kCutKPT];
      float sv[kCutKPT];
#pragma unroll
      for (int j = 0; j < kCutKPT / 2; ++j) {
        const ulonglong2 v = __ldcg(pm + j);
        mv[2 * j] = v.x;
        mv[2 * j + 1] = v.y;
      }
#pragma unroll
      for (int j = 0; j < kCutKPT / 4; ++j) {
        const float4 v = __ldcg(ps + j);
        sv[4 * j] = v.x;
        sv[4 * j + 1] = v.y;
        sv[4 * j + 2] = v.z;
        sv[4 * j + 3] = v.w;
      }
#pragma unroll
      for (int j = 0; j < kCutKPT; ++j)
        k[j] = (static_cast<uint64_t>(__popcll(mv[j])) << 32) | ord_key(sv[j]);
    } else {
#pragma unroll
      for (int j = 0; j < kCutKPT; ++j)
        k[j] = i0 + j < m ? (static_cast<uint64_t>(__popcll(__ldcg(mask + i0 + j))) << 32) |
                                ord_key(__ldcg(sig + i0 + j))
                          : 0ull;
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
    cutoff_kernel(const uint64_t* __restrict__ mask, const float* __restrict__ sigma,
                  const uint32_t* __restrict__ vhist, int32_t* __restrict__ sel, int nc, int64_t nc_pad, int slice,
                  uint32_t K, int c0, int Hq) {
  extern __shared__ __align__(16) uint8_t dyn[];
  CutShared<CS>& S = *reinterpret_cast<CutShared<CS>*>(dyn);
  cg::cluster_group cl = cg::this_cluster();
  const int rank = static_cast<int>(cl.block_rank());
  const int b = blockIdx.x / CS;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i0 = rank * slice;
  pdl_wait();

  CutKeys ks;
  ks.mask = mask + static_cast<int64_t>(b) * nc_pad + i0;
  ks.sig = sigma + static_cast<int64_t>(b) * nc_pad + i0;
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
#pragma unroll 4
      for (int c = 0; c < CS; ++c) t += cl.map_shared_rank(S.hist, c)[rank * seg + tid];
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
cudaError_t launch_cutoff_cs(const uint64_t* mask, const float* sigma, const uint32_t* vhist, int32_t* sel, int B,
                             int nc, int64_t nc_pad, uint32_t K, int c0, int Hq, cudaStream_t stream) {
  const int slice = ((nc + CS - 1) / CS + kCutKPT - 1) / kCutKPT * kCutKPT;
  return launch_dependent(cutoff_kernel<CS>, dim3(static_cast<unsigned>(B * CS)), dim3(kCutThreads),
                          sizeof(CutShared<CS>), stream, CS, mask, sigma, vhist, sel, nc, nc_pad, slice, K, c0, Hq);
}

// K = |C|: every candidate, ascending (no ranking needed).
__global__ void all_candidates_kernel(int32_t* __restrict__ sel, int nc, int c0) {
  pdl_wait();
  const int b = blockIdx.y;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < nc; i += gridDim.x * blockDim.x)
    sel[static_cast<int64_t>(b) * nc + i] = c0 + i;
  pdl_trigger();
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
  int n8 = 0, n16 = 0;
  cudaError_t e;
  if ((e = configure_cutoff<8>(&n8)) != cudaSuccess) return e;
  if (n8 < 1) return cudaErrorNotSupported;
  // 16-CTA clusters where the device schedules them; 8 otherwise
  dev.cut_cluster = configure_cutoff<16>(&n16) == cudaSuccess && n16 >= 1 ? 16 : 8;
  cudaGetLastError();
  return cudaSuccess;
}

SelectLayout select_layout(const qasc_shape& s, const qasc_ts_params& p) {
  SelectLayout L;
  const Regions R = regions_of(s.n, p.sink, p.local);
  L.nc = R.nc();
  L.nc_pad = static_cast<int64_t>(align_up(static_cast<size_t>(L.nc > 0 ? L.nc : 1), 64));
  L.list_cap = band_list_capacity(L.nc, p.K);
  const size_t bh = static_cast<size_t>(s.B) * s.Hq;
  size_t off = 0;
  L.off_qp = off;
  off = align_up(off + bh * kIndexDim * sizeof(float), 256);
  L.off_band = off;
  off = align_up(off + bh * sizeof(float2), 256);
  L.off_theta = off;
  off = align_up(off + bh * sizeof(float), 256);
  L.off_flag = off;
  off = align_up(off + bh * sizeof(int32_t), 256);
  L.off_count = off;
  L.count_words = 2 * bh + static_cast<size_t>(s.B) * kMaxVoteBins;
  off = align_up(off + L.count_words * sizeof(uint32_t), 256);
  L.off_sigma = off;
  off = align_up(off + static_cast<size_t>(s.B) * L.nc_pad * sizeof(float), 256);
  L.off_mask = off;
  off = align_up(off + static_cast<size_t>(s.B) * L.nc_pad * sizeof(uint64_t), 256);
  L.off_list = off;
  off = align_up(off + bh * static_cast<size_t>(L.list_cap) * sizeof(uint2), 256);
  L.total = off;
  return L;
}

int launch_cutoff(const qasc_shape& s, const qasc_ts_params& p, const SelectLayout& L, uint8_t* ws, int32_t* sel,
                  const DeviceInfo& dev, cudaStream_t stream) {
  const Regions R = regions_of(s.n, p.sink, p.local);
  const int nc = static_cast<int>(L.nc);
  const uint32_t K = static_cast<uint32_t>(p.K);
  if (static_cast<int64_t>(K) == L.nc) {
    const unsigned gx = static_cast<unsigned>((nc + 1023) / 1024 < 64 ? (nc + 1023) / 1024 : 64);
    return launch_dependent(all_candidates_kernel, dim3(gx, static_cast<unsigned>(s.B)), dim3(1024), 0, stream, 1,
                            sel, nc, static_cast<int>(R.c0));
  }
  const uint64_t* mask = reinterpret_cast<const uint64_t*>(ws + L.off_mask);
  const float* sigma = reinterpret_cast<const float*>(ws + L.off_sigma);
  const uint32_t* vhist = reinterpret_cast<const uint32_t*>(ws + L.off_count) + 2 * static_cast<size_t>(s.B) * s.Hq;
  return dev.cut_cluster == 16
             ? launch_cutoff_cs<16>(mask, sigma, vhist, sel, s.B, nc, L.nc_pad, K, static_cast<int>(R.c0), s.Hq, stream)
             : launch_cutoff_cs<8>(mask, sigma, vhist, sel, s.B, nc, L.nc_pad, K, static_cast<int>(R.c0), s.Hq, stream);
}

}  // namespace qasc

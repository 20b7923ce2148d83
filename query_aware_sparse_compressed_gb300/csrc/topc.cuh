#pragma once
// Exact top-c of rows of fp32 scores, as the ascending indices of the c
// largest (ties to the lower index), on one thread-block cluster per row.
// Shared by SnapKV's top-c step and the per-KV-head TokenSelect selection.
// Include inside an anonymous namespace of a .cu file, after common.cuh.

// -------------------------------------------------------------- top-c select
// One cluster of CS CTAs per row (8, 4 or 2: the largest whose CTAs fit in
// one wave of the device); CTA r holds the scores of its slice of
// the row as order-preserving keys in shared memory (kPcKPT consecutive per
// thread, each thread reading back only its own).
//  1. Either the producing pass histogrammed the keys' top 12 bits, and
//     every CTA finds the first digit from it; or the row's keys share the
//     leading bits of its smallest and largest key (reduced here from per-CTA
//     partials written by the producing pass), and the digits start below
//     that common prefix: 12 bits, 12 bits, then the rest.  Cluster digit levels
//     (histograms added into rank 0, which finds the digit holding the c-th
//     largest key and broadcasts it) narrow the candidates until rank 0 can
//     hold them.
//  2. The matching keys are pushed to rank 0, which resolves the remaining
//     digits and broadcasts the cut key and the number of ties to take.
//  3. Ordered compaction: a key is kept if it exceeds the cut, or equals it
//     and is among the first ties in index order; every CTA pushes its
//     (greater, equal) counts to all others and writes its kept indices
//     (plus idx_offset) at their ranks (ascending).
constexpr int kPcMaxCS = 8;
constexpr int kPcThreads = 1024;
constexpr int kPcWarps = kPcThreads / 32;
constexpr int kPcKPT = 16;
constexpr int kPcChunk = kPcThreads * kPcKPT;
constexpr int kPcSmemChunks = 2;            // chunks of a slice kept in shared memory (32768 keys)
constexpr int kPcCap = 8192;
constexpr int kPcBins = 4096;               // widest digit: 12 bits

struct TopcShared {
  // chunk c's keys: thread t's float4-group u at keys[(c * kPcKPT / 4 + u) * kPcThreads + t]
  // (a warp's accesses are contiguous, so conflict-free)
  uint4 keys[kPcSmemChunks * kPcChunk / 4];
  uint32_t hist[kPcBins];
  uint32_t recv[kPcBins];        // rank 0: a narrowing level's cluster histogram (sum of the CTAs')
  uint32_t cand[kPcCap];         // rank 0: keys pushed by the cluster
  uint32_t cnt[kPcMaxCS][2];     // (greater, equal) of every CTA
  uint32_t wsum[2][kPcWarps];
  uint32_t scan_tot[2];
  uint32_t ncand;
  uint32_t bcast[3];             // rank 0 -> all: prefix, k, matching count
  int res[2];
};

// Bin of cnt[0, nbins) holding the k-th largest (larger bin = larger keys);
// S.res = {bin, count above}.  Whole block.
__device__ void pc_find_crossing(const uint32_t* cnt, int nbins, uint32_t k, TopcShared& S) {
  const int per = nbins >= kPcThreads ? nbins / kPcThreads : 1;
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
  if (l == 0) S.wsum[0][w] = sfx;
  __syncthreads();
  uint32_t above = sfx - local;
  for (int i = w + 1; i < kPcWarps; ++i) above += S.wsum[0][i];
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

__device__ __forceinline__ uint32_t pc_incl_scan(uint32_t v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

// Block-wide exclusive scans of two counters, and their totals.
__device__ __forceinline__ void pc_excl2(TopcShared& S, uint32_t a, uint32_t b, uint32_t& ea, uint32_t& eb,
                                         uint32_t& ta, uint32_t& tb) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const uint32_t ia = pc_incl_scan(a), ib = pc_incl_scan(b);
  if (lane == 31) {
    S.wsum[0][w] = ia;
    S.wsum[1][w] = ib;
  }
  __syncthreads();
  if (w == 0) {
    const uint32_t xa = lane < kPcWarps ? S.wsum[0][lane] : 0u, xb = lane < kPcWarps ? S.wsum[1][lane] : 0u;
    const uint32_t sa = pc_incl_scan(xa), sb = pc_incl_scan(xb);
    __syncwarp();
    if (lane < kPcWarps) {
      S.wsum[0][lane] = sa - xa;
      S.wsum[1][lane] = sb - xb;
    }
    if (lane == 31) {
      S.scan_tot[0] = sa;
      S.scan_tot[1] = sb;
    }
  }
  __syncthreads();
  ea = S.wsum[0][w] + ia - a;
  eb = S.wsum[1][w] + ib - b;
  ta = S.scan_tot[0];
  tb = S.scan_tot[1];
  __syncthreads();
}

// This CTA's slice of the row as keys: the first kPcSmemChunks chunks staged
// in shared memory (a slice of up to 32768 keys is read from global memory
// once), later chunks reloaded per pass.
struct PcKeys {
  const float* g;
  uint4* sm;
  int m;
  int nchunks;
  __device__ __forceinline__ void load(int c, uint32_t (&k)[kPcKPT]) const {
    const int j0 = c * kPcChunk + static_cast<int>(threadIdx.x) * kPcKPT;
    if (j0 + kPcKPT <= m) {
      const float4* q = reinterpret_cast<const float4*>(g + j0);
#pragma unroll
      for (int t = 0; t < kPcKPT / 4; ++t) {
        const float4 v = __ldcg(q + t);
        k[4 * t + 0] = ord_key(v.x);
        k[4 * t + 1] = ord_key(v.y);
        k[4 * t + 2] = ord_key(v.z);
        k[4 * t + 3] = ord_key(v.w);
      }
    } else {
#pragma unroll
      for (int t = 0; t < kPcKPT; ++t) k[t] = j0 + t < m ? ord_key(__ldcg(g + j0 + t)) : 0u;
    }
  }
  // chunk c (< kPcSmemChunks) from global into shared memory
  __device__ __forceinline__ void stage(int c) const {
    uint32_t k[kPcKPT];
    load(c, k);
#pragma unroll
    for (int u = 0; u < kPcKPT / 4; ++u)
      sm[(c * (kPcKPT / 4) + u) * kPcThreads + threadIdx.x] = make_uint4(k[4 * u], k[4 * u + 1], k[4 * u + 2], k[4 * u + 3]);
  }
  // chunk c's keys into k
  __device__ __forceinline__ void fetch(int c, uint32_t (&k)[kPcKPT]) const {
    if (c < kPcSmemChunks) {
#pragma unroll
      for (int u = 0; u < kPcKPT / 4; ++u) {
        const uint4 v = sm[(c * (kPcKPT / 4) + u) * kPcThreads + threadIdx.x];
        k[4 * u + 0] = v.x;
        k[4 * u + 1] = v.y;
        k[4 * u + 2] = v.z;
        k[4 * u + 3] = v.w;
      }
    } else {
      load(c, k);
    }
  }
};

template <int CS>
__global__ void __cluster_dims__(CS, 1, 1) __launch_bounds__(kPcThreads, 1)
    topc_kernel(const float* __restrict__ p, const uint32_t* __restrict__ prange, int nparts,
                const uint32_t* __restrict__ hist0, int32_t* __restrict__ idx, int64_t n, int64_t n_pad, int c_out,
                int slice, int idx_offset) {
  extern __shared__ __align__(16) uint8_t dyn[];
  TopcShared& S = *reinterpret_cast<TopcShared*>(dyn);
  cg::cluster_group cl = cg::this_cluster();
  const int rank = static_cast<int>(cl.block_rank());
  const int bg = blockIdx.x / CS;
  const int tid = threadIdx.x, lane = tid & 31;
  const int i0 = rank * slice;
  if (tid == 0) S.ncand = 0;
  pdl_wait();
  // the row's first-digit histogram is requested before the keys, so that
  // both reads are in flight together
  constexpr int kHistVec = kPcBins / 4 / kPcThreads;   // uint4 of the histogram per thread
  uint4 hv[kHistVec];
  if (hist0) {
    const uint4* hr = reinterpret_cast<const uint4*>(hist0 + static_cast<int64_t>(bg) * kPcBins);
#pragma unroll
    for (int u = 0; u < kHistVec; ++u) hv[u] = __ldcg(hr + tid + u * kPcThreads);
  }
  PcKeys ks;
  ks.g = p + static_cast<int64_t>(bg) * n_pad + i0;
  ks.sm = S.keys;
  ks.m = max(0, min(static_cast<int>(n) - i0, slice));
  ks.nchunks = (ks.m + kPcChunk - 1) / kPcChunk;
  for (int c = 0; c < ks.nchunks && c < kPcSmemChunks; ++c) ks.stage(c);   // a thread reads back only its own keys
  // visit(f): f(slice index, key) for every key of this thread, in index order
  auto visit = [&](auto&& f) {
    for (int c = 0; c < ks.nchunks; ++c) {
      uint32_t t[kPcKPT];
      ks.fetch(c, t);
      const int j0 = c * kPcChunk + tid * kPcKPT;
#pragma unroll
      for (int j = 0; j < kPcKPT; ++j)
        if (j0 + j < ks.m) f(j0 + j, t[j]);
    }
  };
  int top;
  uint32_t k = static_cast<uint32_t>(c_out);
  uint32_t pmask, prefix, count;   // count: keys matching the fixed digits
  if (hist0) {
    // 1. the first 12-bit digit from the producing pass's histogram of the
    // row (every key counted under key >> 20): each CTA finds the digit
    // holding the c-th largest key itself, no cluster exchange
#pragma unroll
    for (int u = 0; u < kHistVec; ++u) reinterpret_cast<uint4*>(S.hist)[tid + u * kPcThreads] = hv[u];
    __syncthreads();
    pc_find_crossing(S.hist, kPcBins, k, S);
    const uint32_t d = static_cast<uint32_t>(S.res[0]);
    k -= static_cast<uint32_t>(S.res[1]);
    count = S.hist[d];
    top = 20;
    pmask = 0xfff00000u;
    prefix = d << 20;
    __syncthreads();
  } else {
    // 1. digits below the common prefix of the row's keys, from the
    // producing pass's per-CTA key ranges
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    for (int i = tid; i < nparts; i += kPcThreads) {
      const uint2 r = __ldcg(reinterpret_cast<const uint2*>(prange) + static_cast<int64_t>(bg) * nparts + i);
      kmin = min(kmin, r.x);
      kmax = max(kmax, r.y);
    }
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    if (lane == 0) {
      S.wsum[0][tid >> 5] = kmin;
      S.wsum[1][tid >> 5] = kmax;
    }
    __syncthreads();
    for (int w = 0; w < kPcWarps; ++w) {
      kmin = min(kmin, S.wsum[0][w]);
      kmax = max(kmax, S.wsum[1][w]);
    }
    __syncthreads();
    top = kmin == kmax ? 0 : 32 - __clz(kmin ^ kmax);   // bits [top, 32) are common
    pmask = top >= 32 ? 0u : ~0u << top;
    prefix = kmin & pmask;
    count = static_cast<uint32_t>(n);
  }
  auto matches = [&](uint32_t key) { return (key & pmask) == prefix; };
  bool synced = false;   // a cluster barrier has run (every CTA started, rank 0's count zeroed)
  // 1a. narrow with cluster digit levels while rank 0 cannot hold the matching keys
  while (top > 0 && count > static_cast<uint32_t>(kPcCap)) {
    synced = true;
    const int bits = top > 12 ? 12 : top;
    const int shift = top - bits, nb = 1 << bits;
    const uint32_t dmask = static_cast<uint32_t>(nb - 1);
    __syncthreads();
    for (int i = tid; i < nb; i += kPcThreads) S.hist[i] = 0;
    __syncthreads();
    visit([&](int, uint32_t key) {
      if (matches(key)) atomicAdd(&S.hist[(key >> shift) & dmask], 1u);
    });
    cl.sync();   // every CTA's histogram is complete
    if (rank == 0) {
      // rank 0 adds the cluster's histograms with 16-byte loads from every
      // CTA's shared memory (all of a thread's loads in flight together);
      // the others wait at the next cluster barrier, so their histograms
      // stay as they are until this is done
      if (nb >= 4) {
        for (int i = tid; i < nb / 4; i += kPcThreads) {
          uint4 v[CS];
#pragma unroll
          for (int c = 0; c < CS; ++c) v[c] = reinterpret_cast<const uint4*>(cl.map_shared_rank(S.hist, c))[i];
          uint4 t = v[0];
#pragma unroll
          for (int c = 1; c < CS; ++c) {
            t.x += v[c].x;
            t.y += v[c].y;
            t.z += v[c].z;
            t.w += v[c].w;
          }
          reinterpret_cast<uint4*>(S.recv)[i] = t;
        }
      } else if (tid < nb) {
        uint32_t t = 0;
#pragma unroll
        for (int c = 0; c < CS; ++c) t += cl.map_shared_rank(S.hist, c)[tid];
        S.recv[tid] = t;
      }
      if (tid == 0) {
        S.res[0] = 0;
        S.res[1] = 0;
      }
      __syncthreads();
      pc_find_crossing(S.recv, nb, k, S);
      const uint32_t d = static_cast<uint32_t>(S.res[0]);
      const uint32_t nk = k - static_cast<uint32_t>(S.res[1]);
      const uint32_t ncount = S.recv[d];
      if (tid < CS) {
        uint32_t* bc = cl.map_shared_rank(S.bcast, tid);
        bc[0] = prefix | (d << shift);
        bc[1] = nk;
        bc[2] = ncount;
      }
    }
    cl.sync();
    prefix = S.bcast[0];
    k = S.bcast[1];
    count = S.bcast[2];
    pmask |= dmask << shift;
    top = shift;
  }
  // 2. push the matching keys to rank 0 (one remote atomic per warp), which
  // resolves the remaining digits
  if (top > 0) {
    // the first access to another CTA's shared memory waits until every CTA
    // of the cluster runs and rank 0 has zeroed its count (a cluster level's
    // barriers already ordered both)
    if (!synced) cl.sync();
    synced = true;
    uint32_t* n0 = cl.map_shared_rank(&S.ncand, 0);
    uint32_t* c0p = cl.map_shared_rank(S.cand, 0);
    for (int c = 0; c < ks.nchunks; ++c) {
      uint32_t t[kPcKPT];
      ks.fetch(c, t);
      const int j0 = c * kPcChunk + tid * kPcKPT;
      uint32_t mine = 0;
#pragma unroll
      for (int j = 0; j < kPcKPT; ++j) mine += j0 + j < ks.m && matches(t[j]);
      const uint32_t inc = pc_incl_scan(mine);
      const uint32_t wt = __shfl_sync(0xffffffffu, inc, 31);
      uint32_t base = 0;
      if (lane == 31 && wt > 0) base = atomicAdd(n0, wt);
      base = __shfl_sync(0xffffffffu, base, 31) + inc - mine;
      if (mine) {
#pragma unroll
        for (int j = 0; j < kPcKPT; ++j) {
          if (j0 + j >= ks.m) break;
          const uint32_t key = t[j];
          if (matches(key)) {
            if (base < static_cast<uint32_t>(kPcCap)) c0p[base] = key;
            ++base;
          }
        }
      }
    }
    cl.sync();
    if (rank == 0) {
      const int m = static_cast<int>(min(S.ncand, static_cast<uint32_t>(kPcCap)));
      while (top > 0) {
        const int bits = top > 12 ? 12 : top;
        const int shift = top - bits, nb = 1 << bits;
        const uint32_t dmask = static_cast<uint32_t>(nb - 1);
        for (int i = tid; i < nb; i += kPcThreads) S.hist[i] = 0;
        if (tid == 0) {
          S.res[0] = 0;
          S.res[1] = 0;
        }
        __syncthreads();
        for (int i = tid; i < m; i += kPcThreads) {
          const uint32_t x = S.cand[i];
          if ((x & pmask) == prefix) atomicAdd(&S.hist[(x >> shift) & dmask], 1u);
        }
        __syncthreads();
        pc_find_crossing(S.hist, nb, k, S);
        k -= static_cast<uint32_t>(S.res[1]);
        prefix |= static_cast<uint32_t>(S.res[0]) << shift;
        pmask |= dmask << shift;
        top = shift;
        __syncthreads();
      }
      if (tid < CS) {
        uint32_t* bc = cl.map_shared_rank(S.bcast, tid);
        bc[0] = prefix;
        bc[1] = k;
      }
    }
    cl.sync();
    prefix = S.bcast[0];
    k = S.bcast[1];
  }
  const uint32_t cut = prefix, t_take = k;   // the c-th largest key; ties equal to it taken
  // 3. ordered compaction
  uint32_t n_strict = 0, n_tie = 0;
  visit([&](int, uint32_t key) {
    n_strict += key > cut;
    n_tie += key == cut;
  });
  uint32_t e0, e1, cta_strict, cta_tie;
  pc_excl2(S, n_strict, n_tie, e0, e1, cta_strict, cta_tie);
  if (!synced) cl.sync();   // all keys equal: no level or gather ran
  if (tid < CS) {
    uint32_t* d = cl.map_shared_rank(&S.cnt[0][0], tid);
    d[2 * rank + 0] = cta_strict;
    d[2 * rank + 1] = cta_tie;
  }
  cl.sync();   // the last remote access: afterwards each CTA works alone
  uint32_t base = 0, ties_before = 0;
  for (int r = 0; r < rank; ++r) {
    base += S.cnt[r][0] + min(S.cnt[r][1], t_take > ties_before ? t_take - ties_before : 0u);
    ties_before += S.cnt[r][1];
  }
  const uint32_t my_take = min(cta_tie, t_take > ties_before ? t_take - ties_before : 0u);
  int32_t* out = idx + static_cast<int64_t>(bg) * c_out;
  uint32_t strict_base = 0, tie_base = 0;
  for (int c = 0; c < ks.nchunks; ++c) {
    uint32_t t[kPcKPT];
    ks.fetch(c, t);
    const int jb = c * kPcChunk + tid * kPcKPT;
    uint32_t cs = 0, ct = 0;
#pragma unroll
    for (int j = 0; j < kPcKPT; ++j) {
      const bool v = jb + j < ks.m;
      const uint32_t key = t[j];
      cs += v && key > cut;
      ct += v && key == cut;
    }
    uint32_t es, et, ts, tt2;
    pc_excl2(S, cs, ct, es, et, ts, tt2);
    uint32_t sb = strict_base + es, tb = tie_base + et;
#pragma unroll
    for (int j = 0; j < kPcKPT; ++j) {
      if (jb + j >= ks.m) break;
      const uint32_t key = t[j];
      const bool strict = key > cut, tie = key == cut;
      if (strict || (tie && tb < my_take)) {
        const uint32_t pos = base + sb + min(tb, my_take);
        if (pos < static_cast<uint32_t>(c_out)) out[pos] = idx_offset + i0 + jb + j;
      }
      sb += strict;
      tb += tie;
    }
    strict_base += ts;
    tie_base += tt2;
  }
  pdl_trigger();
}


template <int CS>
cudaError_t launch_topc_cs(const float* p, const uint32_t* prange, int nparts, const uint32_t* hist0, int32_t* idx,
                           int rows, int64_t n, int64_t n_pad, int c_out, int idx_offset, cudaStream_t stream) {
  const int slice = static_cast<int>((n + CS - 1) / CS + kPcKPT - 1) / kPcKPT * kPcKPT;
  return launch_dependent(topc_kernel<CS>, dim3(static_cast<unsigned>(rows * CS)), dim3(kPcThreads),
                          sizeof(TopcShared), stream, 1, p, prange, nparts, hist0, idx, n, n_pad, c_out, slice,
                          idx_offset);
}

// Top-c of `rows` rows of n scores (row r at p + r * n_pad; its key-range
// partials at prange + 2 * r * nparts, or, when hist0 is given, the
// histogram of its keys' top 12 bits at hist0 + 4096 r) into idx[r][c_out],
// each index plus idx_offset.  The cluster is the largest of 8, 4 and 2 CTAs of which all
// `rows` clusters are resident at once (max_clusters[0..2]: the device's
// co-resident clusters of 8, 4 and 2, from configure_topc), so that no
// cluster waits for a second wave.
inline cudaError_t launch_topc(const float* p, const uint32_t* prange, int nparts, const uint32_t* hist0, int32_t* idx,
                               int rows, int64_t n, int64_t n_pad, int c_out, int idx_offset, const int* max_clusters,
                               cudaStream_t stream) {
  if (rows <= max_clusters[0])
    return launch_topc_cs<8>(p, prange, nparts, hist0, idx, rows, n, n_pad, c_out, idx_offset, stream);
  if (rows <= max_clusters[1])
    return launch_topc_cs<4>(p, prange, nparts, hist0, idx, rows, n, n_pad, c_out, idx_offset, stream);
  return launch_topc_cs<2>(p, prange, nparts, hist0, idx, rows, n, n_pad, c_out, idx_offset, stream);
}

template <int CS>
cudaError_t configure_topc_cs(int* clusters) {
  cudaError_t e = cudaFuncSetAttribute(topc_kernel<CS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(sizeof(TopcShared)));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CS);
  cfg.blockDim = dim3(kPcThreads);
  cfg.dynamicSmemBytes = sizeof(TopcShared);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(clusters, topc_kernel<CS>, &cfg);
}

// Kernel attributes, and the co-resident clusters of 8, 4 and 2 CTAs.
inline cudaError_t configure_topc(int* max_clusters) {
  cudaError_t e;
  if ((e = configure_topc_cs<8>(&max_clusters[0])) != cudaSuccess) return e;
  if ((e = configure_topc_cs<4>(&max_clusters[1])) != cudaSuccess) return e;
  return configure_topc_cs<2>(&max_clusters[2]);
}

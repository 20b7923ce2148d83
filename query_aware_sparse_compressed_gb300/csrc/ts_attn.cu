// Split-K flash-decode over the attended set T = sink + S + local.
//
// TokenSelect page, section "Token-Level Selection と Sparse Attention",
// equation Attention = softmax(Q K_S^T / sqrt(d)) V_S, with the sink and local
// tokens of the always-included table; section "統合の5ステップ" step 5 merges
// the sparse and local outputs.  Here T is one list per (b, g); pieces of it
// yield (max, sum, unnormalised output) in fp32 and merge_kernel combines them
// exactly (log-sum-exp), which equals a single softmax over T.
//
// Work split: the positions of all (b, g) lists are laid end to end and a
// persistent grid (one CTA per SM) takes equal contiguous ranges of that
// line, so every CTA moves the same number of rows; a range may cross from
// one (b, g) into the next.  A CTA walks its range in tiles of 128 positions.
//
// Roles (288 threads):
//   warps 4-9  loaders, in three pairs: pair s fills ring slot s (tiles
//            t = s mod 3).  They copy the K and V rows of a tile with 16-byte
//            cp.async (a warp instruction moves two whole 256-byte rows, so
//            every row is read coalesced) straight into the MMA operand
//            layout (two 64-column halves, 128-byte swizzle), wait for their
//            own copies and publish the slot, so all three slots' loads are in
//            flight at once.  The pair that loads a (b, g) piece's first tile
//            also stages its queries as the MMA operand.
//   warp 10  MMA (one thread, tcgen05, fp32 accumulators in TMEM):
//              S  = K_tile Q^T      M = 128 tokens, N = 16 (heads), K = d
//              O^T = V_tile^T P     M = 128 dims (V read MN-major), N = 16
//                                   (p_hi and p_lo of each head), K = tokens
//   warps 0-3  softmax: thread r reads token r's logits from TMEM, takes the
//            tile maximum per head (shuffles + one barrier), forms p =
//            exp2(z - m) split into bf16 p_hi + p_lo (~2^-17 relative), writes
//            them as the second MMA's operand, and folds each tile's O^T into
//            fp32 registers (thread r = dimension r): O = O * alpha + O_tile.
// S and O^T are double-buffered in TMEM so that the softmax of tile t overlaps
// the MMAs of tiles t + 1 (S) and t - 1 (O^T).
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace qasc {
namespace {

constexpr int kTile = 128;                       // positions per tile
constexpr int kHalfBytes = kTile * 128;          // 128 rows x 64 bf16 columns
constexpr int kTileBytes = 2 * kHalfBytes;       // one K (or V) tile
constexpr int kStages = 3;
constexpr int kN = 16;                           // MMA N of both products
constexpr int kOpHalf = kN * 128;                // 16 rows x 128 bytes: half of a 16 x 128 operand
constexpr int kSoftWarps = 4;
constexpr int kSoft = 32 * kSoftWarps;
constexpr int kLoadWarps = 6;                    // three pairs, one per ring slot
constexpr int kPairWarps = kLoadWarps / 3;
constexpr int kLoaderRows = kTile / kPairWarps;     // rows of a tile one loader warp copies
constexpr int kLoaderRounds = kLoaderRows / 32;    // row ids per lane
constexpr int kThreads = kSoft + 32 * kLoadWarps + 32;
constexpr int kMmaWarp = kSoftWarps + kLoadWarps;
constexpr int kTmemCols = 64;                    // S[2] at 0, 16; O^T[2] at 32, 48
constexpr int kPartStride = 132;                 // floats per partial: m, l, pad, pad, o[128]
// log2(e) / sqrt(128): logits are kept in base-2 units.
constexpr float kQScale = 1.4426950408889634f * 0.08838834764831845f;

__device__ __forceinline__ int64_t token_at(int64_t j, int64_t sink_end, int64_t K, int64_t local_start,
                                            const int32_t* sel_b) {
  if (j < sink_end) return j;
  if (j < sink_end + K) return sel_b[j - sink_end];
  return local_start + (j - sink_end - K);
}

// Selected entries of list (b, g) in use: all Ksel, or its length when the
// lists carry lengths (clamped to [0, Ksel]).
template <class A>
__device__ __forceinline__ int64_t list_len(const A& a, int b, int g) {
  if (!a.sel_len) return a.Ksel;
  const int64_t v = __ldg(a.sel_len + static_cast<int64_t>(b) * a.len_bstride + static_cast<int64_t>(g) * a.len_gstride);
  return v < 0 ? 0 : (v > a.Ksel ? a.Ksel : v);
}

// Last CTA whose range [c P / G, (c+1) P / G) starts at or before position x,
// i.e. the CTA that holds position x.
__host__ __device__ __forceinline__ int first_cta(int64_t x, int64_t P, int G) {
  int64_t c = ((x + 1) * G + P - 1) / P - 1;
  return static_cast<int>(c < 0 ? 0 : (c >= G ? G - 1 : c));
}

// 16-byte global -> shared copy through L2 (cp.async), with an L2 policy.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "l"(policy)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Byte offset of element (n, k) in a 16-row, 128-column bf16 K-major operand
// stored as two 64-column halves with the 128-byte swizzle.
__device__ __forceinline__ int op_offset(int n, int k) {
  return (k >> 6) * kOpHalf + n * 128 + ((((k & 63) >> 3) ^ (n & 7)) << 4) + (k & 7) * 2;
}

__device__ __forceinline__ uint32_t bf16_rne_bits(float x) {
  uint32_t u = __float_as_uint(x);
  u += 0x7fffu + ((u >> 16) & 1u);
  return u >> 16;
}

struct AttnSmem {
  uint8_t k[kStages][kTileBytes];
  uint8_t v[kStages][kTileBytes];
  uint8_t q[2][2 * kOpHalf];        // queries of a (b, g) piece (rows = heads)
  uint8_t p[2][2 * kOpHalf];        // p_hi (rows 0..GQ-1) and p_lo (rows GQ..2GQ-1) of a tile
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[2], p_empty[2];
  uint64_t o_full[2], o_empty[2];
  float red[2][kSoftWarps][8];      // per-warp head maxima of a tile
  float lred[kSoftWarps][8];        // per-warp head sums of a piece
  uint32_t tmem_base;
};

// Row id of an unused list entry: its K and V rows are zero-filled in shared
// memory, nothing is read.
constexpr int64_t kZeroRow = INT64_MIN;

struct AttnArgs {
  const uint16_t* q;
  const uint16_t* K;
  const uint16_t* V;
  const int32_t* sel;
  int64_t sel_bstride, sel_gstride;   // list of (b, g) at sel + b * sel_bstride + g * sel_gstride
  const int32_t* sel_len;             // optional: entries in use of each list (the rest are masked)
  int64_t len_bstride, len_gstride;
  PageMap pm;        // K / V rows of the main cache (contiguous, or a paged pool)
  const uint16_t* ring_K;   // circular local buffer (ring > 0): token t at slot t mod ring
  const uint16_t* ring_V;
  int64_t ring;
  float* part;       // [B*Hkv][max_splits][GQ][kPartStride]: one partial per covering CTA
  int Hq, Hkv;
  int64_t n_cap, sink_end, Ksel, local_start;
  int64_t T;        // |T| per (b, g)
  int64_t P;        // B * Hkv * T
  int max_splits;   // partial slots per (b, g)
  unsigned* err;
};

// The tiles of this CTA's range, in order: tile counter, bg, first position
// of the tile, rows in the tile, first tile of its piece?, last tile of its
// piece?  A tile made only of unused list entries (past the list's length)
// is skipped by every role alike, unless it ends its piece (each piece keeps
// one tile, so that it still writes its partial); the counter runs over the
// tiles kept.
struct TileInfo {
  int t, bg;
  int64_t q0;
  int rows;
  bool first, last;
};

struct TileIter {
  int64_t p, p_end, seg_end, m0, m1, q0;
  int bg, t;
  bool first;
  __device__ __forceinline__ void start_seg(const AttnArgs& a) {
    bg = static_cast<int>(p / a.T);
    const int64_t base = static_cast<int64_t>(bg) * a.T;
    seg_end = min(p_end, base + a.T);
    // unused entries of this list: positions [m0, m1)
    m0 = base + a.sink_end + list_len(a, bg / a.Hkv, bg % a.Hkv);
    m1 = base + a.sink_end + a.Ksel;
    q0 = p;
    first = true;
  }
  __device__ __forceinline__ void init(const AttnArgs& a, int64_t p_begin, int64_t p_stop) {
    p = p_begin;
    p_end = p_stop;
    t = 0;
    if (p < p_end) start_seg(a);
  }
  __device__ __forceinline__ bool next(const AttnArgs& a, TileInfo& ti) {
    while (p < p_end) {
      if (q0 >= seg_end) {
        p = seg_end;
        if (p < p_end) start_seg(a);
        continue;
      }
      const int rows = static_cast<int>(min(static_cast<int64_t>(kTile), seg_end - q0));
      const bool last = q0 + kTile >= seg_end;
      const int64_t cur = q0;
      q0 += kTile;
      if (!last && cur >= m0 && cur + rows <= m1) continue;
      ti.t = t;
      ti.bg = bg;
      ti.q0 = cur;
      ti.rows = rows;
      ti.first = first;
      ti.last = last;
      ++t;
      first = false;
      return true;
    }
    return false;
  }
};

// f(tile counter, bg, first position, rows, first?, last?) for every tile.
template <class F>
__device__ __forceinline__ void for_each_tile(const AttnArgs& a, int64_t p_begin, int64_t p_end, F&& f) {
  TileIter it;
  it.init(a, p_begin, p_end);
  TileInfo ti;
  while (it.next(a, ti)) f(ti.t, ti.bg, ti.q0, ti.rows, ti.first, ti.last);
}

template <int GQ>
__global__ void __launch_bounds__(kThreads, 1) sparse_attn_kernel(const AttnArgs a) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  AttnSmem& S = *reinterpret_cast<AttnSmem*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int64_t p_begin = static_cast<int64_t>(cta) * a.P / G;
  const int64_t p_end = static_cast<int64_t>(cta + 1) * a.P / G;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.kv_full[s], kPairWarps);
      mbar_init(&S.kv_empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.q_full[i], 1);
      mbar_init(&S.q_empty[i], 1);
      mbar_init(&S.s_full[i], 1);
      mbar_init(&S.s_empty[i], kSoftWarps);
      mbar_init(&S.p_full[i], kSoftWarps);
      mbar_init(&S.p_empty[i], 1);
      mbar_init(&S.o_full[i], 1);
      mbar_init(&S.o_empty[i], kSoftWarps);
    }
    fence_barrier_init();
  }
  // operand padding rows stay zero: queries rows GQ..15, probabilities rows 2GQ..15
  for (int i = tid; i < 2 * 2 * kOpHalf / 16; i += kThreads) {
    const int buf = i / (2 * kOpHalf / 16), r = i - buf * (2 * kOpHalf / 16);
    const int n = (r % (kOpHalf / 16)) / 8;
    if (n >= GQ) reinterpret_cast<uint4*>(S.q[buf])[r] = make_uint4(0, 0, 0, 0);
    if (n >= 2 * GQ) reinterpret_cast<uint4*>(S.p[buf])[r] = make_uint4(0, 0, 0, 0);
  }
  fence_async_smem();
  if (warp == kMmaWarp) tmem_alloc(&S.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  pdl_wait();

  if (warp >= kSoftWarps && warp < kMmaWarp) {
    // ---- loaders: pair s fills ring slot s
    const int lw = warp - kSoftWarps;
    const int pair = lw / kPairWarps, pw = lw % kPairWarps;   // slot, warp within the pair
    const uint64_t pol = policy_evict_first();
    const int half = lane >> 4, c = lane & 15;   // row of the pair, 16-byte chunk of the row
    bool dead = false;
    int seg = -1;
    for_each_tile(a, p_begin, p_end, [&](int t, int bg, int64_t q0, int rows, bool first, bool) {
      if (dead) return;
      if (first) ++seg;
      if (t % kStages != pair) return;
      const int b = bg / a.Hkv, g = bg - b * a.Hkv;
      if (first && pw == 0) {
        const bool ok = mbar_wait(&S.q_empty[seg & 1], ((seg >> 1) & 1u) ^ 1u);
        if (!__all_sync(0xffffffffu, ok)) {
          record_error(a.err, kErrTimeout);
          dead = true;
          return;
        }
        // head n's 128 dims as 16 chunks of 8; chunk c -> half c / 8, column chunk c % 8
        const uint4* qg = reinterpret_cast<const uint4*>(a.q + (static_cast<int64_t>(b) * a.Hq + g * GQ) * kD);
        for (int i = lane; i < GQ * 16; i += 32) {
          const int n = i >> 4, cc = i & 15;
          const uint4 v = __ldg(qg + i);
          *reinterpret_cast<uint4*>(S.q[seg & 1] + (cc >> 3) * kOpHalf + n * 128 + (((cc & 7) ^ (n & 7)) << 4)) = v;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.q_full[seg & 1]);
      }
      const int stage = pair;
      const int32_t* sel_b = a.sel + static_cast<int64_t>(b) * a.sel_bstride + static_cast<int64_t>(g) * a.sel_gstride;
      const int64_t j0 = q0 - static_cast<int64_t>(bg) * a.T;
      // this warp's 64 rows of the tile (two per lane); rows past the end
      // repeat the last valid row; ids outside the cache are clamped so a bad
      // selection cannot fault
      // (positions of a list's unused entries load row 0, which every cache
      // holds, and are masked by the softmax)
      // Row ids: >= 0 a row of the main cache (through the page map);
      // kZeroRow an unused list entry (masked by the softmax), whose shared
      // rows are zero-filled instead of loaded; other negative values
      // (~slot row) a row of the circular local buffer.  A block-table entry
      // outside the pool reads row 0 and records the error.
      const int64_t used_end = a.sink_end + list_len(a, b, g);
      const bool plain = a.pm.table == nullptr && a.ring == 0;   // kernel-uniform: contiguous cache, no ring
      int64_t rowid[kLoaderRounds];
      bool special[kLoaderRounds];
#pragma unroll
      for (int u = 0; u < kLoaderRounds; ++u) {
        const int64_t jp = j0 + min(kLoaderRows * pw + 32 * u + lane, rows - 1);
        const bool masked = jp >= used_end && jp < a.sink_end + a.Ksel;
        int64_t tk = masked ? 0 : token_at(jp, a.sink_end, a.Ksel, a.local_start, sel_b);
        tk = tk < 0 ? 0 : (tk >= a.n_cap ? a.n_cap - 1 : tk);
        int64_t rid;
        if (masked) {
          rid = kZeroRow;
        } else if (plain) {
          rid = static_cast<int64_t>(bg) * a.n_cap + tk;
        } else if (a.ring > 0 && tk >= a.local_start) {
          rid = ~(static_cast<int64_t>(bg) * a.ring + tk % a.ring);
        } else {
          rid = cache_row(a.pm, b, g, a.Hkv, a.n_cap, tk);
          if (rid < 0) {
            record_error(a.err, kErrBadPage);
            rid = 0;
          }
        }
        rowid[u] = rid;
        special[u] = (a.sel_len != nullptr || !plain) && __any_sync(0xffffffffu, rid < 0);
      }
      const bool ok = mbar_wait(&S.kv_empty[stage], ((t / kStages) & 1u) ^ 1u);
      if (!__all_sync(0xffffffffu, ok)) {
        record_error(a.err, kErrTimeout);
        dead = true;
        return;
      }
#pragma unroll
      for (int u = 0; u < kLoaderRounds; ++u) {
        if (!special[u]) {   // warp-uniform: every row of this group in the main cache
#pragma unroll 4
          for (int i = 0; i < 16; ++i) {
            const int r = kLoaderRows * pw + 32 * u + 2 * i + half;   // row in the tile
            const int64_t rid = __shfl_sync(0xffffffffu, rowid[u], 2 * i + half);
            const uint32_t off = (c >> 3) * kHalfBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4);
            cp_async16(S.k[stage] + off, a.K + rid * kD + 8 * c, pol);
            cp_async16(S.v[stage] + off, a.V + rid * kD + 8 * c, pol);
          }
        } else {
#pragma unroll 4
          for (int i = 0; i < 16; ++i) {
            const int r = kLoaderRows * pw + 32 * u + 2 * i + half;
            const int64_t rid = __shfl_sync(0xffffffffu, rowid[u], 2 * i + half);
            const uint32_t off = (c >> 3) * kHalfBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4);
            if (rid == kZeroRow) {
              *reinterpret_cast<uint4*>(S.k[stage] + off) = make_uint4(0u, 0u, 0u, 0u);
              *reinterpret_cast<uint4*>(S.v[stage] + off) = make_uint4(0u, 0u, 0u, 0u);
            } else {
              const uint16_t* kr = rid >= 0 ? a.K + rid * kD : a.ring_K + (~rid) * kD;
              const uint16_t* vr = rid >= 0 ? a.V + rid * kD : a.ring_V + (~rid) * kD;
              cp_async16(S.k[stage] + off, kr + 8 * c, pol);
              cp_async16(S.v[stage] + off, vr + 8 * c, pol);
            }
          }
        }
      }
      cp_async_commit();
      cp_async_wait<0>();
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.kv_full[stage]);
    });
    cp_async_wait<0>();   // nothing of this warp stays in flight past here
  } else if (warp == kMmaWarp) {
    // ---- MMA issue (one thread)
    if (lane == 0) {
      constexpr uint32_t idesc_s = mma_idesc(128, kN);
      constexpr uint32_t idesc_o = mma_idesc_amn(128, kN);
      bool dead = false;
      int seg = -1;
      auto mma_o = [&](int u) {   // O^T of tile u (its probabilities and accumulator ready)
        const int j = u & 1;
        tc_fence_after();
        const uint32_t vb = smem_u32(S.v[u % kStages]);
        const uint32_t pb = smem_u32(S.p[j]);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16(tmem + 32 + 16 * j, sw128_mn_desc(vb + kk * 2048, kHalfBytes, 1024),
                   sw128_desc(pb + (kk >> 2) * kOpHalf + (kk & 3) * 32), idesc_o, kk > 0 ? 1u : 0u);
        mma_commit(&S.o_full[j]);
        mma_commit(&S.p_empty[j]);
        mma_commit(&S.kv_empty[u % kStages]);
      };
      // Each tile's O^T product is issued as soon as its probabilities are
      // in, ahead of the next tile's S product, so that a ring slot is
      // released without waiting for the next tile's rows to arrive; S runs
      // ahead whenever O has nothing to do.
      TileIter sit;
      sit.init(a, p_begin, p_end);
      TileInfo nt;
      bool have = sit.next(a, nt);
      int ns = 0, no = 0;   // tiles whose S / O^T products are issued
      unsigned long long idle_since = globaltimer_ns();
      while (!dead && (have || no < ns)) {
        bool progress = false;
        if (no < ns) {
          const int j = no & 1;
          if (mbar_try_wait(&S.p_full[j], (no >> 1) & 1u) && mbar_try_wait(&S.o_empty[j], ((no >> 1) & 1u) ^ 1u)) {
            mma_o(no);
            ++no;
            progress = true;
          }
        }
        if (!progress && have) {
          const int t = nt.t, j = t & 1, stage = t % kStages;
          if (mbar_try_wait(&S.kv_full[stage], (t / kStages) & 1u) &&
              mbar_try_wait(&S.s_empty[j], ((t >> 1) & 1u) ^ 1u)) {
            if (nt.first) {
              if (seg >= 0) mma_commit(&S.q_empty[seg & 1]);   // the previous piece's queries are free after these
              ++seg;
              if (!mbar_wait(&S.q_full[seg & 1], (seg >> 1) & 1u)) {
                record_error(a.err, kErrTimeout);
                dead = true;
                break;
              }
            }
            tc_fence_after();
            const uint32_t kb = smem_u32(S.k[stage]);
            const uint32_t qb = smem_u32(S.q[seg & 1]);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_bf16(tmem + 16 * j, sw128_desc(kb + (kk >> 2) * kHalfBytes + (kk & 3) * 32),
                       sw128_desc(qb + (kk >> 2) * kOpHalf + (kk & 3) * 32), idesc_s, kk > 0 ? 1u : 0u);
            mma_commit(&S.s_full[j]);
            ++ns;
            have = sit.next(a, nt);
            progress = true;
          }
        }
        if (progress) {
          idle_since = globaltimer_ns();
        } else if (globaltimer_ns() - idle_since > kWaitTimeoutNs) {
          record_error(a.err, kErrTimeout);
          dead = true;
        }
      }
    }
  } else {
    // ---- softmax and output (thread r = TMEM lane r)
    const int r = tid;                          // token row of S, dimension of O^T
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * warp) << 16);
    float M[GQ], lp[GQ], O[GQ], alpha_prev[GQ];
    bool dead = false;
    auto fold = [&](int u) {   // O = O * alpha_prev + O^T of tile u
      const int j = u & 1;
      if (!dead) {
        const bool ok = mbar_wait(&S.o_full[j], (u >> 1) & 1u);
        if (!__all_sync(0xffffffffu, ok)) {
          record_error(a.err, kErrTimeout);
          dead = true;
        }
      }
      if (dead) return;
      tc_fence_after();
      float ot[2 * GQ];
      tmem_ld_cols<2 * GQ>(tl + 32 + 16 * j, ot);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.o_empty[j]);
#pragma unroll
      for (int h = 0; h < GQ; ++h) O[h] = fmaf(O[h], alpha_prev[h], ot[h] + ot[GQ + h]);
    };
    for_each_tile(a, p_begin, p_end, [&](int t, int bg, int64_t q0, int rows, bool first, bool last) {
      const int j = t & 1;
      if (first) {
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
          M[h] = -INFINITY;
          lp[h] = 0.0f;
          O[h] = 0.0f;
          alpha_prev[h] = 1.0f;
        }
      }
      float z[GQ];
      if (!dead) {
        const bool ok = mbar_wait(&S.s_full[j], (t >> 1) & 1u);
        if (!__all_sync(0xffffffffu, ok)) {
          record_error(a.err, kErrTimeout);
          dead = true;
        }
      }
      if (!dead) {
        tc_fence_after();
        tmem_ld_cols<GQ>(tl + 16 * j, z);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.s_empty[j]);
      }
      bool valid = r < rows && !dead;
      if (a.sel_len) {   // unused entries of a list with a length
        const int b = bg / a.Hkv, g = bg - b * a.Hkv;
        const int64_t jp = q0 - static_cast<int64_t>(bg) * a.T + r;
        valid = valid && !(jp >= a.sink_end + list_len(a, b, g) && jp < a.sink_end + a.Ksel);
      }
#pragma unroll
      for (int h = 0; h < GQ; ++h) z[h] = valid ? z[h] * kQScale : -INFINITY;
      // tile maximum per head
#pragma unroll
      for (int h = 0; h < GQ; ++h) {
        float m = warp_max(z[h]);
        if (lane == 0) S.red[j][warp][h] = m;
      }
      named_bar_sync(1, kSoft);
      float al[GQ], pr[GQ];
#pragma unroll
      for (int h = 0; h < GQ; ++h) {
        float mt = S.red[j][0][h];
#pragma unroll
        for (int w = 1; w < kSoftWarps; ++w) mt = fmaxf(mt, S.red[j][w][h]);
        const float mn = fmaxf(M[h], mt);
        al[h] = mn == -INFINITY ? 1.0f : ex2_approx(M[h] - mn);
        pr[h] = mn == -INFINITY ? 0.0f : ex2_approx(z[h] - mn);
        lp[h] = fmaf(lp[h], al[h], pr[h]);
        M[h] = mn;
      }
      // p as the second product's operand: rows h (hi) and GQ + h (lo), column r
      if (!dead) {
        const bool ok = mbar_wait(&S.p_empty[j], ((t >> 1) & 1u) ^ 1u);
        if (!__all_sync(0xffffffffu, ok)) {
          record_error(a.err, kErrTimeout);
          dead = true;
        }
      }
      if (!dead) {
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
          const uint32_t hi = bf16_rne_bits(pr[h]);
          const uint32_t lo = bf16_rne_bits(pr[h] - __uint_as_float(hi << 16));
          *reinterpret_cast<uint16_t*>(S.p[j] + op_offset(h, r)) = static_cast<uint16_t>(hi);
          *reinterpret_cast<uint16_t*>(S.p[j] + op_offset(GQ + h, r)) = static_cast<uint16_t>(lo);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.p_full[j]);
      }
      if (!first) fold(t - 1);
#pragma unroll
      for (int h = 0; h < GQ; ++h) alpha_prev[h] = al[h];
      if (last) {
        fold(t);
        // this CTA's partial of the piece
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
          float l = lp[h];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
          if (lane == 0) S.lred[warp][h] = l;
        }
        named_bar_sync(1, kSoft);
        const int64_t x0 = static_cast<int64_t>(bg) * a.T;
        const int split = cta - first_cta(x0, a.P, G);
        float* base = a.part + (static_cast<int64_t>(bg) * a.max_splits + split) * GQ * kPartStride;
#pragma unroll
        for (int h = 0; h < GQ; ++h) {
          base[h * kPartStride + 4 + r] = O[h];
          if (r == 0) {
            base[h * kPartStride + 0] = M[h];
            base[h * kPartStride + 1] = (S.lred[0][h] + S.lred[1][h]) + (S.lred[2][h] + S.lred[3][h]);
          }
        }
        named_bar_sync(1, kSoft);   // lred is rewritten by the next piece
      }
    });
  }
  tc_fence_before();
  __syncthreads();
  pdl_trigger();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// grid B * Hq, block 512: exact log-sum-exp merge of the partials of every
// CTA that covered this (b, g).  Every load is issued before the first
// barrier: the partials' (max, sum) pairs go to shared memory, and when a
// (b, h) has at most kMergeFast partials each thread also holds the values
// of its output dimension from its partials in registers; so the merge
// costs one round trip to memory.  Four threads per output dimension each
// sum a quarter of the weighted partial outputs, and the quarters are added.
constexpr int kMergeMax = 2048;   // partials per (b, h) the merge can stage
constexpr int kMergeThreads = 4 * kD;
constexpr int kMergeFast = 32;    // partials held in registers (8 per thread)

template <int GQ>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const float* __restrict__ part,
                                                             float* __restrict__ out, float* __restrict__ lse,
                                                             int Hkv, int64_t T, int64_t P, int G, int max_splits) {
  __shared__ float wgt[kMergeMax];
  __shared__ float lsum[kMergeMax];
  __shared__ float red[2][kMergeThreads / 32];
  __shared__ float quarter[3][kD];
  const int bh = blockIdx.x;
  const int Hq = Hkv * GQ;
  pdl_wait();
  const int b = bh / Hq, h = bh - b * Hq;
  const int g = h / GQ, hh = h - g * GQ;
  const int bg = b * Hkv + g;
  const int64_t x0 = static_cast<int64_t>(bg) * T;
  const int c0 = first_cta(x0, P, G);
  const int c1 = first_cta(x0 + T - 1, P, G);
  const int n = min(c1 - c0 + 1, kMergeMax);
  const int64_t pstride = static_cast<int64_t>(GQ) * kPartStride;
  const float* base = part + static_cast<int64_t>(bg) * max_splits * pstride + hh * kPartStride;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int e = tid & (kD - 1), q4 = tid >> 7;
  const bool fast = n <= kMergeFast;
  float v[8];
  if (fast) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int s = q4 + 4 * u;
      v[u] = s < n ? __ldcg(base + s * pstride + 4 + e) : 0.0f;
    }
  }
  float M = -INFINITY;
  for (int s = tid; s < n; s += kMergeThreads) {
    const float ms = __ldcg(base + s * pstride);
    lsum[s] = __ldcg(base + s * pstride + 1);
    wgt[s] = ms;
    M = fmaxf(M, ms);
  }
  M = warp_max(M);
  if (lane == 0) red[0][warp] = M;
  __syncthreads();
  M = red[0][0];
#pragma unroll
  for (int i = 1; i < kMergeThreads / 32; ++i) M = fmaxf(M, red[0][i]);
  float Lp = 0.0f;
  for (int s = tid; s < n; s += kMergeThreads) {
    const float ms = wgt[s];
    const float w = ms == -INFINITY ? 0.0f : exp2f(ms - M);
    wgt[s] = w;
    Lp = fmaf(w, lsum[s], Lp);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Lp += __shfl_xor_sync(0xffffffffu, Lp, o);
  if (lane == 0) red[1][warp] = Lp;
  __syncthreads();
  float L = 0.0f;
#pragma unroll
  for (int i = 0; i < kMergeThreads / 32; ++i) L += red[1][i];
  float O[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
  if (fast) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int s = q4 + 4 * u;
      if (s < n) O[u] = wgt[s] * v[u];
    }
  } else {
    int s = q4;
    for (; s + 28 < n; s += 32) {
      float w8[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) w8[u] = __ldcg(base + (s + 4 * u) * pstride + 4 + e);
#pragma unroll
      for (int u = 0; u < 8; ++u) O[u] = fmaf(wgt[s + 4 * u], w8[u], O[u]);
    }
    for (; s < n; s += 4) O[0] = fmaf(wgt[s], __ldcg(base + s * pstride + 4 + e), O[0]);
  }
  const float Oq = ((O[0] + O[1]) + (O[2] + O[3])) + ((O[4] + O[5]) + (O[6] + O[7]));
  if (q4 > 0) quarter[q4 - 1][e] = Oq;
  __syncthreads();
  if (q4 == 0) {
    out[static_cast<int64_t>(bh) * kD + e] = ((Oq + quarter[0][e]) + (quarter[1][e] + quarter[2][e])) / L;
    if (lse && e == 0) lse[bh] = (M + log2f(L)) * 0.6931471805599453f;
  }
  pdl_trigger();
}

// One CTA per SM, but at least one full tile of positions per CTA.
int grid_for(int64_t P, int num_sms) {
  int64_t G = static_cast<int64_t>(num_sms > 0 ? num_sms : 148);
  const int64_t by_rows = P / kTile;
  if (G > by_rows) G = by_rows;
  if (G < 1) G = 1;
  return static_cast<int>(G);
}

template <int GQ>
int launch_gq(const qasc_shape& s, const qasc_ts_params& p, const AttnLayout& L, const uint16_t* q,
              const uint16_t* K, const uint16_t* V, const int32_t* sel, bool sel_per_kv, const int32_t* sel_len,
              const PageMap& pm, const RingMap& ring, float* out, float* lse, float* part, const DeviceInfo& dev,
              cudaStream_t stream) {
  const Regions R = regions_of(s.n, p.sink, p.local);
  AttnArgs a;
  a.pm = pm;
  a.ring_K = ring.K;
  a.ring_V = ring.V;
  a.ring = ring.K ? ring.R : 0;
  a.q = q;
  a.K = K;
  a.V = V;
  a.sel = sel;
  a.sel_bstride = sel_per_kv ? static_cast<int64_t>(s.Hkv) * p.K : p.K;
  a.sel_gstride = sel_per_kv ? p.K : 0;
  a.sel_len = sel_len;
  a.len_bstride = sel_per_kv ? s.Hkv : 1;
  a.len_gstride = sel_per_kv ? 1 : 0;
  a.part = part;
  a.Hq = s.Hq;
  a.Hkv = s.Hkv;
  a.n_cap = s.n_cap;
  a.sink_end = R.sink_end;
  a.Ksel = p.K;
  a.local_start = R.local_start;
  a.T = L.t_len;
  a.P = L.t_len * s.B * s.Hkv;
  a.max_splits = L.splits;
  a.err = dev.err_word;
  const int G = grid_for(a.P, dev.num_sms);
  cudaError_t e = launch_dependent(sparse_attn_kernel<GQ>, dim3(G), dim3(kThreads), sizeof(AttnSmem) + 1024, stream, 1, a);
  if (e != cudaSuccess) return e;
  return launch_dependent(merge_kernel<GQ>, dim3(s.B * s.Hq), dim3(kMergeThreads), 0, stream, 1,
                          static_cast<const float*>(part), out, lse, s.Hkv, a.T, a.P, G, L.splits);
}

template <int GQ>
cudaError_t configure_gq() {
  return cudaFuncSetAttribute(sparse_attn_kernel<GQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(sizeof(AttnSmem) + 1024));
}

}  // namespace

cudaError_t configure_attn_kernels(const DeviceInfo&) {
  cudaError_t e;
  if ((e = configure_gq<1>()) != cudaSuccess) return e;
  if ((e = configure_gq<2>()) != cudaSuccess) return e;
  if ((e = configure_gq<4>()) != cudaSuccess) return e;
  return configure_gq<8>();
}

AttnLayout attn_layout(const qasc_shape& s, const qasc_ts_params& p, int num_sms) {
  AttnLayout L;
  const Regions R = regions_of(s.n, p.sink, p.local);
  L.t_len = R.sink_end + p.K + (s.n - R.local_start);
  const int64_t bg = static_cast<int64_t>(s.B) * s.Hkv;
  const int64_t P = L.t_len * bg;
  const int G = grid_for(P, num_sms);
  // CTAs overlapping one (b, g) list: every CTA range holds at least
  // floor(P / G) >= 128 positions, so at most (T - 1) / floor(P / G) + 2.
  L.splits = static_cast<int>((L.t_len - 1) / (P / G) + 2);
  L.per_split = 0;
  L.off_part = 0;
  L.total = align_up(static_cast<size_t>(bg) * L.splits * (s.Hq / s.Hkv) * kPartStride * sizeof(float), 256);
  return L;
}

int launch_sparse_attn(const qasc_shape& s, const qasc_ts_params& p, const AttnLayout& L, const uint16_t* q,
                       const uint16_t* K, const uint16_t* V, const int32_t* sel, float* out, float* lse,
                       uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream, bool sel_per_kv,
                       const int32_t* sel_len, const PageMap* pm, const RingMap* ring) {
  float* part = reinterpret_cast<float*>(ws + L.off_part);
  const PageMap m = pm ? *pm : PageMap();
  const RingMap r = ring ? *ring : RingMap();
  switch (s.Hq / s.Hkv) {
    case 1: return launch_gq<1>(s, p, L, q, K, V, sel, sel_per_kv, sel_len, m, r, out, lse, part, dev, stream);
    case 2: return launch_gq<2>(s, p, L, q, K, V, sel, sel_per_kv, sel_len, m, r, out, lse, part, dev, stream);
    case 4: return launch_gq<4>(s, p, L, q, K, V, sel, sel_per_kv, sel_len, m, r, out, lse, part, dev, stream);
    case 8: return launch_gq<8>(s, p, L, q, K, V, sel, sel_per_kv, sel_len, m, r, out, lse, part, dev, stream);
    default: return -1;
  }
}

// ---------------------------------------------------------------------------
// Allocation-free variant, behind ts_sparse_attn_noalloc.
//
// Some callers cannot hand the library a workspace: engines and plugins that
// receive only their input and output buffers, serving runtimes whose memory
// planner owns every device allocation and forbids new ones while requests
// run (an allocation could fail or fragment the pool mid-step), and latency-
// critical loops that cannot afford cudaMalloc's implicit synchronisation.
// For them the split-K partials go to a fixed area compiled into the library.
//
// The area is kNoAllocScratchBytes and stays reserved on every GPU that loads
// the library until the process exits.  Host code cannot use the symbol's
// name as an address, so the first call on each device (with that device
// current) looks the address up with cudaGetSymbolAddress and caches it;
// that first call should happen before any stream capture.  The cached
// address belongs to the device's primary context as it was then: a
// cudaDeviceReset (a new primary context) leaves it stale, and this entry
// point must not be called again after one.  Every call shares
// the area and it keeps whatever the previous call left; nothing in it has to
// start at zero, because each partial the merge reads is written earlier in
// the same call.  Calls that can run at the same time on the GPU race on the
// area, so they must be serialised.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) uint8_t g_attn_noalloc_scratch[kNoAllocScratchBytes];

size_t sparse_attn_noalloc_capacity() { return kNoAllocScratchBytes; }

int launch_sparse_attn_noalloc(const qasc_shape& s, const qasc_ts_params& p, const AttnLayout& L, const uint16_t* q,
                               const uint16_t* K, const uint16_t* V, const int32_t* sel, float* out, float* lse,
                               const DeviceInfo& dev, cudaStream_t stream) {
  static uint8_t* area[64];
  static std::mutex mu;
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
  uint8_t* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!area[dev.device]) {
      void* ptr = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&ptr, g_attn_noalloc_scratch);
      if (e != cudaSuccess) return e;
      area[dev.device] = static_cast<uint8_t*>(ptr);
    }
    ws = area[dev.device];
  }
  return launch_sparse_attn(s, p, L, q, K, V, sel, out, lse, ws, dev, stream);
}

}  // namespace qasc

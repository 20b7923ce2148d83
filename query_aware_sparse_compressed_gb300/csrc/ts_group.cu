// Group-summed index scores of every candidate, for the selection per KV
// head (TokenSelect page, ablation "w/o Voting").
//
// TokenSelect page, section "Query-Key Dot Product Index", equation Score_h:
//   Score_h(i) = q'_h . k_index(i) / sqrt(d'),  q'_h = W_{g(h)}^T q_h (fp32).
// Per (b, g) and candidate i this pass writes sum over the group's heads of
// Score_h(i) (head order), and per (b, g, 512-token block) the smallest and
// largest order-preserving key of those sums (the top-c kernel starts its
// digits below their common leading bits).
//
// The dot products of one (b, g) form a small dense contraction,
// [512 tokens x 32] x [32 x Gq], which runs on the tcgen05 tensor cores:
//   - qprime_kernel first forms q'_h / sqrt(d') (fp32) of every head.  The
//     B operand of group g splits it into three bf16 parts hi + mid + lo
//     (each the round-to-nearest-even of what the earlier parts leave; their
//     sum equals the fp32 value to ~2^-24 relative), as row part * Gq + head
//     of an N-row tile (N = 16, or 32 for Gq = 8; zero padded) in the
//     64-byte-swizzled K-major layout.  The epilogue warps build the operands
//     of every group of a sequence.
//   - The scoring kernel is persistent: one CTA per SM over contiguous runs
//     of units (sequence b, 512-token block); a unit's stages are its Hkv
//     groups in order.  A TMA warp loads each stage's 32 KB of index rows
//     (2-D tensor map, 64-byte swizzle, two 256-row boxes) into a ring; one
//     MMA thread issues eight M=128 x N x K=16 MMAs per stage (four 128-token
//     quarters x two K steps, interleaved so that the four accumulation
//     chains overlap) into TMEM; sixteen epilogue warps (four per TMEM lane
//     quarter) read one token's 3 Gq partial scores per thread, add the parts
//     (lo + mid first) and the group's heads.
#include <cuda.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace qasc {
namespace {

constexpr float kInvSqrtDIdx = 0.17677669529663688f;  // 1 / sqrt(32)
constexpr int kTileTok = kGroupBlock;         // tokens per stage (one block of one group)
constexpr int kTileBytes = kTileTok * kDIdx * 2;
constexpr int kBoxRows = 256;                 // rows per TMA box (two per stage; paged: min(P, 256))
constexpr int kSub = kTileTok / 128;          // 128-token MMA tiles per stage
constexpr int kMaxStages = 4;
constexpr int kAccStages = 4;                 // TMEM accumulators (one stage each)
constexpr int kEpiWarps = 16;                 // four per TMEM lane quarter: one token per thread per stage
constexpr int kEpi = 32 * kEpiWarps;
constexpr int kThreads = kEpi + 64;           // TMA warp, MMA warp, epilogue warps
constexpr int kParts = 3;                     // q' = hi + mid + lo
// MMA N: the 3 Gq rows of (part, head), padded to a multiple of 16.
__host__ __device__ constexpr int mma_n(int gq) { return gq <= 4 ? 16 : 32; }
__host__ __device__ constexpr int tmem_cols(int gq) { return kAccStages * kSub * mma_n(gq); }

// ------------------------------------------------------------ q' kernel
// One CTA of 256 threads per (b, g): q'_h = W_g^T q_h / sqrt(d') in fp32 for
// the group's heads, 8 / Gq threads per output column.
__global__ void __launch_bounds__(256) qprime_kernel(const uint16_t* __restrict__ q, const uint16_t* __restrict__ W,
                                                     float* __restrict__ qp, int Hq, int Hkv) {
  __shared__ __align__(16) uint16_t wst[kD * kDIdx];
  __shared__ float qs[8][kD];
  const int bg = blockIdx.x;
  const int b = bg / Hkv, g = bg - (bg / Hkv) * Hkv;
  const int gq = Hq / Hkv;
  const int tid = threadIdx.x;
  pdl_wait();
  const uint4* w4 = reinterpret_cast<const uint4*>(W + static_cast<int64_t>(g) * kD * kDIdx);
  for (int i = tid; i < kD * kDIdx / 8; i += 256) reinterpret_cast<uint4*>(wst)[i] = __ldg(w4 + i);
  const uint16_t* qsrc = q + (static_cast<int64_t>(b) * Hq + static_cast<int64_t>(g) * gq) * kD;
  for (int i = tid; i < gq * kD; i += 256) qs[i / kD][i % kD] = bf_to_f(qsrc[i]);
  __syncthreads();
  const int tpo = 8 / gq;
  const int o = tid / tpo, part = tid - (tid / tpo) * tpo;
  const int hh = o / kDIdx, c = o - (o / kDIdx) * kDIdx;
  const int span = kD / tpo;
  float acc = 0.0f;
  for (int e = part * span; e < (part + 1) * span; ++e) acc = fmaf(qs[hh][e], bf_to_f(wst[e * kDIdx + c]), acc);
  for (int off = tpo / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (part == 0) qp[(static_cast<int64_t>(b) * Hq + static_cast<int64_t>(g) * gq + hh) * kDIdx + c] = acc * kInvSqrtDIdx;
  pdl_trigger();
}

// ------------------------------------------------------- scoring kernel
struct Misc {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t bfull[2], bempty[2];
  uint64_t acc_full[kAccStages], acc_empty[kAccStages];
  uint32_t tmem_base;
  uint32_t rmin[64], rmax[64];   // key range of each group's sums in the current block
};

// The stage a role works on, advanced without divisions: group g of block
// blk of sequence b (stage order: sequences, blocks, groups).
struct Cursor {
  int g, blk, b;
  __device__ __forceinline__ void init(int u0, int blocks) {
    g = 0;
    b = u0 / blocks;
    blk = u0 - b * blocks;
  }
  __device__ __forceinline__ void next(int Hkv, int blocks) {
    if (++g == Hkv) {
      g = 0;
      if (++blk == blocks) {
        blk = 0;
        ++b;
      }
    }
  }
};

// Shared-memory layout (byte offsets from the 1024-aligned base), chosen on
// the host: the index ring, nbuf B-operand buffers of Hkv groups each, then
// Misc.
struct Plan {
  int stages = 0, nbuf = 0, gbytes = 0;
  uint32_t off_bq = 0, off_misc = 0, bytes = 0;
};

Plan make_plan(int gq, int Hkv, int max_smem) {
  Plan P;
  P.gbytes = mma_n(gq) * 64;
  for (int stages = kMaxStages; stages >= 2; --stages)
    for (int nbuf = 2; nbuf >= 1; --nbuf) {
      uint32_t off = static_cast<uint32_t>(stages) * kTileBytes;
      P.off_bq = off;
      off += static_cast<uint32_t>(nbuf * Hkv * P.gbytes);
      P.off_misc = static_cast<uint32_t>(align_up(off, 16));
      P.bytes = P.off_misc + static_cast<uint32_t>(sizeof(Misc)) + 1024;   // + base alignment
      if (P.bytes <= static_cast<uint32_t>(max_smem)) {
        P.stages = stages;
        P.nbuf = nbuf;
        return P;
      }
    }
  P.stages = 0;
  return P;
}

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

// Where the index rows come from.  Contiguous (table == nullptr): block t of
// (b, g) holds candidates [512 t, ...), i.e. rows c0 + 512 t + [0, 512) of
// the [B][Hkv][n_cap] index, in two 256-row boxes.  Paged: blocks start at
// token 0 (block t holds tokens [512 t, 512 t + 512), so every box of
// box_rows = min(P, 256) rows lies in one page); rows below c0 are skipped,
// and boxes wholly at or above c1 are not loaded.
struct IdxSrc {
  const int32_t* table;      // [B][pages_per_seq], or nullptr
  int64_t pages_per_seq, num_pages;
  int page_shift, box_rows, box_shift;   // box_rows = 2^box_shift
  int pos_shift;             // token of block row 0 minus the candidate index of block row 0 (paged: c0)
  int c1;
};

template <int GQ>
__global__ void __launch_bounds__(kThreads, 1) group_score_kernel(const __grid_constant__ CUtensorMap tmap_idx,
                                                                 const IdxSrc src, const GroupScoreArgs a,
                                                                 const Plan P, int Hq, int Hkv, int64_t n_cap,
                                                                 int c0, int nc, int blocks, int units,
                                                                 unsigned* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* tiles = base;
  uint8_t* bq = base + P.off_bq;
  Misc& M = *reinterpret_cast<Misc*>(base + P.off_misc);
  constexpr int kN = mma_n(GQ);
  const int stages = P.stages, nbuf = P.nbuf, gbytes = P.gbytes;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  // Units per CTA: the first units mod G CTAs take one more.
  const int G = gridDim.x;
  const int uq = units / G, ur = units - (units / G) * G;
  const int u0 = static_cast<int>(blockIdx.x) * uq + min(static_cast<int>(blockIdx.x), ur);
  const int u1 = u0 + uq + (static_cast<int>(blockIdx.x) < ur ? 1 : 0);
  const int it0 = u0 * Hkv, it1 = u1 * Hkv;
  const int b_first = u0 / blocks;
  const int nseg = u1 > u0 ? (u1 - 1) / blocks - b_first + 1 : 0;   // sequences this CTA covers

  if (tid == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(&M.full[s], 1);
      mbar_init(&M.empty[s], 1);
    }
    for (int i = 0; i < nbuf; ++i) {
      mbar_init(&M.bfull[i], 1);
      mbar_init(&M.bempty[i], 1);
    }
    for (int i = 0; i < kAccStages; ++i) {
      mbar_init(&M.acc_full[i], 1);
      mbar_init(&M.acc_empty[i], kEpiWarps);
    }
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&M.tmem_base, tmem_cols(GQ));
  if (warp >= 2) {
    const int etid = tid - 64;
    // operand padding rows 3 GQ .. N-1 of every group stay zero
    constexpr int kPad = (kN - kParts * GQ) * kDIdx;
    for (int i = etid; i < nbuf * Hkv * kPad; i += kEpi) {
      const int grp = i / kPad, r = i - grp * kPad;
      *reinterpret_cast<uint16_t*>(bq + grp * gbytes + sw64_offset(kParts * GQ + r / kDIdx, r % kDIdx)) = 0;
    }
    for (int i = etid; i < 64; i += kEpi) {
      M.rmin[i] = 0xffffffffu;
      M.rmax[i] = 0u;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = M.tmem_base;
  // While the q' pass runs: warm L2 with this CTA's first ring of index
  // stages (contiguous cache; hints only).
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmap_idx);
    if (src.table == nullptr) {
      Cursor cu;
      cu.init(u0, blocks);
      for (int it = it0; it < it1 && it < it0 + stages; ++it, cu.next(Hkv, blocks)) {
        const int g = cu.g, b = cu.b, blk = cu.blk;
        const int row = static_cast<int>((static_cast<int64_t>(b) * Hkv + g) * n_cap + c0 +
                                         static_cast<int64_t>(blk) * kTileTok);
#pragma unroll
        for (int bx = 0; bx < kTileTok / kBoxRows; ++bx) tma_prefetch_2d(&tmap_idx, 0, row + bx * kBoxRows);
      }
    }
  }

  if (warp == 0) {
    // ---- TMA issue.  The index is an input of the call: the q' pass that
    // precedes this grid waited for every earlier kernel before letting it
    // launch, so these loads need no dependency wait of their own.
    const uint64_t pol = policy_evict_first();
    const bool paged = src.table != nullptr;
    int issued = 0;
    Cursor cu;
    cu.init(u0, blocks);
    for (int it = it0; it < it1; ++it, cu.next(Hkv, blocks)) {
      const int k = it - it0;
      const int g = cu.g, b = cu.b, blk = cu.blk;
      const int slot = k % stages;
      int nbox = kTileTok / kBoxRows;
      int32_t page = 0;
      if (paged) {   // boxes that hold tokens below c1, each lane < nbox looking up its box's page
        const int rem = src.c1 - blk * kTileTok;
        nbox = rem >= kTileTok ? (kTileTok >> src.box_shift) : ((rem + src.box_rows - 1) >> src.box_shift);
        if (lane < nbox) {
          const int L = blk * kTileTok + (lane << src.box_shift);
          page = __ldg(src.table + static_cast<int64_t>(b) * src.pages_per_seq + (L >> src.page_shift));
        }
      }
      bool ok = true;
      if (lane == 0) ok = mbar_wait(&M.empty[slot], ((k / stages) & 1u) ^ 1u);
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        if (lane == 0) record_error(err, kErrTimeout);
        break;
      }
      if (!paged) {
        if (lane == 0) {
          mbar_arrive_expect_tx(&M.full[slot], kTileBytes);
          const int row = static_cast<int>((static_cast<int64_t>(b) * Hkv + g) * n_cap + c0 +
                                           static_cast<int64_t>(blk) * kTileTok);
#pragma unroll
          for (int bx = 0; bx < kTileTok / kBoxRows; ++bx)
            tma_load_2d_hint(tiles + slot * kTileBytes + bx * kBoxRows * kDIdx * 2, &tmap_idx, 0, row + bx * kBoxRows,
                             &M.full[slot], pol);
        }
      } else {
        if (lane == 0) mbar_arrive_expect_tx(&M.full[slot], static_cast<uint32_t>(nbox) << (src.box_shift + 6));
        for (int bx = 0; bx < nbox; ++bx) {   // warp-uniform
          int32_t pg = __shfl_sync(0xffffffffu, page, bx);
          if (lane == 0) {
            if (pg < 0 || pg >= src.num_pages) {
              record_error(err, kErrBadPage);
              pg = 0;
            }
            const int L = blk * kTileTok + (bx << src.box_shift);
            const int row = static_cast<int>(((static_cast<int64_t>(pg) * Hkv + g) << src.page_shift) +
                                             (L & ((1 << src.page_shift) - 1)));
            tma_load_2d_hint(tiles + slot * kTileBytes + (bx << (src.box_shift + 6)), &tmap_idx, 0, row,
                             &M.full[slot], pol);
          }
        }
      }
      issued = k + 1;
      __syncwarp();
    }
    // no copy may land after the CTA has left: wait (bounded) for each
    // slot's last stage (already complete unless a wait ran out elsewhere)
    if (lane == 0)
      for (int j = issued > stages ? issued - stages : 0; j < issued; ++j)
        if (!mbar_wait(&M.full[j % stages], (j / stages) & 1u)) {
          record_error(err, kErrTimeout);
          break;
        }
  } else if (warp == 1) {
    // ---- MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = mma_idesc(128, kN);
      int cur_seg = -1;
      Cursor cu;
      cu.init(u0, blocks);
      for (int it = it0; it < it1; ++it, cu.next(Hkv, blocks)) {
        const int k = it - it0;
        const int g = cu.g;
        const int seg = cu.b - b_first;
        if (seg != cur_seg) {
          if (cur_seg >= 0) mma_commit(&M.bempty[cur_seg % nbuf]);   // free once the sequence's MMAs finish
          cur_seg = seg;
          if (!mbar_wait(&M.bfull[seg % nbuf], (seg / nbuf) & 1u)) {
            record_error(err, kErrTimeout);
            break;
          }
        }
        const int slot = k % stages;
        const int ab = k % kAccStages;
        if (!mbar_wait(&M.full[slot], (k / stages) & 1u) ||
            !mbar_wait(&M.acc_empty[ab], ((k / kAccStages) & 1u) ^ 1u)) {
          record_error(err, kErrTimeout);
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(tiles + slot * kTileBytes);
        const uint32_t b0 = smem_u32(bq + ((seg % nbuf) * Hkv + g) * gbytes);
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
#pragma unroll
          for (int sub = 0; sub < kSub; ++sub)
            mma_bf16(tmem + (ab * kSub + sub) * kN, sw64_desc(a0 + sub * 128 * kDIdx * 2 + kk * 32),
                     sw64_desc(b0 + kk * 32), idesc, kk);
        }
        mma_commit(&M.empty[slot]);
        mma_commit(&M.acc_full[ab]);
      }
    }
  } else {
    // ---- epilogue: one token per thread per stage (warp w reads TMEM lane
    // quarter w mod 4 of 128-token tile (w - 2) / 4)
    const int etid = tid - 64;
    const int quarter = warp & 3;
    const int sub = (warp - 2) >> 2;
    const int row = sub * 128 + quarter * 32 + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + sub * kN;
    bool dead = false;   // a bounded wait ran out: skip work but keep every barrier

    // B operands of segment j (sequence b_first + j), every group, into slot j mod nbuf
    auto build_b = [&](int j) {
      const int slot = j % nbuf;
      const int b = b_first + j;
      uint8_t* dst = bq + slot * Hkv * gbytes;
      for (int idx = etid; idx < Hq * kDIdx; idx += kEpi) {
        const int h = idx >> 5, c = idx & (kDIdx - 1);
        const int gg = h / GQ, hh = h - gg * GQ;
        const float x = a.qp[(static_cast<int64_t>(b) * Hq + h) * kDIdx + c];
        const uint32_t hi = bf16_rne_bits(x);
        const float r1 = x - __uint_as_float(hi << 16);
        const uint32_t mid = bf16_rne_bits(r1);
        const float r2 = r1 - __uint_as_float(mid << 16);
        const uint32_t lo = bf16_rne_bits(r2);
        uint8_t* t = dst + gg * gbytes;
        *reinterpret_cast<uint16_t*>(t + sw64_offset(hh, c)) = static_cast<uint16_t>(hi);
        *reinterpret_cast<uint16_t*>(t + sw64_offset(GQ + hh, c)) = static_cast<uint16_t>(mid);
        *reinterpret_cast<uint16_t*>(t + sw64_offset(2 * GQ + hh, c)) = static_cast<uint16_t>(lo);
      }
      fence_async_smem();
      named_bar_sync(2, kEpi);
      if (etid == 0) mbar_arrive(&M.bfull[slot]);
    };

    pdl_wait();   // q' of the q' pass
    for (int j = 0; j < (nseg < nbuf ? nseg : nbuf); ++j) build_b(j);
    named_bar_sync(1, kEpi);

    Cursor cu;
    cu.init(u0, blocks);
    for (int it = it0; it < it1; ++it, cu.next(Hkv, blocks)) {
      const int k = it - it0;
      const int ab = k % kAccStages;
      const int g = cu.g, b = cu.b, blk = cu.blk;
      const int seg = b - b_first;
      const int ci = blk * kTileTok + row - src.pos_shift;   // candidate index of this thread's token
      const bool valid = ci >= 0 && ci < nc;
      if (!dead) {
        const bool ok = mbar_wait(&M.acc_full[ab], (k / kAccStages) & 1u);
        if (!__all_sync(0xffffffffu, ok)) {
          record_error(err, kErrTimeout);
          dead = true;
        }
      }
      if (!dead) {
        tc_fence_after();
        float v[kN];
        tmem_ld_cols<kN>(tl + ab * kSub * kN, v);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&M.acc_empty[ab]);
        float sg = 0.0f;
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) sg += (v[2 * GQ + hh] + v[GQ + hh]) + v[hh];
        uint32_t kmin = 0xffffffffu, kmax = 0u;
        if (valid) {
          a.gsum[(static_cast<int64_t>(b) * Hkv + g) * a.nc_pad + ci] = sg;
          kmin = kmax = ord_key(sg);
        }
        kmin = __reduce_min_sync(0xffffffffu, kmin);
        kmax = __reduce_max_sync(0xffffffffu, kmax);
        if (lane == 0 && kmin <= kmax) {
          atomicMin(&M.rmin[g], kmin);
          atomicMax(&M.rmax[g], kmax);
        }
      }
      if (g != Hkv - 1) continue;
      // ---- the unit is complete
      const bool seg_end = it + 1 == it1 || blk == blocks - 1;
      named_bar_sync(1, kEpi);   // every group's range of the unit is complete
      for (int gg = etid; gg < Hkv; gg += kEpi) {
        a.range[(static_cast<int64_t>(b) * Hkv + gg) * blocks + blk] = make_uint2(M.rmin[gg], M.rmax[gg]);
        M.rmin[gg] = 0xffffffffu;
        M.rmax[gg] = 0u;
      }
      named_bar_sync(1, kEpi);
      // after the last unit of a sequence: the operands of segment seg + nbuf
      if (seg_end && seg + nbuf < nseg) {
        if (etid == 0 && !mbar_wait(&M.bempty[seg % nbuf], (seg / nbuf) & 1u)) record_error(err, kErrTimeout);
        named_bar_sync(2, kEpi);   // nobody writes the slot before its MMAs are done
        build_b(seg + nbuf);
      }
    }
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
int launch_gq(const qasc_shape& s, const Regions& R, const uint16_t* index, const GroupScoreArgs& a,
              const DeviceInfo& dev, cudaStream_t stream) {
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cudaErrorNotSupported;
  const Plan P = make_plan(GQ, s.Hkv, dev.max_smem_optin);
  if (P.stages == 0) return -1;
  alignas(64) CUtensorMap tmap;
  IdxSrc src = {};
  const bool paged = a.pm.table != nullptr;
  uint64_t rows = static_cast<uint64_t>(s.B) * s.Hkv * s.n_cap;
  unsigned box_rows = kBoxRows;
  if (paged) {
    src.table = a.pm.table;
    src.pages_per_seq = a.pm.pages_per_seq;
    src.num_pages = a.pm.num_pages;
    src.page_shift = a.pm.page_shift;
    box_rows = (1u << a.pm.page_shift) < kBoxRows ? (1u << a.pm.page_shift) : kBoxRows;
    src.box_rows = static_cast<int>(box_rows);
    src.box_shift = 0;
    while ((1u << src.box_shift) < box_rows) ++src.box_shift;
    src.pos_shift = static_cast<int>(R.c0);
    src.c1 = static_cast<int>(R.c1);
    rows = static_cast<uint64_t>(a.pm.num_pages) * s.Hkv << a.pm.page_shift;
  }
  if (encode_index_map(&tmap, index, rows, box_rows, enc) != 0) return cudaErrorInvalidValue;
  const int blocks = group_score_blocks(R, paged);
  const int units = blocks * s.B;
  const int grid = units < dev.num_sms ? units : dev.num_sms;
  return launch_dependent(group_score_kernel<GQ>, dim3(grid), dim3(kThreads), P.bytes, stream, 1, tmap, src, a, P,
                          s.Hq, s.Hkv, s.n_cap, static_cast<int>(R.c0), static_cast<int>(R.nc()), blocks, units,
                          dev.err_word);
}

template <int GQ>
cudaError_t configure_gq(int max_smem) {
  return cudaFuncSetAttribute(group_score_kernel<GQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
}

}  // namespace

cudaError_t configure_group_kernels(const DeviceInfo& dev) {
  cudaError_t e;
  if ((e = configure_gq<1>(dev.max_smem_optin)) != cudaSuccess) return e;
  if ((e = configure_gq<2>(dev.max_smem_optin)) != cudaSuccess) return e;
  if ((e = configure_gq<4>(dev.max_smem_optin)) != cudaSuccess) return e;
  return configure_gq<8>(dev.max_smem_optin);
}

int group_score_blocks(const Regions& R, bool paged) {
  const int64_t span = paged ? R.c1 : R.nc();
  const int blocks = static_cast<int>((span + kTileTok - 1) / kTileTok);
  return blocks > 0 ? blocks : 1;
}

int launch_group_scores(const qasc_shape& s, const qasc_ts_params& p, const uint16_t* q, const uint16_t* W,
                        const uint16_t* index, const GroupScoreArgs& a, const DeviceInfo& dev, cudaStream_t stream) {
  const Regions R = regions_of(s.n, p.sink, p.local);
  if (R.nc() <= 0) return 0;
  int rc = launch_dependent(qprime_kernel, dim3(static_cast<unsigned>(s.B) * s.Hkv), dim3(256), 0, stream, 1, q, W,
                            a.qp, s.Hq, s.Hkv);
  if (rc != 0) return rc;
  switch (s.Hq / s.Hkv) {
    case 1: return launch_gq<1>(s, R, index, a, dev, stream);
    case 2: return launch_gq<2>(s, R, index, a, dev, stream);
    case 4: return launch_gq<4>(s, R, index, a, dev, stream);
    case 8: return launch_gq<8>(s, R, index, a, dev, stream);
    default: return -1;
  }
}

}  // namespace qasc

// ts_index_append: compressed key index rows, index = RNE_bf16(K . W).
//
// TokenSelect page, section "Query-Key Dot Product Index": a d' = d/4 key
// index built incrementally during inference.  TokenButler page, section
// "Kernarchitektur": keys projected with a per-layer matrix into that space.
//
// The same kernel serves the paged pool (rows found through the block table)
// and the flush of a circular local buffer (TokenButler, "Inferenzstrategie"
// and "Optimierungen": the newest tokens in a ring, the keys projected in
// batches): it reads K and V from ring slot t mod R, copies them into their
// pages and writes the index rows there.
//
// Correct rounding.  Each product K[e]*W[e][j] of two bf16 values is exact in
// fp32 (8 x 8 significant bits), so every fp32 addition of the dot product
// commits one rounding error bounded by u*|result| (u = 2^-24).  The total
// error is therefore below u/(1-u) times the sum of |every rounded result|,
// which the fast path accumulates alongside (four interleaved FMA chains and
// their combination); 2^-23 times that sum bounds the error rigorously.  If
// both ends of [s - E, s + E] (rounded outward) round to the same bf16, so
// does the exact value, since round-to-nearest-even is monotone.  Otherwise
// (the interval touches a bf16 rounding midpoint) the row is recomputed with
// error-free fp32 transformations (TwoSum), giving hi + lo within about
// 2^-41 of the magnitude sum, and rounded exactly: RNE(hi) unless hi
// itself sits on a midpoint, where the sign of lo decides.
#include "common.cuh"
#include "internal.h"

namespace qasc {
namespace {

constexpr int kAppendWarps = 4;

__device__ __forceinline__ uint16_t bf16_bits_rn(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// RNE to bf16 of the unevaluated sum hi + lo (|lo| <= ulp(hi)/2).  Midpoints
// between bf16 values are fp32 values, so unless hi is one, hi + lo lies on
// the same side of every midpoint as hi.
__device__ __forceinline__ uint16_t bf16_bits_from_pair(float hi, float lo) {
  const uint32_t u = __float_as_uint(hi);
  if ((u & 0xffffu) == 0x8000u && lo != 0.0f) {
    const bool away = (lo > 0.0f) == (hi > 0.0f);   // |hi + lo| above the midpoint
    return static_cast<uint16_t>((u >> 16) + (away ? 1u : 0u));
  }
  return bf16_bits_rn(hi);
}

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

struct AppendArgs {
  const uint16_t* K;     // K rows read: at the destination rows, or the ring's (ring > 0)
  const uint16_t* V;     // ring flush: V rows read from the ring
  const uint16_t* W;
  uint16_t* index;       // index rows written
  uint16_t* K_out;       // ring flush: K and V rows written to the pool (nullptr: no copy)
  uint16_t* V_out;
  PageMap dst;           // rows of token t in the index (and K_out / V_out)
  int64_t ring;          // > 0: token t's K / V rows at slot t mod ring of [B][Hkv][ring]
  int Hkv;
  int64_t n_cap, start, count;
  int tokens_per_cta;
  unsigned* err;
};

// Row of the K (and V) source of token t: the destination row, or its ring slot.
__device__ __forceinline__ int64_t source_row(const AppendArgs& a, int64_t bg, int64_t t, int64_t row) {
  return a.ring > 0 ? bg * a.ring + t % a.ring : row;
}

// Correctly rounded index value from the error-free sum of the exact
// products (TwoSum): hi + lo lies within about 2^-41 of the magnitude sum, so
// RNE(hi) is exact unless hi sits on a midpoint, where the sign of lo decides.
template <class KF, class WF>
__device__ __forceinline__ uint16_t exact_index_value(KF&& kval, WF&& wval) {
  float hi = 0.0f, lo = 0.0f;
#pragma unroll 2
  for (int e = 0; e < kD; ++e) {
    const float p = __fmul_rn(kval(e), wval(e));   // exact
    float tt, err;
    two_sum(hi, p, tt, err);
    hi = tt;
    lo = __fadd_rn(lo, err);
  }
  float h2, l2;
  two_sum(hi, lo, h2, l2);
  return bf16_bits_from_pair(h2, l2);
}

// The same from a K row read in 16-byte chunks and W_g's column j in shared
// memory (the same operations in the same order).
__device__ __forceinline__ uint16_t exact_index_value_row(const uint4* __restrict__ kq4, const float (*ws)[kDIdx],
                                                          int j) {
  float hi = 0.0f, lo = 0.0f;
#pragma unroll 4
  for (int c = 0; c < kD / 8; ++c) {
    const uint4 u = __ldg(kq4 + c);
    const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int h = 0; h < 8; ++h) {
      const float kv = __uint_as_float(h & 1 ? (wd[h >> 1] & 0xffff0000u) : (wd[h >> 1] << 16));
      const float p = __fmul_rn(kv, ws[8 * c + h][j]);   // exact
      float tt, err;
      two_sum(hi, p, tt, err);
      hi = tt;
      lo = __fadd_rn(lo, err);
    }
  }
  float h2, l2;
  two_sum(hi, lo, h2, l2);
  return bf16_bits_from_pair(h2, l2);
}

// W_g widened to fp32 in shared memory ([e][j]), read with independent
// 16-byte loads.
__device__ __forceinline__ void stage_w(const uint16_t* W, int g, float (*ws)[kDIdx]) {
  const uint4* wg = reinterpret_cast<const uint4*>(W + static_cast<int64_t>(g) * kD * kDIdx);
  for (int o = threadIdx.x; o < kD * kDIdx / 8; o += blockDim.x) {
    const uint4 u = __ldg(wg + o);
    const float2 f0 = bf2_to_f2(u.x), f1 = bf2_to_f2(u.y), f2 = bf2_to_f2(u.z), f3 = bf2_to_f2(u.w);
    float* dst = &ws[0][0] + 8 * o;
    dst[0] = f0.x; dst[1] = f0.y; dst[2] = f1.x; dst[3] = f1.y;
    dst[4] = f2.x; dst[5] = f2.y; dst[6] = f3.x; dst[7] = f3.y;
  }
}

// Bulk appends: lane = token (32 per warp), each lane keeps its token's K row
// in registers and 32 column accumulators, and W_g rows are read from shared
// memory as broadcasts; one fp32 chain per column, error bound 2^-23 times the
// sum of its partial sums' magnitudes.  Columns within the bound of a bf16
// midpoint are queued (per warp, across its tokens) and recomputed exactly
// 32 at a time, one per lane, the rest at the end.
// grid: (ceil(count / tokens_per_cta), B * Hkv); block: 32 * kAppendWarps.
__global__ void __launch_bounds__(32 * kAppendWarps) index_append_bulk_kernel(const AppendArgs a) {
  __shared__ float ws[kD][kDIdx];
  __shared__ uint32_t fq[kAppendWarps][32 * kDIdx + 32];   // queued ((token - t0) << 5 | column)
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t bg = blockIdx.y;
  const int g = static_cast<int>(bg % a.Hkv);
  const int b = static_cast<int>(bg / a.Hkv);
  stage_w(a.W, g, ws);
  __syncthreads();

  const int64_t t0 = a.start + static_cast<int64_t>(blockIdx.x) * a.tokens_per_cta;
  const int64_t t1 = min(t0 + a.tokens_per_cta, a.start + a.count);
  uint32_t qn = 0;   // this warp's queued columns (fewer than 32 between rounds)
  auto recompute = [&](uint32_t e) {
    const int64_t tq = t0 + (e >> 5);
    const int j = static_cast<int>(e & 31u);
    const int64_t rq = cache_row(a.dst, b, g, a.Hkv, a.n_cap, tq);
    const uint4* kq4 = reinterpret_cast<const uint4*>(a.K + source_row(a, bg, tq, rq) * kD);
    a.index[rq * kDIdx + j] = exact_index_value_row(kq4, ws, j);
  };
  for (int64_t tb = t0 + static_cast<int64_t>(warp) * 32; tb < t1; tb += kAppendWarps * 32) {
    const int64_t t = tb + lane;
    const int64_t row = t < t1 ? cache_row(a.dst, b, g, a.Hkv, a.n_cap, t) : -2;
    if (row == -1) record_error(a.err, kErrBadPage);   // this token's page is not in the pool
    const bool ok = row >= 0;
    const uint4* ks = reinterpret_cast<const uint4*>(a.K + (ok ? source_row(a, bg, t, row) : 0) * kD);
    if (ok && a.K_out) {   // ring flush: copy the K and V rows into their page
      uint4* kd = reinterpret_cast<uint4*>(a.K_out + row * kD);
      const uint4* vs = reinterpret_cast<const uint4*>(a.V + source_row(a, bg, t, row) * kD);
      uint4* vd = reinterpret_cast<uint4*>(a.V_out + row * kD);
      for (int c = 0; c < kD / 8; ++c) {
        kd[c] = __ldg(ks + c);
        vd[c] = __ldg(vs + c);
      }
    }
    // column accumulators and their magnitude sums in pairs (one packed FMA or
    // add per pair: each half is an ordinary round-to-nearest operation, in
    // the same order as one chain per column)
    float2 sacc2[kDIdx / 2], mag2[kDIdx / 2];
#pragma unroll
    for (int j = 0; j < kDIdx / 2; ++j) sacc2[j] = mag2[j] = make_float2(0.0f, 0.0f);
    // the K row streams through three registers, loaded two chunks ahead
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    uint4 k0 = ok ? __ldg(ks + 0) : zero;
    uint4 k1 = ok ? __ldg(ks + 1) : zero;
#pragma unroll 1
    for (int c = 0; c < kD / 8; ++c) {
      const uint4 k2 = ok && c + 2 < kD / 8 ? __ldg(ks + c + 2) : zero;
      const uint32_t wd[4] = {k0.x, k0.y, k0.z, k0.w};
#pragma unroll
      for (int h = 0; h < 8; ++h) {
        const float k = __uint_as_float(h & 1 ? (wd[h >> 1] & 0xffff0000u) : (wd[h >> 1] << 16));
        const float2 kk = make_float2(k, k);
        const float4* wrow = reinterpret_cast<const float4*>(ws[8 * c + h]);
#pragma unroll
        for (int q4 = 0; q4 < kDIdx / 4; ++q4) {
          const float4 w4 = wrow[q4];
          sacc2[2 * q4 + 0] = __ffma2_rn(kk, make_float2(w4.x, w4.y), sacc2[2 * q4 + 0]);
          sacc2[2 * q4 + 1] = __ffma2_rn(kk, make_float2(w4.z, w4.w), sacc2[2 * q4 + 1]);
          mag2[2 * q4 + 0] = __fadd2_rn(mag2[2 * q4 + 0], make_float2(fabsf(sacc2[2 * q4 + 0].x), fabsf(sacc2[2 * q4 + 0].y)));
          mag2[2 * q4 + 1] = __fadd2_rn(mag2[2 * q4 + 1], make_float2(fabsf(sacc2[2 * q4 + 1].x), fabsf(sacc2[2 * q4 + 1].y)));
        }
      }
      k0 = k1;
      k1 = k2;
    }
    uint32_t amb = 0, packed[kDIdx / 2];
#pragma unroll
    for (int j = 0; j < kDIdx; ++j) {
      const float sj = j & 1 ? sacc2[j >> 1].y : sacc2[j >> 1].x;
      const float bound = (j & 1 ? mag2[j >> 1].y : mag2[j >> 1].x) * 0x1p-23f;
      const uint32_t lo = bf16_bits_rn(__fsub_rd(sj, bound));
      const uint32_t hi = bf16_bits_rn(__fadd_ru(sj, bound));
      if (lo != hi) amb |= 1u << j;
      if (j & 1) packed[j >> 1] |= lo << 16;
      else packed[j >> 1] = lo;
    }
    if (!ok) amb = 0;
    if (ok) {
      uint4* dst = reinterpret_cast<uint4*>(a.index + row * kDIdx);
#pragma unroll
      for (int c = 0; c < kDIdx / 8; ++c)
        dst[c] = make_uint4(packed[4 * c], packed[4 * c + 1], packed[4 * c + 2], packed[4 * c + 3]);
    }
    // queue the ambiguous columns; every full round of 32 is recomputed, one per lane
    const uint32_t cnt = __popc(amb);
    uint32_t inc = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += v;
    }
    const uint32_t total = __shfl_sync(0xffffffffu, inc, 31);
    uint32_t pos = qn + inc - cnt;
    for (uint32_t m = amb; m; m &= m - 1)
      fq[warp][pos++] = (static_cast<uint32_t>(t - t0) << 5) | static_cast<uint32_t>(__ffs(m) - 1);
    qn += total;
    __syncwarp();
    while (qn >= 32) {
      recompute(fq[warp][qn - 32 + lane]);
      qn -= 32;
      __syncwarp();   // those slots take the next appends
    }
  }
  if (lane < qn) recompute(fq[warp][lane]);
}

// grid: (ceil(count / tokens_per_cta), B * Hkv); block: 32 * kAppendWarps.
// Lane j of each warp produces column j of one token's index row.
__global__ void __launch_bounds__(32 * kAppendWarps) index_append_kernel(const AppendArgs a) {
  __shared__ float4 krow[kAppendWarps][kD / 4];
  __shared__ float ws[kD][kDIdx];  // W_g widened to fp32; lane j reads column j
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t bg = blockIdx.y;
  const int g = static_cast<int>(bg % a.Hkv);
  const int b = static_cast<int>(bg / a.Hkv);

  stage_w(a.W, g, ws);
  __syncthreads();
#define w(e) ws[(e)][lane]

  const int64_t t0 = a.start + static_cast<int64_t>(blockIdx.x) * a.tokens_per_cta;
  const int64_t t1 = min(t0 + a.tokens_per_cta, a.start + a.count);
  for (int64_t t = t0 + warp; t < t1; t += kAppendWarps) {
    const int64_t row = cache_row(a.dst, b, g, a.Hkv, a.n_cap, t);
    if (row < 0) {   // the whole warp: this token's page is not in the pool
      if (lane == 0) record_error(a.err, kErrBadPage);
      continue;
    }
    const int64_t src = source_row(a, bg, t, row);
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(a.K + src * kD) + lane);
    if (a.K_out) {
      reinterpret_cast<uint2*>(a.K_out + row * kD)[lane] = raw;
      reinterpret_cast<uint2*>(a.V_out + row * kD)[lane] = __ldg(reinterpret_cast<const uint2*>(a.V + src * kD) + lane);
    }
    const float2 lo2 = bf2_to_f2(raw.x);
    const float2 hi2 = bf2_to_f2(raw.y);
    krow[warp][lane] = make_float4(lo2.x, lo2.y, hi2.x, hi2.y);
    __syncwarp();

    float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
    float a0 = 0.0f, a1 = 0.0f, a2 = 0.0f, a3 = 0.0f;
#pragma unroll 4
    for (int e4 = 0; e4 < kD / 4; ++e4) {
      const float4 k4 = krow[warp][e4];
      s0 = fmaf(k4.x, w(4 * e4 + 0), s0);
      s1 = fmaf(k4.y, w(4 * e4 + 1), s1);
      s2 = fmaf(k4.z, w(4 * e4 + 2), s2);
      s3 = fmaf(k4.w, w(4 * e4 + 3), s3);
      a0 += fabsf(s0);
      a1 += fabsf(s1);
      a2 += fabsf(s2);
      a3 += fabsf(s3);
    }
    const float t01 = __fadd_rn(s0, s1), t23 = __fadd_rn(s2, s3);
    const float s = __fadd_rn(t01, t23);
    const float bound = ((a0 + a1) + (a2 + a3) + fabsf(t01) + fabsf(t23) + fabsf(s)) * 0x1p-23f;
    const uint16_t r_lo = bf16_bits_rn(__fsub_rd(s, bound));
    const uint16_t r_hi = bf16_bits_rn(__fadd_ru(s, bound));
    uint16_t out = r_lo;
    if (r_lo != r_hi) {   // the same error-free sum as exact_index_value, K from the staged row
      float hi = 0.0f, lo = 0.0f;
#pragma unroll 2
      for (int e4 = 0; e4 < kD / 4; ++e4) {
        const float4 k4 = krow[warp][e4];
        const float kk[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float p = __fmul_rn(kk[j], w(4 * e4 + j));   // exact
          float tt, err;
          two_sum(hi, p, tt, err);
          hi = tt;
          lo = __fadd_rn(lo, err);
        }
      }
      float h2, l2;
      two_sum(hi, lo, h2, l2);
      out = bf16_bits_from_pair(h2, l2);
    }
    a.index[row * kDIdx + lane] = out;
    __syncwarp();
  }
#undef w
}

cudaError_t launch_append(const qasc_shape& s, AppendArgs a, cudaStream_t stream) {
  if (a.count <= 0) return cudaSuccess;
  // Small appends (decode) use one CTA per (b, g); bulk appends spread over
  // enough CTAs to cover the GPU a few times.
  const bool bulk = a.count > 64;
  a.tokens_per_cta = bulk ? 32 * kAppendWarps * 4 : static_cast<int>(a.count);
  const int64_t blocks = (a.count + a.tokens_per_cta - 1) / a.tokens_per_cta;
  a.Hkv = s.Hkv;
  dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(s.B * s.Hkv));
  if (bulk)
    index_append_bulk_kernel<<<grid, 32 * kAppendWarps, 0, stream>>>(a);
  else
    index_append_kernel<<<grid, 32 * kAppendWarps, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_index_append(const qasc_shape& s, const uint16_t* K, const uint16_t* W, uint16_t* index,
                                int64_t start, int64_t count, cudaStream_t stream) {
  AppendArgs a = {};
  a.K = K;
  a.W = W;
  a.index = index;
  a.n_cap = s.n_cap;
  a.start = start;
  a.count = count;
  return launch_append(s, a, stream);
}

cudaError_t launch_index_append_paged(const qasc_shape& s, const PageMap& pm, const uint16_t* K, const uint16_t* W,
                                      uint16_t* index, int64_t start, int64_t count, unsigned* err,
                                      cudaStream_t stream) {
  AppendArgs a = {};
  a.K = K;
  a.W = W;
  a.index = index;
  a.dst = pm;
  a.n_cap = s.n_cap;
  a.start = start;
  a.count = count;
  a.err = err;
  return launch_append(s, a, stream);
}

cudaError_t launch_ring_flush(const qasc_shape& s, const PageMap& pm, const RingMap& ring, const uint16_t* W,
                              uint16_t* K_pool, uint16_t* V_pool, uint16_t* index, int64_t start, int64_t count,
                              unsigned* err, cudaStream_t stream) {
  AppendArgs a = {};
  a.K = ring.K;
  a.V = ring.V;
  a.W = W;
  a.index = index;
  a.K_out = K_pool;
  a.V_out = V_pool;
  a.dst = pm;
  a.ring = ring.R;
  a.n_cap = s.n_cap;
  a.start = start;
  a.count = count;
  a.err = err;
  return launch_append(s, a, stream);
}

}  // namespace qasc

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

  // W_g widened to fp32, read with independent 16-byte loads (4 per thread)
  const uint4* wg = reinterpret_cast<const uint4*>(a.W + static_cast<int64_t>(g) * kD * kDIdx);
  for (int o = threadIdx.x; o < kD * kDIdx / 8; o += blockDim.x) {
    const uint4 u = __ldg(wg + o);
    const float2 f0 = bf2_to_f2(u.x), f1 = bf2_to_f2(u.y), f2 = bf2_to_f2(u.z), f3 = bf2_to_f2(u.w);
    float* dst = &ws[0][0] + 8 * o;
    dst[0] = f0.x; dst[1] = f0.y; dst[2] = f1.x; dst[3] = f1.y;
    dst[4] = f2.x; dst[5] = f2.y; dst[6] = f3.x; dst[7] = f3.y;
  }
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
    const int64_t src = a.ring > 0 ? bg * a.ring + t % a.ring : row;
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
    if (r_lo != r_hi) {
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
  a.tokens_per_cta = a.count <= 64 ? static_cast<int>(a.count) : 256;
  const int64_t blocks = (a.count + a.tokens_per_cta - 1) / a.tokens_per_cta;
  a.Hkv = s.Hkv;
  dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(s.B * s.Hkv));
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

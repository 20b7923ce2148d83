// ts_index_append: compressed key index rows, index = RNE_bf16(K . W).
//
// TokenSelect page, section "Query-Key Dot Product Index": a d' = d/4 key
// index built incrementally during inference.  TokenButler page, section
// "Kernarchitektur": keys projected with a per-layer matrix into that space.
//
// Correct rounding.  Each product K[e]*W[e][j] of two bf16 values is exact in
// fp32 (8 x 8 significant bits), so the fp32 FMA chain s_i = fl(s_{i-1} + p_i)
// commits one rounding error per step, bounded by u*|s_i| (u = 2^-24).  The
// total error is therefore at most u/(1-u) * sum_i |s_i| < 2^-23 * A, where A
// is that sum computed in fp32.  If both ends of [s - E, s + E] (rounded
// outward) round to the same bf16, then so does the exact value, because
// round-to-nearest-even is monotone.  Otherwise (rarely: the interval touches
// a bf16 rounding midpoint) the row is recomputed in fp64 and rounded with a
// truncate-plus-sticky rule.
#include "common.cuh"
#include "internal.h"

namespace qasc {
namespace {

constexpr int kAppendWarps = 4;

__device__ __forceinline__ uint16_t bf16_bits_rn(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

// Round-to-nearest-even of an fp64 value to bf16: truncate to fp32, then
// round bits [15:0] with the discarded fp64 tail folded into the sticky bit.
__device__ __forceinline__ uint16_t bf16_bits_from_double(double x) {
  const float f = __double2float_rz(x);
  uint32_t u = __float_as_uint(f);
  const bool sticky = static_cast<double>(f) != x;
  const uint32_t lsb = (u >> 16) & 1u;
  const uint32_t round_bit = (u >> 15) & 1u;
  const bool rest = ((u & 0x7fffu) != 0u) || sticky;
  if (round_bit && (rest || lsb)) u += 0x10000u;
  return static_cast<uint16_t>(u >> 16);
}

// grid: (ceil(count / tokens_per_cta), B * Hkv); block: 32 * kAppendWarps.
// Lane j of each warp produces column j of one token's index row.
__global__ void __launch_bounds__(32 * kAppendWarps) index_append_kernel(
    const uint16_t* __restrict__ K, const uint16_t* __restrict__ W, uint16_t* __restrict__ index, int Hkv,
    int64_t n_cap, int64_t start, int64_t count, int tokens_per_cta) {
  __shared__ float4 krow[kAppendWarps][kD / 4];
  __shared__ float ws[kD][kDIdx];  // W_g widened to fp32; lane j reads column j
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t bg = blockIdx.y;
  const int g = static_cast<int>(bg % Hkv);

  const uint16_t* wg = W + static_cast<int64_t>(g) * kD * kDIdx;
  for (int o = threadIdx.x; o < kD * kDIdx; o += blockDim.x) ws[o / kDIdx][o % kDIdx] = bf_to_f(__ldg(wg + o));
  __syncthreads();
#define w(e) ws[(e)][lane]

  const int64_t t0 = start + static_cast<int64_t>(blockIdx.x) * tokens_per_cta;
  const int64_t t1 = min(t0 + tokens_per_cta, start + count);
  for (int64_t t = t0 + warp; t < t1; t += kAppendWarps) {
    const int64_t row = bg * n_cap + t;
    const uint2 raw = __ldg(reinterpret_cast<const uint2*>(K + row * kD) + lane);
    const float2 a = bf2_to_f2(raw.x);
    const float2 b = bf2_to_f2(raw.y);
    krow[warp][lane] = make_float4(a.x, a.y, b.x, b.y);
    __syncwarp();

    float s = 0.0f, acc = 0.0f;
#pragma unroll 4
    for (int e4 = 0; e4 < kD / 4; ++e4) {
      const float4 k4 = krow[warp][e4];
      s = fmaf(k4.x, w(4 * e4 + 0), s);
      acc += fabsf(s);
      s = fmaf(k4.y, w(4 * e4 + 1), s);
      acc += fabsf(s);
      s = fmaf(k4.z, w(4 * e4 + 2), s);
      acc += fabsf(s);
      s = fmaf(k4.w, w(4 * e4 + 3), s);
      acc += fabsf(s);
    }
    const float bound = acc * 0x1p-23f;
    const uint16_t r_lo = bf16_bits_rn(__fsub_rd(s, bound));
    const uint16_t r_hi = bf16_bits_rn(__fadd_ru(s, bound));
    uint16_t out = r_lo;
    if (r_lo != r_hi) {
      double sd = 0.0;
#pragma unroll 2
      for (int e4 = 0; e4 < kD / 4; ++e4) {
        const float4 k4 = krow[warp][e4];
        sd = fma(static_cast<double>(k4.x), static_cast<double>(w(4 * e4 + 0)), sd);
        sd = fma(static_cast<double>(k4.y), static_cast<double>(w(4 * e4 + 1)), sd);
        sd = fma(static_cast<double>(k4.z), static_cast<double>(w(4 * e4 + 2)), sd);
        sd = fma(static_cast<double>(k4.w), static_cast<double>(w(4 * e4 + 3)), sd);
      }
      out = bf16_bits_from_double(sd);
    }
    index[row * kDIdx + lane] = out;
    __syncwarp();
  }
#undef w
}

}  // namespace

cudaError_t launch_index_append(const qasc_shape& s, const uint16_t* K, const uint16_t* W, uint16_t* index,
                                int64_t start, int64_t count, cudaStream_t stream) {
  if (count <= 0) return cudaSuccess;
  // Small appends (decode) use one CTA per (b, g); bulk appends spread over
  // enough CTAs to cover the GPU a few times.
  int tokens_per_cta = count <= 64 ? static_cast<int>(count) : 256;
  const int64_t blocks = (count + tokens_per_cta - 1) / tokens_per_cta;
  dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(s.B * s.Hkv));
  index_append_kernel<<<grid, 32 * kAppendWarps, 0, stream>>>(K, W, index, s.Hkv, s.n_cap, start, count,
                                                              tokens_per_cta);
  return cudaGetLastError();
}

}  // namespace qasc

// Split-K flash-decode over the attended set T = sink + S + local.
//
// TokenSelect page, section "Token-Level Selection と Sparse Attention",
// equation Attention = softmax(Q K_S^T / sqrt(d)) V_S, with the sink and local
// tokens of the always-included table; section "統合の5ステップ" step 5 merges
// the sparse and local outputs.  Here T is one list, split into contiguous
// pieces per (b, g); each piece yields (max, sum, unnormalised output) in fp32
// and merge_kernel combines them exactly (log-sum-exp), which equals a single
// softmax over T.
//
// Data movement: T's K and V rows (256 bytes each) are gathered by one
// producer warp with one bulk copy per row into a 3-stage ring of 64-token
// stages (32 KB each), completing on an mbarrier; the rows are streamed with
// an evict-first L2 policy.  Compute: four consumer warps form eight
// half-warp groups; a group takes 8 rows of a stage, each lane owning 8 of the
// 128 head dimensions.  Partial q.k products are finished by a butterfly
// reduce-scatter over the 16 lanes (each lane ends up owning whole logits of
// one head), the online softmax runs on those, and probabilities reach the
// P.V update through shared memory.
#include "common.cuh"
#include "internal.h"

namespace qasc {
namespace {

constexpr int kStageTok = 64;
constexpr int kRowBytes = kD * 2;
constexpr int kStages = 3;
constexpr int kConsWarps = 4;
constexpr int kCons = 32 * kConsWarps;
constexpr int kThreads = kCons + 32;
constexpr int kGroups = 2 * kConsWarps;   // half-warp groups
constexpr int kTB = 8;                    // rows per group per stage
constexpr int kPartStride = 132;          // floats per (b, h, split) partial: m, l, pad, pad, o[128]
// log2(e) / sqrt(128): logits are kept in base-2 units.
constexpr float kQScale = 1.4426950408889634f * 0.08838834764831845f;

__device__ __forceinline__ int64_t token_at(int64_t j, int64_t sink_end, int64_t K, int64_t local_start,
                                            const int32_t* sel_b) {
  if (j < sink_end) return j;
  if (j < sink_end + K) return sel_b[j - sink_end];
  return local_start + (j - sink_end - K);
}

template <int GQ>
struct AttnSmem {
  uint8_t k[kStages][kStageTok * kRowBytes];
  uint8_t v[kStages][kStageTok * kRowBytes];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  float q[GQ][kD];
  float p[kGroups][kTB][GQ < 4 ? 4 : GQ];
  float alpha[kGroups][GQ < 4 ? 4 : GQ];
};

template <int GQ>
__global__ void __launch_bounds__(kThreads) sparse_attn_kernel(
    const uint16_t* __restrict__ q, const uint16_t* __restrict__ Kc, const uint16_t* __restrict__ Vc,
    const int32_t* __restrict__ sel, float* __restrict__ part, int Hq, int Hkv, int64_t n_cap, int64_t sink_end,
    int64_t K, int64_t local_start, int64_t t_len, int64_t per_split, int splits, unsigned* err) {
  constexpr int L0 = kTB * GQ;                  // partial logits per lane before the reduce-scatter
  constexpr int R = L0 >= 16 ? L0 / 16 : 1;     // logits owned per lane afterwards
  constexpr int LPH = L0 >= 16 ? 8 / R : 16;    // lanes per head afterwards
  constexpr int PW = GQ < 4 ? 4 : GQ;           // padded head stride in p / alpha
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  AttnSmem<GQ>& S = *reinterpret_cast<AttnSmem<GQ>*>(smem_raw);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int split = blockIdx.x;
  const int bg = blockIdx.y;
  const int b = bg / Hkv, g = bg - b * Hkv;
  const int64_t j_begin = static_cast<int64_t>(split) * per_split;
  const int64_t j_end = min(t_len, j_begin + per_split);
  const int nstage = j_end > j_begin ? static_cast<int>((j_end - j_begin + kStageTok - 1) / kStageTok) : 0;
  const int32_t* sel_b = sel + static_cast<int64_t>(b) * K;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kConsWarps);
    }
    fence_barrier_init();
  }
  for (int o = tid; o < GQ * kD; o += kThreads) {
    const int hh = o / kD, e = o - hh * kD;
    S.q[hh][e] = bf_to_f(q[(static_cast<int64_t>(b) * Hq + g * GQ + hh) * kD + e]) * kQScale;
  }
  __syncthreads();

  if (warp == kConsWarps) {
    // ---- producer warp: gather rows of T
    const uint64_t pol = policy_evict_first();
    const uint16_t* kb = Kc + static_cast<int64_t>(bg) * n_cap * kD;
    const uint16_t* vb = Vc + static_cast<int64_t>(bg) * n_cap * kD;
    for (int st = 0; st < nstage; ++st) {
      const int slot = st % kStages;
      const uint32_t ph = (st / kStages) & 1u;
      const bool ok = mbar_wait(&S.empty[slot], ph ^ 1u);
      if (!__all_sync(0xffffffffu, ok)) {
        record_error(err, kErrTimeout);
        break;
      }
      const int64_t j0 = j_begin + static_cast<int64_t>(st) * kStageTok;
      const int rows = static_cast<int>(min(static_cast<int64_t>(kStageTok), j_end - j0));
      if (lane == 0) mbar_arrive_expect_tx(&S.full[slot], static_cast<uint32_t>(rows) * 2u * kRowBytes);
      __syncwarp();
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int r = lane + 32 * rr;
        if (r < rows) {
          // Ids outside the cache are clamped so a bad selection cannot fault.
          int64_t tok = token_at(j0 + r, sink_end, K, local_start, sel_b);
          tok = tok < 0 ? 0 : (tok >= n_cap ? n_cap - 1 : tok);
          bulk_g2s_hint(&S.k[slot][r * kRowBytes], kb + tok * kD, kRowBytes, &S.full[slot], pol);
          bulk_g2s_hint(&S.v[slot][r * kRowBytes], vb + tok * kD, kRowBytes, &S.full[slot], pol);
        }
      }
    }
    return;
  }

  // ---- consumers
  const int half = lane >> 4, l16 = lane & 15;
  const int gi = warp * 2 + half;
  const unsigned hmask = 0xffffu << (16 * half);
  const int my_head = (l16 * R) / kTB < GQ ? (l16 * R) / kTB : GQ - 1;

  float2 qr[GQ][4];
#pragma unroll
  for (int hh = 0; hh < GQ; ++hh)
#pragma unroll
    for (int j = 0; j < 4; ++j) qr[hh][j] = make_float2(S.q[hh][8 * l16 + 2 * j], S.q[hh][8 * l16 + 2 * j + 1]);

  float2 o[GQ][4];
#pragma unroll
  for (int hh = 0; hh < GQ; ++hh)
#pragma unroll
    for (int j = 0; j < 4; ++j) o[hh][j] = make_float2(0.0f, 0.0f);
  float m_run = -INFINITY;   // running max (base 2) of my_head in this group
  float l_run = 0.0f;        // this lane's share of the running sum

  for (int st = 0; st < nstage; ++st) {
    const int slot = st % kStages;
    const uint32_t ph = (st / kStages) & 1u;
    const bool ok = mbar_wait(&S.full[slot], ph);
    if (!__all_sync(0xffffffffu, ok)) {
      record_error(err, kErrTimeout);
      return;
    }
    const int64_t j0 = j_begin + static_cast<int64_t>(st) * kStageTok;
    const int rows = static_cast<int>(min(static_cast<int64_t>(kStageTok), j_end - j0));
    const int nt = max(0, min(kTB, rows - gi * kTB));
    if (nt > 0) {
      const uint8_t* kst = S.k[slot] + (gi * kTB) * kRowBytes + l16 * 16;
      const uint8_t* vst = S.v[slot] + (gi * kTB) * kRowBytes + l16 * 16;
      // q . k partials: v[h * 8 + t]
      float pv[L0];
#pragma unroll
      for (int t = 0; t < kTB; ++t) {
        uint4 kr = make_uint4(0, 0, 0, 0);
        if (t < nt) kr = *reinterpret_cast<const uint4*>(kst + t * kRowBytes);
        const float2 k0 = bf2_to_f2(kr.x), k1 = bf2_to_f2(kr.y), k2 = bf2_to_f2(kr.z), k3 = bf2_to_f2(kr.w);
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
          float2 a = make_float2(0.0f, 0.0f);
          a = ffma2(qr[hh][0], k0, a);
          a = ffma2(qr[hh][1], k1, a);
          a = ffma2(qr[hh][2], k2, a);
          a = ffma2(qr[hh][3], k3, a);
          pv[hh * kTB + t] = a.x + a.y;
        }
      }
      // Butterfly reduce-scatter over the 16 lanes of the group.
      int len = L0;
#pragma unroll
      for (int off = 8; off >= 1; off >>= 1) {
        if (len >= 2) {
          const int hlen = len / 2;
          const bool upper = (l16 & off) != 0;
#pragma unroll
          for (int i = 0; i < L0 / 2; ++i) {
            if (i < hlen) {
              const float keep = upper ? pv[hlen + i] : pv[i];
              const float give = upper ? pv[i] : pv[hlen + i];
              pv[i] = keep + __shfl_xor_sync(hmask, give, off);
            }
          }
          len = hlen;
        } else {
          pv[0] += __shfl_xor_sync(hmask, pv[0], off);
        }
      }
      // This lane now owns logits idx = l16 * R + i (or l16 / 2 when L0 == 8).
      float z[R];
      float bm = -INFINITY;
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const int idx = L0 >= 16 ? l16 * R + i : (l16 >> 1);
        const int t = idx % kTB;
        z[i] = t < nt ? pv[i] : -INFINITY;
        bm = fmaxf(bm, z[i]);
      }
#pragma unroll
      for (int off = 1; off < LPH; off <<= 1) bm = fmaxf(bm, __shfl_xor_sync(hmask, bm, off));
      const float m_new = fmaxf(m_run, bm);
      const float alpha = m_new == -INFINITY ? 1.0f : exp2f(m_run - m_new);
      float psum = 0.0f;
#pragma unroll
      for (int i = 0; i < R; ++i) {
        const int idx = L0 >= 16 ? l16 * R + i : (l16 >> 1);
        const int t = idx % kTB;
        const float pr = m_new == -INFINITY ? 0.0f : exp2f(z[i] - m_new);
        psum += pr;
        if (L0 >= 16 || (l16 & 1) == 0) S.p[gi][t][my_head] = pr;
      }
      if (L0 < 16 && (l16 & 1)) psum = 0.0f;   // the pair partner holds the same logit
      l_run = l_run * alpha + psum;
      m_run = m_new;
      if ((l16 % LPH) == 0) S.alpha[gi][my_head] = alpha;
      __syncwarp(hmask);
      // Rescale and accumulate P.V.
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) {
        const float a = S.alpha[gi][hh];
        const float2 a2 = make_float2(a, a);
#pragma unroll
        for (int j = 0; j < 4; ++j) o[hh][j] = __fmul2_rn(o[hh][j], a2);
      }
#pragma unroll
      for (int t = 0; t < kTB; ++t) {
        if (t < nt) {
          const uint4 vr = *reinterpret_cast<const uint4*>(vst + t * kRowBytes);
          const float2 v0 = bf2_to_f2(vr.x), v1 = bf2_to_f2(vr.y), v2 = bf2_to_f2(vr.z), v3 = bf2_to_f2(vr.w);
#pragma unroll
          for (int hh = 0; hh < GQ; ++hh) {
            const float pr = S.p[gi][t][hh];
            const float2 p2 = make_float2(pr, pr);
            o[hh][0] = ffma2(p2, v0, o[hh][0]);
            o[hh][1] = ffma2(p2, v1, o[hh][1]);
            o[hh][2] = ffma2(p2, v2, o[hh][2]);
            o[hh][3] = ffma2(p2, v3, o[hh][3]);
          }
        }
      }
      __syncwarp(hmask);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[slot]);
  }

  // ---- combine the eight groups of this CTA (reusing stage memory)
  named_bar_sync(1, kCons);
  float* red_o = reinterpret_cast<float*>(&S.k[0][0]);          // [group][GQ][128]
  float* red_m = reinterpret_cast<float*>(&S.v[0][0]);          // [group][GQ]
  float* red_l = red_m + kGroups * GQ;                          // [group][GQ]
  float lsum = l_run;
#pragma unroll
  for (int off = 1; off < 16; off <<= 1) {
    const float other = __shfl_xor_sync(hmask, lsum, off);
    if (off < LPH) lsum += other;
  }
  if ((l16 % LPH) == 0) {
    red_m[gi * GQ + my_head] = m_run;
    red_l[gi * GQ + my_head] = lsum;
  }
#pragma unroll
  for (int hh = 0; hh < GQ; ++hh) {
    float4* dst = reinterpret_cast<float4*>(red_o + (gi * GQ + hh) * kD + 8 * l16);
    dst[0] = make_float4(o[hh][0].x, o[hh][0].y, o[hh][1].x, o[hh][1].y);
    dst[1] = make_float4(o[hh][2].x, o[hh][2].y, o[hh][3].x, o[hh][3].y);
  }
  named_bar_sync(1, kCons);
  for (int out_i = tid; out_i < GQ * kD; out_i += kCons) {
    const int hh = out_i / kD, e = out_i - hh * kD;
    float M = -INFINITY;
#pragma unroll
    for (int gg = 0; gg < kGroups; ++gg) M = fmaxf(M, red_m[gg * GQ + hh]);
    float Lsum = 0.0f, O = 0.0f;
#pragma unroll
    for (int gg = 0; gg < kGroups; ++gg) {
      const float mg = red_m[gg * GQ + hh];
      const float w = mg == -INFINITY ? 0.0f : exp2f(mg - M);
      Lsum = fmaf(w, red_l[gg * GQ + hh], Lsum);
      O = fmaf(w, red_o[(gg * GQ + hh) * kD + e], O);
    }
    float* dst = part + ((static_cast<int64_t>(b) * Hq + g * GQ + hh) * splits + split) * kPartStride;
    dst[4 + e] = O;
    if (e == 0) {
      dst[0] = M;
      dst[1] = Lsum;
    }
  }
}

// grid B * Hq, block 128: exact log-sum-exp merge of the splits.
__global__ void __launch_bounds__(kD) merge_kernel(const float* __restrict__ part, float* __restrict__ out,
                                                  float* __restrict__ lse, int splits) {
  const int64_t bh = blockIdx.x;
  const float* p = part + bh * splits * kPartStride;
  const int e = threadIdx.x;
  float M = -INFINITY;
  for (int s = 0; s < splits; ++s) M = fmaxf(M, p[s * kPartStride]);
  float L = 0.0f, O = 0.0f;
  for (int s = 0; s < splits; ++s) {
    const float ms = p[s * kPartStride];
    const float w = ms == -INFINITY ? 0.0f : exp2f(ms - M);
    L = fmaf(w, p[s * kPartStride + 1], L);
    O = fmaf(w, p[s * kPartStride + 4 + e], O);
  }
  out[bh * kD + e] = O / L;
  if (lse && e == 0) lse[bh] = (M + log2f(L)) * 0.6931471805599453f;
}

template <int GQ>
int launch_gq(const qasc_shape& s, const qasc_ts_params& p, const AttnLayout& L, const uint16_t* q,
              const uint16_t* K, const uint16_t* V, const int32_t* sel, float* part, const DeviceInfo& dev,
              cudaStream_t stream) {
  const Regions R = regions_of(s.n, p.sink, p.local);
  const size_t smem = sizeof(AttnSmem<GQ>);
  cudaError_t e = cudaFuncSetAttribute(sparse_attn_kernel<GQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(static_cast<unsigned>(L.splits), static_cast<unsigned>(s.B * s.Hkv));
  sparse_attn_kernel<GQ><<<grid, kThreads, smem, stream>>>(q, K, V, sel, part, s.Hq, s.Hkv, s.n_cap, R.sink_end,
                                                          p.K, R.local_start, L.t_len, L.per_split, L.splits,
                                                          dev.err_word);
  return cudaGetLastError();
}

}  // namespace

AttnLayout attn_layout(const qasc_shape& s, const qasc_ts_params& p, int num_sms) {
  AttnLayout L;
  const Regions R = regions_of(s.n, p.sink, p.local);
  L.t_len = R.sink_end + p.K + (s.n - R.local_start);
  const int64_t bg = static_cast<int64_t>(s.B) * s.Hkv;
  // About two CTAs per SM in total, at least one 64-token stage per split.
  const int64_t want = (2 * static_cast<int64_t>(num_sms > 0 ? num_sms : 148) + bg - 1) / bg;
  const int64_t max_splits = (L.t_len + kStageTok - 1) / kStageTok;
  int64_t splits = want < max_splits ? want : max_splits;
  if (splits < 1) splits = 1;
  L.per_split = (L.t_len + splits - 1) / splits;
  L.splits = static_cast<int>((L.t_len + L.per_split - 1) / L.per_split);
  L.off_part = 0;
  L.total = align_up(static_cast<size_t>(s.B) * s.Hq * L.splits * kPartStride * sizeof(float), 256);
  return L;
}

int launch_sparse_attn(const qasc_shape& s, const qasc_ts_params& p, const AttnLayout& L, const uint16_t* q,
                       const uint16_t* K, const uint16_t* V, const int32_t* sel, float* out, float* lse,
                       uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream) {
  float* part = reinterpret_cast<float*>(ws + L.off_part);
  int rc;
  switch (s.Hq / s.Hkv) {
    case 1: rc = launch_gq<1>(s, p, L, q, K, V, sel, part, dev, stream); break;
    case 2: rc = launch_gq<2>(s, p, L, q, K, V, sel, part, dev, stream); break;
    case 4: rc = launch_gq<4>(s, p, L, q, K, V, sel, part, dev, stream); break;
    case 8: rc = launch_gq<8>(s, p, L, q, K, V, sel, part, dev, stream); break;
    default: return -1;
  }
  if (rc != 0) return rc;
  merge_kernel<<<s.B * s.Hq, kD, 0, stream>>>(part, out, lse, L.splits);
  return cudaGetLastError();
}

}  // namespace qasc

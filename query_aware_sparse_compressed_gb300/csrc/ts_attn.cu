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
// persistent grid (three CTAs per SM) takes equal contiguous ranges of that
// line, so every CTA moves the same number of rows; a range may cross from
// one (b, g) into the next.
//
// Data movement: one producer warp gathers the K and V rows (256 bytes each)
// of 64-position stages with TMA tile::gather4 copies (one instruction moves
// four indexed rows of the [B*Hkv*n_cap, 128] tensor; lanes 0-15 issue the K
// row quads and lanes 16-31 the V quads of a stage) into a 2-stage
// shared-memory ring per CTA, completing on an mbarrier.  Token ids of a
// stage are staged in shared memory first.
//
// Compute: four consumer warps form eight half-warp groups; a group takes 8
// rows of a stage, each lane owning 8 of the 128 head dimensions.  Partial
// q.k products are finished by a butterfly reduce-scatter over the 16 lanes
// (each lane ends up owning whole logits of one head), the online softmax
// runs on those, and probabilities reach the P.V update through shared memory.
// Each group writes its own partial for every (b, g) range it covered.
#include <cuda.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace qasc {
namespace {

constexpr int kStageTok = 64;
constexpr int kRowBytes = kD * 2;
constexpr int kStages = 2;
constexpr int kConsWarps = 4;
constexpr int kCons = 32 * kConsWarps;
constexpr int kThreads = kCons + 32;
constexpr int kGroups = 2 * kConsWarps;   // half-warp groups
constexpr int kTB = 8;                    // rows per group per stage
constexpr int kPartStride = 132;          // floats per partial: m, l, pad, pad, o[128]
// CTAs per SM: three (15 warps) when the group's state fits 128 registers,
// one for 8-head groups (their state needs ~250 registers).
__host__ __device__ constexpr int ctas_per_sm(int gq) { return gq <= 4 ? 3 : 1; }
// log2(e) / sqrt(128): logits are kept in base-2 units.
constexpr float kQScale = 1.4426950408889634f * 0.08838834764831845f;

__device__ __forceinline__ int64_t token_at(int64_t j, int64_t sink_end, int64_t K, int64_t local_start,
                                            const int32_t* sel_b) {
  if (j < sink_end) return j;
  if (j < sink_end + K) return sel_b[j - sink_end];
  return local_start + (j - sink_end - K);
}

// Last CTA whose range [c P / G, (c+1) P / G) starts at or before position x,
// i.e. the CTA that holds position x.
__host__ __device__ __forceinline__ int first_cta(int64_t x, int64_t P, int G) {
  int64_t c = ((x + 1) * G + P - 1) / P - 1;
  return static_cast<int>(c < 0 ? 0 : (c >= G ? G - 1 : c));
}

// Four rows (y0..y3) of a 2-D tensor, full 128-column width, into 1 KB of
// shared memory.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* tmap, int y0, int y1, int y2, int y3,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.L2::cache_hint "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(smem_u32(dst)),
      "l"(tmap), "r"(0), "r"(y0), "r"(y1), "r"(y2), "r"(y3), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

template <int GQ>
struct AttnSmem {
  uint8_t k[kStages][kStageTok * kRowBytes];
  uint8_t v[kStages][kStageTok * kRowBytes];
  alignas(16) int32_t ids[kStages][kStageTok];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  float p[kGroups][kTB][GQ < 4 ? 4 : GQ];
  float alpha[kGroups][GQ < 4 ? 4 : GQ];
};

struct AttnArgs {
  const uint16_t* q;
  const uint16_t* K;
  const uint16_t* V;
  const int32_t* sel;
  float* part;
  int Hq, Hkv;
  int64_t n_cap, sink_end, Ksel, local_start;
  int64_t T;        // |T| per (b, g)
  int64_t P;        // B * Hkv * T
  int max_splits;   // partial slots per (b, g)
  unsigned* err;
};

template <int GQ>
__global__ void __launch_bounds__(kThreads, ctas_per_sm(GQ))
    sparse_attn_kernel(const AttnArgs a, const __grid_constant__ CUtensorMap tmap_k,
                       const __grid_constant__ CUtensorMap tmap_v) {
  constexpr int L0 = kTB * GQ;                  // partial logits per lane before the reduce-scatter
  constexpr int R = L0 >= 16 ? L0 / 16 : 1;     // logits owned per lane afterwards
  constexpr int LPH = L0 >= 16 ? 8 / R : 16;    // lanes per head afterwards
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  AttnSmem<GQ>& S = *reinterpret_cast<AttnSmem<GQ>*>(smem_raw);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x, cta = blockIdx.x;
  const int64_t p_begin = static_cast<int64_t>(cta) * a.P / G;
  const int64_t p_end = static_cast<int64_t>(cta + 1) * a.P / G;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kConsWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kConsWarps) {
    // ---- producer warp
    const uint64_t pol = policy_evict_first();
    const int quad = lane & 15;          // which 4-row quad of the stage
    const CUtensorMap* tm = lane < 16 ? &tmap_k : &tmap_v;
    if (lane == 0) {
      prefetch_tensormap(&tmap_k);
      prefetch_tensormap(&tmap_v);
    }
    int st = 0;
    for (int64_t p = p_begin; p < p_end;) {
      const int bg = static_cast<int>(p / a.T);
      const int64_t seg_end = min(p_end, static_cast<int64_t>(bg + 1) * a.T);
      const int b = bg / a.Hkv;
      const int32_t* sel_b = a.sel + static_cast<int64_t>(b) * a.Ksel;
      const int64_t row0 = static_cast<int64_t>(bg) * a.n_cap;
      for (int64_t q0 = p; q0 < seg_end; q0 += kStageTok, ++st) {
        const int slot = st % kStages;
        const uint32_t ph = (st / kStages) & 1u;
        const int rows = static_cast<int>(min(static_cast<int64_t>(kStageTok), seg_end - q0));
        const int nquads = (rows + 3) >> 2;
        const int64_t j0 = q0 - static_cast<int64_t>(bg) * a.T;
        // token ids of this stage (loads issued before the slot wait); rows
        // past the end repeat the last valid row so that quads stay whole
        int64_t t0 = token_at(j0 + min(lane, rows - 1), a.sink_end, a.Ksel, a.local_start, sel_b);
        int64_t t1 = token_at(j0 + min(lane + 32, rows - 1), a.sink_end, a.Ksel, a.local_start, sel_b);
        const bool ok = mbar_wait(&S.empty[slot], ph ^ 1u);
        if (!__all_sync(0xffffffffu, ok)) {
          record_error(a.err, kErrTimeout);
          return;
        }
        // Ids outside the cache are clamped so a bad selection cannot fault.
        t0 = t0 < 0 ? 0 : (t0 >= a.n_cap ? a.n_cap - 1 : t0);
        t1 = t1 < 0 ? 0 : (t1 >= a.n_cap ? a.n_cap - 1 : t1);
        S.ids[slot][lane] = static_cast<int32_t>(row0 + t0);
        S.ids[slot][lane + 32] = static_cast<int32_t>(row0 + t1);
        if (lane == 0) mbar_arrive_expect_tx(&S.full[slot], static_cast<uint32_t>(nquads) * 2u * 4u * kRowBytes);
        __syncwarp();
        if (quad < nquads) {
          const int4 y = *reinterpret_cast<const int4*>(&S.ids[slot][4 * quad]);
          uint8_t* dst = (lane < 16 ? &S.k[slot][0] : &S.v[slot][0]) + quad * 4 * kRowBytes;
          tma_gather4(dst, tm, y.x, y.y, y.z, y.w, &S.full[slot], pol);
        }
        __syncwarp();
      }
      p = seg_end;
    }
    return;
  }

  // ---- consumers
  const int half = lane >> 4, l16 = lane & 15;
  const int gi = warp * 2 + half;
  const unsigned hmask = 0xffffu << (16 * half);
  const int my_head = (l16 * R) / kTB < GQ ? (l16 * R) / kTB : GQ - 1;

  float2 qr[GQ][4];
  float2 o[GQ][4];
  float m_run = -INFINITY;   // running max (base 2) of my_head in this group
  float l_run = 0.0f;        // this lane's share of the running sum

  int st = 0;
  for (int64_t p = p_begin; p < p_end;) {
    const int bg = static_cast<int>(p / a.T);
    const int64_t seg_end = min(p_end, static_cast<int64_t>(bg + 1) * a.T);
    {
      // queries of this KV head's group, pre-scaled into base-2 logit units
      const int b = bg / a.Hkv, g = bg - b * a.Hkv;
      const uint16_t* qb = a.q + (static_cast<int64_t>(b) * a.Hq + g * GQ) * kD + 8 * l16;
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(qb + hh * kD));
        const float2 x0 = bf2_to_f2(raw.x), x1 = bf2_to_f2(raw.y), x2 = bf2_to_f2(raw.z), x3 = bf2_to_f2(raw.w);
        qr[hh][0] = make_float2(x0.x * kQScale, x0.y * kQScale);
        qr[hh][1] = make_float2(x1.x * kQScale, x1.y * kQScale);
        qr[hh][2] = make_float2(x2.x * kQScale, x2.y * kQScale);
        qr[hh][3] = make_float2(x3.x * kQScale, x3.y * kQScale);
#pragma unroll
        for (int j = 0; j < 4; ++j) o[hh][j] = make_float2(0.0f, 0.0f);
      }
      m_run = -INFINITY;
      l_run = 0.0f;
    }
    for (int64_t q0 = p; q0 < seg_end; q0 += kStageTok, ++st) {
      const int slot = st % kStages;
      const uint32_t ph = (st / kStages) & 1u;
      const bool ok = mbar_wait(&S.full[slot], ph);
      if (!__all_sync(0xffffffffu, ok)) {
        record_error(a.err, kErrTimeout);
        return;
      }
      const int rows = static_cast<int>(min(static_cast<int64_t>(kStageTok), seg_end - q0));
      const int nt = max(0, min(kTB, rows - gi * kTB));
      if (nt > 0) {
        const uint8_t* kst = S.k[slot] + (gi * kTB) * kRowBytes + l16 * 16;
        const uint8_t* vst = S.v[slot] + (gi * kTB) * kRowBytes + l16 * 16;
        float pv[L0];   // q . k partials, index h * 8 + t
#pragma unroll
        for (int t = 0; t < kTB; ++t) {
          uint4 kr = make_uint4(0, 0, 0, 0);
          if (t < nt) kr = *reinterpret_cast<const uint4*>(kst + t * kRowBytes);
          const float2 k0 = bf2_to_f2(kr.x), k1 = bf2_to_f2(kr.y), k2 = bf2_to_f2(kr.z), k3 = bf2_to_f2(kr.w);
#pragma unroll
          for (int hh = 0; hh < GQ; ++hh) {
            float2 acc = make_float2(0.0f, 0.0f);
            acc = ffma2(qr[hh][0], k0, acc);
            acc = ffma2(qr[hh][1], k1, acc);
            acc = ffma2(qr[hh][2], k2, acc);
            acc = ffma2(qr[hh][3], k3, acc);
            pv[hh * kTB + t] = acc.x + acc.y;
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
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
          const float al = S.alpha[gi][hh];
          const float2 a2 = make_float2(al, al);
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
    // ---- this group's partial for (bg); the merge kernel combines them
    {
      float lsum = l_run;
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) {
        const float other = __shfl_xor_sync(hmask, lsum, off);
        if (off < LPH) lsum += other;
      }
      const int64_t x0 = static_cast<int64_t>(bg) * a.T;
      const int split = cta - first_cta(x0, a.P, G);
      float* base =
          a.part + ((static_cast<int64_t>(bg) * a.max_splits + split) * kGroups + gi) * GQ * kPartStride;
      if ((l16 % LPH) == 0) {
        base[my_head * kPartStride + 0] = m_run;
        base[my_head * kPartStride + 1] = lsum;
      }
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) {
        float4* dst = reinterpret_cast<float4*>(base + hh * kPartStride + 4 + 8 * l16);
        dst[0] = make_float4(o[hh][0].x, o[hh][0].y, o[hh][1].x, o[hh][1].y);
        dst[1] = make_float4(o[hh][2].x, o[hh][2].y, o[hh][3].x, o[hh][3].y);
      }
    }
    p = seg_end;
  }
}

// grid B * Hq, block 512: exact log-sum-exp merge of every group partial of
// every CTA that covered this (b, g).  The partials' (max, sum) pairs are
// read in parallel into shared memory and turned into weights; then four
// threads per output dimension each sum a quarter of the weighted partial
// outputs with independent loads, and the quarters are added.
constexpr int kMergeMax = 2048;   // partials per (b, h) the merge can stage
constexpr int kMergeThreads = 4 * kD;

template <int GQ>
__global__ void __launch_bounds__(kMergeThreads) merge_kernel(const float* __restrict__ part,
                                                             float* __restrict__ out, float* __restrict__ lse,
                                                             int Hkv, int64_t T, int64_t P, int G, int max_splits) {
  __shared__ float wgt[kMergeMax];
  __shared__ float red[2][kMergeThreads / 32];
  __shared__ float quarter[3][kD];
  const int bh = blockIdx.x;
  const int Hq = Hkv * GQ;
  const int b = bh / Hq, h = bh - b * Hq;
  const int g = h / GQ, hh = h - g * GQ;
  const int bg = b * Hkv + g;
  const int64_t x0 = static_cast<int64_t>(bg) * T;
  const int c0 = first_cta(x0, P, G);
  const int c1 = first_cta(x0 + T - 1, P, G);
  const int n = min((c1 - c0 + 1) * kGroups, kMergeMax);
  const int64_t pstride = static_cast<int64_t>(GQ) * kPartStride;
  const float* base = part + static_cast<int64_t>(bg) * max_splits * kGroups * pstride + hh * kPartStride;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  float M = -INFINITY;
  for (int s = tid; s < n; s += kMergeThreads) {
    const float ms = __ldcg(base + s * pstride);
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
    Lp = fmaf(w, __ldcg(base + s * pstride + 1), Lp);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Lp += __shfl_xor_sync(0xffffffffu, Lp, o);
  if (lane == 0) red[1][warp] = Lp;
  __syncthreads();
  float L = 0.0f;
#pragma unroll
  for (int i = 0; i < kMergeThreads / 32; ++i) L += red[1][i];
  const int e = tid & (kD - 1), q4 = tid >> 7;
  float O[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
  int s = q4;
  for (; s + 28 < n; s += 32) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) v[u] = __ldcg(base + (s + 4 * u) * pstride + 4 + e);
#pragma unroll
    for (int u = 0; u < 8; ++u) O[u] = fmaf(wgt[s + 4 * u], v[u], O[u]);
  }
  for (; s < n; s += 4) O[0] = fmaf(wgt[s], __ldcg(base + s * pstride + 4 + e), O[0]);
  const float Oq = ((O[0] + O[1]) + (O[2] + O[3])) + ((O[4] + O[5]) + (O[6] + O[7]));
  if (q4 > 0) quarter[q4 - 1][e] = Oq;
  __syncthreads();
  if (q4 == 0) {
    out[static_cast<int64_t>(bh) * kD + e] = ((Oq + quarter[0][e]) + (quarter[1][e] + quarter[2][e])) / L;
    if (lse && e == 0) lse[bh] = (M + log2f(L)) * 0.6931471805599453f;
  }
}

// ctas_per_sm(gq) CTAs per SM, but at least one full stage of rows per CTA.
int grid_for(int64_t P, int num_sms, int gq) {
  int64_t G = static_cast<int64_t>(num_sms > 0 ? num_sms : 148) * ctas_per_sm(gq);
  const int64_t by_rows = P / kStageTok;
  if (G > by_rows) G = by_rows;
  if (G < 1) G = 1;
  return static_cast<int>(G);
}

template <int GQ>
int launch_gq(const qasc_shape& s, const qasc_ts_params& p, const AttnLayout& L, const uint16_t* q,
              const uint16_t* K, const uint16_t* V, const int32_t* sel, float* out, float* lse, float* part,
              const DeviceInfo& dev, cudaStream_t stream) {
  const Regions R = regions_of(s.n, p.sink, p.local);
  AttnArgs a;
  a.q = q;
  a.K = K;
  a.V = V;
  a.sel = sel;
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
  const int G = grid_for(a.P, dev.num_sms, GQ);
  // K and V viewed as 2-D [B*Hkv*n_cap rows, 128 columns] bf16 tensors; a box
  // is one full row, fetched four indexed rows at a time.
  EncodeTiledFn enc = encode_tiled_fn();
  if (!enc) return cudaErrorNotSupported;
  alignas(64) CUtensorMap tk, tv;
  const uint64_t gdim[2] = {static_cast<uint64_t>(kD), static_cast<uint64_t>(s.B) * s.Hkv * s.n_cap};
  const uint64_t gstride[1] = {static_cast<uint64_t>(kRowBytes)};
  const unsigned box[2] = {kD, 1};
  const unsigned estr[2] = {1, 1};
  if (enc(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(K), gdim, gstride, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != 0 ||
      enc(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(V), gdim, gstride, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != 0)
    return cudaErrorInvalidValue;
  sparse_attn_kernel<GQ><<<G, kThreads, sizeof(AttnSmem<GQ>), stream>>>(a, tk, tv);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  merge_kernel<GQ><<<s.B * s.Hq, kMergeThreads, 0, stream>>>(part, out, lse, s.Hkv, a.T, a.P, G, L.splits);
  return cudaGetLastError();
}

template <int GQ>
cudaError_t configure_gq() {
  return cudaFuncSetAttribute(sparse_attn_kernel<GQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              static_cast<int>(sizeof(AttnSmem<GQ>)));
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
  const int G = grid_for(P, num_sms, s.Hq / s.Hkv);
  // CTAs overlapping one (b, g) list: every CTA range holds at least
  // floor(P / G) >= 64 positions, so at most (T - 1) / floor(P / G) + 2.
  L.splits = static_cast<int>((L.t_len - 1) / (P / G) + 2);
  L.per_split = 0;
  L.off_part = 0;
  L.total = align_up(static_cast<size_t>(bg) * L.splits * kGroups * (s.Hq / s.Hkv) * kPartStride * sizeof(float),
                     256);
  return L;
}

int launch_sparse_attn(const qasc_shape& s, const qasc_ts_params& p, const AttnLayout& L, const uint16_t* q,
                       const uint16_t* K, const uint16_t* V, const int32_t* sel, float* out, float* lse,
                       uint8_t* ws, const DeviceInfo& dev, cudaStream_t stream) {
  float* part = reinterpret_cast<float*>(ws + L.off_part);
  switch (s.Hq / s.Hkv) {
    case 1: return launch_gq<1>(s, p, L, q, K, V, sel, out, lse, part, dev, stream);
    case 2: return launch_gq<2>(s, p, L, q, K, V, sel, out, lse, part, dev, stream);
    case 4: return launch_gq<4>(s, p, L, q, K, V, sel, out, lse, part, dev, stream);
    case 8: return launch_gq<8>(s, p, L, q, K, V, sel, out, lse, part, dev, stream);
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
// that first call should happen before any stream capture.  Every call shares
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

// spec_verify_sample: the fused rejection-sampling pass of the verify step.
//
// What is computed (quant67 "speculative decoding" section 3.1; "KV Cache +
// Speculative Decoding" sections 7.1-7.3 and 7.6): per sequence b and draft
// position i, p_i = softmax(target_i / T), q_i = softmax(draft_i / T) (or the
// given q_i); x_i is accepted iff u_i q_i(x_i) < p_i(x_i); at the first
// rejection n the token is drawn by inverse CDF (ascending token id, strict
// '>') from max(0, p_n - q_n); if all K are accepted it is drawn from p_K.
//
// GB300 design:
//   * sample_rows_kernel: one thread-block cluster per (sequence, position)
//     row. Each CTA of the cluster pulls its slice of the target row and of
//     the draft row into shared memory with 1-D bulk (TMA) copies, so every
//     logit crosses HBM once. Max and sum-of-exp are reduced across the
//     cluster through distributed shared memory. The accept test and a
//     speculative "if rejected here" inverse-CDF draw (the bonus draw for row
//     K) are evaluated in fp32 together with a bound on their rounding error;
//     the result is one 48-byte record per row.
//   * sample_resolve_kernel: one cluster per sequence walks the K records in
//     order, stops at the first rejection and writes the emitted tokens. A
//     decision whose fp32 margin is inside the rounding bound is recomputed
//     from the logits in float-float arithmetic (about 2^-44 relative error),
//     so emitted tokens agree with exact arithmetic except on a set of
//     uniforms of measure ~1e-12.
#include <cmath>
#include <mutex>
#include <type_traits>

#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kRowThreads = 512;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kResThreads = 512;
constexpr int kResWarps = kResThreads / 32;
constexpr int kResCluster = 8;
constexpr uint32_t kChunkBytes = 16384;
constexpr int kMaxChunks = 32;              // per CTA, target + draft
constexpr size_t kMaxSliceSmem = 200 * 1024;
constexpr size_t kTargetSliceSmem = 64 * 1024;

enum : uint32_t { REC_ACCEPT = 1u, REC_ACC_CERTAIN = 2u };
enum : uint32_t { SMP_FOUND = 1u, SMP_CERTAIN = 2u };

struct RowRec {
  float m_p, s_p, m_q, s_q;  // fast-path row max and sum of exp2((l - m) c)
  float p_x, q_x;            // p_i(x_i), q_i(x_i) in fp32
  float gap, z;              // margin of the fp32 draw and its total mass
  int32_t y;                 // fp32 inverse-CDF draw
  uint32_t acc_flags;        // REC_*
  uint32_t smp_flags;        // SMP_*
  float e_abs;               // rounding bound the margin was compared with
};
static_assert(sizeof(RowRec) == 48, "record layout");

struct SampleParams {
  const void *target;
  const void *draft;
  const int32_t *tokens;
  const float *uniforms;
  float *p_at;
  float *q_at;
  int32_t *out_tokens;
  int32_t *num_acc;
  RowRec *recs;
  int32_t *status;
  int B, K, V;
  int ns;        // elements per CTA slice in the rows kernel (multiple of 8)
  int aligned;   // rows are 16-byte aligned: bulk copies usable
  unsigned flags;
  float c;       // log2(e) / T
  float invT_hi, invT_lo;
  int unitT;
  float log2e_hi, log2e_lo, ln2_hi, ln2_lo;
  float2 tbl[64];  // 2^(j/64) split into (hi, lo)
};

// ------------------------------------------------------------ fp32 path ---

template <typename T>
__device__ __forceinline__ void load8(const T *s, int g, float (&x)[8]);

template <>
__device__ __forceinline__ void load8<float>(const float *s, int g, float (&x)[8]) {
  const float4 a = reinterpret_cast<const float4 *>(s)[2 * g];
  const float4 b = reinterpret_cast<const float4 *>(s)[2 * g + 1];
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16 *s, int g, float (&x)[8]) {
  const uint4 v = reinterpret_cast<const uint4 *>(s)[g];
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    x[2 * k] = __uint_as_float(w[k] << 16);
    x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
  }
}

template <>
__device__ __forceinline__ void load8<__half>(const __half *s, int g, float (&x)[8]) {
  const uint4 v = reinterpret_cast<const uint4 *>(s)[g];
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const __half2 h = *reinterpret_cast<const __half2 *>(&w[k]);
    const float2 f = __half22float2(h);
    x[2 * k] = f.x;
    x[2 * k + 1] = f.y;
  }
}

template <typename T>
__device__ __forceinline__ T pad_value(bool is_prob) {
  if (is_prob) return T(0.f);
  return T(-INFINITY);
}

// Block-wide reduction of one float (all threads get the result).
template <bool MAX>
__device__ __forceinline__ float block_reduce(float v, float *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = MAX ? warp_max(v) : warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  const int nw = blockDim.x >> 5;
  float r = lane < nw ? red[lane] : (MAX ? -INFINITY : 0.f);
  r = MAX ? warp_max(r) : warp_sum(r);
  return r;
}

// Reduce a published per-CTA float across the cluster (same result and
// same order of operations in every CTA). `pub` is this CTA's shared copy.
template <bool MAX>
__device__ __forceinline__ float cluster_reduce(const float *pub, int cs) {
  const int lane = threadIdx.x & 31;
  float v = MAX ? -INFINITY : 0.f;
  if (lane < cs) v = ld_dsmem_f32(mapa(pub, lane));
  return MAX ? warp_max(v) : warp_sum(v);
}

template <typename TT, int DK>
__global__ void __launch_bounds__(kRowThreads) sample_rows_kernel(const __grid_constant__ SampleParams P) {
  using TD = typename std::conditional<DK == 0, TT, float>::type;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kMaxChunks];
  __shared__ float red[32];
  __shared__ float pub_max_p, pub_max_q, pub_sum_p, pub_sum_q, pub_tot, pub_q2;
  __shared__ float wsum[kRowWarps];

  const int cs = gridDim.x;
  const int rank = (int)cluster_ctarank();
  const int i = blockIdx.y, b = blockIdx.z;
  const int K = P.K, V = P.V;
  const bool has_draft = i < K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const TT *trow = static_cast<const TT *>(P.target) + ((int64_t)b * (K + 1) + i) * V;
  const TD *drow = has_draft ? static_cast<const TD *>(P.draft) + ((int64_t)b * K + i) * V : nullptr;
  const int e0 = rank * P.ns;
  const int n_loc = max(0, min(V, e0 + P.ns) - e0);
  const int n_grp = (n_loc + 7) >> 3;
  TT *st = reinterpret_cast<TT *>(smem);
  TD *sd = reinterpret_cast<TD *>(smem + align_up((size_t)P.ns * sizeof(TT), 128));

  // ---- stage the slice into shared memory --------------------------------
  const uint32_t nb_t = (uint32_t)n_loc * sizeof(TT);
  const uint32_t nb_d = has_draft ? (uint32_t)n_loc * sizeof(TD) : 0u;
  const int nch_t = P.aligned ? (int)((nb_t + kChunkBytes - 1) / kChunkBytes) : 0;
  const int nch_d = P.aligned ? (int)((nb_d + kChunkBytes - 1) / kChunkBytes) : 0;
  // padding of the last group: -inf logits / zero probabilities
  for (int e = n_loc + tid; e < n_grp * 8; e += blockDim.x) {
    st[e] = pad_value<TT>(false);
    if (has_draft) sd[e] = pad_value<TD>(DK == 1);
  }
  if (P.aligned) {
    if (tid == 0) {
      for (int k = 0; k < nch_t + nch_d; ++k) mbar_init(&bars[k], 1);
      fence_mbarrier_init();
    }
    __syncthreads();
    if (tid == 0) {
      const uint8_t *gt = reinterpret_cast<const uint8_t *>(trow + e0);
      for (int k = 0; k < nch_t; ++k) {
        const uint32_t off = k * kChunkBytes, nb = min(kChunkBytes, nb_t - off);
        mbar_arrive_expect_tx(&bars[k], nb);
        bulk_g2s(reinterpret_cast<uint8_t *>(st) + off, gt + off, nb, &bars[k]);
      }
      if (has_draft) {
        const uint8_t *gd = reinterpret_cast<const uint8_t *>(drow + e0);
        for (int k = 0; k < nch_d; ++k) {
          const uint32_t off = k * kChunkBytes, nb = min(kChunkBytes, nb_d - off);
          mbar_arrive_expect_tx(&bars[nch_t + k], nb);
          bulk_g2s(reinterpret_cast<uint8_t *>(sd) + off, gd + off, nb, &bars[nch_t + k]);
        }
      }
    }
  } else {
    for (int e = tid; e < n_loc; e += blockDim.x) {
      st[e] = trow[e0 + e];
      if (has_draft) sd[e] = drow[e0 + e];
    }
    __syncthreads();
  }

  // ---- pass 1: row maxima (overlapped with the arriving chunks) ----------
  bool timed_out = false;
  float mt = -INFINITY, md = -INFINITY;
  {
    constexpr int gpc_t = kChunkBytes / (8 * sizeof(TT));  // groups per chunk
    const int nchunks = P.aligned ? nch_t : 1;
    for (int k = 0; k < nchunks; ++k) {
      if (P.aligned && !timed_out && !mbar_wait(&bars[k], 0)) timed_out = true;
      const int g_end = P.aligned ? min(n_grp, (k + 1) * gpc_t) : n_grp;
      for (int g = (P.aligned ? k * gpc_t : 0) + tid; g < g_end; g += blockDim.x) {
        float x[8];
        load8(st, g, x);
#pragma unroll
        for (int j = 0; j < 8; ++j) mt = fmaxf(mt, x[j]);
      }
    }
  }
  if (has_draft) {
    constexpr int gpc_d = kChunkBytes / (8 * sizeof(TD));
    const int nchunks = P.aligned ? nch_d : 1;
    for (int k = 0; k < nchunks; ++k) {
      if (P.aligned && !timed_out && !mbar_wait(&bars[nch_t + k], 0)) timed_out = true;
      if (DK == 0) {
        const int g_end = P.aligned ? min(n_grp, (k + 1) * gpc_d) : n_grp;
        for (int g = (P.aligned ? k * gpc_d : 0) + tid; g < g_end; g += blockDim.x) {
          float x[8];
          load8(sd, g, x);
#pragma unroll
          for (int j = 0; j < 8; ++j) md = fmaxf(md, x[j]);
        }
      }
    }
  }
  if (timed_out) atomic_or_status(P.status, SV_DEV_TIMEOUT);
  mt = block_reduce<true>(mt, red);
  if (has_draft && DK == 0) md = block_reduce<true>(md, red);
  if (tid == 0) { pub_max_p = mt; pub_max_q = md; }
  cluster_sync();
  const float m_p = cluster_reduce<true>(&pub_max_p, cs);
  const float m_q = (has_draft && DK == 0) ? cluster_reduce<true>(&pub_max_q, cs) : 0.f;

  // ---- pass 2: sums of exp2((l - m) c) ------------------------------------
  const float c = P.c;
  const float mcp = m_p * c, mcq = m_q * c;
  float sp = 0.f, sq = 0.f;
  for (int g = tid; g < n_grp; g += blockDim.x) {
    float x[8];
    load8(st, g, x);
#pragma unroll
    for (int j = 0; j < 8; ++j) sp += exp2f(fmaf(x[j], c, -mcp));
    if (has_draft && DK == 0) {
      load8(sd, g, x);
#pragma unroll
      for (int j = 0; j < 8; ++j) sq += exp2f(fmaf(x[j], c, -mcq));
    }
  }
  sp = block_reduce<false>(sp, red);
  if (has_draft && DK == 0) sq = block_reduce<false>(sq, red);
  if (tid == 0) { pub_sum_p = sp; pub_sum_q = sq; }
  cluster_sync();
  const float S_p = cluster_reduce<false>(&pub_sum_p, cs);
  const float S_q = (has_draft && DK == 0) ? cluster_reduce<false>(&pub_sum_q, cs) : 1.f;
  const float inv_sp = 1.f / S_p, inv_sq = 1.f / S_q;

  RowRec *rec = P.recs + (int64_t)b * (K + 1) + i;
  const float *uv = P.uniforms + ((int64_t)b * (K + 1) + i) * 2;
  if (!(fabsf(m_p) <= 3.0e38f) || (has_draft && DK == 0 && !(fabsf(m_q) <= 3.0e38f))) {
    if (tid == 0 && rank == 0) atomic_or_status(P.status, SV_DEV_NONFINITE);
  }

  // ---- accept test (rank 0) ----------------------------------------------
  if (rank == 0 && tid == 0) {
    rec->m_p = m_p; rec->s_p = S_p; rec->m_q = m_q; rec->s_q = S_q;
    uint32_t af = 0;
    float p_x = 0.f, q_x = 0.f;
    if (has_draft) {
      int x = P.tokens[(int64_t)b * K + i];
      if (x < 0 || x >= V) {
        atomic_or_status(P.status, SV_DEV_BAD_TOKEN);
        x = min(max(x, 0), V - 1);
      }
      p_x = exp2f(fmaf(to_f32(trow[x]), c, -mcp)) * inv_sp;
      if (DK == 0) q_x = exp2f(fmaf(to_f32(drow[x]), c, -mcq)) * inv_sq;
      else q_x = to_f32(drow[x]);
      const float lhs = uv[0] * q_x;
      if (lhs < p_x) af |= REC_ACCEPT;
      // relative rounding bound of p_x and u q_x (exp2, argument rounding,
      // row sums): a decision this far from the boundary is exact.
      if (fabsf(p_x - lhs) > 4e-6f * fmaxf(p_x, lhs) && p_x > 0.f && q_x > 0.f) af |= REC_ACC_CERTAIN;
      if (P.p_at) P.p_at[(int64_t)b * K + i] = p_x;
      if (P.q_at) P.q_at[(int64_t)b * K + i] = q_x;
    }
    rec->p_x = p_x; rec->q_x = q_x;
    rec->acc_flags = af;
  }

  // ---- pass 3: weights of the speculative draw, per-warp range sums -------
  // weight w(y) = max(0, p(y) - q(y)) for a draft row, p(y) for the bonus row.
  auto weight8 = [&](int g, float (&w)[8], float &q2) {
    float xp[8];
    load8(st, g, xp);
    if (has_draft) {
      float xq[8];
      load8(sd, g, xq);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float p = exp2f(fmaf(xp[j], c, -mcp)) * inv_sp;
        const float q = DK == 0 ? exp2f(fmaf(xq[j], c, -mcq)) * inv_sq : xq[j];
        w[j] = fmaxf(p - q, 0.f);
        q2 = fmaf(p, p, fmaf(q, q, q2));
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float p = exp2f(fmaf(xp[j], c, -mcp)) * inv_sp;
        w[j] = p;
        q2 = fmaf(p, p, q2);
      }
    }
  };
  const int gpw = (n_grp + kRowWarps - 1) / kRowWarps;  // groups per warp range
  const int g_lo = warp * gpw, g_hi = min(n_grp, g_lo + gpw);
  float run = 0.f, q2 = 0.f;
  for (int s0 = g_lo; s0 < g_hi; s0 += 32) {
    const int g = s0 + lane;
    float v = 0.f;
    if (g < g_hi) {
      float w[8];
      weight8(g, w, q2);
#pragma unroll
      for (int j = 0; j < 8; ++j) v += w[j];
    }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float t = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += t;
    }
    run += __shfl_sync(0xffffffffu, v, 31);
  }
  if (lane == 0) wsum[warp] = run;
  q2 = block_reduce<false>(q2, red);   // contains __syncthreads: wsum visible
  float tot_cta = 0.f;
  for (int w = 0; w < kRowWarps; ++w) tot_cta += wsum[w];
  if (tid == 0) { pub_tot = tot_cta; pub_q2 = q2; }
  cluster_sync();
  // exclusive prefix over ranks (same chain in every CTA)
  float off_c = 0.f, Z = 0.f;
  for (int r = 0; r < cs; ++r) {
    const float t = ld_dsmem_f32(mapa(&pub_tot, r));
    if (r == rank) off_c = Z;
    Z += t;
  }
  const float Q2 = cluster_reduce<false>(&pub_q2, cs);
  const float v = uv[1];
  const float thr = v * Z;
  const float e_abs = 1.9073486e-06f * sqrtf(Q2) + 4.7683716e-07f * (Z + 1.f);  // 2^-19, 2^-21
  const bool draw_ok = Z > 0.f && thr < Z && fabsf(m_p) <= 3.0e38f;
  if (rank == 0 && tid == 0) {
    rec->z = Z;
    rec->e_abs = e_abs;
    if (!draw_ok) { rec->y = -1; rec->smp_flags = 0; rec->gap = 0.f; }
  }
  if (draw_ok && off_c <= thr && thr < off_c + tot_cta) {
    // owner warp: A_w <= thr < A_{w+1}
    float woff = 0.f;
    int owner = kRowWarps - 1;
    float a_w = off_c;
    for (int w = 0; w < kRowWarps; ++w) {
      const float a_next = off_c + (woff + wsum[w]);
      if (thr < a_next || w == kRowWarps - 1) { owner = w; a_w = off_c + woff; break; }
      woff += wsum[w];
    }
    if (warp == owner) {
      float base = a_w;
      int y = -1;
      float c_lo = 0.f, c_hi = 0.f;
      for (int s0 = g_lo; s0 < g_hi && y < 0; s0 += 32) {
        const int g = s0 + lane;
        float w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        float dummy = 0.f, vsum = 0.f;
        if (g < g_hi) {
          weight8(g, w, dummy);
#pragma unroll
          for (int j = 0; j < 8; ++j) vsum += w[j];
        }
        float incl = vsum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float t = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += t;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, base + incl > thr);
        if (hit) {
          const int L = __ffs(hit) - 1;
          if (lane == L) {
            float run_c = base + (incl - vsum);
            for (int j = 0; j < 8; ++j) {
              const float nxt = run_c + w[j];
              if (nxt > thr) { y = (e0 + 8 * g + j); c_lo = run_c; c_hi = nxt; break; }
              run_c = nxt;
            }
            if (y < 0) y = -2;   // rounding moved the crossing: not found
          }
          y = __shfl_sync(0xffffffffu, y, L);
          c_lo = __shfl_sync(0xffffffffu, c_lo, L);
          c_hi = __shfl_sync(0xffffffffu, c_hi, L);
          if (y < 0) break;
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) {
        if (y >= 0 && y < V) {
          const float gap = fminf(thr - c_lo, c_hi - thr);
          rec->y = y;
          rec->gap = gap;
          rec->smp_flags = SMP_FOUND | (gap > e_abs ? SMP_CERTAIN : 0u);
        } else {
          rec->y = -1;
          rec->gap = 0.f;
          rec->smp_flags = 0;
        }
      }
    }
  }
  // the accept test and the draw of an out-of-range draft row are resolved
  // exactly by the resolve kernel (flags left uncertain)
  cluster_sync();   // no CTA leaves while a peer may still read its shared memory
}

// ------------------------------------------------- float-float arithmetic ---
// A value is hi + lo with |lo| <= ulp(hi)/2; error-free transformations
// (Knuth two-sum, fma-based two-product) give ~2^-44 relative accuracy.

struct ff {
  float hi, lo;
};

__device__ __forceinline__ ff two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  const float e = (a - (s - bb)) + (b - bb);
  return {s, e};
}

__device__ __forceinline__ ff quick_two_sum(float a, float b) {
  const float s = a + b;
  return {s, b - (s - a)};
}

__device__ __forceinline__ ff ff_add(ff a, ff b) {
  ff s = two_sum(a.hi, b.hi);
  const ff t = two_sum(a.lo, b.lo);
  s.lo += t.hi;
  s = quick_two_sum(s.hi, s.lo);
  s.lo += t.lo;
  return quick_two_sum(s.hi, s.lo);
}

__device__ __forceinline__ ff ff_neg(ff a) { return {-a.hi, -a.lo}; }

__device__ __forceinline__ ff ff_mul(ff a, ff b) {
  const float p = a.hi * b.hi;
  float e = fmaf(a.hi, b.hi, -p);
  e = fmaf(a.hi, b.lo, e);
  e = fmaf(a.lo, b.hi, e);
  return quick_two_sum(p, e);
}

__device__ __forceinline__ bool ff_gt(ff a, ff b) {  // a > b
  const ff d = ff_add(a, ff_neg(b));
  return d.hi > 0.f || (d.hi == 0.f && d.lo > 0.f);
}

__device__ __forceinline__ ff ff_max0(ff a) {
  return (a.hi > 0.f || (a.hi == 0.f && a.lo > 0.f)) ? a : ff{0.f, 0.f};
}

__device__ __forceinline__ ff shfl_ff(ff v, int src) {
  return {__shfl_sync(0xffffffffu, v.hi, src), __shfl_sync(0xffffffffu, v.lo, src)};
}

// exp((l - m) / T) for l <= m in float-float: reduce t = x log2(e) to
// n/64 + r with |r| <= 1/128, 2^r = e^(r ln2) by its Taylor series to the
// 5th power (truncation < 1e-14), 2^(j/64) from a float-float table.
__device__ __forceinline__ ff ff_exp(float l, float m, const SampleParams &P, const float2 *tbl) {
  ff x = two_sum(l, -m);
  if (!P.unitT) x = ff_mul(x, ff{P.invT_hi, P.invT_lo});
  if (!(x.hi > -87.f)) return ff{0.f, 0.f};   // below the fp32 normal range: negligible
  const ff t = ff_mul(x, ff{P.log2e_hi, P.log2e_lo});
  const float n = rintf(t.hi * 64.f);
  const float rh = fmaf(-n, 0.015625f, t.hi);  // exact
  const ff r = two_sum(rh, t.lo);
  const ff y = ff_mul(r, ff{P.ln2_hi, P.ln2_lo});  // |y| <= 0.0055
  const float yh = y.hi;
  const float poly = yh * yh * (0.5f + yh * (0.16666667f + yh * (0.041666668f + yh * 0.0083333338f)));
  const ff s = two_sum(yh, y.lo + (poly + yh * y.lo));  // e^y - 1
  const int ni = (int)n;
  const float2 T = tbl[ni & 63];
  const ff Tf{T.x, T.y};
  ff res = ff_add(Tf, ff_mul(Tf, s));
  const int k = ni >> 6;                           // floor(n / 64)
  res.hi = ldexpf(res.hi, k);
  res.lo = ldexpf(res.lo, k);
  return res;
}

// Block reduction of a float-float sum (result in all threads).
__device__ __forceinline__ ff block_reduce_ff(ff v, ff *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = ff_add(v, ff{__shfl_xor_sync(0xffffffffu, v.hi, o),
                                                     __shfl_xor_sync(0xffffffffu, v.lo, o)});
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  ff r = ff{0.f, 0.f};
  const int nw = blockDim.x >> 5;
  for (int w = 0; w < nw; ++w) r = ff_add(r, red[w]);
  return r;
}

struct ExactShared {
  ff red[32];
  ff wsum[kResWarps];
  ff pub_sp, pub_sq, pub_tot;
  int pub_y, pub_last;
  float2 tbl[64];
};

// Exact-arithmetic evaluation of row i of sequence b by the whole cluster
// (every thread of every CTA calls it with the same arguments). Returns the
// accept decision when need_accept (and stops there if accepted); otherwise
// *y_out receives the inverse-CDF draw of the row.
template <typename TT, int DK>
__device__ bool exact_row(const SampleParams &P, int b, int i, const RowRec &rec, bool need_accept,
                          int *y_out, ExactShared &sh) {
  using TD = typename std::conditional<DK == 0, TT, float>::type;
  const int K = P.K, V = P.V;
  const int cs = gridDim.x;
  const int rank = (int)cluster_ctarank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool has_draft = i < K;
  const TT *trow = static_cast<const TT *>(P.target) + ((int64_t)b * (K + 1) + i) * V;
  const TD *drow = has_draft ? static_cast<const TD *>(P.draft) + ((int64_t)b * K + i) * V : nullptr;
  const float m_p = rec.m_p, m_q = rec.m_q;
  const int nsp = ((V + cs - 1) / cs + 31) / 32 * 32;
  const int e0 = min(V, rank * nsp), e1 = min(V, e0 + nsp);

  // pass A: float-float row sums of exp((l - m) / T)
  ff sp{0.f, 0.f}, sq{0.f, 0.f};
  for (int e = e0 + tid; e < e1; e += blockDim.x) {
    sp = ff_add(sp, ff_exp(to_f32(trow[e]), m_p, P, sh.tbl));
    if (has_draft && DK == 0) sq = ff_add(sq, ff_exp(to_f32(drow[e]), m_q, P, sh.tbl));
  }
  sp = block_reduce_ff(sp, sh.red);
  sq = block_reduce_ff(sq, sh.red);
  if (tid == 0) { sh.pub_sp = sp; sh.pub_sq = sq; }
  cluster_sync();
  ff Sp{0.f, 0.f}, Sq{0.f, 0.f};
  for (int r = 0; r < cs; ++r) {
    const uint32_t a = mapa(&sh.pub_sp, r), q = mapa(&sh.pub_sq, r);
    Sp = ff_add(Sp, ff{ld_dsmem_f32(a), ld_dsmem_f32(a + 4)});
    Sq = ff_add(Sq, ff{ld_dsmem_f32(q), ld_dsmem_f32(q + 4)});
  }
  cluster_sync();   // every peer has read the published sums
  if (DK == 1 || !has_draft) Sq = ff{1.f, 0.f};
  const float *uv = P.uniforms + ((int64_t)b * (K + 1) + i) * 2;

  if (need_accept && has_draft) {
    int x = P.tokens[(int64_t)b * K + i];
    x = min(max(x, 0), V - 1);
    const ff epx = ff_exp(to_f32(trow[x]), m_p, P, sh.tbl);
    // u q(x) < p(x)  <=>  u e_q(x) S_p < e_p(x) S_q   (draft logits)
    //                <=>  u q(x) S_p < e_p(x)         (draft probabilities)
    ff lhs, rhs;
    if (DK == 0) {
      const ff eqx = ff_exp(to_f32(drow[x]), m_q, P, sh.tbl);
      lhs = ff_mul(ff_mul(ff{uv[0], 0.f}, eqx), Sp);
      rhs = ff_mul(epx, Sq);
    } else {
      lhs = ff_mul(ff{uv[0], 0.f}, ff_mul(ff{to_f32(drow[x]), 0.f}, Sp));
      rhs = epx;
    }
    if (ff_gt(rhs, lhs)) return true;
  }

  // pass B: scaled weights w'(y) = S_p S_q w(y) and the inverse CDF.
  // mode 0: target row (bonus, or the zero-mass fallback), 1: residual of
  // two softmaxes, 2: residual against given draft probabilities.
  int mode = !has_draft ? 0 : (DK == 0 ? 1 : 2);
  const int wr = ((nsp + kResWarps - 1) / kResWarps + 31) / 32 * 32;
  const int w_lo = min(e1, e0 + warp * wr), w_hi = min(e1, w_lo + wr);
  auto weight = [&](int e) -> ff {
    const ff ep = ff_exp(to_f32(trow[e]), m_p, P, sh.tbl);
    if (mode == 0) return ep;
    if (mode == 1) {
      const ff eq = ff_exp(to_f32(drow[e]), m_q, P, sh.tbl);
      return ff_max0(ff_add(ff_mul(ep, Sq), ff_neg(ff_mul(eq, Sp))));
    }
    return ff_max0(ff_add(ep, ff_neg(ff_mul(ff{to_f32(drow[e]), 0.f}, Sp))));
  };
  auto scan32 = [&](ff v) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const ff t{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
      if (lane >= o) v = ff_add(t, v);
    }
    return v;
  };

  int y = -1;
  for (int attempt = 0; attempt < 2; ++attempt) {
    // per-warp totals over contiguous ranges, and the last positive index
    ff run{0.f, 0.f};
    int last_pos = -1;
    for (int s0 = w_lo; s0 < w_hi; s0 += 32) {
      const int e = s0 + lane;
      const ff w = e < w_hi ? weight(e) : ff{0.f, 0.f};
      const unsigned pos = __ballot_sync(0xffffffffu, w.hi > 0.f);
      if (pos) last_pos = s0 + 31 - __clz(pos);
      run = ff_add(run, shfl_ff(scan32(w), 31));
    }
    if (lane == 0) {
      sh.wsum[warp] = run;
      if (last_pos >= 0) atomicMax(&sh.pub_last, last_pos);
    }
    __syncthreads();
    ff tot{0.f, 0.f};
    for (int w = 0; w < kResWarps; ++w) tot = ff_add(tot, sh.wsum[w]);
    if (tid == 0) sh.pub_tot = tot;
    cluster_sync();
    ff off_c{0.f, 0.f}, Z{0.f, 0.f};
    int last_all = -1;
    for (int r = 0; r < cs; ++r) {
      const uint32_t a = mapa(&sh.pub_tot, r);
      const ff t{ld_dsmem_f32(a), ld_dsmem_f32(a + 4)};
      if (r == rank) off_c = Z;
      Z = ff_add(Z, t);
      last_all = max(last_all, ld_dsmem_s32(mapa(&sh.pub_last, r)));
    }
    cluster_sync();   // peers have read pub_tot / pub_last
    if (tid == 0) sh.pub_last = -1;
    if (!(Z.hi > 0.f)) {   // zero residual mass: draw from p_n instead
      __syncthreads();
      if (mode == 0) break;
      mode = 0;
      continue;
    }
    const ff thr = ff_mul(ff{uv[1], 0.f}, Z);
    const ff end_c = ff_add(off_c, tot);
    if (!ff_gt(off_c, thr) && ff_gt(end_c, thr)) {
      ff woff{0.f, 0.f};
      int owner = kResWarps - 1;
      ff a_w = off_c;
      for (int w = 0; w < kResWarps; ++w) {
        const ff nxt = ff_add(woff, sh.wsum[w]);
        if (ff_gt(ff_add(off_c, nxt), thr) || w == kResWarps - 1) {
          owner = w;
          a_w = ff_add(off_c, woff);
          break;
        }
        woff = nxt;
      }
      if (warp == owner) {
        ff base = a_w;
        int found = -1, last_p = -1;
        for (int s0 = w_lo; s0 < w_hi && found < 0; s0 += 32) {
          const int e = s0 + lane;
          const ff w = e < w_hi ? weight(e) : ff{0.f, 0.f};
          const unsigned pos = __ballot_sync(0xffffffffu, w.hi > 0.f);
          if (pos) last_p = s0 + 31 - __clz(pos);
          const ff incl = scan32(w);
          const unsigned hit =
              __ballot_sync(0xffffffffu, w.hi > 0.f && ff_gt(ff_add(base, incl), thr));
          if (hit) found = s0 + __ffs(hit) - 1;
          base = ff_add(base, shfl_ff(incl, 31));
        }
        if (found < 0) found = last_p;   // crossing within rounding of the range end
        if (lane == 0) sh.pub_y = found;
      }
    }
    cluster_sync();
    for (int r = 0; r < cs; ++r) y = max(y, ld_dsmem_s32(mapa(&sh.pub_y, r)));
    if (y < 0) y = last_all;   // v Z at the very top of the range (rounding)
    cluster_sync();            // peers have read pub_y
    if (tid == 0) sh.pub_y = -1;
    __syncthreads();
    break;
  }
  *y_out = y;
  return false;
}

template <typename TT, int DK>
__global__ void __launch_bounds__(kResThreads) sample_resolve_kernel(const __grid_constant__ SampleParams P) {
  __shared__ ExactShared sh;
  const int b = blockIdx.y;
  const int K = P.K;
  const int tid = threadIdx.x;
  if (tid < 64) sh.tbl[tid] = P.tbl[tid];
  if (tid == 0) { sh.pub_y = -1; sh.pub_last = -1; }
  __syncthreads();
  cluster_sync();   // peers initialised before any distributed read
  const bool force = (P.flags & SV_SAMPLE_FORCE_EXACT) != 0;
  int n = K, y = -1;
  bool have_y = false;
  for (int i = 0; i < K; ++i) {
    const RowRec rec = P.recs[(int64_t)b * (K + 1) + i];
    bool acc;
    if (!force && (rec.acc_flags & REC_ACC_CERTAIN)) {
      acc = (rec.acc_flags & REC_ACCEPT) != 0;
    } else {
      int yy = -1;
      acc = exact_row<TT, DK>(P, b, i, rec, true, &yy, sh);
      if (!acc) { y = yy; have_y = true; }
    }
    if (!acc) { n = i; break; }
  }
  if (!have_y) {
    const RowRec rec = P.recs[(int64_t)b * (K + 1) + n];
    if (!force && (rec.smp_flags & SMP_CERTAIN)) y = rec.y;
    else exact_row<TT, DK>(P, b, n, rec, false, &y, sh);
  }
  if (cluster_ctarank() == 0) {
    for (int j = tid; j < K + 1; j += blockDim.x)
      P.out_tokens[(int64_t)b * (K + 1) + j] = j < n ? P.tokens[(int64_t)b * K + j] : (j == n ? y : -1);
    if (tid == 0) P.num_acc[b] = n;
  }
}

// ------------------------------------------------------------------ host ---

size_t records_bytes(int B, int K) { return align_up((size_t)B * (K + 1) * sizeof(RowRec), 256); }

void split_ff(double d, float &hi, float &lo) {
  hi = (float)d;
  lo = (float)(d - (double)hi);
}

template <typename TT, int DK>
sv_status launch_sample(const SampleParams &P, int cs, size_t smem, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(sample_rows_kernel<TT, DK>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)(kMaxSliceSmem + 1024));
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(sample_rows_kernel<TT, DK>,
                                      cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
  if (attr_err != cudaSuccess)
    return fail(SV_ERR_CUDA, "spec_verify_sample: cudaFuncSetAttribute: %s", cudaGetErrorString(attr_err));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, P.K + 1, P.B);
  cfg.blockDim = dim3(kRowThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, sample_rows_kernel<TT, DK>, P);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_sample rows launch: %s", cudaGetErrorString(e));
  attr[0].val.clusterDim.x = kResCluster;
  cfg.gridDim = dim3(kResCluster, P.B);
  cfg.blockDim = dim3(kResThreads);
  cfg.dynamicSmemBytes = 0;
  e = cudaLaunchKernelEx(&cfg, sample_resolve_kernel<TT, DK>, P);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_sample resolve launch: %s", cudaGetErrorString(e));
  return ok();
}

}  // namespace
}  // namespace sv

extern "C" size_t spec_verify_sample_workspace_size(int B, int K, int V) {
  (void)V;
  if (B < 0 || K < 0) return 0;
  return sv::records_bytes(B, K);
}

extern "C" sv_status spec_verify_sample_ex(const void *target_logits, sv_dtype logit_dtype,
                                           const void *draft, sv_dtype draft_dtype, int draft_is_probs,
                                           const int32_t *draft_tokens, const float *uniforms, int B,
                                           int K, int V, float temperature, int32_t *out_tokens,
                                           int32_t *num_accepted, float *p_at_draft, float *q_at_draft,
                                           void *workspace, size_t workspace_bytes,
                                           int32_t *dev_status, unsigned flags, sv_stream_t stream) {
  using namespace sv;
  if (B < 0 || K < 0 || V < 1)
    return fail(SV_ERR_INVALID_ARG, "spec_verify_sample: bad sizes B=%d K=%d V=%d", B, K, V);
  if (B > 65535 || K + 1 > 65535)
    return fail(SV_ERR_UNSUPPORTED, "spec_verify_sample: B and K+1 must be <= 65535");
  if (!(temperature > 0.f) || !std::isfinite(temperature))
    return fail(SV_ERR_INVALID_ARG, "spec_verify_sample: temperature must be finite and > 0");
  if (!target_logits || !uniforms || !out_tokens || !num_accepted)
    return fail(SV_ERR_INVALID_ARG, "spec_verify_sample: null pointer argument");
  if (K > 0 && (!draft || !draft_tokens))
    return fail(SV_ERR_INVALID_ARG, "spec_verify_sample: draft and draft_tokens are required for K > 0");
  if (logit_dtype != SV_F32 && logit_dtype != SV_BF16 && logit_dtype != SV_F16)
    return fail(SV_ERR_UNSUPPORTED, "spec_verify_sample: logits must be f32, bf16 or f16");
  if (draft_is_probs) {
    if (K > 0 && draft_dtype != SV_F32)
      return fail(SV_ERR_UNSUPPORTED, "spec_verify_sample: draft probabilities must be f32");
  } else if (K > 0 && draft_dtype != logit_dtype) {
    return fail(SV_ERR_UNSUPPORTED, "spec_verify_sample: draft logits must have the target's dtype");
  }
  if (!workspace || workspace_bytes < records_bytes(B, K))
    return fail(SV_ERR_WORKSPACE, "spec_verify_sample: workspace needs %zu bytes", records_bytes(B, K));
  if (!aligned(workspace, 256)) return fail(SV_ERR_WORKSPACE, "spec_verify_sample: workspace not 256-byte aligned");
  if (B == 0) return ok();

  const int es_t = dtype_bytes(logit_dtype);
  const int es_d = K > 0 ? (draft_is_probs ? 4 : es_t) : 0;
  int cs = 0;
  int ns = 0;
  size_t smem = 0;
  auto smem_for = [&](int c, int &ns_out) {
    ns_out = (int)align_up((size_t)((V + c - 1) / c), 8);
    return align_up((size_t)ns_out * es_t, 128) + (size_t)ns_out * es_d;
  };
  for (int c = 1; c <= 16; c *= 2) {
    int n;
    const size_t sm = smem_for(c, n);
    if (sm <= kTargetSliceSmem) { cs = c; ns = n; smem = sm; break; }
  }
  if (!cs) {
    for (int c = 1; c <= 16; c *= 2) {
      int n;
      const size_t sm = smem_for(c, n);
      if (sm <= kMaxSliceSmem) { cs = c; ns = n; smem = sm; break; }
    }
  }
  if (!cs) return fail(SV_ERR_UNSUPPORTED, "spec_verify_sample: vocabulary of %d too large", V);

  SampleParams P = {};
  P.target = target_logits; P.draft = draft; P.tokens = draft_tokens; P.uniforms = uniforms;
  P.p_at = p_at_draft; P.q_at = q_at_draft; P.out_tokens = out_tokens; P.num_acc = num_accepted;
  P.recs = static_cast<RowRec *>(workspace); P.status = dev_status;
  P.B = B; P.K = K; P.V = V; P.ns = ns; P.flags = flags;
  P.aligned = aligned(target_logits, 16) && ((size_t)V * es_t) % 16 == 0 &&
              (K == 0 || (aligned(draft, 16) && ((size_t)V * es_d) % 16 == 0));
  const double log2e = 1.4426950408889634074, ln2 = 0.69314718055994530942;
  P.c = (float)(log2e / (double)temperature);
  P.unitT = temperature == 1.0f;
  split_ff(1.0 / (double)temperature, P.invT_hi, P.invT_lo);
  split_ff(log2e, P.log2e_hi, P.log2e_lo);
  split_ff(ln2, P.ln2_hi, P.ln2_lo);
  for (int j = 0; j < 64; ++j) split_ff(std::exp2((double)j / 64.0), P.tbl[j].x, P.tbl[j].y);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool probs = draft_is_probs && K > 0;
  switch (logit_dtype) {
    case SV_F32: return probs ? launch_sample<float, 1>(P, cs, smem, s) : launch_sample<float, 0>(P, cs, smem, s);
    case SV_BF16:
      return probs ? launch_sample<__nv_bfloat16, 1>(P, cs, smem, s)
                   : launch_sample<__nv_bfloat16, 0>(P, cs, smem, s);
    default:
      return probs ? launch_sample<__half, 1>(P, cs, smem, s) : launch_sample<__half, 0>(P, cs, smem, s);
  }
}

extern "C" sv_status spec_verify_sample(const void *target_logits, sv_dtype logit_dtype, const void *draft,
                                        sv_dtype draft_dtype, int draft_is_probs,
                                        const int32_t *draft_tokens, const float *uniforms, int B, int K,
                                        int V, float temperature, int32_t *out_tokens,
                                        int32_t *num_accepted, float *p_at_draft, float *q_at_draft,
                                        void *workspace, size_t workspace_bytes, int32_t *dev_status,
                                        sv_stream_t stream) {
  return spec_verify_sample_ex(target_logits, logit_dtype, draft, draft_dtype, draft_is_probs, draft_tokens,
                               uniforms, B, K, V, temperature, out_tokens, num_accepted, p_at_draft,
                               q_at_draft, workspace, workspace_bytes, dev_status, 0u, stream);
}

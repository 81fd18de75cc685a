// spec_verify_sample: the fused rejection-sampling pass of the verify step.
//
// What is computed (quant67 "speculative decoding" section 3.1; "KV Cache +
// Speculative Decoding" sections 7.1-7.3 and 7.6): per sequence b and draft
// position i, p_i = softmax(target_i / T), q_i = softmax(draft_i / T) (or the
// given q_i); x_i is accepted iff u_i q_i(x_i) < p_i(x_i); at the first
// rejection n the token is drawn by inverse CDF (ascending token id, strict
// '>') from max(0, p_n - q_n); if all K are accepted it is drawn from p_K.
//
// GB300 design: sample_init_kernel (one CTA) zeroes the call's counters;
// sample_fused_kernel does the work; sample_exact_kernel resolves, in
// float-float arithmetic, the rare sequences the fused kernel could not
// certify. Every CTA of the two working kernels takes a ticket from a global
// counter when it starts; the ticket names its work item, so a CTA only ever
// waits for CTAs holding smaller tickets, which are already running or done.
//   * statistics items, (chunk c, position i) of sequence b: the 8192-logit
//     chunk of target row i and of draft row i, loaded with 16-byte loads
//     straight into registers (every logit crosses HBM once); exact maxima,
//     fp32 sums of exponentials (the two rows paired in packed fp32
//     arithmetic); one (max, sum) pair per row and chunk. The last item of a
//     sequence to finish combines them, evaluates the accept tests in fp32
//     with a certificate that each lies outside its rounding bound, walks to
//     the first rejection (or the bonus row) and publishes the row drawn from.
//   * draw items, (chunk c) of sequence b, ticketed a few sequences behind
//     b's statistics so that draws run while other sequences still stream:
//     each waits for b's decisions, streams its chunk of the row drawn from
//     (the residual max(0, p - q), or the bonus row) and publishes per-warp
//     sums of the weights; the last draw item of the sequence locates v Z
//     (chunk, warp, then one warp's 1024 logits reloaded from L2) and
//     certifies the token.
//   * a decision that is not certified (a few percent of sequences at a
//     128K vocabulary) goes to sample_exact_kernel, which re-evaluates it in
//     float-float arithmetic (~1e-9 relative error per term), so emitted
//     tokens are those of exact arithmetic except for uniforms within
//     ~1e-10 of a boundary.
#include <cmath>
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kFThreads = 256;
constexpr int kFWarps = kFThreads / 32;
constexpr int kChunk = 8192;                          // logits of a row per item
constexpr int kChunkGroups = kChunk / 8;              // groups of eight
constexpr int kGrp = kChunkGroups / kFThreads;        // groups per thread (4)
constexpr int kMaxChunks = 32;                        // V <= 262144
constexpr int kMaxPos = 64;                           // K + 1 <= 64
static_assert(kGrp == 4 && kChunkGroups == 32 * kGrp * kFWarps, "draw layout: warp, block of 32 groups, lane");

// per-sequence words (zeroed by sample_init_kernel): statistics items done,
// draw items done, decisions published
enum : int { SEQ_STATS = 0, SEQ_DRAW = 1, SEQ_DEC = 2, SEQ_WORDS = 4 };
// what the decisions leave to the draw items: the draw, or nothing (the
// sequence went to the float-float kernel)
enum : int { DEC_DRAW = 1, DEC_EXACT = 2 };
// the call's words: tickets of the two kernels, the pending count, then one
// barrier counter per float-float group
enum : int { SYNC_TICKET = 0, SYNC_XTICKET = 1, SYNC_PCOUNT = 2, SYNC_XBAR = 4, SYNC_WORDS = 64 };
constexpr int kWtStride = 12;   // per chunk of a draw: kFWarps warp totals, the chunk total, padding

struct SampleParams {
  const void *target;     // [B][K+1][V]
  const void *draft;      // [B][K][V] logits (target dtype) or f32 probabilities
  const int32_t *tokens;  // [B][K]
  const float *uniforms;  // [B][K+1][2]
  float *p_at;
  float *q_at;
  int32_t *out_tokens;
  int32_t *num_acc;
  float4 *part;           // [B][K+1][nc] (max, sum) of the target and draft chunks; the float-float
                          // kernel reuses a pending sequence's rows for (S_p hi, lo, S_q hi, lo)
  float4 *rowrec;         // [B][K+1] (m_p, S_p, m_q, S_q) of each row
  int *rowflag;           // [B][K+1] accept test: bit 0 accepted, bit 1 certified
  float *wtot;            // [B][nc][kWtStride] per-warp and chunk totals of the draw
  float4 *xtot;           // [B][nc] float-float chunk totals (hi, lo) and last positive index
  int2 *dec;              // [B] (row drawn from, DEC_*)
  int2 *pend;             // [B] sequences left to the float-float kernel: (b, first row to resolve)
  unsigned *seq;          // [B][SEQ_WORDS]
  unsigned *sync;         // [SYNC_WORDS]
  int32_t *status;
  int B, K, V, nc;
  int lag;                // sequences a draw item is ticketed behind its statistics
  int aligned;            // rows are 16-byte aligned: vector loads
  unsigned flags;
  float c;                // log2(e) / T
  float invT_hi, invT_lo;
  int unitT;
  float log2e_hi, log2e_lo;
  float2 tbl[64];         // 2^(j/64) split into (hi, lo)
};

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

__device__ __forceinline__ bool ff_pos(ff a) { return a.hi > 0.f || (a.hi == 0.f && a.lo > 0.f); }

__device__ __forceinline__ bool ff_gt(ff a, ff b) { return ff_pos(ff_add(a, ff_neg(b))); }

__device__ __forceinline__ ff ff_max0(ff a) { return ff_pos(a) ? a : ff{0.f, 0.f}; }


__device__ __forceinline__ ff scan32_ff(ff v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const ff t{__shfl_up_sync(0xffffffffu, v.hi, o), __shfl_up_sync(0xffffffffu, v.lo, o)};
    if (lane >= o) v = ff_add(t, v);
  }
  return v;
}

// ------------------------------------------------------------ fp32 path ---

// 2^x on the SFU (flushes results below 2^-126, i.e. weights < 1e-38 of the
// row maximum, to zero). Its relative error on [-30, 0] measured on GB300 is
// below 1.5e-7.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Block sum of a float-float value (result in every thread): butterflies
// within each warp, then over the warp partials (identical bits everywhere).
__device__ __forceinline__ ff warp_sum_ff(ff v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = ff_add(v, ff{__shfl_xor_sync(0xffffffffu, v.hi, o),
                                                     __shfl_xor_sync(0xffffffffu, v.lo, o)});
  return v;
}

__device__ __forceinline__ ff block_sum_ff(ff v, ff *red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_ff(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  return warp_sum_ff(lane < (int)(blockDim.x >> 5) ? red[lane] : ff{0.f, 0.f});
}

__device__ __forceinline__ int warp_max_s32(int v) {
  int r;
  asm volatile("redux.sync.max.s32 %0, %1, 0xffffffff;" : "=r"(r) : "r"(v));
  return r;
}


// warp maximum on the reduction unit (NaN inputs are ignored, like fmaxf)
__device__ __forceinline__ float warp_max_redux(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

template <typename H2>
__device__ __forceinline__ H2 as_h2(uint32_t w) {
  H2 h;
  memcpy(&h, &w, 4);
  return h;
}

// Negated rounded reference -fl(m c) of a partial maximum (0 for an empty or
// all -inf partial: its exponents are then 2^-inf = 0).
__device__ __forceinline__ float neg_ref(float m, float c) { return m == -INFINITY ? 0.f : -__fmul_rn(m, c); }

// Rescale a partial sum taken against fl(m c) to the reference fl(mx c).
__device__ __forceinline__ float rescale(float s, float m, float mx, float c) {
  return m == -INFINITY ? 0.f : s * ex2(__fmul_rn(m, c) - __fmul_rn(mx, c));
}

// Warp-wide (max, sum) of a partial pair: identical bits in every lane.
__device__ __forceinline__ void warp_ms(float &m, float &s, float c) {
  const float mx = warp_max_redux(m);
  s = warp_sum(rescale(s, m, mx, c));
  m = mx;
}

// raw bits of 8 logits: one 16-byte word for 16-bit types, two for f32
template <typename T> struct Raw8 { uint4 w[sizeof(T) / 2]; };

template <typename T>
__device__ __forceinline__ uint32_t neg_inf_bits();
template <> __device__ __forceinline__ uint32_t neg_inf_bits<float>() { return 0xff800000u; }
template <> __device__ __forceinline__ uint32_t neg_inf_bits<__nv_bfloat16>() { return 0xff80ff80u; }
template <> __device__ __forceinline__ uint32_t neg_inf_bits<__half>() { return 0xfc00fc00u; }

// group g (elements 8g .. 8g+7) of a row; elements at or past e1 read as -inf
// (as 0 for given probabilities: pad_zero)
template <typename T>
__device__ __forceinline__ Raw8<T> raw_load(const T *row, int g, int e1, bool vec, bool pad_zero) {
  Raw8<T> r;
  if (vec && 8 * g + 8 <= e1) {
    const uint4 *p = reinterpret_cast<const uint4 *>(row + 8 * g);
#pragma unroll
    for (int k = 0; k < (int)(sizeof(T) / 2); ++k) r.w[k] = __ldg(p + k);
    return r;
  }
  T v[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int e = 8 * g + j;
    if (e < e1) {
      v[j] = row[e];
    } else {
      const uint32_t bits = pad_zero ? 0u : neg_inf_bits<T>();
      memcpy(&v[j], &bits, sizeof(T));
    }
  }
  memcpy(&r, v, sizeof(v));
  return r;
}

template <typename T>
__device__ __forceinline__ void unpack8(const Raw8<T> &r, float (&x)[8]) {
  if constexpr (std::is_same<T, float>::value) {
    x[0] = __uint_as_float(r.w[0].x); x[1] = __uint_as_float(r.w[0].y);
    x[2] = __uint_as_float(r.w[0].z); x[3] = __uint_as_float(r.w[0].w);
    x[4] = __uint_as_float(r.w[1].x); x[5] = __uint_as_float(r.w[1].y);
    x[6] = __uint_as_float(r.w[1].z); x[7] = __uint_as_float(r.w[1].w);
  } else {
    const uint32_t w[4] = {r.w[0].x, r.w[0].y, r.w[0].z, r.w[0].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      if constexpr (std::is_same<T, __nv_bfloat16>::value) {
        x[2 * k] = __uint_as_float(w[k] << 16);
        x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
      } else {
        const float2 f = __half22float2(as_h2<__half2>(w[k]));
        x[2 * k] = f.x;
        x[2 * k + 1] = f.y;
      }
    }
  }
}

// exact maximum of 8 logits (a selection: the packed 16-bit forms are exact)
template <typename T>
__device__ __forceinline__ float max8(const Raw8<T> &r) {
  if constexpr (std::is_same<T, float>::value) {
    float x[8];
    unpack8(r, x);
    return fmaxf(max3f(x[0], x[1], x[2]), max3f(max3f(x[3], x[4], x[5]), x[6], x[7]));
  } else if constexpr (std::is_same<T, __nv_bfloat16>::value) {
    const __nv_bfloat162 a = __hmax2(as_h2<__nv_bfloat162>(r.w[0].x), as_h2<__nv_bfloat162>(r.w[0].y));
    const __nv_bfloat162 bb = __hmax2(as_h2<__nv_bfloat162>(r.w[0].z), as_h2<__nv_bfloat162>(r.w[0].w));
    const __nv_bfloat162 m = __hmax2(a, bb);
    return fmaxf(__low2float(m), __high2float(m));
  } else {
    const __half2 a = __hmax2(as_h2<__half2>(r.w[0].x), as_h2<__half2>(r.w[0].y));
    const __half2 bb = __hmax2(as_h2<__half2>(r.w[0].z), as_h2<__half2>(r.w[0].w));
    const __half2 m = __hmax2(a, bb);
    return fmaxf(__low2float(m), __high2float(m));
  }
}

// sum of eight fp32 weights, pairwise in packed arithmetic
__device__ __forceinline__ float sum8f(const float (&w)[8]) {
  const float2 a = __fadd2_rn(make_float2(w[0], w[1]), make_float2(w[2], w[3]));
  const float2 bb = __fadd2_rn(make_float2(w[4], w[5]), make_float2(w[6], w[7]));
  const float2 t = __fadd2_rn(a, bb);
  return t.x + t.y;
}

__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// fp32 weights of one group of eight elements of the row drawn from, in
// units of S_p times probability: max(0, e_p - r e_q) with r = S_p / S_q
// (draft logits) or r = S_p (draft probabilities, e_q = q), e_p alone for
// the bonus row; padding reads as -inf (logits) or 0 (probabilities)
template <typename TT, typename TD, int DK>
__device__ __forceinline__ void draw_weights8(const Raw8<TT> &rt, const Raw8<TD> &rd, bool has_draft, float c,
                                              float mcp, float mcq, float r_pq, float (&w)[8]) {
  float xp[8];
  unpack8(rt, xp);
  const float2 cc = make_float2(c, c);
  if (has_draft) {
    float xq[8];
    unpack8(rd, xq);
    const float2 nref = make_float2(-mcp, -mcq);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      float ep, eq;
      if (DK == 0) {
        const float2 y = __ffma2_rn(make_float2(xp[j], xq[j]), cc, nref);
        ep = ex2(y.x);
        eq = ex2(y.y);
      } else {
        ep = ex2(fmaf(xp[j], c, -mcp));
        eq = xq[j];
      }
      w[j] = fmaxf(fmaf(-r_pq, eq, ep), 0.f);
    }
  } else {
    const float2 np = make_float2(-mcp, -mcp);
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      const float2 y = __ffma2_rn(make_float2(xp[j], xp[j + 1]), cc, np);
      w[j] = ex2(y.x);
      w[j + 1] = ex2(y.y);
    }
  }
}

// ------------------------------------------- float-float re-evaluation ---
// Lean float-float exp: exp((l - m)/T) for l <= m as an unevaluated pair
// hi + lo with ~1e-9 relative error: t = (l - m) log2(e) split into
// n/64 + r (|r| <= 1/128), 2^r - 1 by its Taylor series to r^5, 2^(j/64)
// from the (hi, lo) table, 2^k by exponent construction. Values below e^-87
// relative to the row maximum are returned as 0.
// The float-float pass runs rarely, with the instruction cache cold for its
// code, so the exponential and the weights are single out-of-line copies
// called from rolled loops.
struct FfK {
  float inv_hi, inv_lo;     // 1/T
  float l2e_hi, l2e_lo;     // log2(e)
  int unitT;                // T == 1
};

__device__ __noinline__ ff ffx_exp(float l, float m, FfK k, const float2 *tbl) {
  if (!(l > -INFINITY)) return ff{0.f, 0.f};
  ff x = two_sum(l, -m);
  if (!k.unitT) x = ff_mul(x, ff{k.inv_hi, k.inv_lo});
  if (!(x.hi > -87.f)) return ff{0.f, 0.f};
  const float t_hi = x.hi * k.l2e_hi;
  const float t_lo = fmaf(x.hi, k.l2e_hi, -t_hi) + fmaf(x.hi, k.l2e_lo, x.lo * k.l2e_hi);
  const float n = rintf(t_hi * 64.f);
  const float r = fmaf(-n, 0.015625f, t_hi) + t_lo;
  const float y = r * 0.69314718f;
  const float s = fmaf(y * y, 0.5f + y * (0.16666667f + y * (0.041666668f + y * 0.0083333338f)), y);
  const int ni = (int)n;
  const float2 T = tbl[ni & 63];
  const float scale = __int_as_float(((ni >> 6) + 127) << 23);
  return ff{T.x * scale, fmaf(T.x, s, T.y) * scale};
}

// sum of nonnegative pairs: two-sum on the high parts, low parts added
__device__ __forceinline__ void acc_add(ff &a, ff v) {
  const ff s = two_sum(a.hi, v.hi);
  a.hi = s.hi;
  a.lo += s.lo + v.lo;
}

__device__ __forceinline__ ff ff_norm(ff a) { return quick_two_sum(a.hi, a.lo); }

// float-float weight of one element (target logit lp, draft value lq) of the
// row drawn from: mode 0 the target row (e_p), 1 two softmaxes
// (max(0, e_p S_q - e_q S_p)), 2 given draft probabilities
// (max(0, e_p - q S_p)); a padding element (lp = -inf) weighs 0
__device__ __noinline__ ff resid_weight(int mode, float lp, float lq, float m_p, float m_q, ff Sp, ff Sq, FfK k,
                                        const float2 *tbl) {
  const ff ep = ffx_exp(lp, m_p, k, tbl);
  if (mode == 0) return ep;
  if (mode == 1) return ff_max0(ff_add(ff_mul(ep, Sq), ff_neg(ff_mul(ffx_exp(lq, m_q, k, tbl), Sp))));
  return ff_max0(ff_add(ep, ff_neg(ff_mul(ff{lq > -INFINITY ? lq : 0.f, 0.f}, Sp))));
}

// ------------------------------------------------- cross-CTA signalling ---

__device__ __forceinline__ unsigned ld_acquire(const unsigned *p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void red_release_add(unsigned *p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_release(unsigned *p, unsigned v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned atom_add_acq_rel(unsigned *p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Thread 0 polls *ctr until it reaches target (acquire), at most the wait
// limit; every thread of the CTA gets the result through *flag. Counters are
// zeroed for each call and only grow.
__device__ __forceinline__ bool cta_wait_geq(const unsigned *ctr, unsigned target, unsigned *flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned ok = 1u;
    const uint64_t t0 = global_ns();
    while (ld_acquire(ctr) < target) {
      if (global_ns() - t0 > kWaitLimitNs) { ok = 0u; break; }
      __nanosleep(64);
    }
    *flag = ok;
  }
  __syncthreads();
  return *flag != 0u;
}

// The CTA's global writes so far become visible to whoever sees the count.
__device__ __forceinline__ void cta_arrive(unsigned *ctr) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) red_release_add(ctr, 1u);
}

// sequence b is left to the float-float kernel, from row i0 on
__device__ __forceinline__ void push_pending(const SampleParams &P, int b, int i0) {
  const unsigned slot = atomicAdd(P.sync + SYNC_PCOUNT, 1u);
  P.pend[slot] = make_int2(b, i0);
}

// emitted tokens of sequence b: the n accepted drafts, then y, then -1
__device__ __forceinline__ void write_outputs(const SampleParams &P, int b, int n, int y) {
  const int K = P.K;
  for (int j = 0; j <= K; ++j)
    P.out_tokens[(int64_t)b * (K + 1) + j] = j < n ? P.tokens[(int64_t)b * K + j] : (j == n ? y : -1);
  P.num_acc[b] = n;
}

struct FusedShared {
  int kind, b, i, c;            // the decoded ticket (kind 0 statistics, 1 draw, -1 none)
  unsigned flag;                // result of thread 0's wait
  int last;                     // this CTA was the last of its kind to arrive for the sequence
  float red[4][kFWarps];        // statistics reductions
  float4 rs[kMaxPos];           // decision: (m_p, S_p, m_q, S_q) of every row of the sequence
  int rfl[kMaxPos];             // decision: accept test, bit 0 accepted, bit 1 certified
  float btot[kFWarps][kGrp];    // draw: block totals
};

// ------------------------------------------------------ statistics item ---

// combined (max, sum) of target (and draft) row i of sequence b from its
// chunk pairs: every lane of the warp ends with the same bits
__device__ __forceinline__ void row_stats(const SampleParams &P, int b, int i, bool q_logits, float &m_p, float &S_p,
                                          float &m_q, float &S_q) {
  const int lane = threadIdx.x & 31;
  const float4 *pr = P.part + ((int64_t)b * (P.K + 1) + i) * P.nc;
  m_p = -INFINITY; S_p = 0.f; m_q = -INFINITY; S_q = 0.f;
  for (int c0 = 0; c0 < P.nc; c0 += 32) {
    float a = -INFINITY, sa = 0.f, d = -INFINITY, sd = 0.f;
    if (c0 + lane < P.nc) {
      const float4 v = __ldcg(pr + c0 + lane);
      a = v.x; sa = v.y; d = v.z; sd = v.w;
    }
    warp_ms(a, sa, P.c);
    const float mp = fmaxf(m_p, a);
    S_p = rescale(S_p, m_p, mp, P.c) + rescale(sa, a, mp, P.c);
    m_p = mp;
    if (q_logits) {
      warp_ms(d, sd, P.c);
      const float mq = fmaxf(m_q, d);
      S_q = rescale(S_q, m_q, mq, P.c) + rescale(sd, d, mq, P.c);
      m_q = mq;
    }
  }
}

// The decisions of sequence b, taken once by the last statistics CTA of the
// sequence: every row's statistics, the accept tests in fp32 with their
// certificates, and the walk (the first rejection stops it; an uncertified
// test sends the sequence to the float-float kernel from that row on). The
// row drawn from is published for the draw items.
template <typename TT, int DK>
__device__ __noinline__ void decide(const SampleParams &P, FusedShared &sh, int b) {
  using TD = typename std::conditional<DK == 0, TT, float>::type;
  const int K = P.K, V = P.V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float cl = P.c;
  for (int i = warp; i <= K; i += kFWarps) {
    const bool ql = i < K && DK == 0;
    float m_p, S_p, m_q, S_q;
    row_stats(P, b, i, ql, m_p, S_p, m_q, S_q);
    if (!ql) { m_q = 0.f; S_q = 1.f; }
    const bool finite = fabsf(m_p) <= 3.0e38f && (!ql || fabsf(m_q) <= 3.0e38f) && S_p > 0.f;
    int fl = 0;
    if (i < K) {
      int x = P.tokens[(int64_t)b * K + i];
      if (x < 0 || x >= V) {
        if (lane == 0) atomic_or_status(P.status, SV_DEV_BAD_TOKEN);
        x = min(max(x, 0), V - 1);
      }
      const float lp_x = to_f32(static_cast<const TT *>(P.target)[((int64_t)b * (K + 1) + i) * V + x]);
      const float lq_x = to_f32(static_cast<const TD *>(P.draft)[((int64_t)b * K + i) * V + x]);
      const float u = P.uniforms[((int64_t)b * (K + 1) + i) * 2];
      const float mcp = __fmul_rn(m_p, cl), mcq = __fmul_rn(m_q, cl);
      const float p_x = ex2(fmaf(lp_x, cl, -mcp)) / S_p;
      const float q_x = DK == 0 ? ex2(fmaf(lq_x, cl, -mcq)) / S_q : lq_x;
      const float lhs = u * q_x;
      const bool accept = lhs < p_x;
      // p_x and u q_x each carry < 2e-6 relative rounding (exp2, argument
      // rounding, row sums): a decision this far from the boundary is exact
      const bool cert = fabsf(p_x - lhs) > 4e-6f * fmaxf(p_x, lhs) && p_x > 0.f && q_x > 0.f && finite;
      fl = (accept ? 1 : 0) | (cert ? 2 : 0);
      if (lane == 0) {
        if (P.p_at) P.p_at[(int64_t)b * K + i] = p_x;
        if (P.q_at) P.q_at[(int64_t)b * K + i] = q_x;
      }
    }
    if (lane == 0) {
      if (!finite) atomic_or_status(P.status, SV_DEV_NONFINITE);
      sh.rs[i] = make_float4(m_p, S_p, m_q, S_q);
      sh.rfl[i] = fl;
      P.rowrec[(int64_t)b * (K + 1) + i] = make_float4(m_p, S_p, m_q, S_q);
      P.rowflag[(int64_t)b * (K + 1) + i] = fl;
    }
  }
  __syncthreads();
  if (tid == 0) {
    int n = K, unc = -1;
    for (int i = 0; i < K; ++i) {
      const int fl = sh.rfl[i];
      if (!(fl & 2)) { unc = i; break; }
      if (!(fl & 1)) { n = i; break; }
    }
    if (P.flags & SV_SAMPLE_FORCE_EXACT) unc = 0;
    const float4 r = sh.rs[n];
    const bool finite = fabsf(r.x) <= 3.0e38f && fabsf(r.z) <= 3.0e38f && r.y > 0.f;
    int state = DEC_DRAW;
    if (unc >= 0 || !finite) {
      state = DEC_EXACT;
      push_pending(P, b, unc >= 0 ? unc : n);
    }
    P.dec[b] = make_int2(n, state);
    __threadfence();
    st_release(P.seq + (size_t)b * SEQ_WORDS + SEQ_DEC, 1u);
  }
}

// (chunk c, position i) of sequence b: each thread holds 32 logits of the
// target row and of the draft row in registers (16-byte loads, all issued
// before any arithmetic), takes exact maxima, then sums of
// 2^(l c - fl(m c)) with the two rows paired in packed fp32 arithmetic.
template <typename TT, int DK>
__device__ __forceinline__ void stats_item(const SampleParams &P, FusedShared &sh, int b, int i, int c) {
  using TD = typename std::conditional<DK == 0, TT, float>::type;
  const int K = P.K, V = P.V;
  const bool q_logits = i < K && DK == 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float cl = P.c;
  const TT *trow = static_cast<const TT *>(P.target) + ((int64_t)b * (K + 1) + i) * V;
  const TD *drow = q_logits ? static_cast<const TD *>(P.draft) + ((int64_t)b * K + i) * V : nullptr;
  const int e0 = c * kChunk, e1 = min(V, e0 + kChunk);
  const int g0 = e0 / 8, g1 = (e1 + 7) / 8;
  const bool vec = P.aligned != 0;

  Raw8<TT> rt[kGrp];
  Raw8<TD> rd[kGrp];
#pragma unroll
  for (int k = 0; k < kGrp; ++k) {
    const int g = g0 + tid + k * kFThreads;
    if (g < g1) {
      rt[k] = raw_load(trow, g, e1, vec, false);
      if (q_logits) rd[k] = raw_load(drow, g, e1, vec, false);
    }
  }
  float mt = -INFINITY, md = -INFINITY;
#pragma unroll
  for (int k = 0; k < kGrp; ++k) {
    if (g0 + tid + k * kFThreads < g1) {
      mt = fmaxf(mt, max8(rt[k]));
      if (q_logits) md = fmaxf(md, max8(rd[k]));
    }
  }
  float s_t = 0.f, s_d = 0.f;
  {
    const float2 cc = make_float2(cl, cl);
    const float2 nm = make_float2(neg_ref(mt, cl), neg_ref(md, cl));
    float2 a0 = make_float2(0.f, 0.f), a1 = a0;
#pragma unroll
    for (int k = 0; k < kGrp; ++k) {
      if (g0 + tid + k * kFThreads >= g1) continue;
      float xt[8];
      unpack8(rt[k], xt);
      if (q_logits) {
        float xd[8];
        unpack8(rd[k], xd);
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
          const float2 y0 = __ffma2_rn(make_float2(xt[j], xd[j]), cc, nm);
          const float2 y1 = __ffma2_rn(make_float2(xt[j + 1], xd[j + 1]), cc, nm);
          a0 = __fadd2_rn(a0, make_float2(ex2(y0.x), ex2(y0.y)));
          a1 = __fadd2_rn(a1, make_float2(ex2(y1.x), ex2(y1.y)));
        }
      } else {
        const float2 nt = make_float2(nm.x, nm.x);
#pragma unroll
        for (int j = 0; j < 8; j += 4) {
          const float2 y0 = __ffma2_rn(make_float2(xt[j], xt[j + 1]), cc, nt);
          const float2 y1 = __ffma2_rn(make_float2(xt[j + 2], xt[j + 3]), cc, nt);
          a0 = __fadd2_rn(a0, make_float2(ex2(y0.x), ex2(y0.y)));
          a1 = __fadd2_rn(a1, make_float2(ex2(y1.x), ex2(y1.y)));
        }
      }
    }
    if (q_logits) {
      s_t = a0.x + a1.x;
      s_d = a0.y + a1.y;
    } else {
      s_t = (a0.x + a0.y) + (a1.x + a1.y);
    }
  }
  warp_ms(mt, s_t, cl);
  if (q_logits) warp_ms(md, s_d, cl);
  if (lane == 0) { sh.red[0][warp] = mt; sh.red[1][warp] = s_t; sh.red[2][warp] = md; sh.red[3][warp] = s_d; }
  __syncthreads();
  if (warp == 0) {
    float m1 = lane < kFWarps ? sh.red[0][lane] : -INFINITY, s1 = lane < kFWarps ? sh.red[1][lane] : 0.f;
    float m2 = lane < kFWarps ? sh.red[2][lane] : -INFINITY, s2 = lane < kFWarps ? sh.red[3][lane] : 0.f;
    warp_ms(m1, s1, cl);
    if (q_logits) warp_ms(m2, s2, cl);
    if (lane == 0) {
      P.part[((int64_t)b * (K + 1) + i) * P.nc + c] = make_float4(m1, s1, m2, s2);
      __threadfence();
      const unsigned NS = (unsigned)(P.nc * (K + 1));
      sh.last = atom_add_acq_rel(P.seq + (size_t)b * SEQ_WORDS + SEQ_STATS, 1u) == NS - 1;
    }
  }
  __syncthreads();
  if (sh.last) decide<TT, DK>(P, sh, b);
}

// ------------------------------------------------------------ draw item ---

// Group gbase + 32 k (k < kGrp) of chunk c is lane `lane`'s group of block
// k of warp `warp`: element order within a chunk is (warp, block, lane,
// element), i.e. token order.
__device__ __forceinline__ int draw_gbase(int c, int warp, int lane) {
  return c * kChunkGroups + warp * (32 * kGrp) + lane;
}

// weights and totals the draw of sequence b shares between its items
struct DrawRow {
  int n;
  bool has_draft, q_logits, finite;
  float m_p, S_p, m_q, S_q, mcp, mcq, r_pq;
};

__device__ __forceinline__ DrawRow draw_row(const SampleParams &P, int b, int n, int DK) {
  DrawRow d;
  d.n = n;
  d.has_draft = n < P.K;
  d.q_logits = d.has_draft && DK == 0;
  const float4 r = __ldcg(P.rowrec + (int64_t)b * (P.K + 1) + n);
  d.m_p = r.x; d.S_p = r.y; d.m_q = r.z; d.S_q = r.w;
  d.finite = fabsf(d.m_p) <= 3.0e38f && (!d.q_logits || fabsf(d.m_q) <= 3.0e38f) && d.S_p > 0.f;
  d.mcp = __fmul_rn(d.m_p, P.c);
  d.mcq = __fmul_rn(d.m_q, P.c);
  d.r_pq = d.q_logits ? d.S_p / d.S_q : d.S_p;
  return d;
}

// The token of sequence b, found by the last of its draw items: the prefix
// of the chunk totals locates v Z, the per-warp totals of that chunk the
// warp, and one warp reloads that warp's 1024 logits (from L2) to find the
// block, the lane and the element. The draw is certified against its
// rounding bound, or the sequence goes to the float-float kernel.
template <typename TT, int DK>
__device__ __noinline__ void locate(const SampleParams &P, int b, const DrawRow &d) {
  using TD = typename std::conditional<DK == 0, TT, float>::type;
  const int K = P.K, V = P.V, nc = P.nc;
  const int lane = threadIdx.x & 31;
  const float cl = P.c;
  const float *wt = P.wtot + (int64_t)b * nc * kWtStride;
  const float t_r = lane < nc ? __ldcg(wt + lane * kWtStride + kFWarps) : 0.f;
  float Z = 0.f;
  for (int rr = 0; rr < nc; ++rr) Z += __shfl_sync(0xffffffffu, t_r, rr);
  const float v_u = P.uniforms[((int64_t)b * (K + 1) + d.n) * 2 + 1];
  const float thr = v_u * Z;
  float o = 0.f, base = 0.f;
  int own = -1;
  for (int rr = 0; rr < nc; ++rr) {
    const float t = __shfl_sync(0xffffffffu, t_r, rr);
    if (own < 0 && t > 0.f && o <= thr && thr < o + t) { own = rr; base = o; }
    o += t;
  }
  if (!(d.finite && Z > 0.f && own >= 0)) {   // zero mass, non-finite, or rounding
    if (lane == 0) push_pending(P, b, d.n);
    return;
  }
  // the warp of the owner chunk (per-warp totals in order)
  const float wv = lane < kFWarps ? __ldcg(wt + own * kWtStride + lane) : 0.f;
  int ow = kFWarps - 1;
  for (int w = 0; w < kFWarps; ++w) {
    const float t = __shfl_sync(0xffffffffu, wv, w);
    if (thr < base + t || w == kFWarps - 1) { ow = w; break; }
    base += t;
  }
  // that warp's four blocks of 32 groups, from L2
  const TT *trow = static_cast<const TT *>(P.target) + ((int64_t)b * (K + 1) + d.n) * V;
  const TD *drow = d.has_draft ? static_cast<const TD *>(P.draft) + ((int64_t)b * K + d.n) * V : nullptr;
  const int ngr = (V + 7) >> 3;
  const bool vec = P.aligned != 0;
  const int gb = draw_gbase(own, ow, lane);
  Raw8<TT> rt[kGrp];
  Raw8<TD> rd[kGrp];
#pragma unroll
  for (int k = 0; k < kGrp; ++k) {
    const int g = gb + 32 * k;
    if (g < ngr) {
      rt[k] = raw_load(trow, g, V, vec, false);
      if (d.has_draft) rd[k] = raw_load(drow, g, V, vec, DK == 1);
    }
  }
  float ls[kGrp], w8[kGrp][8];
#pragma unroll
  for (int k = 0; k < kGrp; ++k) {
#pragma unroll
    for (int j = 0; j < 8; ++j) w8[k][j] = 0.f;
    if (gb + 32 * k < ngr) draw_weights8<TT, TD, DK>(rt[k], rd[k], d.has_draft, cl, d.mcp, d.mcq, d.r_pq, w8[k]);
    ls[k] = sum8f(w8[k]);
  }
  int ob = kGrp - 1;
  float vs = ls[kGrp - 1];
#pragma unroll
  for (int k = 0; k < kGrp; ++k) {
    const float t = warp_sum_f(ls[k]);
    if (ob == kGrp - 1 && k < kGrp - 1) {
      if (thr < base + t) { ob = k; vs = ls[k]; }
      else base += t;
    }
  }
  // the lane, then the element, within block ob
  const int g = gb + 32 * ob;
  float inc = vs;
#pragma unroll
  for (int s = 1; s < 32; s <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, inc, s);
    if (lane >= s) inc += t;
  }
  const unsigned hit = __ballot_sync(0xffffffffu, g < ngr && base + inc > thr);
  int y = -1;
  float c_lo = 0.f, c_hi = 0.f;
  if (hit) {
    const int L = __ffs(hit) - 1;
    if (lane == L) {
      float run_c = base + (inc - vs);
#pragma unroll
      for (int k = 0; k < kGrp; ++k) {
        if (k != ob) continue;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float nxt = run_c + w8[k][j];
          if (y < 0 && nxt > thr) { y = 8 * g + j; c_lo = run_c; c_hi = nxt; }
          run_c = nxt;
        }
      }
    }
    y = __shfl_sync(0xffffffffu, y, L);
    c_lo = __shfl_sync(0xffffffffu, c_lo, L);
    c_hi = __shfl_sync(0xffffffffu, c_hi, L);
  }
  if (lane == 0) {
    // rounding bound of the fp32 CDF near thr, in units of w' = S_p w:
    // per-element exp / argument / ratio errors (~2^-22 relative, random:
    // sqrt(sum p^2) <= sqrt(max p) = sqrt(1/S)), and the rounding of the
    // running sums (~2^-24 per addition)
    const float e_abs = 4.7683716e-07f * d.S_p * sqrtf(1.f / d.S_p + (d.q_logits ? 1.f / d.S_q : 0.f)) +
                        1.1920929e-07f * (Z + d.S_p);   // 2^-21, 2^-23
    const bool found = y >= 0 && y < V;   // else: rounding moved the crossing
    const float gap = found ? fminf(thr - c_lo, c_hi - thr) : 0.f;
    if (found && gap > e_abs) write_outputs(P, b, d.n, y);
    else push_pending(P, b, d.n);
  }
}

// (chunk c) of sequence b: once the sequence's decisions are out, the chunk
// of the row drawn from (the residual max(0, p - q) of the first rejection,
// or the bonus row) is streamed into registers, its weights summed per warp;
// the last draw item of the sequence locates the token.
template <typename TT, int DK>
__device__ __forceinline__ void draw_item(const SampleParams &P, FusedShared &sh, int b, int c) {
  using TD = typename std::conditional<DK == 0, TT, float>::type;
  const int K = P.K, V = P.V, nc = P.nc;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  unsigned *sq = P.seq + (size_t)b * SEQ_WORDS;
  if (!cta_wait_geq(sq + SEQ_DEC, 1u, &sh.flag)) {
    if (tid == 0) atomic_or_status(P.status, SV_DEV_TIMEOUT);
    return;
  }
  const int2 dec = __ldcg(P.dec + b);
  if (dec.y != DEC_DRAW) return;
  const DrawRow d = draw_row(P, b, dec.x, DK);
  const TT *trow = static_cast<const TT *>(P.target) + ((int64_t)b * (K + 1) + d.n) * V;
  const TD *drow = d.has_draft ? static_cast<const TD *>(P.draft) + ((int64_t)b * K + d.n) * V : nullptr;
  const int ngr = (V + 7) >> 3;
  const bool vec = P.aligned != 0;
  const int gb = draw_gbase(c, warp, lane);
  Raw8<TT> rt[kGrp];
  Raw8<TD> rd[kGrp];
#pragma unroll
  for (int k = 0; k < kGrp; ++k) {
    const int g = gb + 32 * k;
    if (g < ngr) {
      rt[k] = raw_load(trow, g, V, vec, false);
      if (d.has_draft) rd[k] = raw_load(drow, g, V, vec, DK == 1);
    }
  }
#pragma unroll
  for (int k = 0; k < kGrp; ++k) {
    float w[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (gb + 32 * k < ngr) draw_weights8<TT, TD, DK>(rt[k], rd[k], d.has_draft, P.c, d.mcp, d.mcq, d.r_pq, w);
    const float t = warp_sum_f(sum8f(w));
    if (lane == 0) sh.btot[warp][k] = t;
  }
  __syncthreads();
  if (tid == 0) {   // warp totals (blocks in order), then the chunk's
    float *wt = P.wtot + ((int64_t)b * nc + c) * kWtStride;
    float tc = 0.f;
    for (int w = 0; w < kFWarps; ++w) {
      float t = 0.f;
      for (int k = 0; k < kGrp; ++k) t += sh.btot[w][k];
      wt[w] = t;
      tc += t;
    }
    wt[kFWarps] = tc;
    __threadfence();
    sh.last = atom_add_acq_rel(sq + SEQ_DRAW, 1u) == (unsigned)(nc - 1);
  }
  __syncthreads();
  if (sh.last && warp == 0) locate<TT, DK>(P, b, d);
}

// ---------------------------------------------------------------- kernels ---

// Work item of a ticket. Per sequence: NS = nc (K+1) statistics items and
// ND = nc draw items. Tickets run in steps s = 0, 1, ...: step s holds the
// statistics items of sequence s (s < B), then the draw items of sequence
// s - lag (0 <= s - lag < B).
__device__ __forceinline__ void decode_ticket(const SampleParams &P, unsigned t, int &kind, int &b, int &i, int &c) {
  const int nc = P.nc, NS = nc * (P.K + 1), ND = nc, B = P.B, L = P.lag;
  const long long c1 = (long long)min(L, B) * NS;
  const long long c2 = (long long)max(0, B - L) * (NS + ND);
  const long long tt = t;
  kind = -1; b = 0; i = 0; c = 0;
  if (tt < c1) {
    b = (int)(tt / NS);
    const int r = (int)(tt % NS);
    kind = 0; i = r / nc; c = r % nc;
  } else if (tt < c1 + c2) {
    const long long u = tt - c1;
    const int s = L + (int)(u / (NS + ND)), r = (int)(u % (NS + ND));
    if (r < NS) { kind = 0; b = s; i = r / nc; c = r % nc; }
    else { kind = 1; b = s - L; c = r - NS; }
  } else {
    const long long u = tt - c1 - c2;
    b = max(0, B - L) + (int)(u / ND);
    c = (int)(u % ND);
    kind = b < B ? 1 : -1;
  }
}

template <typename TT, int DK>
__global__ void __launch_bounds__(kFThreads, sizeof(TT) == 4 ? 3 : 4) sample_fused_kernel(const __grid_constant__ SampleParams P) {
  __shared__ FusedShared sh;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) {
    int kind, b, i, c;
    decode_ticket(P, atomicAdd(P.sync + SYNC_TICKET, 1u), kind, b, i, c);
    sh.kind = kind; sh.b = b; sh.i = i; sh.c = c;
  }
  __syncthreads();
  const int kind = sh.kind, b = sh.b, i = sh.i, c = sh.c;
  if (kind == 0) stats_item<TT, DK>(P, sh, b, i, c);
  else if (kind == 1) draw_item<TT, DK>(P, sh, b, c);
}

// ------------------------------------------------ float-float kernel -------
// The sequences the fused kernel could not certify, resolved in float-float
// arithmetic by kXGroups groups of nc CTAs (CTA c of a group owns chunk c of
// every row); a group takes pending sequences j = group, group + kXGroups, ...
// For each, from row i0 on:
//   A. float-float sums of e_p and e_q over this CTA's chunk of each row
//      i0 .. j_end (j_end: the first certified rejection at or after i0,
//      else K; the walk cannot pass it) -> group barrier;
//   B. every CTA forms the same row sums and takes the exact accept tests in
//      walk order (certified ones keep their fp32 outcome), which fixes the
//      row n2 drawn from; float-float weights of this chunk of row n2, kept
//      per (warp, block, lane) group in registers -> group barrier;
//   C. every CTA forms the same prefix over chunks; the chunk holding v Z
//      finds the token (warp, block, lane from the totals, then the crossing
//      lane's eight elements in order) and writes the outputs.
// With zero residual mass (reading R9) the draw falls back to p_n2, whose
// chunk sums are those of step A. Group barriers are counters that only
// grow; a CTA waits only for CTAs of its own group.
constexpr int kXGroups = 4;

struct ExactShared {
  unsigned flag;
  float4 rs[kMaxPos];
  int rfl[kMaxPos];
  ff fbt[kFWarps][kGrp];        // float-float block totals
  ff fws[kFWarps];
  ff fred[kFWarps];
  int wlast[kFWarps];
  ff rowS[kMaxPos][2];          // float-float row sums (S_p, S_q)
  ff xz, xthr, xoff;
  int n2, xown, xlast;
  float2 tbl[64];
};

template <typename TT, int DK>
__device__ void exact_sequence(const SampleParams &P, ExactShared &sh, int b, int c, int i0, unsigned *bar,
                               unsigned base) {
  using TD = typename std::conditional<DK == 0, TT, float>::type;
  const int K = P.K, V = P.V, nc = P.nc;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool force = (P.flags & SV_SAMPLE_FORCE_EXACT) != 0;
  const bool vec = P.aligned != 0;
  const FfK fk{P.invT_hi, P.invT_lo, P.log2e_hi, P.log2e_lo, P.unitT};
  const int ngr = (V + 7) >> 3;
  const int gb = draw_gbase(c, warp, lane);
  int j_end = K;
  if (!force)
    for (int j = i0; j < K; ++j)
      if ((sh.rfl[j] & 3) == 2) { j_end = j; break; }

  // ---- A: float-float row sums over this chunk -----------------------------
  for (int j = i0; j <= j_end; ++j) {
    const bool ql = j < K && DK == 0;
    const TT *trow = static_cast<const TT *>(P.target) + ((int64_t)b * (K + 1) + j) * V;
    const TD *drow = ql ? static_cast<const TD *>(P.draft) + ((int64_t)b * K + j) * V : nullptr;
    const float m_p = sh.rs[j].x, m_q = sh.rs[j].z;
    ff sp{0.f, 0.f}, sqs{0.f, 0.f};
#pragma unroll 1
    for (int k = 0; k < kGrp; ++k) {
      const int g = gb + 32 * k;
      if (g >= ngr) continue;
      float x[8];
      unpack8(raw_load(trow, g, V, vec, false), x);
#pragma unroll 1
      for (int e = 0; e < 8; ++e) acc_add(sp, ffx_exp(x[e], m_p, fk, sh.tbl));
      if (ql) {
        unpack8(raw_load(drow, g, V, vec, false), x);
#pragma unroll 1
        for (int e = 0; e < 8; ++e) acc_add(sqs, ffx_exp(x[e], m_q, fk, sh.tbl));
      }
    }
    sp = block_sum_ff(ff_norm(sp), sh.fred);
    sqs = block_sum_ff(ff_norm(sqs), sh.fred);
    if (tid == 0) P.part[((int64_t)b * (K + 1) + j) * nc + c] = make_float4(sp.hi, sp.lo, sqs.hi, sqs.lo);
  }
  cta_arrive(bar);
  if (!cta_wait_geq(bar, base + (unsigned)nc, &sh.flag)) {
    if (tid == 0) atomic_or_status(P.status, SV_DEV_TIMEOUT);
    return;
  }

  // ---- B: row sums, exact walk, float-float weights of the drawn row -------
  for (int j = i0 + warp; j <= j_end; j += kFWarps) {
    const float4 v = lane < nc ? __ldcg(P.part + ((int64_t)b * (K + 1) + j) * nc + lane)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    const ff sp = warp_sum_ff(ff{v.x, v.y}), sqs = warp_sum_ff(ff{v.z, v.w});
    if (lane == 0) {
      sh.rowS[j][0] = sp;
      sh.rowS[j][1] = (j < K && DK == 0) ? sqs : ff{1.f, 0.f};
    }
  }
  __syncthreads();
  if (tid == 0) {
    int n2 = j_end;
    for (int j = i0; j < j_end; ++j) {
      if (!force && (sh.rfl[j] & 2)) continue;   // a certified acceptance (j < j_end)
      // u q(x) < p(x)  <=>  u e_q(x) S_p < e_p(x) S_q   (draft logits)
      //                <=>  u q(x) S_p < e_p(x)         (draft probabilities)
      const int x = min(max(P.tokens[(int64_t)b * K + j], 0), V - 1);
      const float lp_x = to_f32(static_cast<const TT *>(P.target)[((int64_t)b * (K + 1) + j) * V + x]);
      const float lq_x = to_f32(static_cast<const TD *>(P.draft)[((int64_t)b * K + j) * V + x]);
      const float u = P.uniforms[((int64_t)b * (K + 1) + j) * 2];
      const ff Sp = sh.rowS[j][0], Sq = sh.rowS[j][1];
      const ff epx = ff_norm(ffx_exp(lp_x, sh.rs[j].x, fk, sh.tbl));
      ff lhs, rhs;
      if (DK == 0) {
        lhs = ff_mul(ff_mul(ff{u, 0.f}, ff_norm(ffx_exp(lq_x, sh.rs[j].z, fk, sh.tbl))), Sp);
        rhs = ff_mul(epx, Sq);
      } else {
        lhs = ff_mul(ff{u, 0.f}, ff_mul(ff{lq_x, 0.f}, Sp));
        rhs = epx;
      }
      if (!ff_gt(rhs, lhs)) { n2 = j; break; }
    }
    sh.n2 = n2;
  }
  __syncthreads();
  const int n2 = sh.n2;
  const int mode = n2 < K ? (DK == 0 ? 1 : 2) : 0;
  const float m_p = sh.rs[n2].x, m_q = sh.rs[n2].z;
  const ff Sp = sh.rowS[n2][0], Sqn = mode == 1 ? sh.rowS[n2][1] : ff{1.f, 0.f};
  const TT *trow = static_cast<const TT *>(P.target) + ((int64_t)b * (K + 1) + n2) * V;
  const TD *drow = n2 < K ? static_cast<const TD *>(P.draft) + ((int64_t)b * K + n2) * V : nullptr;
  // weights of group g of row n2 in the given mode, summed; last positive index
  auto group_sum = [&](int g, int md, ff &s, int &last) {
    s = ff{0.f, 0.f};
    if (g >= ngr) return;
    float xp[8], xq[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    unpack8(raw_load(trow, g, V, vec, false), xp);
    if (md != 0) unpack8(raw_load(drow, g, V, vec, DK == 1), xq);
#pragma unroll 1
    for (int e = 0; e < 8; ++e) {
      const ff w = resid_weight(md, xp[e], xq[e], m_p, m_q, Sp, Sqn, fk, sh.tbl);
      acc_add(s, w);
      if (w.hi > 0.f) last = 8 * g + e;
    }
    s = ff_norm(s);
  };
  // the chunk's group sums (registers), block and warp totals (shared)
  ff gs[kGrp];
  auto chunk_sums = [&](int md) {
    int last = -1;
#pragma unroll
    for (int k = 0; k < kGrp; ++k) {
      group_sum(gb + 32 * k, md, gs[k], last);
      const ff t = warp_sum_ff(gs[k]);
      if (lane == 0) sh.fbt[warp][k] = t;
    }
    last = warp_max_s32(last);
    if (lane == 0) sh.wlast[warp] = last;
    __syncthreads();
    if (tid == 0) {
      int lc = -1;
      for (int w = 0; w < kFWarps; ++w) {
        ff t{0.f, 0.f};
        for (int k = 0; k < kGrp; ++k) t = ff_add(t, sh.fbt[w][k]);
        sh.fws[w] = t;
        lc = max(lc, sh.wlast[w]);
      }
      sh.xlast = lc;
    }
    __syncthreads();
  };
  chunk_sums(mode);
  if (tid == 0) {
    ff tc{0.f, 0.f};
    for (int w = 0; w < kFWarps; ++w) tc = ff_add(tc, sh.fws[w]);
    P.xtot[(int64_t)b * nc + c] = make_float4(tc.hi, tc.lo, __int_as_float(sh.xlast), 0.f);
  }
  cta_arrive(bar);
  if (!cta_wait_geq(bar, base + 2u * (unsigned)nc, &sh.flag)) {
    if (tid == 0) atomic_or_status(P.status, SV_DEV_TIMEOUT);
    return;
  }

  // ---- C: prefix over chunks (the same bits in every CTA), owner, token ----
  const float v_u = P.uniforms[((int64_t)b * (K + 1) + n2) * 2 + 1];
  // chunk weights: the row's own, or p_n2's (step A's sums) when the residual
  // has no mass
  auto prefix = [&](bool from_p) {
    if (warp == 0) {
      ff tv{0.f, 0.f};
      if (lane < nc) {
        if (from_p) {
          const float4 v = __ldcg(P.part + ((int64_t)b * (K + 1) + n2) * nc + lane);
          tv = ff{v.x, v.y};
        } else {
          const float4 v = __ldcg(P.xtot + (int64_t)b * nc + lane);
          tv = ff{v.x, v.y};
        }
      }
      ff XZ{0.f, 0.f};
      for (int rr = 0; rr < nc; ++rr)
        XZ = ff_add(XZ, ff{__shfl_sync(0xffffffffu, tv.hi, rr), __shfl_sync(0xffffffffu, tv.lo, rr)});
      const ff thr = ff_mul(ff{v_u, 0.f}, XZ);
      ff o{0.f, 0.f}, off{0.f, 0.f};
      int own = -1, lastc = -1;
      for (int rr = 0; rr < nc; ++rr) {
        const ff t{__shfl_sync(0xffffffffu, tv.hi, rr), __shfl_sync(0xffffffffu, tv.lo, rr)};
        if (rr == c) off = o;
        const ff nx = ff_add(o, t);
        if (ff_pos(t)) {
          lastc = rr;
          if (own < 0 && ff_gt(nx, thr)) own = rr;
        }
        o = nx;
      }
      // v Z past the last CDF value through rounding (reading R10): the last
      // chunk with weight, whose search then ends on its last positive token
      if (own < 0) own = lastc;
      if (lane == 0) {
        sh.xz = XZ;
        sh.xthr = thr;
        sh.xoff = off;
        sh.xown = own;
      }
    }
    __syncthreads();
  };
  prefix(false);
  bool from_p = false;
  if (!ff_pos(sh.xz)) {
    if (mode == 0) {   // a bonus row without mass (non-finite logits; flagged): no token
      if (c == 0 && tid == 0) write_outputs(P, b, n2, -1);
      return;
    }
    from_p = true;     // zero residual mass (reading R9): draw from p_n2
    __syncthreads();
    prefix(true);
  }
  const int own = sh.xown;
  if (own < 0) {   // no token carries weight (non-finite logits; flagged)
    if (c == 0 && tid == 0) write_outputs(P, b, n2, -1);
    return;
  }
  if (own != c) return;
  if (from_p) chunk_sums(0);
  const ff thr = sh.xthr;
  ff fb = sh.xoff;
  int ow = kFWarps - 1;
  for (int w = 0; w < kFWarps; ++w) {
    const ff nb = ff_add(fb, sh.fws[w]);
    if (ff_gt(nb, thr) || w == kFWarps - 1) { ow = w; break; }
    fb = nb;
  }
  int ob = kGrp - 1;
  for (int k = 0; k < kGrp; ++k) {
    const ff nb = ff_add(fb, sh.fbt[ow][k]);
    if (ff_gt(nb, thr) || k == kGrp - 1) { ob = k; break; }
    fb = nb;
  }
  if (warp == ow) {
    ff vs{0.f, 0.f};
#pragma unroll
    for (int k = 0; k < kGrp; ++k)
      if (k == ob) vs = gs[k];
    const ff incl = scan32_ff(vs, lane);
    const ff tex{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
    const ff excl = lane == 0 ? ff{0.f, 0.f} : tex;
    const int g = gb + 32 * ob;
    const unsigned hit = __ballot_sync(0xffffffffu, g < ngr && ff_gt(ff_add(fb, incl), thr));
    int y = -1;
    if (hit) {
      const int L = __ffs(hit) - 1;
      if (lane == L) {
        float xp[8], xq[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const int md = from_p ? 0 : mode;
        unpack8(raw_load(trow, g, V, vec, false), xp);
        if (md != 0) unpack8(raw_load(drow, g, V, vec, DK == 1), xq);
        ff run = ff_add(fb, excl);
        int lastp = -1;
        for (int e = 0; e < 8 && y < 0; ++e) {
          const ff w = resid_weight(md, xp[e], xq[e], m_p, m_q, Sp, Sqn, fk, sh.tbl);
          const ff nxt = ff_add(run, w);
          if (w.hi > 0.f) {
            lastp = 8 * g + e;
            if (ff_gt(nxt, thr)) y = 8 * g + e;
          }
          run = nxt;
        }
        if (y < 0) y = lastp;   // the crossing within rounding of this group's end
      }
      y = __shfl_sync(0xffffffffu, y, L);
    }
    if (y < 0) y = sh.xlast;   // ... or of the chunk's
    if (lane == 0) write_outputs(P, b, n2, y);
  }
}

template <typename TT, int DK>
__global__ void __launch_bounds__(kFThreads) sample_exact_kernel(const __grid_constant__ SampleParams P) {
  __shared__ ExactShared sh;
  __shared__ int s_grp, s_c, s_np;
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x < 64) sh.tbl[threadIdx.x] = P.tbl[threadIdx.x];
  if (threadIdx.x == 0) {
    const unsigned t = atomicAdd(P.sync + SYNC_XTICKET, 1u);
    s_grp = (int)(t / (unsigned)P.nc);
    s_c = (int)(t % (unsigned)P.nc);
    s_np = (int)min(__ldcg(P.sync + SYNC_PCOUNT), (unsigned)P.B);
  }
  __syncthreads();
  const int grp = s_grp, c = s_c, np = s_np;
  unsigned *bar = P.sync + SYNC_XBAR + grp;
  unsigned base = 0;
  for (int j = grp; j < np; j += kXGroups) {
    const int2 pe = __ldcg(P.pend + j);
    const int b = pe.x, i0 = pe.y;
    for (int i = threadIdx.x; i <= P.K; i += blockDim.x) {
      sh.rs[i] = __ldcg(P.rowrec + (int64_t)b * (P.K + 1) + i);
      sh.rfl[i] = __ldcg(P.rowflag + (int64_t)b * (P.K + 1) + i);
    }
    __syncthreads();
    exact_sequence<TT, DK>(P, sh, b, c, i0, bar, base);
    base += 2u * (unsigned)P.nc;
    __syncthreads();
  }
}

// Zeroes the call's tickets, pending count, group barriers and per-sequence
// counters once the previous kernel of the stream (which may be an earlier
// call on this workspace) has completed.
__global__ void __launch_bounds__(1024) sample_init_kernel(unsigned *sync, unsigned *seq, int n_words) {
  pdl_trigger();
  pdl_wait();
  for (int j = threadIdx.x; j < n_words; j += blockDim.x) seq[j] = 0u;
  if (threadIdx.x < SYNC_WORDS) sync[threadIdx.x] = 0u;
}

// ------------------------------------------------------------------ host ---

int stat_chunks(int V) { return (V + kChunk - 1) / kChunk; }

size_t parts_bytes(int B, int K, int V) { return align_up((size_t)B * (K + 1) * stat_chunks(V) * sizeof(float4), 256); }
size_t rows_bytes(int B, int K) { return align_up((size_t)B * (K + 1) * (sizeof(float4) + sizeof(int)), 256); }
size_t wtot_bytes(int B, int V) { return align_up((size_t)B * stat_chunks(V) * kWtStride * sizeof(float), 256); }
size_t xtot_bytes(int B, int V) { return align_up((size_t)B * stat_chunks(V) * sizeof(float4), 256); }
size_t small_bytes(int B) {   // decisions, pending list, per-sequence counters, then the call's words
  return align_up((size_t)B * sizeof(int2), 256) * 2 + align_up((size_t)B * SEQ_WORDS * sizeof(unsigned), 256) + 256;
}

size_t workspace_bytes_for(int B, int K, int V) {
  return parts_bytes(B, K, V) + rows_bytes(B, K) + wtot_bytes(B, V) + xtot_bytes(B, V) + small_bytes(B);
}

int sm_count() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
  });
  return n;
}

void split_ff(double d, float &hi, float &lo) {
  hi = (float)d;
  lo = (float)(d - (double)hi);
}

template <typename TT, int DK>
sv_status launch_sample(SampleParams &P, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int per_sm = 0;
  std::call_once(once, [] {
    attr_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sample_fused_kernel<TT, DK>, kFThreads, 0);
  });
  if (attr_err != cudaSuccess)
    return fail(SV_ERR_CUDA, "spec_verify_sample: occupancy query: %s", cudaGetErrorString(attr_err));
  // draw items of a sequence are ticketed after the statistics items of the
  // sequences that fill the GPU's CTA slots once more, so that by the time
  // they run the sequence's decisions are normally out
  const int NS = P.nc * (P.K + 1);
  const long long slots = (long long)sm_count() * std::max(per_sm, 1);
  P.lag = (int)std::min<long long>(P.B, std::max<long long>(1, (slots + NS - 1) / NS + 1));
  cudaError_t e = launch_k(sample_init_kernel, dim3(1), dim3(1024), 0, s, 1, P.sync, P.seq, P.B * SEQ_WORDS);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_sample init launch: %s", cudaGetErrorString(e));
  const long long items = (long long)P.B * (NS + P.nc);
  if (items > 0x7fffffffLL) return fail(SV_ERR_UNSUPPORTED, "spec_verify_sample: %lld work items", items);
  e = launch_k(sample_fused_kernel<TT, DK>, dim3((unsigned)items), dim3(kFThreads), 0, s, 1, P);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_sample launch: %s", cudaGetErrorString(e));
  e = launch_k(sample_exact_kernel<TT, DK>, dim3(kXGroups * P.nc), dim3(kFThreads), 0, s, 1, P);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_sample float-float launch: %s", cudaGetErrorString(e));
  return ok();
}

// Host checks of spec_verify_sample's arguments (everything but the workspace).
sv_status check_sample_args(const void *target_logits, sv_dtype logit_dtype, const void *draft,
                            sv_dtype draft_dtype, int draft_is_probs, const int32_t *draft_tokens,
                            const float *uniforms, int B, int K, int V, float temperature,
                            const int32_t *out_tokens, const int32_t *num_accepted) {
  if (B < 0 || K < 0 || V < 1)
    return fail(SV_ERR_INVALID_ARG, "spec_verify_sample: bad sizes B=%d K=%d V=%d", B, K, V);
  if (B > 65535 || K + 1 > kMaxPos)
    return fail(SV_ERR_UNSUPPORTED, "spec_verify_sample: B must be <= 65535 and K + 1 <= %d", kMaxPos);
  if (V > kMaxChunks * kChunk)
    return fail(SV_ERR_UNSUPPORTED, "spec_verify_sample: vocabulary of %d too large (at most %d)", V,
                kMaxChunks * kChunk);
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
  return SV_OK;
}

}  // namespace
}  // namespace sv

extern "C" size_t spec_verify_sample_workspace_size(int B, int K, int V) {
  if (B < 0 || K < 0 || V < 1) return 0;
  return sv::workspace_bytes_for(B, K, V);
}

extern "C" sv_status spec_verify_sample_ex(const void *target_logits, sv_dtype logit_dtype,
                                           const void *draft, sv_dtype draft_dtype, int draft_is_probs,
                                           const int32_t *draft_tokens, const float *uniforms, int B,
                                           int K, int V, float temperature, int32_t *out_tokens,
                                           int32_t *num_accepted, float *p_at_draft, float *q_at_draft,
                                           void *workspace, size_t workspace_bytes,
                                           int32_t *dev_status, unsigned flags, sv_stream_t stream) {
  using namespace sv;
  {
    const sv_status st = check_sample_args(target_logits, logit_dtype, draft, draft_dtype, draft_is_probs,
                                           draft_tokens, uniforms, B, K, V, temperature, out_tokens, num_accepted);
    if (st != SV_OK) return st;
  }
  if (!workspace || workspace_bytes < workspace_bytes_for(B, K, V))
    return fail(SV_ERR_WORKSPACE, "spec_verify_sample: workspace needs %zu bytes", workspace_bytes_for(B, K, V));
  if (!aligned(workspace, 256)) return fail(SV_ERR_WORKSPACE, "spec_verify_sample: workspace not 256-byte aligned");
  if (B == 0) return ok();

  const int es_t = dtype_bytes(logit_dtype);
  const int es_buf_d = (draft_is_probs && K > 0) ? 4 : es_t;

  SampleParams P = {};
  P.target = target_logits; P.draft = draft; P.tokens = draft_tokens; P.uniforms = uniforms;
  P.p_at = p_at_draft; P.q_at = q_at_draft; P.out_tokens = out_tokens; P.num_acc = num_accepted;
  P.status = dev_status;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  P.part = reinterpret_cast<float4 *>(ws);
  ws += parts_bytes(B, K, V);
  P.rowrec = reinterpret_cast<float4 *>(ws);
  P.rowflag = reinterpret_cast<int *>(ws + (size_t)B * (K + 1) * sizeof(float4));
  ws += rows_bytes(B, K);
  P.wtot = reinterpret_cast<float *>(ws);
  ws += wtot_bytes(B, V);
  P.xtot = reinterpret_cast<float4 *>(ws);
  ws += xtot_bytes(B, V);
  P.dec = reinterpret_cast<int2 *>(ws);
  ws += align_up((size_t)B * sizeof(int2), 256);
  P.pend = reinterpret_cast<int2 *>(ws);
  ws += align_up((size_t)B * sizeof(int2), 256);
  P.seq = reinterpret_cast<unsigned *>(ws);
  ws += align_up((size_t)B * SEQ_WORDS * sizeof(unsigned), 256);
  P.sync = reinterpret_cast<unsigned *>(ws);
  P.nc = stat_chunks(V);
  P.B = B; P.K = K; P.V = V; P.flags = flags;
  P.aligned = aligned(target_logits, 16) && ((size_t)V * es_t) % 16 == 0 &&
              (K == 0 || (aligned(draft, 16) && ((size_t)V * es_buf_d) % 16 == 0));
  const double log2e = 1.4426950408889634074;
  P.c = (float)(log2e / (double)temperature);
  P.unitT = temperature == 1.0f;
  split_ff(1.0 / (double)temperature, P.invT_hi, P.invT_lo);
  split_ff(log2e, P.log2e_hi, P.log2e_lo);
  for (int j = 0; j < 64; ++j) split_ff(std::exp2((double)j / 64.0), P.tbl[j].x, P.tbl[j].y);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool probs = draft_is_probs && K > 0;
  switch (logit_dtype) {
    case SV_F32: return probs ? launch_sample<float, 1>(P, s) : launch_sample<float, 0>(P, s);
    case SV_BF16: return probs ? launch_sample<__nv_bfloat16, 1>(P, s) : launch_sample<__nv_bfloat16, 0>(P, s);
    default: return probs ? launch_sample<__half, 1>(P, s) : launch_sample<__half, 0>(P, s);
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

// ------------------------------------------------------------- top-p ---
// The target rows (and, on request, the draft logit rows) go through the
// top-p filter into the front of the workspace; the sampling kernels then
// read the filtered rows. The statistics kernel waits for the filter before
// its first load.
namespace {
size_t topp_rows_bytes(int B, int K, int V, sv_dtype dt, int draft_topp) {
  const size_t es = (size_t)sv::dtype_bytes(dt);
  size_t n = sv::align_up((size_t)B * (K + 1) * V * es, 256);
  if (draft_topp && K > 0) n += sv::align_up((size_t)B * K * V * es, 256);
  return n;
}
}  // namespace

extern "C" size_t spec_verify_sample_topp_workspace_size(int B, int K, int V, sv_dtype logit_dtype,
                                                         int draft_topp) {
  if (B < 0 || K < 0 || V < 1) return 0;
  if (logit_dtype != SV_F32 && logit_dtype != SV_BF16 && logit_dtype != SV_F16) return 0;
  return topp_rows_bytes(B, K, V, logit_dtype, draft_topp) + sv::workspace_bytes_for(B, K, V);
}

extern "C" sv_status spec_verify_sample_topp(const void *target_logits, sv_dtype logit_dtype, const void *draft,
                                             sv_dtype draft_dtype, int draft_is_probs,
                                             const int32_t *draft_tokens, const float *uniforms, int B, int K,
                                             int V, float temperature, float top_p, int draft_topp,
                                             int32_t *out_tokens, int32_t *num_accepted, float *p_at_draft,
                                             float *q_at_draft, void *workspace, size_t workspace_bytes,
                                             int32_t *dev_status, sv_stream_t stream) {
  using namespace sv;
  if (!(top_p > 0.f) || !(top_p <= 1.f))
    return fail(SV_ERR_INVALID_ARG, "spec_verify_sample_topp: top_p must be in (0, 1]");
  if (draft_topp && draft_is_probs)
    return fail(SV_ERR_INVALID_ARG, "spec_verify_sample_topp: draft_topp needs draft logits, not probabilities");
  if (top_p >= 1.f)
    return spec_verify_sample_ex(target_logits, logit_dtype, draft, draft_dtype, draft_is_probs, draft_tokens,
                                 uniforms, B, K, V, temperature, out_tokens, num_accepted, p_at_draft, q_at_draft,
                                 workspace, workspace_bytes, dev_status, 0u, stream);
  {
    const sv_status st = check_sample_args(target_logits, logit_dtype, draft, draft_dtype, draft_is_probs,
                                           draft_tokens, uniforms, B, K, V, temperature, out_tokens, num_accepted);
    if (st != SV_OK) return st;
  }
  if (V > (1 << 28)) return fail(SV_ERR_UNSUPPORTED, "spec_verify_sample_topp: V = %d above 2^28", V);
  const size_t front = topp_rows_bytes(B, K, V, logit_dtype, draft_topp);
  const size_t need = front + workspace_bytes_for(B, K, V);
  if (!workspace || workspace_bytes < need)
    return fail(SV_ERR_WORKSPACE, "spec_verify_sample_topp: workspace needs %zu bytes", need);
  if (!aligned(workspace, 256)) return fail(SV_ERR_WORKSPACE, "spec_verify_sample_topp: workspace not 256-byte aligned");
  if (B == 0) return ok();
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  const size_t es = (size_t)dtype_bytes(logit_dtype);
  void *ft = ws;
  void *fd = (draft_topp && K > 0) ? ws + align_up((size_t)B * (K + 1) * V * es, 256) : nullptr;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const sv_status st = launch_topp_filter(logit_dtype, target_logits, ft, B * (K + 1), draft, fd,
                                          fd ? B * K : 0, V, temperature, top_p, dev_status, s);
  if (st != SV_OK) return st;
  return spec_verify_sample_ex(ft, logit_dtype, fd ? fd : draft, draft_dtype, draft_is_probs, draft_tokens, uniforms,
                               B, K, V, temperature, out_tokens, num_accepted, p_at_draft, q_at_draft, ws + front,
                               workspace_bytes - front, dev_status, 0u, stream);
}

// ------------------------------------------------- allocation-free entry ---
// Some callers cannot allocate device memory when they verify a round: for
// example an engine that reserves all of the GPU's memory for its KV pool at
// start-up and forbids allocations afterwards, or a caller whose fixed C
// interface has no way to pass a workspace. For them the records live in
// this static device array (every GPU that loads the library keeps it until
// the process exits).
namespace {
constexpr size_t kStaticScratchBytes = 1u << 20;   // 1 MiB
__device__ __align__(256) uint8_t g_sample_scratch[kStaticScratchBytes];
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
// the array's device address per device, and the id of the context it was
// resolved in: a context that was destroyed and created again (after a
// cudaDeviceReset, say) loads the module anew, possibly at another address
struct ScratchAddr {
  unsigned long long ctx_id;
  void *ptr;
};
ScratchAddr g_scratch[kMaxDevices] = {};

typedef int (*PfnCtxGetCurrent)(void **ctx);
typedef int (*PfnCtxGetId)(void *ctx, unsigned long long *id);

// id of the calling thread's current context (0 if the driver cannot say, in
// which case the address is resolved again on every call)
unsigned long long current_ctx_id() {
  static PfnCtxGetCurrent get_cur = nullptr;
  static PfnCtxGetId get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_cur = reinterpret_cast<PfnCtxGetCurrent>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PfnCtxGetId>(p);
  });
  void *ctx = nullptr;
  unsigned long long id = 0;
  if (!get_cur || !get_id || get_cur(&ctx) != 0 || !ctx || get_id(ctx, &id) != 0) return 0;
  return id;
}
}  // namespace

extern "C" sv_status spec_verify_sample_static(const void *target_logits, sv_dtype logit_dtype,
                                               const void *draft, sv_dtype draft_dtype, int draft_is_probs,
                                               const int32_t *draft_tokens, const float *uniforms, int B, int K,
                                               int V, float temperature, int32_t *out_tokens,
                                               int32_t *num_accepted, float *p_at_draft, float *q_at_draft,
                                               int32_t *dev_status, sv_stream_t stream) {
  using namespace sv;
  if (B < 0 || K < 0 || V < 1)
    return fail(SV_ERR_INVALID_ARG, "spec_verify_sample_static: bad sizes B=%d K=%d V=%d", B, K, V);
  const size_t need = workspace_bytes_for(B, K, V);
  if (need > kStaticScratchBytes)
    return fail(SV_ERR_UNSUPPORTED,
                "spec_verify_sample_static: B = %d sequences of %d rows need %zu bytes (%d 16-byte chunk "
                "statistics per row and per sequence, 16 bytes per sequence), more than the static scratch "
                "of %zu bytes; use spec_verify_sample with a caller workspace",
                B, K + 1, need, stat_chunks(V), kStaticScratchBytes);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_sample_static: cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(SV_ERR_UNSUPPORTED, "spec_verify_sample_static: device %d", dev);
  void *ptr = nullptr;
  {
    // first call on a device (or in a new context of it): resolve the array's
    // device address, with that device current
    const unsigned long long ctx = current_ctx_id();
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch[dev].ptr || ctx == 0 || g_scratch[dev].ctx_id != ctx) {
      void *addr = nullptr;
      e = cudaGetSymbolAddress(&addr, g_sample_scratch);
      if (e != cudaSuccess) {
        g_scratch[dev] = ScratchAddr{0ull, nullptr};
        return fail(SV_ERR_CUDA, "spec_verify_sample_static: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
      }
      g_scratch[dev] = ScratchAddr{ctx, addr};
    }
    ptr = g_scratch[dev].ptr;
  }
  return spec_verify_sample(target_logits, logit_dtype, draft, draft_dtype, draft_is_probs, draft_tokens,
                            uniforms, B, K, V, temperature, out_tokens, num_accepted, p_at_draft, q_at_draft, ptr,
                            kStaticScratchBytes, dev_status, stream);
}

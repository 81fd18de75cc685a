// spec_verify_sample: the fused rejection-sampling pass of the verify step.
//
// What is computed (quant67 "speculative decoding" section 3.1; "KV Cache +
// Speculative Decoding" sections 7.1-7.3 and 7.6): per sequence b and draft
// position i, p_i = softmax(target_i / T), q_i = softmax(draft_i / T) (or the
// given q_i); x_i is accepted iff u_i q_i(x_i) < p_i(x_i); at the first
// rejection n the token is drawn by inverse CDF (ascending token id, strict
// '>') from max(0, p_n - q_n); if all K are accepted it is drawn from p_K.
//
// GB300 design (three launches, no host round trip):
//   * sample_stats_kernel: a streaming reduction. One CTA per (8192-logit
//     chunk, position, sequence) loads its chunk of the target row and of
//     the draft row with 16-byte loads straight into registers, takes exact
//     maxima and fp32 sums of exponentials (target and draft paired in
//     packed fp32 arithmetic) and writes one (max, sum) pair per row; every
//     logit crosses HBM once.
//   * sample_draw_kernel: one cluster per sequence combines the chunk
//     statistics, evaluates every accept test in fp32 with a certificate
//     that it lies outside its rounding bound, and finds the position whose
//     draw is used (the first certified rejection, or the bonus row). Only
//     that row is read again; its residual weights are formed over the
//     cluster's shared-memory slices and the inverse-CDF draw gets its own
//     certificate. One 48-byte record per (sequence, position) results.
//   * sample_finish_kernel: a few clusters walk each sequence's records in
//     order, stop at the first rejection and write the emitted tokens. The
//     rare decision that is not certified (a few percent of sequences) is
//     re-evaluated from that row's logits in float-float arithmetic (~1e-9
//     relative error per term), so emitted tokens are those of exact
//     arithmetic except for uniforms within ~1e-10 of a boundary.
#include <cmath>
#include <algorithm>
#include <mutex>
#include <type_traits>

#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kRowThreads = 256;
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kResThreads = 512;   // finish kernel
constexpr int kResWarps = kResThreads / 32;
constexpr uint32_t kChunkBytes = 16384;
constexpr int kMaxChunks = 32;              // per CTA, target + draft
constexpr size_t kMaxSliceSmem = 200 * 1024;
constexpr size_t kTargetSliceSmem = 64 * 1024;
constexpr int kFinishClusters = 8;

enum : uint32_t {
  REC_ACCEPT = 1u,       // fp32 accept decision of the draft at this position
  REC_ACC_CERT = 2u,     // ... certified: outside the rounding bound
  REC_DRAW_CERT = 4u,    // the fp32 draw was found and certified
  REC_EXACT_ACC = 8u,    // set by the finish kernel: accept re-evaluated in float-float
  REC_EXACT_DRAW = 16u,  // set by the finish kernel: draw re-evaluated in float-float
};

struct RowRec {
  float m_p, s_p, m_q, s_q;  // row max and sum of exp2((l - m) c) (fp32)
  float p_x, q_x;            // p_i(x_i), q_i(x_i) in fp32
  float gap, z;              // margin of the fp32 draw and the mass it was drawn from
  int32_t y;                 // fp32 draw of this row (-1 if not found)
  uint32_t flags;            // REC_*
  int32_t y_exact;           // float-float draw (finish kernel; -1 if not evaluated)
  float e_abs;               // rounding bound the fp32 margin was compared with
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
  float4 *part;  // [B][K+1][nc] (max, sum) of the target and draft chunks
  int32_t *status;
  int B, K, V;
  int nc;        // statistics chunks per row
  int ns;        // elements per CTA slice of the draw kernel (multiple of 8)
  int ns_x;      // elements per CTA slice in the finish kernel
  int aligned;   // rows are 16-byte aligned: bulk copies usable
  int cache_x;   // finish kernel keeps the float-float exponentials in shared memory
  unsigned flags;
  float c;       // log2(e) / T
  float invT_hi, invT_lo;
  int unitT;
  float log2e_hi, log2e_lo, ln2_hi, ln2_lo;
  float2 tbl[64];  // 2^(j/64) split into (hi, lo)
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

// (m, s) pairs of an online softmax: s = sum 2^(fl(x c - fl(m c))). Every
// exponent is taken against the rounded reference fl(m c), the same one the
// weights of pass B use, so sums and weights share one scale. Commutative,
// so butterfly reductions leave the same bits in every lane.
__device__ __forceinline__ void ms_combine(float &m, float &s, float m2, float s2, float c) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) { m = mn; s = 0.f; return; }
  // __fmul_rn: the references must be the rounded products, never fused
  // into an fma (a fused m c - fl(m c) would rescale the leading partial by
  // its rounding residual at every reduction level)
  const float rc = __fmul_rn(mn, c);
  s = s * ex2(__fmul_rn(m, c) - rc) + s2 * ex2(__fmul_rn(m2, c) - rc);
  m = mn;
}


// Warp-wide combination of (m, s) pairs: the maximum first, then every lane
// rescales its own sum to it (one ex2), then a plain sum. Butterfly
// reductions leave identical bits in every lane.
__device__ __forceinline__ void warp_ms_fast(float &m, float &s, float c) {
  const float mx = warp_max(m);
  s = (m == -INFINITY) ? 0.f : s * ex2(__fmul_rn(m, c) - __fmul_rn(mx, c));
  s = warp_sum(s);
  m = mx;
}

template <typename T>
__device__ __forceinline__ void online8(const T *buf, int g, float c, float &m, float &s) {
  float x[8];
  load8(buf, g, x);
  float mx = fmaxf(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])), fmaxf(fmaxf(x[4], x[5]), fmaxf(x[6], x[7])));
  if (mx > m) {
    s = (m == -INFINITY) ? 0.f : s * ex2(__fmul_rn(m, c) - __fmul_rn(mx, c));
    m = mx;
  }
  if (m == -INFINITY) return;
  const float mc = __fmul_rn(m, c);
#pragma unroll
  for (int j = 0; j < 8; ++j) s += ex2(fmaf(x[j], c, -mc));
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

__device__ __forceinline__ ff ld_dsmem_ff(const ff *p, int rank) {
  const uint32_t a = mapa(p, rank);
  return ff{ld_dsmem_f32(a), ld_dsmem_f32(a + 4)};
}

__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
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

// Thread-local maximum over groups g0, g0 + stride, ... of a slice. A maximum
// is a selection, so the packed 16-bit forms are exact.
template <typename T>
__device__ __forceinline__ float slice_max(const T *buf, int g0, int n_grp, int stride);

template <>
__device__ __forceinline__ float slice_max<float>(const float *buf, int g0, int n_grp, int stride) {
  float r0 = -INFINITY, r1 = -INFINITY;
  const float4 *p = reinterpret_cast<const float4 *>(buf);
  for (int g = g0; g < n_grp; g += stride) {
    const float4 a = p[2 * g], b = p[2 * g + 1];
    r0 = max3f(r0, a.x, a.y);
    r1 = max3f(r1, a.z, a.w);
    r0 = max3f(r0, b.x, b.y);
    r1 = max3f(r1, b.z, b.w);
  }
  return fmaxf(r0, r1);
}

template <typename H2>
__device__ __forceinline__ H2 as_h2(uint32_t w) {
  H2 h;
  memcpy(&h, &w, 4);
  return h;
}

template <>
__device__ __forceinline__ float slice_max<__nv_bfloat16>(const __nv_bfloat16 *buf, int g0, int n_grp, int stride) {
  const __nv_bfloat162 ninf = __floats2bfloat162_rn(-INFINITY, -INFINITY);
  __nv_bfloat162 r0 = ninf, r1 = ninf;
  const uint4 *p = reinterpret_cast<const uint4 *>(buf);
  for (int g = g0; g < n_grp; g += stride) {
    const uint4 v = p[g];
    r0 = __hmax2(r0, as_h2<__nv_bfloat162>(v.x));
    r1 = __hmax2(r1, as_h2<__nv_bfloat162>(v.y));
    r0 = __hmax2(r0, as_h2<__nv_bfloat162>(v.z));
    r1 = __hmax2(r1, as_h2<__nv_bfloat162>(v.w));
  }
  r0 = __hmax2(r0, r1);
  return fmaxf(__low2float(r0), __high2float(r0));
}

template <>
__device__ __forceinline__ float slice_max<__half>(const __half *buf, int g0, int n_grp, int stride) {
  const __half2 ninf = __floats2half2_rn(-INFINITY, -INFINITY);
  __half2 r0 = ninf, r1 = ninf;
  const uint4 *p = reinterpret_cast<const uint4 *>(buf);
  for (int g = g0; g < n_grp; g += stride) {
    const uint4 v = p[g];
    r0 = __hmax2(r0, as_h2<__half2>(v.x));
    r1 = __hmax2(r1, as_h2<__half2>(v.y));
    r0 = __hmax2(r0, as_h2<__half2>(v.z));
    r1 = __hmax2(r1, as_h2<__half2>(v.w));
  }
  r0 = __hmax2(r0, r1);
  return fmaxf(__low2float(r0), __high2float(r0));
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

// ------------------------------------------------------ statistics pass ---
// sample_stats_kernel: one CTA per (8192-logit chunk, position, sequence).
// Each thread holds 32 logits of the target row and of the draft row in
// registers (16-byte loads, all issued before any arithmetic), takes exact
// maxima, then sums of 2^(l c - fl(m c)) with the two rows paired in packed
// fp32 arithmetic; the CTA's (max, sum) pairs go to the workspace. No
// shared-memory staging and no cluster: a streaming reduction.
constexpr int kStatThreads = 256;
constexpr int kStatChunk = 8192;                               // logits per CTA per row
constexpr int kStatGroups = kStatChunk / (8 * kStatThreads);   // groups of 8 per thread

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

template <typename TT, int DK>
__global__ void __launch_bounds__(kStatThreads) sample_stats_kernel(const __grid_constant__ SampleParams P) {
  pdl_wait();
  pdl_trigger();
  using TD = typename std::conditional<DK == 0, TT, float>::type;
  __shared__ float red[4][kStatThreads / 32];
  const int c = blockIdx.x, i = blockIdx.y, b = blockIdx.z;
  const int K = P.K, V = P.V;
  const bool q_logits = i < K && DK == 0;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float cl = P.c;
  const TT *trow = static_cast<const TT *>(P.target) + ((int64_t)b * (K + 1) + i) * V;
  const TD *drow = q_logits ? static_cast<const TD *>(P.draft) + ((int64_t)b * K + i) * V : nullptr;
  const int e0 = c * kStatChunk, e1 = min(V, e0 + kStatChunk);
  const int g0 = e0 / 8, g1 = (e1 + 7) / 8;
  const bool vec = P.aligned != 0;

  Raw8<TT> rt[kStatGroups];
  Raw8<TD> rd[kStatGroups];
#pragma unroll
  for (int k = 0; k < kStatGroups; ++k) {
    const int g = g0 + tid + k * kStatThreads;
    if (g < g1) {
      rt[k] = raw_load(trow, g, e1, vec, false);
      if (q_logits) rd[k] = raw_load(drow, g, e1, vec, false);
    }
  }
  float mt = -INFINITY, md = -INFINITY;
#pragma unroll
  for (int k = 0; k < kStatGroups; ++k) {
    if (g0 + tid + k * kStatThreads < g1) {
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
    for (int k = 0; k < kStatGroups; ++k) {
      if (g0 + tid + k * kStatThreads >= g1) continue;
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
  if (lane == 0) { red[0][warp] = mt; red[1][warp] = s_t; red[2][warp] = md; red[3][warp] = s_d; }
  __syncthreads();
  if (warp == 0) {
    constexpr int nw = kStatThreads / 32;
    float m1 = lane < nw ? red[0][lane] : -INFINITY, s1 = lane < nw ? red[1][lane] : 0.f;
    float m2 = lane < nw ? red[2][lane] : -INFINITY, s2 = lane < nw ? red[3][lane] : 0.f;
    warp_ms(m1, s1, cl);
    if (q_logits) warp_ms(m2, s2, cl);
    if (lane == 0) P.part[((int64_t)b * (K + 1) + i) * P.nc + c] = make_float4(m1, s1, m2, s2);
  }
}

// ------------------------------------------------- decide and draw pass ---
// sample_draw_kernel: one cluster per sequence. Every CTA combines the chunk
// statistics of each row (lanes over chunks, the same order everywhere, so
// every CTA holds the same bits) and the accept tests are evaluated in fp32
// with their rounding certificates; CTA 0 writes every row's record. The
// first position that rejects (or whose test is not certified) stops the
// walk; only the row drawn from is read again: the residual of the first
// certified rejection, or the bonus row when every draft is accepted. Its
// weights w'(y) = max(0, e_p(y) - r e_q(y)) are formed over the cluster's
// slices, one warp scan of lane totals and the cluster's prefix locate v Z,
// and the draw gets its own certificate. Anything uncertified is left to
// the finish kernel.
struct DrawShared {
  uint64_t bar;
  int stop;               // 2 * position + (0: not certified, 1: certified rejection)
  float row_m_p, row_s_p, row_m_q, row_s_q;
  float pub_tot;          // this CTA's draw mass
  float wsum[kRowWarps];
};

// combined (max, sum) of target (and draft) row i of sequence b: every lane
// of the warp ends with the same bits
__device__ __forceinline__ void row_stats(const SampleParams &P, int b, int i, bool q_logits, float &m_p, float &S_p,
                                          float &m_q, float &S_q) {
  const int lane = threadIdx.x & 31;
  const float4 *pr = P.part + ((int64_t)b * (P.K + 1) + i) * P.nc;
  m_p = -INFINITY; S_p = 0.f; m_q = -INFINITY; S_q = 0.f;
  for (int c0 = 0; c0 < P.nc; c0 += 32) {
    float a = -INFINITY, sa = 0.f, d = -INFINITY, sd = 0.f;
    if (c0 + lane < P.nc) {
      const float4 v = pr[c0 + lane];
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

template <typename TT, int DK>
__global__ void __launch_bounds__(kRowThreads) sample_draw_kernel(const __grid_constant__ SampleParams P) {
  pdl_wait();
  pdl_trigger();
  using TD = typename std::conditional<DK == 0, TT, float>::type;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ DrawShared sh;

  const int cs = (int)cluster_nctarank(), rank = (int)cluster_ctarank();
  const int b = blockIdx.y;
  const int K = P.K, V = P.V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float c = P.c;
  const bool force = (P.flags & SV_SAMPLE_FORCE_EXACT) != 0;
  if (tid == 0) sh.stop = 2 * K + 1;
  __syncthreads();

  // ---- accept tests of every draft position --------------------------------
  for (int i = warp; i < K; i += kRowWarps) {
    float m_p, S_p, m_q, S_q;
    row_stats(P, b, i, DK == 0, m_p, S_p, m_q, S_q);
    if (DK != 0) { m_q = 0.f; S_q = 1.f; }
    int x = P.tokens[(int64_t)b * K + i];
    if (x < 0 || x >= V) {
      if (rank == 0 && lane == 0) atomic_or_status(P.status, SV_DEV_BAD_TOKEN);
      x = min(max(x, 0), V - 1);
    }
    const float lp_x = to_f32(static_cast<const TT *>(P.target)[((int64_t)b * (K + 1) + i) * V + x]);
    const float lq_x = to_f32(static_cast<const TD *>(P.draft)[((int64_t)b * K + i) * V + x]);
    const float u = P.uniforms[((int64_t)b * (K + 1) + i) * 2];
    const bool finite = fabsf(m_p) <= 3.0e38f && (DK != 0 || fabsf(m_q) <= 3.0e38f) && S_p > 0.f;
    const float mcp = __fmul_rn(m_p, c), mcq = __fmul_rn(m_q, c);
    const float p_x = ex2(fmaf(lp_x, c, -mcp)) / S_p;
    const float q_x = DK == 0 ? ex2(fmaf(lq_x, c, -mcq)) / S_q : lq_x;
    const float lhs = u * q_x;
    const bool accept = lhs < p_x;
    // p_x and u q_x each carry < 2e-6 relative rounding (exp2, argument
    // rounding, row sums): a decision this far from the boundary is exact
    const bool acc_cert = fabsf(p_x - lhs) > 4e-6f * fmaxf(p_x, lhs) && p_x > 0.f && q_x > 0.f && finite;
    if (lane == 0) {
      if (!acc_cert) atomicMin(&sh.stop, 2 * i);
      else if (!accept) atomicMin(&sh.stop, 2 * i + 1);
      if (rank == 0) {
        RowRec *rec = P.recs + (int64_t)b * (K + 1) + i;
        if (!finite) atomic_or_status(P.status, SV_DEV_NONFINITE);
        rec->m_p = m_p; rec->s_p = S_p; rec->m_q = m_q; rec->s_q = S_q;
        rec->p_x = p_x; rec->q_x = q_x;
        rec->y = -1; rec->y_exact = -1; rec->gap = 0.f; rec->z = 0.f; rec->e_abs = 0.f;
        rec->flags = (accept ? REC_ACCEPT : 0u) | (acc_cert ? REC_ACC_CERT : 0u);
        if (P.p_at) P.p_at[(int64_t)b * K + i] = p_x;
        if (P.q_at) P.q_at[(int64_t)b * K + i] = q_x;
      }
    }
  }
  __syncthreads();
  const int stop = sh.stop;
  // the row drawn from: a certified rejection, or the bonus row (K)
  const bool certain = (stop & 1) != 0;
  const int n = stop >> 1;
  const bool has_draft = n < K;
  const bool q_logits = has_draft && DK == 0;
  if (warp == 0 && certain) {   // statistics of the row drawn from
    float m_p, S_p, m_q, S_q;
    row_stats(P, b, n, q_logits, m_p, S_p, m_q, S_q);
    if (!q_logits) { m_q = 0.f; S_q = 1.f; }
    if (lane == 0) { sh.row_m_p = m_p; sh.row_s_p = S_p; sh.row_m_q = m_q; sh.row_s_q = S_q; }
  }
  if (warp == 1 && rank == 0) {
    // the bonus row's record (the finish kernel may walk to it)
    float m_p, S_p, m_q, S_q;
    row_stats(P, b, K, false, m_p, S_p, m_q, S_q);
    if (lane == 0) {
      RowRec *rec = P.recs + (int64_t)b * (K + 1) + K;
      rec->m_p = m_p; rec->s_p = S_p; rec->m_q = 0.f; rec->s_q = 1.f;
      rec->p_x = 0.f; rec->q_x = 0.f;
      rec->y = -1; rec->y_exact = -1; rec->gap = 0.f; rec->z = 0.f; rec->e_abs = 0.f;
      rec->flags = 0u;
      if (!(fabsf(m_p) <= 3.0e38f && S_p > 0.f)) atomic_or_status(P.status, SV_DEV_NONFINITE);
    }
  }
  __syncthreads();
  // identical in every CTA of the cluster: no shared memory of a peer is
  // read on this path
  if (!certain || force) return;
  const float m_p = sh.row_m_p, S_p = sh.row_s_p, m_q = sh.row_m_q, S_q = sh.row_s_q;
  const bool finite = fabsf(m_p) <= 3.0e38f && (!q_logits || fabsf(m_q) <= 3.0e38f) && S_p > 0.f;

  // ---- the draw: slices of row n -------------------------------------------
  const TT *trow = static_cast<const TT *>(P.target) + ((int64_t)b * (K + 1) + n) * V;
  const TD *drow = has_draft ? static_cast<const TD *>(P.draft) + ((int64_t)b * K + n) * V : nullptr;
  const int e0 = rank * P.ns;
  const int n_loc = max(0, min(V, e0 + P.ns) - e0);
  const int n_grp = (n_loc + 7) >> 3;
  TT *st = reinterpret_cast<TT *>(smem);
  TD *sd = reinterpret_cast<TD *>(smem + align_up((size_t)P.ns * sizeof(TT), 128));
  for (int e = n_loc + tid; e < n_grp * 8; e += kRowThreads) {   // pad the last group
    st[e] = pad_value<TT>(false);
    if (has_draft) sd[e] = pad_value<TD>(DK == 1);
  }
  bool timed_out = false;
  if (P.aligned) {
    if (tid == 0) {
      mbar_init(&sh.bar, 1);
      fence_mbarrier_init();
      const uint32_t nb_t = (uint32_t)n_loc * sizeof(TT), nb_d = has_draft ? (uint32_t)n_loc * sizeof(TD) : 0u;
      mbar_arrive_expect_tx(&sh.bar, nb_t + nb_d);
      const uint8_t *gt = reinterpret_cast<const uint8_t *>(trow + e0);
      for (uint32_t off = 0; off < nb_t; off += kChunkBytes)
        bulk_g2s(reinterpret_cast<uint8_t *>(st) + off, gt + off, min(kChunkBytes, nb_t - off), &sh.bar);
      if (has_draft) {
        const uint8_t *gd = reinterpret_cast<const uint8_t *>(drow + e0);
        for (uint32_t off = 0; off < nb_d; off += kChunkBytes)
          bulk_g2s(reinterpret_cast<uint8_t *>(sd) + off, gd + off, min(kChunkBytes, nb_d - off), &sh.bar);
      }
    }
    __syncthreads();   // the barrier is initialised before anyone waits on it
    if (n_loc > 0 && !mbar_wait(&sh.bar, 0)) timed_out = true;
  } else {
    for (int e = tid; e < n_loc; e += kRowThreads) {
      st[e] = trow[e0 + e];
      if (has_draft) sd[e] = drow[e0 + e];
    }
    __syncthreads();
  }
  if (timed_out) atomic_or_status(P.status, SV_DEV_TIMEOUT);

  const float mcp = __fmul_rn(m_p, c), mcq = __fmul_rn(m_q, c);
  const float r_pq = q_logits ? S_p / S_q : S_p;
  const float v_u = P.uniforms[((int64_t)b * (K + 1) + n) * 2 + 1];
  const float2 cc = make_float2(c, c);
  const float2 nref = make_float2(-mcp, -mcq);
  auto weight8 = [&](int g, float (&w)[8]) {
    float xp[8];
    load8(st, g, xp);
    if (has_draft) {
      float xq[8];
      load8(sd, g, xq);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float eq, ep;
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
  };
  auto sum8 = [](const float (&w)[8]) {
    const float2 a = __fadd2_rn(make_float2(w[0], w[1]), make_float2(w[2], w[3]));
    const float2 bb = __fadd2_rn(make_float2(w[4], w[5]), make_float2(w[6], w[7]));
    const float2 t = __fadd2_rn(a, bb);
    return t.x + t.y;
  };
  // warp `warp` owns groups [g_lo, g_hi); lane l owns the run
  // [g_lo + l G, g_lo + (l+1) G) of it, visited in a lane-rotated order so
  // the 16-byte shared-memory reads of a quarter warp hit distinct banks
  const int gpw = (n_grp + kRowWarps - 1) / kRowWarps;
  const int g_lo = min(n_grp, warp * gpw), g_hi = min(n_grp, g_lo + gpw);
  const int G = (gpw + 31) >> 5;
  const int r_lo = min(g_hi, g_lo + lane * G), r_hi = min(g_hi, r_lo + G);
  float t_l = 0.f;
  const int rot = G > 0 ? lane % G : 0;
  for (int s = 0; s < G; ++s) {
    int k = s + rot;
    k = k >= G ? k - G : k;
    const int g = r_lo + k;
    if (g < r_hi) {
      float w[8];
      weight8(g, w);
      t_l += sum8(w);
    }
  }
  float incl = t_l;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) sh.wsum[warp] = incl;
  __syncthreads();
  float tot_cta = 0.f;
  for (int w = 0; w < kRowWarps; ++w) tot_cta += sh.wsum[w];
  if (tid == 0) sh.pub_tot = tot_cta;
  cluster_sync();   // masses published
  const float t_r = lane < cs ? ld_dsmem_f32(mapa(&sh.pub_tot, lane)) : 0.f;
  // the last distributed read of this launch is done: arrive now, wait at exit
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  float off_c = 0.f, Z = 0.f;
  for (int rr = 0; rr < cs; ++rr) {
    const float t = __shfl_sync(0xffffffffu, t_r, rr);
    if (rr == rank) off_c = Z;
    Z += t;
  }
  const float thr = v_u * Z;
  // rounding bound of the fp32 CDF near thr, in units of w' = S_p w:
  // per-element exp / argument / ratio errors (~2^-22 relative, random:
  // sqrt(sum p^2) <= sqrt(max p) = sqrt(1/S)), and the rounding of the
  // running sums (~2^-24 per addition)
  const float e_abs = 4.7683716e-07f * S_p * sqrtf(1.f / S_p + (q_logits ? 1.f / S_q : 0.f)) +
                      1.1920929e-07f * (Z + S_p);   // 2^-21, 2^-23
  const bool draw_ok = finite && Z > 0.f && thr < Z;
  RowRec *rec = P.recs + (int64_t)b * (K + 1) + n;
  const uint32_t acc_flags = has_draft ? REC_ACC_CERT : 0u;   // a certified rejection (or the bonus row)
  if (rank == 0 && tid == 0) {
    rec->z = Z; rec->e_abs = e_abs;
    if (!draw_ok) { rec->y = -1; rec->gap = 0.f; rec->flags = acc_flags; }
  }
  if (draw_ok && off_c <= thr && thr < off_c + tot_cta) {
    float woff = 0.f, base = off_c;
    int owner = kRowWarps - 1;
    for (int w = 0; w < kRowWarps; ++w) {
      const float nxt = woff + sh.wsum[w];
      if (thr < off_c + nxt || w == kRowWarps - 1) { owner = w; base = off_c + woff; break; }
      woff = nxt;
    }
    if (warp == owner) {
      // the lane whose run holds thr, then its groups rescanned in order
      const unsigned hit = __ballot_sync(0xffffffffu, base + incl > thr);
      int y = -1;
      float c_lo = 0.f, c_hi = 0.f;
      if (hit) {
        const int L = __ffs(hit) - 1;
        float start = base + __shfl_sync(0xffffffffu, incl - t_l, L);
        const int L_lo = __shfl_sync(0xffffffffu, r_lo, L), L_hi = __shfl_sync(0xffffffffu, r_hi, L);
        for (int g0 = L_lo; g0 < L_hi && y < 0; g0 += 32) {   // one pass while G <= 32
          const int g = g0 + lane;
          float w[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          float vsum = 0.f;
          if (g < L_hi) {
            weight8(g, w);
            vsum = ((w[0] + w[1]) + (w[2] + w[3])) + ((w[4] + w[5]) + (w[6] + w[7]));
          }
          float inc2 = vsum;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const float t = __shfl_up_sync(0xffffffffu, inc2, o);
            if (lane >= o) inc2 += t;
          }
          const unsigned h2 = __ballot_sync(0xffffffffu, g < L_hi && start + inc2 > thr);
          if (h2) {
            const int L2 = __ffs(h2) - 1;
            if (lane == L2) {
              float run_c = start + (inc2 - vsum);
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const float nxt = run_c + w[j];
                if (y < 0 && nxt > thr) { y = e0 + 8 * g + j; c_lo = run_c; c_hi = nxt; }
                run_c = nxt;
              }
            }
            y = __shfl_sync(0xffffffffu, y, L2);
            c_lo = __shfl_sync(0xffffffffu, c_lo, L2);
            c_hi = __shfl_sync(0xffffffffu, c_hi, L2);
          }
          start += __shfl_sync(0xffffffffu, inc2, 31);
        }
      }
      if (lane == 0) {
        const bool found = y >= 0 && y < V;   // else: rounding moved the crossing
        const float gap = found ? fminf(thr - c_lo, c_hi - thr) : 0.f;
        rec->y = found ? y : -1;
        rec->gap = gap;
        rec->flags = acc_flags | ((found && gap > e_abs) ? REC_DRAW_CERT : 0u);
      }
    }
  }
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ------------------------------------------- float-float re-evaluation ---
// Lean float-float exp: exp((l - m)/T) for l <= m as an unevaluated pair
// hi + lo with ~1e-9 relative error: t = (l - m) log2(e) split into
// n/64 + r (|r| <= 1/128), 2^r - 1 by its Taylor series to r^5, 2^(j/64)
// from the (hi, lo) table, 2^k by exponent construction. Values below e^-87
// relative to the row maximum are returned as 0.
__device__ __forceinline__ ff ffx_exp(float l, float m, const SampleParams &P, const float2 *tbl) {
  if (!(l > -INFINITY)) return ff{0.f, 0.f};
  ff x = two_sum(l, -m);
  if (!P.unitT) x = ff_mul(x, ff{P.invT_hi, P.invT_lo});
  if (!(x.hi > -87.f)) return ff{0.f, 0.f};
  const float t_hi = x.hi * P.log2e_hi;
  const float t_lo = fmaf(x.hi, P.log2e_hi, -t_hi) + fmaf(x.hi, P.log2e_lo, x.lo * P.log2e_hi);
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

struct ExactShared {
  ff red[32];
  ff wsum[kResWarps];    // per-warp weight totals
  ff wincl[kResWarps];   // their inclusive prefix
  ff pub_sp, pub_sq, pub_tot;
  int pub_y, pub_last;
  float2 tbl[64];
};

// Exact-arithmetic (float-float) evaluation of row i of sequence b: the
// accept test (when need_acc) and, unless accepted, the inverse-CDF draw.
// Called by every thread of every CTA of the cluster; st / sd hold this CTA's
// slice [e0, e0 + n_grp*8) of the row (padded like the rows kernel does).
template <typename TT, int DK>
__device__ bool exact_row(const SampleParams &P, ExactShared &sh, const TT *st,
                          const typename std::conditional<DK == 0, TT, float>::type *sd, ff *cp, ff *cq,
                          int n_grp, int e0, bool has_draft, bool need_acc, float m_p, float m_q, float lp_x,
                          float lq_x, float u, float v_u, int *y_out) {
  const int cs = (int)cluster_nctarank(), rank = (int)cluster_ctarank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool q_logits = has_draft && DK == 0;
  // cp / cq (when not null) keep e_p, e_q of element j of group g at
  // [j * n_grp + g] for the weights pass
  ff sp{0.f, 0.f}, sq{0.f, 0.f};
  for (int g = tid; g < n_grp; g += blockDim.x) {
    float x[8];
    load8(st, g, x);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const ff e = ffx_exp(x[j], m_p, P, sh.tbl);
      if (cp) cp[j * n_grp + g] = e;
      acc_add(sp, e);
    }
    if (q_logits) {
      load8(sd, g, x);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const ff e = ffx_exp(x[j], m_q, P, sh.tbl);
        if (cp) cq[j * n_grp + g] = e;
        acc_add(sq, e);
      }
    }
  }
  sp = block_sum_ff(ff_norm(sp), sh.red);
  sq = block_sum_ff(ff_norm(sq), sh.red);
  if (tid == 0) { sh.pub_sp = sp; sh.pub_sq = sq; }
  cluster_sync();
  ff Sp = lane < cs ? ld_dsmem_ff(&sh.pub_sp, lane) : ff{0.f, 0.f};
  ff Sq = lane < cs ? ld_dsmem_ff(&sh.pub_sq, lane) : ff{0.f, 0.f};
  Sp = warp_sum_ff(Sp);
  Sq = warp_sum_ff(Sq);
  cluster_sync();   // peers have read the published sums
  if (!q_logits) Sq = ff{1.f, 0.f};
  if (need_acc && has_draft) {
    // u q(x) < p(x)  <=>  u e_q(x) S_p < e_p(x) S_q   (draft logits)
    //                <=>  u q(x) S_p < e_p(x)         (draft probabilities)
    const ff epx = ff_norm(ffx_exp(lp_x, m_p, P, sh.tbl));
    ff lhs, rhs;
    if (DK == 0) {
      lhs = ff_mul(ff_mul(ff{u, 0.f}, ff_norm(ffx_exp(lq_x, m_q, P, sh.tbl))), Sp);
      rhs = ff_mul(epx, Sq);
    } else {
      lhs = ff_mul(ff{u, 0.f}, ff_mul(ff{lq_x, 0.f}, Sp));
      rhs = epx;
    }
    if (ff_gt(rhs, lhs)) return true;
  }
  // scaled weights w'(y) = S_p S_q w(y); mode 0: target row (bonus, or the
  // zero-mass fallback), 1: two softmaxes, 2: given probabilities
  int mode = !has_draft ? 0 : (DK == 0 ? 1 : 2);
  auto wx8 = [&](int g, ff (&w)[8]) {
    float xp[8], xq[8];
    if (!cp) load8(st, g, xp);
    if (has_draft && (mode == 2 || !cp)) load8(sd, g, xq);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const ff ep = cp ? cp[j * n_grp + g] : ffx_exp(xp[j], m_p, P, sh.tbl);
      if (mode == 0) {
        w[j] = ep;
      } else if (mode == 1) {
        const ff eq = cp ? cq[j * n_grp + g] : ffx_exp(xq[j], m_q, P, sh.tbl);
        w[j] = ff_max0(ff_add(ff_mul(ep, Sq), ff_neg(ff_mul(eq, Sp))));
      } else {
        w[j] = ff_max0(ff_add(ep, ff_neg(ff_mul(ff{xq[j], 0.f}, Sp))));
      }
    }
  };
  // Each warp owns groups [g_lo, g_hi); lane l owns the run [r_lo, r_hi) of
  // them, so one warp scan of the lane totals and one scan of the warp
  // totals give every run its offset; the owner of v Z is found by ballots.
  const int nw = (int)(blockDim.x >> 5);
  const int gpw = (n_grp + nw - 1) / nw;
  const int g_lo = min(n_grp, warp * gpw), g_hi = min(n_grp, g_lo + gpw);
  const int G = (gpw + 31) >> 5;
  const int r_lo = min(g_hi, g_lo + lane * G), r_hi = min(g_hi, r_lo + G);
  int y = -1;
  for (int attempt = 0; attempt < 2; ++attempt) {
    ff t_l{0.f, 0.f};
    int last_pos = -1;
    for (int g = r_lo; g < r_hi; ++g) {
      ff w[8];
      wx8(g, w);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        acc_add(t_l, w[j]);
        if (w[j].hi > 0.f) last_pos = e0 + 8 * g + j;
      }
    }
    t_l = ff_norm(t_l);
    const ff incl = scan32_ff(t_l, lane);
    last_pos = warp_max_s32(last_pos);
    if (lane == 31) sh.wsum[warp] = incl;
    if (lane == 0 && last_pos >= 0) atomicMax(&sh.pub_last, last_pos);
    __syncthreads();
    if (warp == 0) {
      // inclusive prefix of the warp totals; the CTA total is published
      const ff wi = scan32_ff(lane < nw ? sh.wsum[lane] : ff{0.f, 0.f}, lane);
      if (lane < nw) sh.wincl[lane] = wi;
      if (lane == nw - 1) sh.pub_tot = wi;
    }
    __syncthreads();
    cluster_sync();   // totals published
    // CTA r owns [sum of the totals before r, + its total): a sequential
    // prefix in rank order, the same in every CTA
    const ff t_r = lane < cs ? ld_dsmem_ff(&sh.pub_tot, lane) : ff{0.f, 0.f};
    const int last_all = warp_max_s32(lane < cs ? ld_dsmem_s32(mapa(&sh.pub_last, lane)) : -1);
    cluster_sync();   // peers have read the totals
    if (tid == 0) sh.pub_last = -1;
    ff xoff{0.f, 0.f}, XZ{0.f, 0.f};
    for (int r = 0; r < cs; ++r) {
      const ff t{__shfl_sync(0xffffffffu, t_r.hi, r), __shfl_sync(0xffffffffu, t_r.lo, r)};
      if (r == rank) xoff = XZ;
      XZ = ff_add(XZ, t);
    }
    if (!ff_pos(XZ)) {   // zero residual mass: draw from p_n instead
      __syncthreads();
      if (mode == 0) break;
      mode = 0;
      continue;
    }
    const ff xthr = ff_mul(ff{v_u, 0.f}, XZ);
    const ff tot{__shfl_sync(0xffffffffu, t_r.hi, rank), __shfl_sync(0xffffffffu, t_r.lo, rank)};
    if (!ff_gt(xoff, xthr) && ff_gt(ff_add(xoff, tot), xthr)) {
      // the first warp whose inclusive total passes v Z (the last one if
      // rounding leaves none)
      const bool past = lane < nw && ff_gt(ff_add(xoff, sh.wincl[lane]), xthr);
      const unsigned wb = __ballot_sync(0xffffffffu, past);
      const int owner = wb ? __ffs(wb) - 1 : nw - 1;
      if (warp == owner) {
        const ff base = owner > 0 ? ff_add(xoff, sh.wincl[owner - 1]) : xoff;
        const unsigned lb = __ballot_sync(0xffffffffu, ff_gt(ff_add(base, incl), xthr));
        const int L = lb ? __ffs(lb) - 1 : 31;
        const ff excl{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
        ff start = ff_add(base, lane == 0 ? ff{0.f, 0.f} : excl);
        start = ff{__shfl_sync(0xffffffffu, start.hi, L), __shfl_sync(0xffffffffu, start.lo, L)};
        const int L_lo = __shfl_sync(0xffffffffu, r_lo, L), L_hi = __shfl_sync(0xffffffffu, r_hi, L);
        // the run's groups, one per lane, in ascending order
        int found = -1, last_p = -1;
        for (int g0 = L_lo; g0 < L_hi && found < 0; g0 += 32) {
          const int g = g0 + lane;
          ff w[8];
          ff gs{0.f, 0.f};
#pragma unroll
          for (int j = 0; j < 8; ++j) w[j] = ff{0.f, 0.f};
          if (g < L_hi) {
            wx8(g, w);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc_add(gs, w[j]);
          }
          gs = ff_norm(gs);
          const ff inc2 = scan32_ff(gs, lane);
          int cand = -1;
          ff run_c = ff_add(start, ff_add(inc2, ff_neg(gs)));
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const ff nxt = ff_add(run_c, w[j]);
            if (cand < 0 && w[j].hi > 0.f && ff_gt(nxt, xthr)) cand = e0 + 8 * g + j;
            if (w[j].hi > 0.f) last_p = max(last_p, e0 + 8 * g + j);
            run_c = nxt;
          }
          const unsigned hit = __ballot_sync(0xffffffffu, cand >= 0);
          if (hit) found = __shfl_sync(0xffffffffu, cand, __ffs(hit) - 1);
          start = ff_add(start, ff{__shfl_sync(0xffffffffu, inc2.hi, 31), __shfl_sync(0xffffffffu, inc2.lo, 31)});
        }
        last_p = warp_max_s32(last_p);
        if (found < 0) found = last_p;   // crossing within rounding of the run's end
        if (lane == 0) sh.pub_y = found;
      }
    }
    cluster_sync();   // the draw is published
    y = warp_max_s32(lane < cs ? ld_dsmem_s32(mapa(&sh.pub_y, lane)) : -1);
    if (y < 0) y = last_all;   // v Z at the very top of the range (rounding)
    cluster_sync();   // peers have read pub_y
    if (tid == 0) sh.pub_y = -1;
    __syncthreads();
    break;
  }
  *y_out = y;
  return false;
}

// Every cluster walks every sequence (one thread per sequence, in rounds of
// kResThreads sequences): certified accepts, then the first rejection or the
// bonus row. All CTAs build the same ordered list of sequences whose next
// needed decision is not certified, and cluster c re-evaluates entries
// c, c + ncl, ... (the row's slices copied into shared memory, float-float
// arithmetic, continuing the walk), so the rare exact rows spread over all
// clusters. The tokens of a fully certified sequence b are written by
// cluster b % ncl.
constexpr int kFinishMaxSeq = kResThreads;   // sequences per walk round

template <typename TT, int DK>
__global__ void __launch_bounds__(kResThreads) sample_finish_kernel(const __grid_constant__ SampleParams P) {
  pdl_wait();
  pdl_trigger();
  using TD = typename std::conditional<DK == 0, TT, float>::type;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ ExactShared sh;
  __shared__ __align__(8) uint64_t bar;
  __shared__ int list_n;
  __shared__ int list_b[kFinishMaxSeq], list_i[kFinishMaxSeq];
  __shared__ int warp_cnt[kResWarps];
  const int cs = (int)cluster_nctarank(), rank = (int)cluster_ctarank();
  const int cid = blockIdx.x / cs, ncl = gridDim.x / cs;
  const int K = P.K, V = P.V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool force = (P.flags & SV_SAMPLE_FORCE_EXACT) != 0;
  const int ns = P.ns_x;
  const int e0 = min(V, rank * ns);
  const int n_loc = max(0, min(V, e0 + ns) - e0);
  const int n_grp = (n_loc + 7) >> 3;
  TT *st = reinterpret_cast<TT *>(smem);
  TD *sd = reinterpret_cast<TD *>(smem + align_up((size_t)ns * sizeof(TT), 128));
  ff *cp = nullptr, *cq = nullptr;
  if (P.cache_x) {
    cp = reinterpret_cast<ff *>(smem + align_up((size_t)ns * sizeof(TT), 128) + align_up((size_t)ns * sizeof(TD), 128));
    cq = cp + ns;
  }
  if (tid < 64) sh.tbl[tid] = P.tbl[tid];
  if (tid == 0) {
    sh.pub_y = -1; sh.pub_last = -1;
    mbar_init(&bar, 1);
    fence_mbarrier_init();
  }
  __syncthreads();
  cluster_sync();   // peers initialised before any distributed read

  uint32_t phase = 0;
  const bool vec = P.aligned != 0;
  for (int round0 = 0; round0 < P.B; round0 += kFinishMaxSeq) {
    // ---- parallel walk: one thread per sequence ---------------------------
    const int b = round0 + tid;
    int start = -1;   // first position whose decision needs the float-float pass
    if (b < P.B) {
      const RowRec *recs = P.recs + (int64_t)b * (K + 1);
      int n = K, ysel = -1;
      bool done = false;
      for (int i0 = 0; i0 <= K && !done; i0 += 8) {
        uint32_t f[8];
        int yv[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {   // independent loads: one round trip
          const int i = i0 + j;
          f[j] = i <= K ? recs[i].flags : 0u;
          yv[j] = i <= K ? recs[i].y : -1;
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = i0 + j;
          if (done || i > K) continue;
          if (i < K && (force || !(f[j] & REC_ACC_CERT))) {
            start = i;
            done = true;
          } else if (i == K || !(f[j] & REC_ACCEPT)) {
            n = i;
            done = true;
            if (!force && (f[j] & REC_DRAW_CERT)) ysel = yv[j];
            else start = n;
          }
        }
      }
      if (start < 0 && rank == 0 && b % ncl == cid) {
        for (int j = 0; j <= K; ++j)
          P.out_tokens[(int64_t)b * (K + 1) + j] = j < n ? P.tokens[(int64_t)b * K + j] : (j == n ? ysel : -1);
        P.num_acc[b] = n;
      }
    }
    // deterministic compaction (same order in every CTA of every cluster)
    const unsigned vote = __ballot_sync(0xffffffffu, start >= 0);
    if (lane == 0) warp_cnt[warp] = __popc(vote);
    __syncthreads();
    if (tid == 0) {
      int acc = 0;
      for (int w = 0; w < kResWarps; ++w) { const int t = warp_cnt[w]; warp_cnt[w] = acc; acc += t; }
      list_n = acc;
    }
    __syncthreads();
    if (start >= 0) {
      const int pos = warp_cnt[warp] + __popc(vote & ((1u << lane) - 1u));
      list_b[pos] = b;
      list_i[pos] = start;
    }
    __syncthreads();

    // ---- float-float re-evaluation of this cluster's list entries ---------
    for (int li = cid; li < list_n; li += ncl) {
      const int bb = list_b[li];
      const RowRec *recs = P.recs + (int64_t)bb * (K + 1);
      const int32_t *toks = P.tokens + (int64_t)bb * K;
      int i = list_i[li], n = K, y = -1;
      for (;;) {
        // next position needing evaluation from i on (certified accepts skipped)
        int need = -1;
        bool need_acc = false;
        for (; i < K; ++i) {
          const uint32_t f = recs[i].flags;
          if (force || !(f & REC_ACC_CERT)) { need = i; need_acc = true; break; }
          if (!(f & REC_ACCEPT)) break;
        }
        n = min(i, K);
        if (need < 0) {
          if (!force && (recs[n].flags & REC_DRAW_CERT)) { y = recs[n].y; break; }
          need = n;
        }
        const bool has_draft = need < K;
        const TT *trow = static_cast<const TT *>(P.target) + ((int64_t)bb * (K + 1) + need) * V;
        const TD *drow = has_draft ? static_cast<const TD *>(P.draft) + ((int64_t)bb * K + need) * V : nullptr;
        // slice -> shared memory (bulk copy when rows are 16-byte aligned)
        for (int e = n_loc + tid; e < n_grp * 8; e += blockDim.x) {
          st[e] = pad_value<TT>(false);
          if (has_draft) sd[e] = pad_value<TD>(DK == 1);
        }
        if (vec) {
          if (tid == 0 && n_loc > 0) {
            const uint32_t nbt = (uint32_t)n_loc * sizeof(TT), nbd = has_draft ? (uint32_t)n_loc * sizeof(TD) : 0u;
            fence_proxy_async_shared();
            mbar_arrive_expect_tx(&bar, nbt + nbd);
            bulk_g2s(st, trow + e0, nbt, &bar);
            if (has_draft) bulk_g2s(sd, drow + e0, nbd, &bar);
          }
          if (n_loc > 0) {
            if (!mbar_wait(&bar, phase) && tid == 0) atomic_or_status(P.status, SV_DEV_TIMEOUT);
            phase ^= 1u;
          }
        } else {
          for (int e = tid; e < n_loc; e += blockDim.x) {
            st[e] = trow[e0 + e];
            if (has_draft) sd[e] = drow[e0 + e];
          }
        }
        __syncthreads();
        const RowRec rr = recs[need];
        const float *uv = P.uniforms + ((int64_t)bb * (K + 1) + need) * 2;
        float lp_x = 0.f, lq_x = 0.f;
        if (has_draft) {
          const int x = min(max(toks[need], 0), V - 1);
          lp_x = to_f32(trow[x]);
          lq_x = to_f32(drow[x]);
        }
        int yy = -1;
        const bool acc = exact_row<TT, DK>(P, sh, st, sd, cp, cq, n_grp, e0, has_draft, need_acc, rr.m_p,
                                           rr.m_q, lp_x, lq_x, uv[0], uv[1], &yy);
        if (rank == 0 && tid == 0) {
          RowRec *w = P.recs + (int64_t)bb * (K + 1) + need;
          w->flags = rr.flags | (need_acc ? REC_EXACT_ACC : 0u) | (acc ? 0u : REC_EXACT_DRAW);
          if (!acc) w->y_exact = yy;
        }
        __syncthreads();   // the slice buffers are rewritten next
        if (need_acc && acc) { i = need + 1; continue; }   // accepted: continue the walk
        n = need;
        y = yy;
        break;
      }
      if (rank == 0) {
        for (int j = tid; j <= K; j += blockDim.x)
          P.out_tokens[(int64_t)bb * (K + 1) + j] = j < n ? toks[j] : (j == n ? y : -1);
        if (tid == 0) P.num_acc[bb] = n;
      }
    }
    __syncthreads();   // the list is rebuilt in the next round
  }
  cluster_sync();   // no CTA leaves while a peer may still read its shared memory
}

// ------------------------------------------------------------------ host ---

size_t records_bytes(int B, int K) { return align_up((size_t)B * (K + 1) * sizeof(RowRec), 256); }

int stat_chunks(int V) { return (V + kStatChunk - 1) / kStatChunk; }

// per-row records, then the chunk statistics
size_t workspace_bytes_for(int B, int K, int V) {
  return records_bytes(B, K) + align_up((size_t)B * (K + 1) * stat_chunks(V) * sizeof(float4), 256);
}

void split_ff(double d, float &hi, float &lo) {
  hi = (float)d;
  lo = (float)(d - (double)hi);
}


template <typename TT, int DK>
sv_status launch_sample(const SampleParams &P, int cs, size_t smem, int cs_x, size_t smem_x, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    const int lim = (int)(kMaxSliceSmem + 1024);
    attr_err = cudaFuncSetAttribute(sample_draw_kernel<TT, DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(sample_draw_kernel<TT, DK>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(sample_finish_kernel<TT, DK>, cudaFuncAttributeMaxDynamicSharedMemorySize, lim);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(sample_finish_kernel<TT, DK>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  });
  if (attr_err != cudaSuccess)
    return fail(SV_ERR_CUDA, "spec_verify_sample: cudaFuncSetAttribute: %s", cudaGetErrorString(attr_err));
  cudaError_t e = launch_k(sample_stats_kernel<TT, DK>, dim3(P.nc, P.K + 1, P.B), dim3(kStatThreads), 0, s, 1, P);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_sample statistics launch: %s", cudaGetErrorString(e));
  e = launch_k(sample_draw_kernel<TT, DK>, dim3(cs, P.B), dim3(kRowThreads), smem, s, cs, P);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_sample draw launch: %s", cudaGetErrorString(e));
  const int ncl = std::max(1, std::min(P.B, kFinishClusters));
  e = launch_k(sample_finish_kernel<TT, DK>, dim3(cs_x * ncl), dim3(kResThreads), smem_x, s, cs_x, P);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_sample finish launch: %s", cudaGetErrorString(e));
  return ok();
}

}  // namespace
}  // namespace sv

extern "C" size_t spec_verify_sample_workspace_size(int B, int K, int V) {
  (void)V;
  if (B < 0 || K < 0) return 0;
  if (V < 1) return 0;
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
  if (!workspace || workspace_bytes < workspace_bytes_for(B, K, V))
    return fail(SV_ERR_WORKSPACE, "spec_verify_sample: workspace needs %zu bytes", workspace_bytes_for(B, K, V));
  if (!aligned(workspace, 256)) return fail(SV_ERR_WORKSPACE, "spec_verify_sample: workspace not 256-byte aligned");
  if (B == 0) return ok();

  const int es_t = dtype_bytes(logit_dtype);
  int cs = 0;
  int ns = 0;
  size_t smem = 0;
  // rows kernel: the smallest cluster whose slices take <= 64 KB (three CTAs
  // per SM), else the smallest that fits at all
  const int es_buf_d = (draft_is_probs && K > 0) ? 4 : es_t;
  auto slice_smem = [&](int c, int &n) {
    n = (int)align_up((size_t)((V + c - 1) / c), 8);
    return align_up((size_t)n * es_t, 128) + align_up((size_t)n * es_buf_d, 128);
  };
  for (int c = 1; c <= 16 && !cs; c *= 2) {
    int n;
    const size_t sm = slice_smem(c, n);
    if (sm <= kTargetSliceSmem) { cs = c; ns = n; smem = sm; }
  }
  if (!cs) {
    int n;
    const size_t sm = slice_smem(16, n);
    if (sm <= kMaxSliceSmem) { cs = 16; ns = n; smem = sm; }
  }
  // finish kernel: 16-CTA clusters (8 for small vocabularies)
  const int cs_x = V >= 65536 ? 16 : 8;
  int ns_x = 0;
  size_t smem_x = slice_smem(cs_x, ns_x);
  // float-float exponentials of both rows cached when they fit
  const size_t cache_bytes = (size_t)ns_x * sizeof(ff) * ((draft_is_probs && K > 0) ? 1 : 2);
  const bool cache_x = smem_x + cache_bytes <= kMaxSliceSmem;
  if (cache_x) smem_x += cache_bytes;
  if (cs && smem_x > kMaxSliceSmem) cs = 0;
  if (!cs) return fail(SV_ERR_UNSUPPORTED, "spec_verify_sample: vocabulary of %d too large", V);

  SampleParams P = {};
  P.target = target_logits; P.draft = draft; P.tokens = draft_tokens; P.uniforms = uniforms;
  P.p_at = p_at_draft; P.q_at = q_at_draft; P.out_tokens = out_tokens; P.num_acc = num_accepted;
  P.recs = static_cast<RowRec *>(workspace); P.status = dev_status;
  P.part = reinterpret_cast<float4 *>(static_cast<uint8_t *>(workspace) + records_bytes(B, K));
  P.nc = stat_chunks(V);
  P.B = B; P.K = K; P.V = V; P.ns = ns; P.ns_x = ns_x; P.flags = flags; P.cache_x = cache_x ? 1 : 0;
  P.aligned = aligned(target_logits, 16) && ((size_t)V * es_t) % 16 == 0 &&
              (K == 0 || (aligned(draft, 16) && ((size_t)V * es_buf_d) % 16 == 0));
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
    case SV_F32: return probs ? launch_sample<float, 1>(P, cs, smem, cs_x, smem_x, s) : launch_sample<float, 0>(P, cs, smem, cs_x, smem_x, s);
    case SV_BF16:
      return probs ? launch_sample<__nv_bfloat16, 1>(P, cs, smem, cs_x, smem_x, s)
                   : launch_sample<__nv_bfloat16, 0>(P, cs, smem, cs_x, smem_x, s);
    default:
      return probs ? launch_sample<__half, 1>(P, cs, smem, cs_x, smem_x, s) : launch_sample<__half, 0>(P, cs, smem, cs_x, smem_x, s);
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

// ------------------------------------------------- allocation-free entry ---
// Some callers cannot allocate device memory when they verify a round: for
// example an engine that reserves all of the GPU's memory for its KV pool at
// start-up and forbids allocations afterwards, or a caller whose fixed C
// interface has no way to pass a workspace. For them the records live in
// this static device array (every GPU that loads the library keeps it until
// the process exits).
namespace {
constexpr size_t kStaticScratchBytes = 1u << 20;   // 1 MiB: 48 + 16 ceil(V / 8192) bytes per (sequence, position)
__device__ __align__(256) uint8_t g_sample_scratch[kStaticScratchBytes];
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices] = {};
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
                "spec_verify_sample_static: B*(K+1) = %lld rows need %zu bytes (a %zu-byte record and %d "
                "16-byte chunk statistics per row), more than the static scratch of %zu bytes; use "
                "spec_verify_sample with a caller workspace",
                (long long)B * (K + 1), need, sizeof(RowRec), stat_chunks(V), kStaticScratchBytes);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_sample_static: cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(SV_ERR_UNSUPPORTED, "spec_verify_sample_static: device %d", dev);
  void *ptr = nullptr;
  {
    // first call on a device: resolve the array's device address (the
    // device is current here)
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
      e = cudaGetSymbolAddress(&g_scratch_ptr[dev], g_sample_scratch);
      if (e != cudaSuccess) {
        g_scratch_ptr[dev] = nullptr;
        return fail(SV_ERR_CUDA, "spec_verify_sample_static: cudaGetSymbolAddress: %s", cudaGetErrorString(e));
      }
    }
    ptr = g_scratch_ptr[dev];
  }
  return spec_verify_sample(target_logits, logit_dtype, draft, draft_dtype, draft_is_probs, draft_tokens,
                            uniforms, B, K, V, temperature, out_tokens, num_accepted, p_at_draft, q_at_draft, ptr,
                            kStaticScratchBytes, dev_status, stream);
}

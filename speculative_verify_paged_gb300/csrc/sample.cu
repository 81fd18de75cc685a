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
//     that row is read again, 16-byte loads straight into registers (no
//     shared-memory slices, so every CTA of the grid is resident at once);
//     its residual weights are summed per block of 256 elements, the
//     cluster's prefix locates v Z, the owning warp rescans one block, and
//     the inverse-CDF draw gets its own certificate. One 48-byte record per
//     (sequence, position) results; certified sequences write their tokens.
//   * sample_finish_kernel: one CTA per SM (cooperative launch) resolves the
//     sequences the draw kernel queued. The rare decision that is not
//     certified (a few percent of sequences) is
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
  int gpc;       // groups of eight elements per CTA slice of the draw kernel
  int aligned;   // rows are 16-byte aligned: bulk copies usable
  unsigned *fin_sync;   // finish grid barrier: arrival count, generation; [2] pending count
  int2 *pend;           // [B] sequences left to the finish grid: (b, first row to resolve)
  float2 *fin_sum;      // [kMaxUnits][kMaxFinCtas][2] chunk sums of e_p, e_q (float-float)
  float2 *fin_tot;      // [kMaxEntries][kMaxFinCtas] chunk totals of the weights
  int *fin_last;        // [kMaxEntries][kMaxFinCtas] last positive weight of a chunk
  unsigned flags;
  uint64_t wait_ns;     // limit of each wait on another CTA's arrival
  unsigned withhold;    // test hook: SV_TEST_WITHHOLD_ARRIVALS keeps CTA 0 of the finish grid from arriving
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

// Resident CTAs per SM: five for 16-bit logits with draft logits (8B shape
// 23.2 -> 22.2 us per sampling call, 70B 71.4 -> 70.8 us), three for the
// others (fp32 rows spill at five: 277 -> 373 us on the fp8 workload, and
// reach 88 registers, two CTAs, with no bound: 300 us)
template <typename TT, int DK>
__global__ void __launch_bounds__(kStatThreads, sizeof(TT) == 2 && DK == 0 ? 5 : 3)
    sample_stats_kernel(const __grid_constant__ SampleParams P) {
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
  if (tid == 0 && c == 0 && i == 0 && b == 0) P.fin_sync[2] = 0u;   // no sequence pending yet
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
// weights w'(y) = max(0, e_p(y) - r e_q(y)) are formed from register loads
// of each CTA's slice; block totals, warp totals and the cluster's prefix
// locate v Z, the owning warp rescans one block, and the draw gets its own
// certificate. Anything uncertified is left to the finish kernel.

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

constexpr int kMaxDrawBlocks = 64;   // blocks of 32 groups per CTA slice (2048 groups)
constexpr int kDrawRowCache = 64;    // rows whose statistics the draw kernel keeps from its accept tests

struct DrawShared {
  int stop;               // 2 * position + (0: not certified, 1: certified rejection)
  float pub_tot;          // this CTA's draw mass
  float wsum[kRowWarps];  // per warp
  float btot[kMaxDrawBlocks];   // per block of 32 groups
};

// combined (max, sum) of target (and draft) row i of sequence b: every lane
// of the warp ends with the same bits
// emitted tokens of sequence b: the n accepted drafts, then y, then -1
__device__ __forceinline__ void write_outputs(const SampleParams &P, int b, int n, int y) {
  const int K = P.K;
  for (int j = 0; j <= K; ++j)
    P.out_tokens[(int64_t)b * (K + 1) + j] = j < n ? P.tokens[(int64_t)b * K + j] : (j == n ? y : -1);
  P.num_acc[b] = n;
}

// hands sequence b to the finish grid, to be resolved from row `start` on
__device__ __forceinline__ void push_pending(const SampleParams &P, int b, int start) {
  const unsigned slot = atomicAdd(&P.fin_sync[2], 1u);
  P.pend[slot] = make_int2(b, start);
}

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
__global__ void __launch_bounds__(kRowThreads, 4) sample_draw_kernel(const __grid_constant__ SampleParams P) {
  using TD = typename std::conditional<DK == 0, TT, float>::type;
  __shared__ DrawShared sh;
  __shared__ float4 s_rs[kDrawRowCache];   // (m_p, S_p, m_q, S_q) of the first rows

  const int cs = (int)cluster_nctarank(), rank = (int)cluster_ctarank();
  const int b = blockIdx.y;
  const int K = P.K, V = P.V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float c = P.c;
  const bool force = (P.flags & SV_SAMPLE_FORCE_EXACT) != 0;
  // The inputs of this warp's first accept test are loaded before the wait
  // on the statistics pass: the caller's arrays, or rows the top-p filter
  // wrote, which had finished before any CTA of the statistics pass let
  // this grid start.
  int x0 = 0;
  bool bad0 = false;
  float lp0 = 0.f, lq0 = 0.f, u0 = 0.f;
  if (warp < K) {
    x0 = P.tokens[(int64_t)b * K + warp];
    bad0 = x0 < 0 || x0 >= V;
    x0 = min(max(x0, 0), V - 1);
    lp0 = to_f32(static_cast<const TT *>(P.target)[((int64_t)b * (K + 1) + warp) * V + x0]);
    lq0 = to_f32(static_cast<const TD *>(P.draft)[((int64_t)b * K + warp) * V + x0]);
    u0 = P.uniforms[((int64_t)b * (K + 1) + warp) * 2];
  }
  pdl_wait();
  pdl_trigger();
  if (tid == 0) sh.stop = 2 * K + 1;
  if (tid == 0 && blockIdx.x == 0 && b == 0) P.fin_sync[0] = 0u;   // the finish grid barrier starts empty
  __syncthreads();

  // ---- accept tests of every draft position, and the bonus row's record ---
  // (each row's statistics are kept for the draw that follows)
  for (int i = warp; i <= K; i += kRowWarps) {
    float m_p, S_p, m_q, S_q;
    if (i == K) {   // the bonus row: the finish kernel may walk to it
      row_stats(P, b, K, false, m_p, S_p, m_q, S_q);
      if (lane == 0) {
        if (K < kDrawRowCache) s_rs[K] = make_float4(m_p, S_p, 0.f, 1.f);
        if (rank == 0) {
          RowRec *rec = P.recs + (int64_t)b * (K + 1) + K;
          rec->m_p = m_p; rec->s_p = S_p; rec->m_q = 0.f; rec->s_q = 1.f;
          rec->p_x = 0.f; rec->q_x = 0.f;
          rec->y = -1; rec->y_exact = -1; rec->gap = 0.f; rec->z = 0.f; rec->e_abs = 0.f;
          rec->flags = 0u;
          if (!(fabsf(m_p) <= 3.0e38f && S_p > 0.f)) atomic_or_status(P.status, SV_DEV_NONFINITE);
        }
      }
      continue;
    }
    row_stats(P, b, i, DK == 0, m_p, S_p, m_q, S_q);
    if (DK != 0) { m_q = 0.f; S_q = 1.f; }
    int x;
    float lp_x, lq_x, u;
    bool bad;
    if (i == warp) {
      x = x0; bad = bad0; lp_x = lp0; lq_x = lq0; u = u0;
    } else {
      x = P.tokens[(int64_t)b * K + i];
      bad = x < 0 || x >= V;
      x = min(max(x, 0), V - 1);
      lp_x = to_f32(static_cast<const TT *>(P.target)[((int64_t)b * (K + 1) + i) * V + x]);
      lq_x = to_f32(static_cast<const TD *>(P.draft)[((int64_t)b * K + i) * V + x]);
      u = P.uniforms[((int64_t)b * (K + 1) + i) * 2];
    }
    if (bad && rank == 0 && lane == 0) atomic_or_status(P.status, SV_DEV_BAD_TOKEN);
    if (i < kDrawRowCache && lane == 0) s_rs[i] = make_float4(m_p, S_p, m_q, S_q);
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
  // identical in every CTA of the cluster: no shared memory of a peer is
  // read on this path
  if (!certain || force) {   // the first uncertified accept test (or all, forced)
    if (rank == 0 && tid == 0) push_pending(P, b, force ? 0 : n);
    return;
  }
  if (n >= kDrawRowCache) {   // statistics of the row drawn from, when not kept
    if (warp == 0) {
      float a0, a1, a2, a3;
      row_stats(P, b, n, q_logits, a0, a1, a2, a3);
      if (!q_logits) { a2 = 0.f; a3 = 1.f; }
      if (lane == 0) s_rs[0] = make_float4(a0, a1, a2, a3);
    }
    __syncthreads();
  }
  const float4 rs = s_rs[n < kDrawRowCache ? n : 0];
  const float m_p = rs.x, S_p = rs.y, m_q = rs.z, S_q = rs.w;
  const bool finite = fabsf(m_p) <= 3.0e38f && (!q_logits || fabsf(m_q) <= 3.0e38f) && S_p > 0.f;

  // ---- the draw: this CTA's slice of row n, straight into registers -------
  // The slice is groups [gs0, gs1) of eight elements; warp w takes blocks
  // [w bpw, (w+1) bpw) of 32 consecutive groups (lane l: group 32 k + l of
  // the block), so element order is (warp, block, lane, element).
  const TT *trow = static_cast<const TT *>(P.target) + ((int64_t)b * (K + 1) + n) * V;
  const TD *drow = has_draft ? static_cast<const TD *>(P.draft) + ((int64_t)b * K + n) * V : nullptr;
  const int ngr = (V + 7) >> 3;
  const int gs0 = min(ngr, rank * P.gpc), gs1 = min(ngr, gs0 + P.gpc);
  const int nblk = (gs1 - gs0 + 31) >> 5;
  const int bpw = (nblk + kRowWarps - 1) / kRowWarps;
  const bool vec = P.aligned != 0;
  const float mcp = __fmul_rn(m_p, c), mcq = __fmul_rn(m_q, c);
  const float r_pq = q_logits ? S_p / S_q : S_p;
  const float v_u = P.uniforms[((int64_t)b * (K + 1) + n) * 2 + 1];
  constexpr int kFly = sizeof(TT) == 4 || sizeof(TD) == 4 ? 2 : 4;   // blocks in flight per warp
  for (int k0 = warp * bpw; k0 < min(nblk, (warp + 1) * bpw); k0 += kFly) {
    Raw8<TT> rt[kFly];
    Raw8<TD> rd[kFly];
#pragma unroll
    for (int f = 0; f < kFly; ++f) {
      const int g = gs0 + (k0 + f) * 32 + lane;
      if (k0 + f < (warp + 1) * bpw && g < gs1) {
        rt[f] = raw_load(trow, g, V, vec, false);
        if (has_draft) rd[f] = raw_load(drow, g, V, vec, DK == 1);
      }
    }
#pragma unroll
    for (int f = 0; f < kFly; ++f) {
      const int k = k0 + f;
      if (k >= min(nblk, (warp + 1) * bpw)) break;
      float w[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (gs0 + k * 32 + lane < gs1) draw_weights8<TT, TD, DK>(rt[f], rd[f], has_draft, c, mcp, mcq, r_pq, w);
      const float t = warp_sum_f(sum8f(w));
      if (lane == 0) sh.btot[k] = t;
    }
  }
  __syncthreads();
  if (warp == 0) {   // warp totals (blocks in order), then the CTA's
    float t = 0.f;
    if (lane < kRowWarps)
      for (int k = lane * bpw; k < min(nblk, (lane + 1) * bpw); ++k) t += sh.btot[k];
    if (lane < kRowWarps) sh.wsum[lane] = t;
    __syncwarp();
    if (lane == 0) {
      float tc = 0.f;
      for (int w = 0; w < kRowWarps; ++w) tc += sh.wsum[w];
      sh.pub_tot = tc;
    }
  }
  cluster_sync();   // masses published
  const float tot_cta = sh.pub_tot;
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
    if (!draw_ok) { rec->y = -1; rec->gap = 0.f; rec->flags = acc_flags; push_pending(P, b, n); }
  }
  if (draw_ok && off_c <= thr && thr < off_c + tot_cta) {
    // the owner warp and block (prefixes in element order), the same in
    // every thread of the CTA
    float base = off_c;
    int ow = kRowWarps - 1;
    for (int w = 0; w < kRowWarps; ++w) {
      if (thr < base + sh.wsum[w] || w == kRowWarps - 1) { ow = w; break; }
      base += sh.wsum[w];
    }
    const int kb0 = ow * bpw, kb1 = min(nblk, (ow + 1) * bpw);
    int ob = max(kb0, kb1 - 1);
    for (int k = kb0; k < kb1; ++k) {
      if (thr < base + sh.btot[k] || k == kb1 - 1) { ob = k; break; }
      base += sh.btot[k];
    }
    if (warp == ow) {
      // rescan of block ob: lane sums, their prefix, then the crossing lane's
      // eight elements in order
      const int g = gs0 + ob * 32 + lane;
      float w[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      if (ob < kb1 && g < gs1) {
        Raw8<TT> rt = raw_load(trow, g, V, vec, false);
        Raw8<TD> rd;
        if (has_draft) rd = raw_load(drow, g, V, vec, DK == 1);
        draw_weights8<TT, TD, DK>(rt, rd, has_draft, c, mcp, mcq, r_pq, w);
      }
      const float vs = ((w[0] + w[1]) + (w[2] + w[3])) + ((w[4] + w[5]) + (w[6] + w[7]));
      float inc2 = vs;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, inc2, o);
        if (lane >= o) inc2 += t;
      }
      const unsigned h2 = __ballot_sync(0xffffffffu, g < gs1 && base + inc2 > thr);
      int y = -1;
      float c_lo = 0.f, c_hi = 0.f;
      if (h2) {
        const int L2 = __ffs(h2) - 1;
        if (lane == L2) {
          float run_c = base + (inc2 - vs);
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const float nxt = run_c + w[j];
            if (y < 0 && nxt > thr) { y = 8 * g + j; c_lo = run_c; c_hi = nxt; }
            run_c = nxt;
          }
        }
        y = __shfl_sync(0xffffffffu, y, L2);
        c_lo = __shfl_sync(0xffffffffu, c_lo, L2);
        c_hi = __shfl_sync(0xffffffffu, c_hi, L2);
      }
      if (lane == 0) {
        const bool found = y >= 0 && y < V;   // else: rounding moved the crossing
        const float gap = found ? fminf(thr - c_lo, c_hi - thr) : 0.f;
        const bool cert = found && gap > e_abs;
        rec->y = found ? y : -1;
        rec->gap = gap;
        rec->flags = acc_flags | (cert ? REC_DRAW_CERT : 0u);
        if (cert) write_outputs(P, b, n, y);
        else push_pending(P, b, n);
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
// The finish grid runs its code once per call, with the instruction cache
// cold, so the exponential and the weights are single out-of-line copies
// called from rolled loops.
struct FfK {
  float inv_hi, inv_lo;     // 1/T
  float l2e_hi, l2e_lo;     // log2(e)
  int unitT;                // T == 1
};
__device__ __forceinline__ FfK ff_consts(const SampleParams &P) {
  return FfK{P.invT_hi, P.invT_lo, P.log2e_hi, P.log2e_lo, P.unitT};
}

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

// ------------------------------------------------ cooperative finish pass ---
// sample_finish_kernel: one CTA per SM, launched cooperatively (all CTAs
// resident), so the grid can meet at barriers.
//   * Every CTA walks every sequence's records (certified accepts, then the
//     first rejection or the bonus row) and builds the same ordered list of
//     sequences whose walk reaches a decision that is not certified; the
//     tokens of the others are written by CTA b % gridDim.x.
//   * Listed sequences are resolved in rounds. A round takes, for each one,
//     the rows its walk may still need (uncertified accept tests and the row
//     it ends on), at most kMaxUnits rows in all, and evaluates them together:
//     every CTA sums e_p and e_q over its contiguous chunk of each row ->
//     grid barrier -> every CTA forms the same row sums, takes the exact
//     accept tests in walk order, picks each sequence's draw row and sums its
//     residual weights over the chunk -> grid barrier -> every CTA forms the
//     same prefix over chunks; the CTA whose chunk holds v Z finds the token
//     and writes that sequence's outputs. Sequences whose rows ran past the
//     round's budget continue in the next round.
// Cross-CTA values go through the workspace and are read from L2; every CTA
// combines them in the same order, so all CTAs take the same decisions.
constexpr int kFinThreads = 512;
constexpr int kFinWarps = kFinThreads / 32;
constexpr int kMaxEntries = 32;     // sequences resolved together
constexpr int kMaxUnits = 32;       // rows evaluated per round
constexpr int kMaxFinCtas = 160;    // CTAs of the finish grid (one per SM)
static_assert(kMaxUnits >= kMaxEntries && kMaxUnits <= 2 * kFinWarps, "unit slots per warp");

// sequence phases: walk its records from e_i, redraw row e_i from p (zero
// residual mass), or finished
enum : int { ENT_WALK = 0, ENT_REDRAW = 1, ENT_DONE = 2 };

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

// Grid barrier of the cooperative launch: one arrival count in global memory
// (zeroed before the launch); barrier j of the launch completes when the
// count reaches j * gridDim.x, so the count is never reset. Bounded wait
// (limit_ns); returns false after a timeout. (Test hook: withheld, this
// CTA does not arrive, so every CTA's wait runs out.)
__device__ __forceinline__ bool grid_sync(unsigned *count, unsigned &target, int *flag, uint64_t limit_ns,
                                          bool withhold) {
  __syncthreads();
  if (threadIdx.x == 0) {
    bool ok = true;
    target += gridDim.x;
    __threadfence();
    if (!withhold) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(count) : "memory");
    const uint64_t t0 = global_ns();
    for (;;) {
      unsigned v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(count) : "memory");
      if ((int)(v - target) >= 0) break;
      if (global_ns() - t0 > limit_ns) { ok = false; break; }
      __nanosleep(16);
    }
    __threadfence();
    *flag = ok ? 1 : 0;
  }
  __syncthreads();
  return *flag != 0;
}

__device__ __forceinline__ ff ldcg_ff(const float2 *p) {
  const float2 v = __ldcg(p);
  return ff{v.x, v.y};
}

// exclusive block prefix (element order = thread order) and total of ff
// values; every thread gets its exclusive prefix and the block total
__device__ __forceinline__ void block_scan_ff(ff v, ff *wtot, ff &excl, ff &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const ff incl = scan32_ff(v, lane);
  __syncthreads();
  if (lane == 31) wtot[warp] = incl;
  __syncthreads();
  const ff wi = scan32_ff(lane < kFinWarps ? wtot[lane] : ff{0.f, 0.f}, lane);   // every warp, same bits
  const ff wex{__shfl_sync(0xffffffffu, wi.hi, (warp + 31) & 31), __shfl_sync(0xffffffffu, wi.lo, (warp + 31) & 31)};
  const ff w_off = warp == 0 ? ff{0.f, 0.f} : wex;
  const ff tex{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
  excl = ff_add(w_off, lane == 0 ? ff{0.f, 0.f} : tex);
  total = ff{__shfl_sync(0xffffffffu, wi.hi, kFinWarps - 1), __shfl_sync(0xffffffffu, wi.lo, kFinWarps - 1)};
}

// Warps of a CTA shared among n items (rows or draws): with n <= kFinWarps,
// item j gets warps j, j + n, j + 2n, ...; with more, warp w takes items w
// and w + kFinWarps alone. For warp w: its first item, its index in the
// item's group and the group's size in warps.
struct WarpShare { int first, gi, gn; };
__device__ __forceinline__ WarpShare warp_share(int warp, int n) {
  if (n <= kFinWarps) return {warp % n, warp / n, (kFinWarps - 1 - warp % n) / n + 1};
  return {warp, 0, 1};
}

// the per-warp partials of item j, in a fixed order: sum of slot[w][k] over
// the warps of its group
__device__ __forceinline__ ff group_sum(const ff (*slot)[2], int j, int n) {
  if (n > kFinWarps) return slot[j % kFinWarps][j / kFinWarps];
  ff s{0.f, 0.f};
  for (int w = j; w < kFinWarps; w += n) s = ff_add(s, slot[w][0]);
  return s;
}

// stages row[a + t * stride] (-inf from e1 on) for t < 8 into this thread's
// slots st[t][threadIdx.x]: the eight loads are issued together
template <typename T>
__device__ __forceinline__ void stage8(float (*st)[kFinThreads], const T *row, int a, int stride, int e1) {
  float x[8];
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    const int at = a + t * stride;
    x[t] = at < e1 ? to_f32(row[at]) : -INFINITY;
  }
#pragma unroll
  for (int t = 0; t < 8; ++t) st[t][threadIdx.x] = x[t];
}

template <typename TT, int DK>
__global__ void __launch_bounds__(kFinThreads, 1) sample_finish_kernel(const __grid_constant__ SampleParams P) {
  pdl_wait();
  pdl_trigger();
  using TD = typename std::conditional<DK == 0, TT, float>::type;
  __shared__ ff red[32];
  __shared__ float2 tbl[64];
  __shared__ int sync_flag, n_units, n_draws, n_pend;
  // sequences being resolved (the same in every CTA)
  __shared__ int e_b[kMaxEntries], e_i[kMaxEntries], e_state[kMaxEntries];
  __shared__ int e_nu[kMaxEntries], e_u0[kMaxEntries], e_du[kMaxEntries], e_dr[kMaxEntries];
  // rows evaluated this round: sequence, row, whether it is an accept test,
  // the test's inputs, its verdict and the row sums
  __shared__ int u_e[kMaxUnits], u_row[kMaxUnits], u_test[kMaxUnits], u_acc[kMaxUnits];
  __shared__ float u_lpx[kMaxUnits], u_lqx[kMaxUnits], u_u[kMaxUnits];
  __shared__ ff u_sp[kMaxUnits], u_sq[kMaxUnits];
  // draws of this round: sequence, unit, weight mode, owner CTA, its lower
  // bound, the threshold v Z
  __shared__ int d_e[kMaxEntries], d_u[kMaxEntries], d_mode[kMaxEntries], d_own[kMaxEntries];
  __shared__ ff d_off[kMaxEntries], d_thr[kMaxEntries];
  // per-warp partials (two slots: a warp serves at most two items)
  __shared__ ff w_a[kFinWarps][2], w_b[kFinWarps][2];
  __shared__ int w_last[kFinWarps][2];
  __shared__ int pick, found;
  // per-thread staging of a batch of eight loaded logits (target, draft)
  __shared__ float stg[2][8][kFinThreads];

  const int nb = gridDim.x, cta = blockIdx.x;
  const int K = P.K, V = P.V;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool force = (P.flags & SV_SAMPLE_FORCE_EXACT) != 0;
  if (tid < 64) tbl[tid] = P.tbl[tid];
  if (tid == 0) n_pend = min((int)__ldcg(&P.fin_sync[2]), P.B);
  unsigned gen = 0;   // arrivals the next barrier waits for (thread 0)
  const FfK fk = ff_consts(P);
  // this CTA's chunk of every row; in the owner's search thread t takes
  // elements [a0, a1) of it
  const int chunk = (int)align_up((size_t)((V + nb - 1) / nb), 8);
  const int e0 = min(V, cta * chunk), e1 = min(V, e0 + chunk);
  const int per_t = (chunk + kFinThreads - 1) / kFinThreads;
  const int a0 = min(e1, e0 + tid * per_t), a1 = min(e1, a0 + per_t);
  bool grid_ok = true;
  __syncthreads();
  const int np = n_pend;

  for (int base = 0; base < np; base += kMaxEntries) {
    const int ne = min(kMaxEntries, np - base);
    if (tid < ne) {
      const int2 pe = __ldcg(P.pend + base + tid);
      e_b[tid] = pe.x;
      e_i[tid] = pe.y;
      e_state[tid] = ENT_WALK;
    }
    __syncthreads();
    // every round resolves a sequence or moves its walk past one row at least
    for (int iter = 0; iter <= K + 2; ++iter) {
      // ---- rows each sequence may still need -------------------------------
      if (tid < ne) {
        int nu = 0;
        if (e_state[tid] == ENT_REDRAW) {
          nu = 1;
        } else if (e_state[tid] == ENT_WALK) {
          const RowRec *recs = P.recs + (int64_t)e_b[tid] * (K + 1);
          for (int r = e_i[tid]; r <= K; ++r) {
            const uint32_t f = recs[r].flags;
            if (r < K && (force || !(f & REC_ACC_CERT))) { ++nu; continue; }
            if (r < K && (f & REC_ACCEPT)) continue;
            if (force || !(f & REC_DRAW_CERT)) ++nu;
            else if (nu == 0) {   // the walk ends on a certified draw
              e_state[tid] = ENT_DONE;
              if (cta == 0) write_outputs(P, e_b[tid], r, recs[r].y);
            }
            break;
          }
        }
        e_nu[tid] = nu;
      }
      __syncthreads();
      if (tid == 0) {   // shares of the round's rows, in list order
        int left = 0, used = 0;
        for (int e = 0; e < ne; ++e) left += e_nu[e] > 0;
        for (int e = 0; e < ne; ++e) {
          if (e_nu[e] == 0) continue;
          --left;
          const int take = min(e_nu[e], kMaxUnits - used - left);
          e_u0[e] = used;
          e_nu[e] = take;
          used += take;
        }
        n_units = used;
      }
      __syncthreads();
      const int U = n_units;
      if (U == 0) break;
      if (tid < ne && e_nu[tid] > 0) {   // this sequence's units
        int k = e_u0[tid];
        const int kend = k + e_nu[tid];
        if (e_state[tid] == ENT_REDRAW) {
          u_e[k] = tid; u_row[k] = e_i[tid]; u_test[k] = 0;
        } else {
          const RowRec *recs = P.recs + (int64_t)e_b[tid] * (K + 1);
          for (int r = e_i[tid]; r <= K && k < kend; ++r) {
            const uint32_t f = recs[r].flags;
            const bool test = r < K && (force || !(f & REC_ACC_CERT));
            if (!test && r < K && (f & REC_ACCEPT)) continue;
            if (!test && !force && (f & REC_DRAW_CERT)) break;   // certified: no unit
            u_e[k] = tid; u_row[k] = r; u_test[k] = test ? 1 : 0;
            ++k;
            if (!test) break;
          }
        }
      }
      __syncthreads();

      // ---- step 1: chunk sums of e_p and e_q of every unit ------------------
      {
        const WarpShare ws = warp_share(warp, U);
        for (int k = ws.first, slot = 0; k < U; k += kFinWarps, ++slot) {
          const int bb = e_b[u_e[k]], r = u_row[k];
          const bool q_logits = DK == 0 && r < K && e_state[u_e[k]] == ENT_WALK;
          const TT *trow = static_cast<const TT *>(P.target) + ((int64_t)bb * (K + 1) + r) * V;
          const TD *drow = r < K ? static_cast<const TD *>(P.draft) + ((int64_t)bb * K + r) * V : nullptr;
          if (ws.gi == 0 && lane == 0 && u_test[k]) {   // inputs of the accept test
            const int x = min(max(P.tokens[(int64_t)bb * K + r], 0), V - 1);
            u_lpx[k] = to_f32(trow[x]);
            u_lqx[k] = to_f32(drow[x]);
            u_u[k] = P.uniforms[((int64_t)bb * (K + 1) + r) * 2];
          }
          const float m_p = P.recs[(int64_t)bb * (K + 1) + r].m_p, m_q = P.recs[(int64_t)bb * (K + 1) + r].m_q;
          const int stride = ws.gn * 32;
          ff sp{0.f, 0.f}, sq{0.f, 0.f};
          for (int a = e0 + ws.gi * 32 + lane; a < e1; a += 8 * stride) {
            stage8(stg[0], trow, a, stride, e1);
            if (q_logits) stage8(stg[1], drow, a, stride, e1);
#pragma unroll 1
            for (int t = 0; t < 8; ++t) {
              acc_add(sp, ffx_exp(stg[0][t][tid], m_p, fk, tbl));
              if (q_logits) acc_add(sq, ffx_exp(stg[1][t][tid], m_q, fk, tbl));
            }
          }
          sp = warp_sum_ff(ff_norm(sp));
          sq = warp_sum_ff(ff_norm(sq));
          if (lane == 0) { w_a[warp][slot] = sp; w_b[warp][slot] = sq; }
        }
        __syncthreads();
        if (tid < U) {
          const ff sp = group_sum(w_a, tid, U), sq = group_sum(w_b, tid, U);
          float4 *dst = reinterpret_cast<float4 *>(P.fin_sum + ((size_t)tid * kMaxFinCtas + cta) * 2);
          *dst = make_float4(sp.hi, sp.lo, sq.hi, sq.lo);
        }
      }
      grid_ok = grid_sync(P.fin_sync, gen, &sync_flag, P.wait_ns,
                          cta == 0 && (P.withhold & SV_TEST_WITHHOLD_ARRIVALS)) && grid_ok;
      if (!grid_ok) break;   // a barrier gave up: no further waits in this launch

      // ---- step 2: row sums and exact accept tests (warp per unit; lanes
      // stride the CTAs, the same order in every CTA) -------------------------
      for (int k = warp; k < U; k += kFinWarps) {
        float4 v[(kMaxFinCtas + 31) / 32];
#pragma unroll
        for (int q = 0; q < (kMaxFinCtas + 31) / 32; ++q) {
          const int c = lane + 32 * q;
          v[q] = c < nb ? __ldcg(reinterpret_cast<const float4 *>(P.fin_sum + ((size_t)k * kMaxFinCtas + c) * 2))
                        : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        ff sp{0.f, 0.f}, sq{0.f, 0.f};
#pragma unroll
        for (int q = 0; q < (kMaxFinCtas + 31) / 32; ++q) {
          sp = ff_add(sp, ff{v[q].x, v[q].y});
          sq = ff_add(sq, ff{v[q].z, v[q].w});
        }
        sp = warp_sum_ff(sp);
        sq = warp_sum_ff(sq);
        if (lane == 0) {
          const int bb = e_b[u_e[k]], r = u_row[k];
          if (!(DK == 0 && r < K && e_state[u_e[k]] == ENT_WALK)) sq = ff{1.f, 0.f};
          u_sp[k] = sp;
          u_sq[k] = sq;
          int acc = 0;
          if (u_test[k]) {
            // u q(x) < p(x)  <=>  u e_q(x) S_p < e_p(x) S_q   (draft logits)
            //                <=>  u q(x) S_p < e_p(x)         (draft probabilities)
            const RowRec &rr = P.recs[(int64_t)bb * (K + 1) + r];
            const float u = u_u[k], lq_x = u_lqx[k];
            const ff epx = ff_norm(ffx_exp(u_lpx[k], rr.m_p, fk, tbl));
            ff lhs, rhs;
            if (DK == 0) {
              lhs = ff_mul(ff_mul(ff{u, 0.f}, ff_norm(ffx_exp(lq_x, rr.m_q, fk, tbl))), sp);
              rhs = ff_mul(epx, sq);
            } else {
              lhs = ff_mul(ff{u, 0.f}, ff_mul(ff{lq_x, 0.f}, sp));
              rhs = epx;
            }
            acc = ff_gt(rhs, lhs) ? 1 : 0;
          }
          u_acc[k] = acc;
        }
      }
      __syncthreads();
      // each sequence walks its units: the first exact rejection, or the row
      // it ends on, is its draw; a walk that runs out of units continues next
      // round
      if (tid < ne) {
        int du = -1, dr = -1;
        if (e_nu[tid] > 0) {
          const int bb = e_b[tid];
          int k = e_u0[tid];
          const int kend = k + e_nu[tid];
          if (e_state[tid] == ENT_REDRAW) {
            du = k; dr = e_i[tid];
          } else {
            RowRec *recs = P.recs + (int64_t)bb * (K + 1);
            int r = e_i[tid];
            for (; r <= K; ++r) {
              const uint32_t f = recs[r].flags;
              const bool test = r < K && (force || !(f & REC_ACC_CERT));
              if (!test && r < K && (f & REC_ACCEPT)) continue;
              if (!test && !force && (f & REC_DRAW_CERT)) {   // ends on a certified draw
                e_state[tid] = ENT_DONE;
                if (cta == 0) write_outputs(P, bb, r, recs[r].y);
                break;
              }
              if (k == kend) break;   // out of units: resume here
              if (test) {
                if (cta == 0) recs[r].flags = f | REC_EXACT_ACC;
                if (u_acc[k]) { ++k; continue; }
              }
              du = k; dr = r;
              break;
            }
            if (du < 0 && e_state[tid] == ENT_WALK) e_i[tid] = r;
          }
        }
        e_du[tid] = du;
        e_dr[tid] = dr;
      }
      __syncthreads();
      if (tid == 0) {   // draws of this round, in list order
        int nd = 0;
        for (int e = 0; e < ne; ++e) {
          if (e_du[e] < 0) continue;
          d_e[nd] = e;
          d_u[nd] = e_du[e];
          d_mode[nd] = e_state[e] == ENT_WALK && e_dr[e] < K ? (DK == 0 ? 1 : 2) : 0;
          ++nd;
        }
        n_draws = nd;
      }
      __syncthreads();
      const int D = n_draws;
      // chunk totals of the residual weights and their last positive index
      {
        const WarpShare ws = warp_share(warp, max(D, 1));
        for (int j = ws.first, slot = 0; j < D; j += kFinWarps, ++slot) {
          const int e = d_e[j], k = d_u[j], mode = d_mode[j];
          const int bb = e_b[e], r = e_dr[e];
          const float m_p = P.recs[(int64_t)bb * (K + 1) + r].m_p, m_q = P.recs[(int64_t)bb * (K + 1) + r].m_q;
          const TT *trow = static_cast<const TT *>(P.target) + ((int64_t)bb * (K + 1) + r) * V;
          const TD *drow = r < K ? static_cast<const TD *>(P.draft) + ((int64_t)bb * K + r) * V : nullptr;
          const ff Sp = u_sp[k], Sq = u_sq[k];
          const int stride = ws.gn * 32;
          ff t{0.f, 0.f};
          int last = -1;
          for (int a = e0 + ws.gi * 32 + lane; a < e1; a += 8 * stride) {
            stage8(stg[0], trow, a, stride, e1);
            if (mode != 0) stage8(stg[1], drow, a, stride, e1);
#pragma unroll 1
            for (int s8 = 0; s8 < 8; ++s8) {
              const ff w = resid_weight(mode, stg[0][s8][tid], mode != 0 ? stg[1][s8][tid] : 0.f, m_p, m_q, Sp, Sq,
                                        fk, tbl);
              acc_add(t, w);
              if (w.hi > 0.f) last = a + s8 * stride;
            }
          }
          t = warp_sum_ff(ff_norm(t));
          last = warp_max_s32(last);
          if (lane == 0) { w_a[warp][slot] = t; w_last[warp][slot] = last; }
        }
        __syncthreads();
        if (tid < D) {
          const ff t = group_sum(w_a, tid, D);
          int m = -1;
          if (D > kFinWarps) m = w_last[tid % kFinWarps][tid / kFinWarps];
          else for (int w = tid; w < kFinWarps; w += D) m = max(m, w_last[w][0]);
          P.fin_tot[(size_t)tid * kMaxFinCtas + cta] = make_float2(t.hi, t.lo);
          P.fin_last[(size_t)tid * kMaxFinCtas + cta] = m;
        }
      }
      grid_ok = grid_sync(P.fin_sync, gen, &sync_flag, P.wait_ns,
                          cta == 0 && (P.withhold & SV_TEST_WITHHOLD_ARRIVALS)) && grid_ok;
      if (!grid_ok) break;   // a barrier gave up: no further waits in this launch

      // ---- step 3: prefix over chunks (warp per draw) -----------------------
      // lane l sums CTAs [l per_l, (l+1) per_l) in order, lanes are scanned
      // in a fixed order, and the CTAs of the lane holding v Z chain their
      // boundaries in order (the last one closes on the next lane's start)
      for (int j = warp; j < D; j += kFinWarps) {
        const int e = d_e[j], bb = e_b[e], r = e_dr[e];
        const float2 *tot = P.fin_tot + (size_t)j * kMaxFinCtas;
        const int per_l = (nb + 31) / 32;   // <= 5
        ff tv[(kMaxFinCtas + 31) / 32];
        ff run{0.f, 0.f};
#pragma unroll
        for (int q = 0; q < (kMaxFinCtas + 31) / 32; ++q) {
          const int c = lane * per_l + q;
          tv[q] = q < per_l && c < nb ? ldcg_ff(tot + c) : ff{0.f, 0.f};
        }
        const float v_u = P.uniforms[((int64_t)bb * (K + 1) + r) * 2 + 1];
#pragma unroll
        for (int q = 0; q < (kMaxFinCtas + 31) / 32; ++q) run = ff_add(run, tv[q]);
        const ff incl = scan32_ff(run, lane);
        const ff XZ{__shfl_sync(0xffffffffu, incl.hi, 31), __shfl_sync(0xffffffffu, incl.lo, 31)};
        const ff tex{__shfl_up_sync(0xffffffffu, incl.hi, 1), __shfl_up_sync(0xffffffffu, incl.lo, 1)};
        const ff excl = lane == 0 ? ff{0.f, 0.f} : tex;
        int own = -2;   // zero residual mass
        ff s0{0.f, 0.f}, xthr{0.f, 0.f};
        if (ff_pos(XZ)) {
          xthr = ff_mul(ff{v_u, 0.f}, XZ);
          const unsigned past = __ballot_sync(0xffffffffu, ff_gt(incl, xthr));
          const int L = past ? __ffs(past) - 1 : 31;
          int mine = -1;
          ff lo = excl;
          if (lane == L) {
            const int c_first = L * per_l, c_last = min(nb, (L + 1) * per_l) - 1;
            mine = max(0, c_last);
#pragma unroll
            for (int q = 0; q < (kMaxFinCtas + 31) / 32; ++q) {
              if (c_first + q >= c_last) break;
              const ff s1 = ff_add(lo, tv[q]);
              if (ff_gt(s1, xthr)) { mine = c_first + q; break; }
              lo = s1;
            }
          }
          own = __shfl_sync(0xffffffffu, mine, L);
          s0 = ff{__shfl_sync(0xffffffffu, lo.hi, L), __shfl_sync(0xffffffffu, lo.lo, L)};
        }
        if (lane == 0) { d_own[j] = own; d_off[j] = s0; d_thr[j] = xthr; }
      }
      __syncthreads();
      // the owner CTA finds the token within its chunk and writes the outputs
      for (int j = 0; j < D; ++j) {
        const int e = d_e[j], mode = d_mode[j];
        const int bb = e_b[e], r = e_dr[e];
        if (d_own[j] == -2) {   // zero residual mass: the draw falls back to p
          if (mode == 0 && cta == 0 && tid == 0) {
            write_outputs(P, bb, r, -1);
            P.recs[(int64_t)bb * (K + 1) + r].flags |= REC_EXACT_DRAW;
            P.recs[(int64_t)bb * (K + 1) + r].y_exact = -1;
          }
          continue;
        }
        if (d_own[j] != cta) continue;
        const int k = d_u[j];
        const float m_p = P.recs[(int64_t)bb * (K + 1) + r].m_p, m_q = P.recs[(int64_t)bb * (K + 1) + r].m_q;
        const TT *trow = static_cast<const TT *>(P.target) + ((int64_t)bb * (K + 1) + r) * V;
        const TD *drow = r < K ? static_cast<const TD *>(P.draft) + ((int64_t)bb * K + r) * V : nullptr;
        const ff Sp = u_sp[k], Sq = u_sq[k], xthr = d_thr[j];
        ff t{0.f, 0.f};
        int lastp = -1;
        for (int a = a0; a < a1; a += 8) {
          stage8(stg[0], trow, a, 1, a1);
          if (mode != 0) stage8(stg[1], drow, a, 1, a1);
#pragma unroll 1
          for (int s8 = 0; s8 < 8; ++s8) {
            const ff w = resid_weight(mode, stg[0][s8][tid], mode != 0 ? stg[1][s8][tid] : 0.f, m_p, m_q, Sp, Sq,
                                      fk, tbl);
            acc_add(t, w);
            if (w.hi > 0.f) lastp = a + s8;
          }
        }
        t = ff_norm(t);
        ff excl, total;
        block_scan_ff(t, red, excl, total);
        // the first thread whose upper bound passes v Z
        const ff lo = ff_add(d_off[j], excl);
        const unsigned wb = __ballot_sync(0xffffffffu, ff_gt(ff_add(lo, t), xthr));
        if (lane == 0) w_last[warp][0] = wb ? warp * 32 + __ffs(wb) - 1 : 1 << 30;
        __syncthreads();
        if (tid == 0) {
          int first = 1 << 30;
          for (int w = 0; w < kFinWarps; ++w) first = min(first, w_last[w][0]);
          pick = first;
          found = -1;
        }
        __syncthreads();
        if (tid == pick) {
          int cand = -1;
          ff runc = lo;
          for (int a = a0; a < a1 && cand < 0; ++a) {
            const ff w = resid_weight(mode, to_f32(trow[a]), mode != 0 ? to_f32(drow[a]) : 0.f, m_p, m_q, Sp, Sq, fk,
                                      tbl);
            const ff nxt = ff_add(runc, w);
            if (w.hi > 0.f && ff_gt(nxt, xthr)) cand = a;
            runc = nxt;
          }
          if (cand < 0) cand = lastp;   // crossing within rounding of this thread's end
          found = cand;
        }
        __syncthreads();
        if (tid == 0) {
          // v Z within rounding of the chunk's top: its last positive weight,
          // else the row's
          int y = found;
          if (y < 0) y = __ldcg(P.fin_last + (size_t)j * kMaxFinCtas + cta);
          for (int c = 0; c < nb && y < 0; ++c) y = max(y, __ldcg(P.fin_last + (size_t)j * kMaxFinCtas + c));
          write_outputs(P, bb, r, y);
          P.recs[(int64_t)bb * (K + 1) + r].flags |= REC_EXACT_DRAW;
          P.recs[(int64_t)bb * (K + 1) + r].y_exact = y;
        }
        __syncthreads();
      }
      if (tid < D) {   // state changes, the same in every CTA
        const int e = d_e[tid];
        if (d_own[tid] == -2 && d_mode[tid] != 0) { e_state[e] = ENT_REDRAW; e_i[e] = e_dr[e]; }
        else e_state[e] = ENT_DONE;
      }
      __syncthreads();
    }
    __syncthreads();
    if (!grid_ok) break;
  }
  if (!grid_ok && tid == 0 && cta == 0) atomic_or_status(P.status, SV_DEV_TIMEOUT);
}

// ------------------------------------------------------------------ host ---

size_t records_bytes(int B, int K) { return align_up((size_t)B * (K + 1) * sizeof(RowRec), 256); }

int stat_chunks(int V) { return (V + kStatChunk - 1) / kStatChunk; }

// scratch of the finish grid: barrier words, per-CTA row sums of every unit,
// per-CTA weight totals and last positive indices of every draw
constexpr size_t kFinSyncBytes = 256;
constexpr size_t kFinSumBytes = (size_t)kMaxUnits * kMaxFinCtas * 2 * sizeof(float2);
constexpr size_t kFinTotBytes = (size_t)kMaxEntries * kMaxFinCtas * sizeof(float2);
constexpr size_t kFinLastBytes = (size_t)kMaxEntries * kMaxFinCtas * sizeof(int);
constexpr size_t kFinScratchBytes = kFinSyncBytes + kFinSumBytes + kFinTotBytes + kFinLastBytes;

size_t parts_bytes(int B, int K, int V) { return align_up((size_t)B * (K + 1) * stat_chunks(V) * sizeof(float4), 256); }

size_t pending_bytes(int B) { return align_up((size_t)B * sizeof(int2), 256); }

// per-row records, the chunk statistics, the finish grid's scratch, then the
// list of sequences pending for it
size_t workspace_bytes_for(int B, int K, int V) {
  return records_bytes(B, K) + parts_bytes(B, K, V) + kFinScratchBytes + pending_bytes(B);
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

// Cooperative launch of the finish grid (every CTA resident), staged behind
// the previous launch when the driver accepts both attributes together.
template <typename KernelT>
cudaError_t launch_coop(KernelT kernel, int nb, cudaStream_t s, const SampleParams &P) {
  static int pdl_ok = 1;
  for (;;) {
    cudaLaunchAttribute attr[2];
    int n = 0;
    attr[n].id = cudaLaunchAttributeCooperative;
    attr[n].val.cooperative = 1;
    ++n;
    if (pdl_ok) {
      attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[n].val.programmaticStreamSerializationAllowed = 1;
      ++n;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nb);
    cfg.blockDim = dim3(kFinThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = (unsigned)n;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, P);
    if (e == cudaSuccess) launch_counter().fetch_add(1, std::memory_order_relaxed);
    if (e == cudaSuccess || !pdl_ok) return e;
    (void)cudaGetLastError();   // retry as a plain cooperative launch
    pdl_ok = 0;
  }
}

void split_ff(double d, float &hi, float &lo) {
  hi = (float)d;
  lo = (float)(d - (double)hi);
}


template <typename TT, int DK>
sv_status launch_sample(const SampleParams &P, int cs, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int fin_blocks = 0;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(sample_draw_kernel<TT, DK>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    int per_sm = 0;
    if (attr_err == cudaSuccess)
      attr_err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sample_finish_kernel<TT, DK>, kFinThreads, 0);
    // one CTA per SM (the kernel is bound to one by its registers), all resident
    fin_blocks = std::min(kMaxFinCtas, sm_count() * std::min(per_sm, 1));
  });
  if (attr_err != cudaSuccess)
    return fail(SV_ERR_CUDA, "spec_verify_sample: kernel attributes: %s", cudaGetErrorString(attr_err));
  if (fin_blocks < 1) return fail(SV_ERR_CUDA, "spec_verify_sample: the finish grid does not fit on the device");
  cudaError_t e = launch_k(sample_stats_kernel<TT, DK>, dim3(P.nc, P.K + 1, P.B), dim3(kStatThreads), 0, s, 1, P);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_sample statistics launch: %s", cudaGetErrorString(e));
  e = launch_k(sample_draw_kernel<TT, DK>, dim3(cs, P.B), dim3(kRowThreads), 0, s, cs, P);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_sample draw launch: %s", cudaGetErrorString(e));
  e = launch_coop(sample_finish_kernel<TT, DK>, fin_blocks, s, P);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_sample finish launch: %s", cudaGetErrorString(e));
  return ok();
}

}  // namespace
}  // namespace sv

namespace sv {
namespace {
// Draw-kernel cluster: the smallest (up to 16 CTAs) whose slices take at most
// eight groups of eight elements per thread; gpc = groups per CTA slice.
void draw_shape(int V, int &cs, int &gpc) {
  const int ngr = (V + 7) / 8;
  cs = 1;
  while (cs < 16 && (ngr + cs - 1) / cs > 8 * kRowThreads) cs *= 2;
  gpc = (ngr + cs - 1) / cs;
}

// Host checks of spec_verify_sample's arguments (everything but the workspace).
sv_status check_sample_args(const void *target_logits, sv_dtype logit_dtype, const void *draft,
                            sv_dtype draft_dtype, int draft_is_probs, const int32_t *draft_tokens,
                            const float *uniforms, int B, int K, int V, float temperature,
                            const int32_t *out_tokens, const int32_t *num_accepted) {
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
  int cs, gpc;
  draw_shape(V, cs, gpc);
  if (gpc > kMaxDrawBlocks * 32)
    return fail(SV_ERR_UNSUPPORTED, "spec_verify_sample: vocabulary of %d too large (at most %d)", V,
                16 * kMaxDrawBlocks * 32 * 8);
  return SV_OK;
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
  int cs, gpc;
  draw_shape(V, cs, gpc);

  SampleParams P = {};
  P.target = target_logits; P.draft = draft; P.tokens = draft_tokens; P.uniforms = uniforms;
  P.p_at = p_at_draft; P.q_at = q_at_draft; P.out_tokens = out_tokens; P.num_acc = num_accepted;
  P.recs = static_cast<RowRec *>(workspace); P.status = dev_status;
  P.part = reinterpret_cast<float4 *>(static_cast<uint8_t *>(workspace) + records_bytes(B, K));
  P.nc = stat_chunks(V);
  {
    uint8_t *fin = static_cast<uint8_t *>(workspace) + records_bytes(B, K) + parts_bytes(B, K, V);
    P.fin_sync = reinterpret_cast<unsigned *>(fin);
    P.fin_sum = reinterpret_cast<float2 *>(fin + kFinSyncBytes);
    P.fin_tot = reinterpret_cast<float2 *>(fin + kFinSyncBytes + kFinSumBytes);
    P.fin_last = reinterpret_cast<int *>(fin + kFinSyncBytes + kFinSumBytes + kFinTotBytes);
    P.pend = reinterpret_cast<int2 *>(fin + kFinScratchBytes);
  }
  P.B = B; P.K = K; P.V = V; P.gpc = gpc; P.flags = flags;
  P.wait_ns = wait_limit_ns();
  P.withhold = test_withhold();
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
    case SV_F32: return probs ? launch_sample<float, 1>(P, cs, s) : launch_sample<float, 0>(P, cs, s);
    case SV_BF16: return probs ? launch_sample<__nv_bfloat16, 1>(P, cs, s) : launch_sample<__nv_bfloat16, 0>(P, cs, s);
    default: return probs ? launch_sample<__half, 1>(P, cs, s) : launch_sample<__half, 0>(P, cs, s);
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
constexpr size_t kStaticScratchBytes = 1u << 20;   // 1 MiB: 48 + 16 ceil(V / 8192) bytes per (sequence, position)
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

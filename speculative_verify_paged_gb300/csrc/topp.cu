// Top-p filter of logit rows: every logit outside the row's top-p set becomes
// -inf, so that softmax(filtered / T) is p = softmax(logits / T) truncated to
// that set and renormalised ("KV Cache + Speculative Decoding", section 7.5
// and Q21: under top-p the target distribution is p cut to its own top-p set
// and renormalised, and rejection sampling stays exact with it).
//
// The set: order the tokens by logit, largest first, equal logits by
// ascending token id; keep the shortest prefix whose mass reaches top_p.
// Every token x gets the composite key (ordered logit bits << 32) | (2^32 - 1
// - x), so that order is plain descending order of the composite, and the set
// is {x : composite(x) >= cut} for one cut value.
//
// Masses are the weights 2^((l - m) log2(e) / T) of the row (m its maximum),
// rounded to multiples of 2^-40 and summed as 64-bit integers: the sums, and
// so the set, do not depend on the order of the additions (the kernel is
// deterministic). Each weight is within about 2.2e-7 (relative) of its exact
// value (the SFU exp2, the first-order correction, the rounding to 2^-40), so
// a cumulative mass as a fraction of the row mass is within 5e-7: the set is
// exact unless top_p lies that close to a cumulative mass.
//
// One 512-thread CTA per row. The first pass reads the row from memory; the
// later passes read it again, from L2 (the rows in flight, two CTAs per SM,
// take about a half of it at 128K bf16 logits per row). Passes:
//   1. the row maximum m;
//   2. every thread adds the masses of its logits into its own row of 8
//      coarse bins of 8 binades of weight each (shared memory, no atomics);
//      the block sums them, giving Z and the coarse bin where the running
//      mass reaches ceil(top_p Z);
//   3. a histogram of that coarse bin in fine bins of 1/32 of a binade
//      (shared atomics, only for the logits of that bin) gives the fine bin
//      of the crossing;
//   4. the fine bin's tokens are gathered (if more than 512, the bin is
//      first split by the composite's bits, 8 at a time, until at most 512
//      remain) and ranked by direct comparison of composites: the cut;
//   5. the row is written: logits in fine bins above the cut's bin stay,
//      those below go, the composite decides within it.
// Bins come from one fma of the logit and are non-increasing in it; only
// pass 2 (and the gathered tokens) compute the precise weights.

#include <cmath>
#include <mutex>

#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kTpThreads = 512;
constexpr int kTpWarps = kTpThreads / 32;
constexpr int kTpCoarse = 8;          // coarse bins of kTpFinePer fine bins
constexpr int kTpFinePer = 256;       // 8 binades of 1/32 each
constexpr int kTpFineAll = kTpCoarse * kTpFinePer;
constexpr int kTpCap = 512;           // candidates ranked directly
constexpr int kTpUnroll = 4;          // 16-byte loads in flight per thread
constexpr float kTpQuant = 1099511627776.0f;  // 2^40

typedef unsigned long long u64;

struct TpParams {
  const void *in0;
  void *out0;
  int rows0;
  const void *in1;
  void *out1;
  int V;
  int vec;            // rows are 16-byte aligned: vector loads and stores
  float c_hi, c_lo;   // log2(e) / T as a float-float pair
  double top_p;
  int32_t *status;
};

template <typename T>
struct TpType;
template <>
struct TpType<float> {
  static constexpr int G = 4;
  static constexpr uint32_t kSign = 0x80000000u, kMag = 0x7fffffffu, kInf = 0x7f800000u;
  static constexpr uint32_t kNegInf = 0xff800000u, kKeyMask = 0xffffffffu;
  static constexpr bool kExactDiff = false;   // x - m needs a two-sum
  static __device__ __forceinline__ uint32_t get(const uint4 &r, int k) { return (&r.x)[k]; }
  static __device__ __forceinline__ float val(uint32_t b) { return __uint_as_float(b); }
  static __device__ __forceinline__ uint32_t ld1(const void *p, int e) {
    return __float_as_uint(__ldg(static_cast<const float *>(p) + e));
  }
  static __device__ __forceinline__ void st1(void *p, int e, uint32_t b) { static_cast<uint32_t *>(p)[e] = b; }
};
template <>
struct TpType<__nv_bfloat16> {
  static constexpr int G = 8;
  static constexpr uint32_t kSign = 0x8000u, kMag = 0x7fffu, kInf = 0x7f80u;
  static constexpr uint32_t kNegInf = 0xff80u, kKeyMask = 0xffffu;
  // x - m of two bf16 values is exact in fp32 unless their binades are more
  // than 16 apart; then |x| < 2^-16 |m| and the rounding (an ulp of m) moves
  // the weight of such a token by ~1e-6 relative, and such tokens carry a
  // negligible share of the mass
  static constexpr bool kExactDiff = true;
  static __device__ __forceinline__ uint32_t get(const uint4 &r, int k) {
    const uint32_t w = (&r.x)[k >> 1];
    return (k & 1) ? (w >> 16) : (w & 0xffffu);
  }
  static __device__ __forceinline__ float val(uint32_t b) { return __uint_as_float(b << 16); }
  static __device__ __forceinline__ uint32_t ld1(const void *p, int e) {
    return (uint32_t)__ldg(static_cast<const unsigned short *>(p) + e);
  }
  static __device__ __forceinline__ void st1(void *p, int e, uint32_t b) {
    static_cast<unsigned short *>(p)[e] = (unsigned short)b;
  }
};
template <>
struct TpType<__half> {
  static constexpr int G = 8;
  static constexpr uint32_t kSign = 0x8000u, kMag = 0x7fffu, kInf = 0x7c00u;
  static constexpr uint32_t kNegInf = 0xfc00u, kKeyMask = 0xffffu;
  static constexpr bool kExactDiff = true;    // 11-bit significands: as for bf16
  static __device__ __forceinline__ uint32_t get(const uint4 &r, int k) {
    const uint32_t w = (&r.x)[k >> 1];
    return (k & 1) ? (w >> 16) : (w & 0xffffu);
  }
  static __device__ __forceinline__ float val(uint32_t b) {
    return __half2float(__ushort_as_half((unsigned short)b));
  }
  static __device__ __forceinline__ uint32_t ld1(const void *p, int e) {
    return (uint32_t)__ldg(static_cast<const unsigned short *>(p) + e);
  }
  static __device__ __forceinline__ void st1(void *p, int e, uint32_t b) {
    static_cast<unsigned short *>(p)[e] = (unsigned short)b;
  }
};

__device__ __forceinline__ float tp_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Canonical bits: NaN becomes -inf (and is reported), -0 becomes +0.
template <typename T>
__device__ __forceinline__ uint32_t tp_canon(uint32_t b, bool &nan) {
  using TT = TpType<T>;
  nan = (b & TT::kMag) > TT::kInf;
  if (nan) b = TT::kNegInf;
  if (b == TT::kSign) b = 0u;
  return b;
}

template <typename T>
__device__ __forceinline__ u64 tp_composite(uint32_t canon, int id) {
  using TT = TpType<T>;
  const uint32_t key = (canon & TT::kSign) ? (~canon & TT::kKeyMask) : (canon | TT::kSign);
  return ((u64)key << 32) | (u64)(0xffffffffu - (uint32_t)id);
}

// Calls f(e0, r, nv) for every group of a row of V elements: r holds the
// elements e0 .. e0 + nv - 1 packed as in memory (nv = G except in the last
// group). Full 16-byte groups go round-robin over the threads, kTpUnroll
// loads in flight per thread; the ragged end (and the whole row when it is
// not 16-byte aligned) is loaded one element at a time.
template <typename T, typename F>
__device__ __forceinline__ void tp_row_groups(const void *row, int V, int vec, F f) {
  using TT = TpType<T>;
  constexpr int G = TT::G;
  const int ng = vec ? V / G : 0;
  const uint4 *rv = static_cast<const uint4 *>(row);
  int g = threadIdx.x;
  for (; g + (kTpUnroll - 1) * kTpThreads < ng; g += kTpUnroll * kTpThreads) {
    uint4 r[kTpUnroll];
#pragma unroll
    for (int u = 0; u < kTpUnroll; ++u) r[u] = __ldg(rv + g + u * kTpThreads);
#pragma unroll
    for (int u = 0; u < kTpUnroll; ++u) f((g + u * kTpThreads) * G, r[u], G);
  }
  for (; g < ng; g += kTpThreads) f(g * G, __ldg(rv + g), G);
  for (int h = ng + (int)threadIdx.x; h * G < V; h += kTpThreads) {
    const int nv = min(G, V - h * G);
    uint4 r = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int k = 0; k < G; ++k) {
      if (k < nv) {
        const uint32_t b = TT::ld1(row, h * G + k);
        if (sizeof(T) == 4) (&r.x)[k] = b;
        else (&r.x)[k >> 1] |= b << ((k & 1) * 16);
      }
    }
    f(h * G, r, nv);
  }
}

// Exclusive scan over the block of one u64 per thread; *total is the sum.
__device__ __forceinline__ u64 tp_block_excl_scan(u64 v, u64 *s_warp, u64 *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  u64 incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const u64 t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[warp] = incl;
  __syncthreads();
  u64 before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kTpWarps; ++w) {
    const u64 x = s_warp[w];
    if (w < warp) before += x;
    tot += x;
  }
  __syncthreads();
  *total = tot;
  return before + incl - v;
}

// Over entries h[phys(0)], h[phys(1)], ... (n <= kTpThreads of them, thread
// i holding entry i), the entry where the running mass from `above` first
// reaches thr: writes phys(i) to *s_sel and the mass before it to *s_above.
template <typename Phys>
__device__ __forceinline__ void tp_cross(const u64 *h, int n, Phys phys, u64 above, u64 thr, u64 *s_warp,
                                         int *s_sel, u64 *s_above) {
  const int i = threadIdx.x;
  const u64 mine = i < n ? h[phys(i)] : 0ull;
  u64 tot;
  const u64 cum = above + tp_block_excl_scan(mine, s_warp, &tot);
  if (i < n && cum < thr && thr <= cum + mine) {
    *s_sel = phys(i);
    *s_above = cum;
  }
  __syncthreads();
}

template <typename T>
__global__ void __launch_bounds__(kTpThreads, 2) topp_row_kernel(const __grid_constant__ TpParams P) {
  using TT = TpType<T>;
  __shared__ u64 acc[kTpCoarse][kTpThreads];   // per-thread coarse masses
  __shared__ u64 h_fine[256];                  // fine (or radix) histogram
  __shared__ u64 c_comp[kTpCap];               // gathered candidates
  __shared__ u64 c_q[kTpCap];
  __shared__ u64 s_warp64[kTpWarps];
  __shared__ float s_wmax[kTpWarps];
  __shared__ int s_wflag[kTpWarps];
  __shared__ int s_sel;
  __shared__ u64 s_above;
  __shared__ u64 s_cut;
  __shared__ unsigned s_count;

  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x;
  const void *in;
  void *out;
  if (row < P.rows0) {
    in = static_cast<const T *>(P.in0) + (int64_t)row * P.V;
    out = static_cast<T *>(P.out0) + (int64_t)row * P.V;
  } else {
    in = static_cast<const T *>(P.in1) + (int64_t)(row - P.rows0) * P.V;
    out = static_cast<T *>(P.out1) + (int64_t)(row - P.rows0) * P.V;
  }
  const int V = P.V;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  // ---- 1. row maximum (NaN is flagged; fmaxf ignores it) ----
  float mx = -INFINITY;
  int flag = 0;
  tp_row_groups<T>(in, V, P.vec, [&](int, const uint4 &r, int nv) {
#pragma unroll
    for (int k = 0; k < TT::G; ++k) {
      if (k < nv) {
        const uint32_t b = TT::get(r, k);
        const float x = TT::val(b);
        flag |= ((b & TT::kMag) > TT::kInf) ? 1 : 0;
        flag |= (x == INFINITY) ? 2 : 0;
        mx = fmaxf(mx, x);
      }
    }
  });
  mx = warp_max(mx);
  flag = (int)__reduce_or_sync(0xffffffffu, (unsigned)flag);
  if (lane == 0) { s_wmax[warp] = mx; s_wflag[warp] = flag; }
  for (int i = threadIdx.x; i < kTpCoarse * kTpThreads; i += kTpThreads) (&acc[0][0])[i] = 0ull;
  if (threadIdx.x == 0) { s_count = 0u; s_sel = -1; s_above = 0ull; s_cut = 0ull; }
  __syncthreads();
  float m = -INFINITY;
  flag = 0;
#pragma unroll
  for (int w = 0; w < kTpWarps; ++w) { m = fmaxf(m, s_wmax[w]); flag |= s_wflag[w]; }
  if (flag && threadIdx.x == 0) atomic_or_status(P.status, SV_DEV_NONFINITE);

  if (!(m > -INFINITY) || m == INFINITY) {
    // nothing to rank (no finite logit, or a +inf one): the row is passed
    // through unchanged and the sampling flags it
    if (out != in)
      tp_row_groups<T>(in, V, 0, [&](int e0, const uint4 &r, int nv) {
#pragma unroll
        for (int k = 0; k < TT::G; ++k)
          if (k < nv) TT::st1(out, e0 + k, TT::get(r, k));
      });
    return;
  }

  // Fine bin of a logit x: round(32 (fl(m c_hi) - x c_hi)) from one fma onto
  // the integer grid of [2^23, 2^24), capped at the last fine bin; it is
  // non-increasing in x, needs no conversion instruction, and puts -inf and
  // NaN (fminf drops the NaN) in the last bin, which takes no mass.
  // Weight: 2^ex with ex = (x - m) c taken as hi + lo (c = c_hi + c_lo, an fma
  // for the product's rounding, a two-sum for x - m where it is not exact);
  // 2^hi from the SFU (relative error below 1.5e-7 on [-30, 0]), 2^lo as the
  // first-order factor 1 + lo ln 2 (|lo| is about an ulp of hi).
  const float c_hi = P.c_hi, c_lo = P.c_lo;
  const float mc = __fmul_rn(m, c_hi);
  const float c32 = 32.f * c_hi;                    // exact (a power of two)
  const float mc32 = fmaf(32.f, mc, 8388608.f);     // 32 mc + 2^23, exact when |32 mc| < 2^22
  const float top = 8388608.f + (float)(kTpFineAll - 1);
  // (fminf first, so NaN goes to the last bin; the fmaxf keeps bins >= 0 when
  // the rounding of mc32 at huge |m c| pushes the maximum just below 2^23)
  auto fine_of = [&](float x) {
    return __float_as_int(fmaxf(fminf(fmaf(-x, c32, mc32), top), 8388608.f)) - 0x4B000000;
  };
  auto mass_of = [&](float x) -> u64 {
    const float d = x - m;
    float d_lo = 0.f;
    if (!TT::kExactDiff) {
      const float bb = d - x;
      d_lo = (x - (d - bb)) + (-m - bb);
    }
    const float h = d * c_hi;
    float l = fmaf(d, c_hi, -h);
    l = fmaf(d, c_lo, l);
    if (!TT::kExactDiff) l = fmaf(d_lo, c_hi, l);
    const float t = tp_ex2(h);
    if (!(t > 0.f)) return 0ull;   // also -inf and NaN
    return __float2ull_rn(fmaf(t, l * 0.693147180559945309f, t) * kTpQuant);
  };
  auto comp_of = [&](uint32_t b, int e) {
    bool nan;
    return tp_composite<T>(tp_canon<T>(b, nan), e);
  };

  // ---- 2. coarse masses, private per thread ----
  u64 *my_acc = &acc[0][threadIdx.x];
  tp_row_groups<T>(in, V, P.vec, [&](int, const uint4 &r, int nv) {
#pragma unroll
    for (int k = 0; k < TT::G; ++k) {
      if (k < nv) {
        const float x = TT::val(TT::get(r, k));
        const int fb = fine_of(x);
        if (fb < kTpFineAll - 1) my_acc[(fb >> 8) * kTpThreads] += mass_of(x);
      }
    }
  });
  __syncthreads();
  // block sums of the coarse bins: warp w adds half of bin w / 2
  {
    const int cb = warp >> 1, base = (warp & 1) * (kTpThreads / 2);
    u64 sum = 0;
#pragma unroll
    for (int j = 0; j < kTpThreads / 64; ++j) sum += acc[cb][base + lane + 32 * j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane == 0) s_warp64[warp] = sum;
  }
  __syncthreads();
  u64 coarse[kTpCoarse];
  u64 Z = 0;
#pragma unroll
  for (int c = 0; c < kTpCoarse; ++c) {
    coarse[c] = s_warp64[2 * c] + s_warp64[2 * c + 1];
    Z += coarse[c];
  }
  u64 thr = (u64)ceil(P.top_p * (double)Z);
  thr = thr < 1ull ? 1ull : (thr > Z ? Z : thr);
  int cbin = -1;
  u64 above = 0;
  {
    u64 cum = 0;
#pragma unroll
    for (int c = 0; c < kTpCoarse; ++c) {
      if (cbin < 0 && cum < thr && thr <= cum + coarse[c]) { cbin = c; above = cum; }
      cum += coarse[c];
    }
  }
  __syncthreads();   // s_warp64 is reused below

  // ---- 3. fine histogram of the crossing coarse bin ----
  for (int i = threadIdx.x; i < kTpFinePer; i += kTpThreads) h_fine[i] = 0ull;
  __syncthreads();
  const int f0 = cbin * kTpFinePer;
  tp_row_groups<T>(in, V, P.vec, [&](int, const uint4 &r, int nv) {
#pragma unroll
    for (int k = 0; k < TT::G; ++k) {
      if (k < nv) {
        const float x = TT::val(TT::get(r, k));
        const unsigned rel = (unsigned)(fine_of(x) - f0);
        if (rel < (unsigned)kTpFinePer) {
          const u64 q = mass_of(x);
          if (q) atomicAdd(&h_fine[rel], q);
        }
      }
    }
  });
  __syncthreads();
  tp_cross(h_fine, kTpFinePer, [](int i) { return i; }, above, thr, s_warp64, &s_sel, &s_above);
  const int fbin = s_sel >= 0 ? f0 + s_sel : -1;   // -1 only if nothing reached thr (not expected)
  above = s_above;

  // ---- 4. gather the fine bin's tokens (one vote per group) and rank them ----
  int sh = 64;        // radix split: the composite's bits at and above sh equal pfx
  u64 pfx = 0ull;
  auto gather_pass = [&]() {
    tp_row_groups<T>(in, V, P.vec, [&](int e0, const uint4 &r, int nv) {
      unsigned cm = 0;
#pragma unroll
      for (int k = 0; k < TT::G; ++k) {
        if (k < nv && fine_of(TT::val(TT::get(r, k))) == fbin &&
            (sh >= 64 || (comp_of(TT::get(r, k), e0 + k) >> sh) == pfx))
          cm |= 1u << k;
      }
      const unsigned am = __activemask();
      if (!__ballot_sync(am, cm != 0u)) return;
#pragma unroll 1
      for (int k = 0; k < TT::G; ++k) {
        const bool cand = (cm >> k) & 1u;
        const unsigned bal = __ballot_sync(am, cand);
        if (!bal) continue;
        const int leader = __ffs(bal) - 1;
        unsigned base = 0;
        if (lane == leader) base = atomicAdd(&s_count, (unsigned)__popc(bal));
        base = __shfl_sync(am, base, leader);
        if (cand) {
          const unsigned slot = base + (unsigned)__popc(bal & ((1u << lane) - 1u));
          if (slot < (unsigned)kTpCap) {
            const uint32_t b = TT::get(r, k);
            c_comp[slot] = comp_of(b, e0 + k);
            c_q[slot] = mass_of(TT::val(b));
          }
        }
      }
    });
    __syncthreads();
  };
  gather_pass();
  int n_all = (int)s_count;
  while (n_all > kTpCap && sh > 0) {
    // Rare: more than kTpCap tokens in the fine bin (many equal or nearly
    // equal logits). Split them by the next 8 bits of the composite, keep the
    // part where the running mass reaches thr, and gather again.
    const int nsh = sh > 8 ? sh - 8 : 0;
    const int width = sh - nsh;
    for (int i = threadIdx.x; i < 256; i += kTpThreads) h_fine[i] = 0ull;
    if (threadIdx.x == 0) { s_count = 0u; s_sel = -1; }
    __syncthreads();
    tp_row_groups<T>(in, V, P.vec, [&](int e0, const uint4 &r, int nv) {
#pragma unroll
      for (int k = 0; k < TT::G; ++k) {
        if (k < nv) {
          const uint32_t b = TT::get(r, k);
          const float x = TT::val(b);
          if (fine_of(x) != fbin) continue;
          const u64 comp = comp_of(b, e0 + k);
          if (sh < 64 && (comp >> sh) != pfx) continue;
          const u64 q = mass_of(x);
          if (q) atomicAdd(&h_fine[(int)((comp >> nsh) & ((1ull << width) - 1ull))], q);
        }
      }
    });
    __syncthreads();
    tp_cross(h_fine, 256, [](int i) { return 255 - i; }, above, thr, s_warp64, &s_sel, &s_above);
    above = s_above;
    pfx = (sh >= 64 ? 0ull : (pfx << width)) | (u64)(s_sel < 0 ? 0 : s_sel);
    sh = nsh;
    gather_pass();
    n_all = (int)s_count;
  }
  if (n_all <= kTpCap) {
    // candidate i is the cut iff the mass before it (everything in higher
    // bins and radix parts, plus every candidate with a larger composite) is
    // below thr and reaches thr with it
    for (int i = threadIdx.x; i < n_all; i += kTpThreads) {
      const u64 ci = c_comp[i], qi = c_q[i];
      u64 before = 0;
      for (int j = 0; j < n_all; ++j) before += (c_comp[j] > ci) ? c_q[j] : 0ull;
      if (above + before < thr && thr <= above + before + qi) s_cut = ci;
    }
  }
  __syncthreads();
  const u64 cut = s_cut;   // 0: no cut found, the row is kept whole

  // ---- 5. write the filtered row: fine bins above the cut's stay, bins
  // below go (NaN and -inf are in the last bin), the composite decides in it ----
  tp_row_groups<T>(in, V, P.vec, [&](int e0, const uint4 &r, int nv) {
    uint32_t ob[TT::G];
#pragma unroll
    for (int k = 0; k < TT::G; ++k) {
      const uint32_t b = TT::get(r, k);
      const int fb = fine_of(TT::val(b));
      const bool nan = (b & TT::kMag) > TT::kInf;
      const bool keep = cut == 0ull ? !nan : (fb < fbin || (fb == fbin && comp_of(b, e0 + k) >= cut));
      ob[k] = keep ? b : TT::kNegInf;
    }
    if (P.vec && nv == TT::G) {
      uint4 o;
      if (sizeof(T) == 4) {
        o = make_uint4(ob[0], ob[1 % TT::G], ob[2 % TT::G], ob[3 % TT::G]);
      } else {
#pragma unroll
        for (int k = 0; k < TT::G; k += 2) (&o.x)[k >> 1] = ob[k] | (ob[(k + 1) % TT::G] << 16);
      }
      *reinterpret_cast<uint4 *>(static_cast<T *>(out) + e0) = o;
    } else {
#pragma unroll
      for (int k = 0; k < TT::G; ++k)
        if (k < nv) TT::st1(out, e0 + k, ob[k]);
    }
  });
}

}  // namespace

// Launches the filter over rows0 rows of in0 -> out0 followed by rows1 rows of
// in1 -> out1 (all [rows][V] of one dtype). Host checks are the caller's.
// In place (out == in) is allowed: a row's CTA reads its row in every pass but
// writes it only in the last, and no CTA touches another row.
sv_status launch_topp_filter(sv_dtype dtype, const void *in0, void *out0, int rows0, const void *in1, void *out1,
                             int rows1, int V, float temperature, float top_p, int32_t *status, cudaStream_t s) {
  const int es = dtype_bytes(dtype);
  if (rows0 + rows1 == 0) return ok();
  TpParams P = {};
  P.in0 = in0; P.out0 = out0; P.rows0 = rows0;
  P.in1 = in1; P.out1 = out1;
  P.V = V;
  P.vec = aligned(in0, 16) && aligned(out0, 16) && (rows1 == 0 || (aligned(in1, 16) && aligned(out1, 16))) &&
          ((size_t)V * es) % 16 == 0;
  const double cd = 1.4426950408889634074 / (double)temperature;
  P.c_hi = (float)cd;
  P.c_lo = (float)(cd - (double)P.c_hi);
  P.top_p = (double)top_p;
  P.status = status;
  cudaError_t e = cudaSuccess;
  const dim3 grid(rows0 + rows1);
  switch (dtype) {
    case SV_F32: e = launch_k(topp_row_kernel<float>, grid, dim3(kTpThreads), 0, s, 1, P); break;
    case SV_BF16: e = launch_k(topp_row_kernel<__nv_bfloat16>, grid, dim3(kTpThreads), 0, s, 1, P); break;
    case SV_F16: e = launch_k(topp_row_kernel<__half>, grid, dim3(kTpThreads), 0, s, 1, P); break;
    default: return fail(SV_ERR_UNSUPPORTED, "top-p filter: logits must be f32, bf16 or f16");
  }
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "top-p filter launch: %s", cudaGetErrorString(e));
  return ok();
}

}  // namespace sv

extern "C" sv_status spec_topp_filter(const void *logits, sv_dtype dtype, int rows, int V, float temperature,
                                      float top_p, void *out, int32_t *dev_status, sv_stream_t stream) {
  using namespace sv;
  if (rows < 0 || V < 1) return fail(SV_ERR_INVALID_ARG, "spec_topp_filter: bad sizes rows=%d V=%d", rows, V);
  if (!logits || !out) return fail(SV_ERR_INVALID_ARG, "spec_topp_filter: null pointer argument");
  if (!(temperature > 0.f) || !std::isfinite(temperature))
    return fail(SV_ERR_INVALID_ARG, "spec_topp_filter: temperature must be finite and > 0");
  if (!(top_p > 0.f) || !(top_p <= 1.f)) return fail(SV_ERR_INVALID_ARG, "spec_topp_filter: top_p must be in (0, 1]");
  if (dtype != SV_F32 && dtype != SV_BF16 && dtype != SV_F16)
    return fail(SV_ERR_UNSUPPORTED, "spec_topp_filter: logits must be f32, bf16 or f16");
  if (V > (1 << 28)) return fail(SV_ERR_UNSUPPORTED, "spec_topp_filter: V = %d above 2^28", V);
  if (rows == 0) return ok();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (top_p >= 1.f) {
    if (out == logits) return ok();
    const cudaError_t e = cudaMemcpyAsync(out, logits, (size_t)rows * V * dtype_bytes(dtype), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_topp_filter copy: %s", cudaGetErrorString(e));
    return ok();
  }
  return launch_topp_filter(dtype, logits, out, rows, nullptr, nullptr, 0, V, temperature, top_p, dev_status, s);
}

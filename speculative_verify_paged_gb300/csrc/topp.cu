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
// Masses are the weights w = 2^((l - m) log2(e) / T) of the row (m its
// maximum); each is within about 2.2e-7 (relative) of its exact value (the
// SFU exp2 and a first-order correction for the rounding of the exponent).
// Sums that decide the set are compensated fp32 sums per thread (within two
// ulps) combined in fp64 in a fixed order, and sums of the few tokens ranked
// directly are exact 64-bit sums of masses in 2^-40 fixed point, so a
// cumulative mass as a fraction of the row mass is within 5e-7 of exact, and
// the kernel is deterministic: the set is exact unless top_p lies that close
// to a cumulative mass.
//
// One 512-thread CTA per row, two per SM. The first pass reads the row from
// memory, the other two from L2. Passes:
//   1. the row maximum m, with packed two-lane max instructions (a second,
//      NaN-propagating max flags NaN);
//   2. Z, the row's mass; and an approximate mass for each of 2048 fine bins
//      of 1/32 of a binade of weight: every w of bin f is scaled by
//      2^(f/32 + s), rounded to an integer and added with a 32-bit shared
//      atomic (exact integer sums: deterministic, and within 2^-(s+1) of the
//      bin's mass, relative). A block scan gives the window of bins
//      [f_lo, f_hi] where the running mass can reach top_p Z, given that
//      error bound (one bin in nearly every row);
//   3. the row is written: logits in bins above the window stay (their
//      masses summed into `above`), those below go, and the window's logits
//      are written as kept and gathered (composite, mass, position). The
//      gathered tokens (at most 512; more only with many equal or nearly
//      equal logits, then the window is split by the composite's bits, 8 at
//      a time, over extra passes) are ranked by direct comparison: the cut.
//      Those below it are then overwritten with -inf.
// A logit's bin is round(32 (m - x) c) from the same roundings in every pass,
// so it is non-increasing in x and a bin boundary never separates equal
// logits; NaN and -inf fall in the last bin, which takes no mass.
//
// That is the general kernel, topp_row_kernel. Rows of at most 188000 logits
// (every vocabulary the workloads use) run topp_bin_kernel instead, which
// keeps exact per-bin masses in pass 2 (a count and quantised offsets from
// each bin's nominal weight, two 32-bit atomics per logit), so that Z, the
// window and the mass above it are exact sums and the write pass only
// compares logits with two thresholds.

#include <cmath>
#include <mutex>

#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kTpThreads = 512;
constexpr int kTpWarps = kTpThreads / 32;
constexpr int kTpBins = 2048;         // 64 binades of weight in steps of 1/32
constexpr int kTpBinsPer = kTpBins / kTpThreads;
constexpr int kTpCap = 512;           // candidates ranked directly
constexpr int kTpUnroll = 4;          // 16-byte loads in flight per thread
constexpr int kTpUnroll1 = 8;         // the same in the maximum passes and topp_bin_kernel's binning pass
constexpr float kTpQuant = 1099511627776.0f;  // 2^40
static_assert(kTpBinsPer * kTpThreads == kTpBins, "bins per thread");

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
  int qbits;          // s: pass 2 scales bin f's weights by 2^(f/32 + s)
  double win_eps;     // relative error bound of pass 2's cumulative masses
  int32_t *status;
  unsigned long long base[128];   // topp_bin_kernel: 2^(-j/128) in 2^-62 fixed point
};

// Per logit type: the element at position k of a 16-byte group, its value,
// scalar loads and stores, and the packed maxima of pass 1 over one 32-bit
// word (two 16-bit logits or one f32 logit).
template <typename T>
struct TpType;
template <>
struct TpType<float> {
  static constexpr int G = 4;
  static constexpr uint32_t kSign = 0x80000000u, kMag = 0x7fffffffu, kInf = 0x7f800000u;
  static constexpr uint32_t kNegInf = 0xff800000u, kKeyMask = 0xffffffffu;
  static constexpr uint32_t kNegInfWord = 0xff800000u;
  static constexpr bool kExactDiff = false;   // x - m needs a two-sum
  static __device__ __forceinline__ uint32_t get(const uint4 &r, int k) { return (&r.x)[k]; }
  static __device__ __forceinline__ float val(uint32_t b) { return __uint_as_float(b); }
  static __device__ __forceinline__ uint32_t ld1(const void *p, int e) {
    return __float_as_uint(__ldg(static_cast<const float *>(p) + e));
  }
  static __device__ __forceinline__ void st1(void *p, int e, uint32_t b) { static_cast<uint32_t *>(p)[e] = b; }
  static __device__ __forceinline__ uint32_t pmax(uint32_t a, uint32_t b) {
    uint32_t y;
    asm("max.f32 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
    return y;
  }
  static __device__ __forceinline__ uint32_t pmax_nan(uint32_t a, uint32_t b) {
    uint32_t y;
    asm("max.NaN.f32 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
    return y;
  }
  static __device__ __forceinline__ float word_max(uint32_t w) { return __uint_as_float(w); }
  static __device__ __forceinline__ bool word_nan(uint32_t w) { return (w & kMag) > kInf; }
};
template <>
struct TpType<__nv_bfloat16> {
  static constexpr int G = 8;
  static constexpr uint32_t kSign = 0x8000u, kMag = 0x7fffu, kInf = 0x7f80u;
  static constexpr uint32_t kNegInf = 0xff80u, kKeyMask = 0xffffu;
  static constexpr uint32_t kNegInfWord = 0xff80ff80u;
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
  static __device__ __forceinline__ uint32_t pmax(uint32_t a, uint32_t b) {
    uint32_t y;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
    return y;
  }
  static __device__ __forceinline__ uint32_t pmax_nan(uint32_t a, uint32_t b) {
    uint32_t y;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
    return y;
  }
  static __device__ __forceinline__ float word_max(uint32_t w) {
    return fmaxf(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
  }
  static __device__ __forceinline__ bool word_nan(uint32_t w) {
    return (w & kMag) > kInf || ((w >> 16) & kMag) > kInf;
  }
};
template <>
struct TpType<__half> {
  static constexpr int G = 8;
  static constexpr uint32_t kSign = 0x8000u, kMag = 0x7fffu, kInf = 0x7c00u;
  static constexpr uint32_t kNegInf = 0xfc00u, kKeyMask = 0xffffu;
  static constexpr uint32_t kNegInfWord = 0xfc00fc00u;
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
  static __device__ __forceinline__ uint32_t pmax(uint32_t a, uint32_t b) {
    uint32_t y;
    asm("max.f16x2 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
    return y;
  }
  static __device__ __forceinline__ uint32_t pmax_nan(uint32_t a, uint32_t b) {
    uint32_t y;
    asm("max.NaN.f16x2 %0, %1, %2;" : "=r"(y) : "r"(a), "r"(b));
    return y;
  }
  static __device__ __forceinline__ float word_max(uint32_t w) {
    return fmaxf(val(w & 0xffffu), val(w >> 16));
  }
  static __device__ __forceinline__ bool word_nan(uint32_t w) {
    return (w & kMag) > kInf || ((w >> 16) & kMag) > kInf;
  }
};

__device__ __forceinline__ float tp_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Canonical bits: NaN becomes -inf, -0 becomes +0.
template <typename T>
__device__ __forceinline__ uint32_t tp_canon(uint32_t b) {
  using TT = TpType<T>;
  if ((b & TT::kMag) > TT::kInf) b = TT::kNegInf;
  if (b == TT::kSign) b = 0u;
  return b;
}

template <typename T>
__device__ __forceinline__ u64 tp_composite(uint32_t b, int id) {
  using TT = TpType<T>;
  const uint32_t canon = tp_canon<T>(b);
  const uint32_t key = (canon & TT::kSign) ? (~canon & TT::kKeyMask) : (canon | TT::kSign);
  return ((u64)key << 32) | (u64)(0xffffffffu - (uint32_t)id);
}

// Calls f(e0, r, nv) for every group of a row of V elements: r holds the
// elements e0 .. e0 + nv - 1 packed as in memory (nv = G except in the last
// group); the lanes of a short group past nv hold -inf. Full 16-byte groups go
// round-robin over the threads, U loads in flight per thread; the ragged end
// (and the whole row when it is not 16-byte aligned) is loaded one element at
// a time.
template <typename T, bool LAST = false, int U = kTpUnroll, typename F>
__device__ __forceinline__ void tp_row_groups(const void *row, int V, int vec, F f) {
  using TT = TpType<T>;
  constexpr int G = TT::G;
  const int ng = vec ? V / G : 0;
  const uint4 *rv = static_cast<const uint4 *>(row);
  // LAST: the pass that reads the row for the last time loads it evict-first
  auto ld = [](const uint4 *p) { return LAST ? __ldcs(p) : __ldg(p); };
  int g = threadIdx.x;
  for (; g + (U - 1) * kTpThreads < ng; g += U * kTpThreads) {
    uint4 r[U];
#pragma unroll
    for (int u = 0; u < U; ++u) r[u] = ld(rv + g + u * kTpThreads);
#pragma unroll
    for (int u = 0; u < U; ++u) f((g + u * kTpThreads) * G, r[u], G);
  }
  for (; g < ng; g += kTpThreads) f(g * G, ld(rv + g), G);
  for (int h = ng + (int)threadIdx.x; h * G < V; h += kTpThreads) {
    const int nv = min(G, V - h * G);
    uint4 r = make_uint4(TT::kNegInfWord, TT::kNegInfWord, TT::kNegInfWord, TT::kNegInfWord);
#pragma unroll
    for (int k = 0; k < G; ++k) {
      if (k < nv) {
        const uint32_t b = TT::ld1(row, h * G + k);
        if (sizeof(T) == 4) {
          (&r.x)[k] = b;
        } else {
          const int sh = (k & 1) * 16;
          (&r.x)[k >> 1] = ((&r.x)[k >> 1] & ~(0xffffu << sh)) | (b << sh);
        }
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

// Compensated (Kahan) addition of w to the fp32 pair (s, c): s - c tracks
// the exact sum to about two ulps of it.
__device__ __forceinline__ void tp_kahan(float &s, float &c, float w) {
  const float y = w - c;
  const float t = s + y;
  c = (t - s) - y;
  s = t;
}

// Sum over the block of one double per thread, in a fixed order (so every
// run gives the same bits); every thread gets the total.
__device__ __forceinline__ double tp_block_sum_d(double v, double *s_wd) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if (lane == 0) s_wd[warp] = v;
  __syncthreads();
  double tot = 0.0;
#pragma unroll
  for (int w = 0; w < kTpWarps; ++w) tot += s_wd[w];
  __syncthreads();
  return tot;
}

template <typename T>
__global__ void __launch_bounds__(kTpThreads, 2) topp_row_kernel(const __grid_constant__ TpParams P) {
  using TT = TpType<T>;
  constexpr int G = TT::G;
  __shared__ unsigned hist[kTpBins];           // approximate masses per fine bin, fixed point
  __shared__ float s_tbl[kTpBins];             // 2^(f/32 + s): the fixed-point scale of bin f
  __shared__ u64 rhist[256];                   // masses per radix digit (the rare split)
  __shared__ u64 c_comp[kTpCap];               // gathered candidates
  __shared__ u64 c_q[kTpCap];
  __shared__ int c_pos[kTpCap];
  __shared__ u64 s_warp64[kTpWarps];
  __shared__ double s_wd[kTpWarps];
  __shared__ float s_wmax[kTpWarps];
  __shared__ int s_wflag[kTpWarps];
  __shared__ int s_flo, s_fhi, s_sel;
  __shared__ u64 s_above_q, s_cut, s_cmax, s_cmin;
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

  // ---- 1. row maximum (max ignores NaN; max.NaN propagates it, for the flag) ----
  uint32_t wmax = TT::kNegInfWord, wnan = TT::kNegInfWord;
  tp_row_groups<T, false, kTpUnroll1>(in, V, P.vec, [&](int, const uint4 &r, int) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      wmax = TT::pmax(wmax, (&r.x)[j]);
      wnan = TT::pmax_nan(wnan, (&r.x)[j]);
    }
  });
  for (int i = threadIdx.x; i < kTpBins; i += kTpThreads) {
    hist[i] = 0u;
    s_tbl[i] = exp2f((float)i * 0.03125f + (float)P.qbits);
  }
  if (threadIdx.x == 0) {
    s_count = 0u; s_sel = -1; s_flo = 0; s_fhi = kTpBins - 2;
    s_above_q = 0ull; s_cut = 0ull; s_cmax = 0ull; s_cmin = ~0ull;
  }
  {
    float mx = warp_max(TT::word_max(wmax));
    int flag = TT::word_nan(wnan) ? 1 : 0;
    flag = (int)__reduce_or_sync(0xffffffffu, (unsigned)flag);
    if (lane == 0) { s_wmax[warp] = mx; s_wflag[warp] = flag; }
  }
  __syncthreads();
  float m = -INFINITY;
  int flag = 0;
#pragma unroll
  for (int w = 0; w < kTpWarps; ++w) { m = fmaxf(m, s_wmax[w]); flag |= s_wflag[w]; }
  if ((flag || m == INFINITY) && threadIdx.x == 0) atomic_or_status(P.status, SV_DEV_NONFINITE);

  if (!(m > -INFINITY) || m == INFINITY) {
    // nothing to rank (no finite logit, or a +inf one): the row is passed
    // through unchanged and the sampling flags it
    if (out != in)
      tp_row_groups<T>(in, V, 0, [&](int e0, const uint4 &r, int nv) {
#pragma unroll
        for (int k = 0; k < G; ++k)
          if (k < nv) TT::st1(out, e0 + k, TT::get(r, k));
      });
    return;
  }

  // Bin of a logit x: d = x - m (<= 0), h = d c_hi (<= 0, the exponent of the
  // weight), bin = round(-32 h) from one fma onto the integer grid of
  // [2^23, 2^24), capped at the last bin. Each step rounds monotonically, so
  // the bin is non-increasing in x; -inf and NaN (fminf drops the NaN) land in
  // the last bin, as do weights below 2^-63.98, which take no part.
  // Weight: 2^(d c) with d c taken as h + lo (c = c_hi + c_lo, an fma for the
  // product's rounding, a two-sum for x - m where it is not exact); 2^h from
  // the SFU (relative error below 1.5e-7 on [-64, 0]), 2^lo as the first-order
  // factor 1 + lo ln 2 (|lo| is about an ulp of h).
  const float c_hi = P.c_hi, c_lo = P.c_lo;
  const float top = 8388608.f + (float)(kTpBins - 1);
  auto bin_of = [&](float x, float &d, float &h) {
    d = __fsub_rn(x, m);
    h = __fmul_rn(d, c_hi);
    return __float_as_int(fminf(fmaf(h, -32.f, 8388608.f), top)) - 0x4B000000;
  };
  auto weight_of = [&](float x, float d, float h) -> float {
    float l = fmaf(d, c_hi, -h);
    l = fmaf(d, c_lo, l);
    if (!TT::kExactDiff) {
      const float bb = d - x;
      const float d_lo = (x - (d - bb)) + (-m - bb);
      l = fmaf(d_lo, c_hi, l);
    }
    const float t = tp_ex2(h);
    return fmaf(t, l * 0.693147180559945309f, t);
  };

  // ---- 2. Z, and approximate masses per bin ----
  // Z: compensated fp32 sums per thread, combined in fp64. Bin f: the weights
  // w (within 2^(+-1/64) of 2^(-f/32)) scaled by 2^(f/32 + s) and rounded to
  // integers, summed with 32-bit shared atomics (order-independent); with s
  // chosen so that V 2^(s + 1/64) < 2^31 the sums cannot overflow, and a bin's
  // sum over 2^(f/32 + s) is within 2^-(s+1) 2^(1/64) (relative) of the exact
  // mass of the bin.
  float zs = 0.f, zc = 0.f;
  tp_row_groups<T>(in, V, P.vec, [&](int, const uint4 &r, int) {
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const float x = TT::val(TT::get(r, k));
      float d, h;
      const int fb = bin_of(x, d, h);
      if (fb < kTpBins - 1) {
        const float w = weight_of(x, d, h);
        tp_kahan(zs, zc, w);
        const float v = fmaf(w, s_tbl[fb], 8388608.f);   // round(w 2^(f/32 + s)) + 2^23
        atomicAdd(&hist[fb], (unsigned)__float_as_uint(v) - 0x4B000000u);
      }
    }
  });
  const double Z = tp_block_sum_d((double)zs - (double)zc, s_wd);   // also orders hist's atomics
  const double thr = P.top_p * Z;
  {
    // the window [f_lo, f_hi] that must hold the bin where the running mass
    // reaches thr: cumulative approximate masses in 2^-32 fixed point (exact
    // u64 scan), widened by their error bound
    u64 a[kTpBinsPer];
    u64 part = 0;
#pragma unroll
    for (int j = 0; j < kTpBinsPer; ++j) {
      const int f = threadIdx.x * kTpBinsPer + j;
      a[j] = __float2ull_rn((float)hist[f] / s_tbl[f] * 4294967296.f);
      part += a[j];
    }
    u64 tot;
    u64 cum = tp_block_excl_scan(part, s_warp64, &tot);
    const double err = Z * 4294967296.0 * P.win_eps;
    const double lo_t = thr * 4294967296.0 - err, hi_t = thr * 4294967296.0 + err;
    const u64 lo_u = lo_t <= 0.0 ? 0ull : (u64)lo_t, hi_u = (u64)ceil(hi_t);
#pragma unroll
    for (int j = 0; j < kTpBinsPer; ++j) {
      const int f = threadIdx.x * kTpBinsPer + j;
      if (cum < lo_u && lo_u <= cum + a[j]) s_flo = f;
      if (cum < hi_u && hi_u <= cum + a[j]) s_fhi = f;
      cum += a[j];
    }
  }
  __syncthreads();
  const int f_lo = s_flo, f_hi = max(s_flo, min(s_fhi, kTpBins - 2));

  // ---- 3. write the row: bins above the window stay (their accurate masses
  // summed, compensated, into `above`), bins below go (NaN and -inf are in
  // the last bin), the window's tokens stay for now and are gathered
  // (composite, mass in 2^-40 fixed point, position) ----
  float as = 0.f, ac = 0.f;
  tp_row_groups<T>(in, V, P.vec, [&](int e0, const uint4 &r, int nv) {
    uint32_t ob[G];
    unsigned cm = 0;
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const uint32_t b = TT::get(r, k);
      const float x = TT::val(b);
      float d, h;
      const int fb = bin_of(x, d, h);
      const float w = weight_of(x, d, h);
      tp_kahan(as, ac, fb < f_lo ? w : 0.f);
      ob[k] = fb <= f_hi ? b : TT::kNegInf;
      cm |= (fb >= f_lo && fb <= f_hi && k < nv) ? 1u << k : 0u;
    }
    if (P.vec && nv == G) {
      uint4 o;
      if (sizeof(T) == 4) {
        o = make_uint4(ob[0], ob[1 % G], ob[2 % G], ob[3 % G]);
      } else {
#pragma unroll
        for (int k = 0; k < G; k += 2) (&o.x)[k >> 1] = ob[k] | (ob[(k + 1) % G] << 16);
      }
      *reinterpret_cast<uint4 *>(static_cast<T *>(out) + e0) = o;
    } else {
#pragma unroll
      for (int k = 0; k < G; ++k)
        if (k < nv) TT::st1(out, e0 + k, ob[k]);
    }
    if (cm) {
      unsigned slot = atomicAdd(&s_count, (unsigned)__popc(cm));
#pragma unroll
      for (int k = 0; k < G; ++k) {
        if (((cm >> k) & 1u) && slot < (unsigned)kTpCap) {
          const uint32_t b = TT::get(r, k);
          const float x = TT::val(b);
          float d, h;
          bin_of(x, d, h);
          c_comp[slot] = tp_composite<T>(b, e0 + k);
          c_q[slot] = __float2ull_rn(weight_of(x, d, h) * kTpQuant);
          c_pos[slot] = e0 + k;
        }
        slot += (cm >> k) & 1u;
      }
    }
  });
  // the mass above the window, in 2^-40 units as a double (the block sum
  // also orders the gathers above before the reads below)
  const double above = tp_block_sum_d((double)as - (double)ac, s_wd) * (double)kTpQuant;
  const double thr_q = thr * (double)kTpQuant;

  // ---- the rare split: more than kTpCap tokens in the window (many equal
  // or nearly equal logits). Histogram them by the next 8 bits of the
  // composite, keep the digit where the running mass reaches thr, and gather
  // again. Bins outside the window were final after pass 3 and the window's
  // logits are unchanged in `in` (also when out == in), so the passes read
  // `in`. ----
  int sh = 64;        // the composite's bits at and above sh equal pfx
  u64 pfx = 0ull;
  u64 above_q = 0ull; // exact mass of the window's tokens above the prefix
  int n_all = (int)s_count;
  auto in_window = [&](uint32_t b, int e, u64 &comp) {
    float d, h;
    const int fb = bin_of(TT::val(b), d, h);
    if (fb < f_lo || fb > f_hi) return false;
    comp = tp_composite<T>(b, e);
    return sh >= 64 || (comp >> sh) == pfx;
  };
  while (n_all > kTpCap && sh > 0) {
    const int nsh = sh > 8 ? sh - 8 : 0;
    const int width = sh - nsh;
    __syncthreads();   // every thread has read s_count and s_sel before they are reset
    for (int i = threadIdx.x; i < 256; i += kTpThreads) rhist[i] = 0ull;
    if (threadIdx.x == 0) { s_count = 0u; s_sel = -1; }
    __syncthreads();
    tp_row_groups<T>(in, V, P.vec, [&](int e0, const uint4 &r, int nv) {
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const uint32_t b = TT::get(r, k);
        u64 comp;
        if (k < nv && in_window(b, e0 + k, comp)) {
          const float x = TT::val(b);
          float d, h;
          bin_of(x, d, h);
          atomicAdd(&rhist[(int)((comp >> nsh) & ((1ull << width) - 1ull))],
                    __float2ull_rn(weight_of(x, d, h) * kTpQuant));
        }
      }
    });
    __syncthreads();
    {
      // digits in descending order: entry i is digit 255 - i
      const int i = threadIdx.x;
      const u64 mine = i < 256 ? rhist[255 - i] : 0ull;
      u64 tot;
      const u64 cum = above_q + tp_block_excl_scan(mine, s_warp64, &tot);
      if (i < 256 && mine > 0ull && above + (double)cum < thr_q && thr_q <= above + (double)(cum + mine)) {
        s_sel = 255 - i;
        s_above_q = cum;
      }
      __syncthreads();
      const int sel0 = s_sel;
      __syncthreads();   // read by every thread before thread 0 may write it
      if (sel0 < 0) {
        if (threadIdx.x == 0) {
          const bool before_all = above + (double)above_q >= thr_q;
          u64 c = above_q;
          for (int dgt = 255; dgt >= 0; --dgt) {
            if (rhist[dgt] == 0ull) continue;
            if (before_all) { s_sel = dgt; s_above_q = c; break; }
            s_sel = dgt; s_above_q = c;   // keeps the last nonempty digit
            c += rhist[dgt];
          }
        }
        __syncthreads();
      }
    }
    above_q = s_above_q;
    pfx = (sh >= 64 ? 0ull : (pfx << width)) | (u64)(s_sel < 0 ? 0 : s_sel);
    sh = nsh;
    tp_row_groups<T>(in, V, P.vec, [&](int e0, const uint4 &r, int nv) {
      unsigned cm = 0;
#pragma unroll
      for (int k = 0; k < G; ++k) {
        u64 comp;
        if (k < nv && in_window(TT::get(r, k), e0 + k, comp)) cm |= 1u << k;
      }
      if (cm) {
        unsigned slot = atomicAdd(&s_count, (unsigned)__popc(cm));
#pragma unroll
        for (int k = 0; k < G; ++k) {
          if (((cm >> k) & 1u) && slot < (unsigned)kTpCap) {
            const uint32_t b = TT::get(r, k);
            const float x = TT::val(b);
            float d, h;
            bin_of(x, d, h);
            c_comp[slot] = tp_composite<T>(b, e0 + k);
            c_q[slot] = __float2ull_rn(weight_of(x, d, h) * kTpQuant);
            c_pos[slot] = e0 + k;
          }
          slot += (cm >> k) & 1u;
        }
      }
    });
    __syncthreads();
    n_all = (int)s_count;
  }

  // ---- the cut: candidate i is the cut iff the mass before it (everything
  // above the window and the prefix, plus every candidate with a larger
  // composite) is below thr and reaches thr with it ----
  if (n_all <= kTpCap) {
    for (int i = threadIdx.x; i < n_all; i += kTpThreads) {
      const u64 ci = c_comp[i], qi = c_q[i];
      u64 before = above_q;
      for (int j = 0; j < n_all; ++j) before += (c_comp[j] > ci) ? c_q[j] : 0ull;
      if (above + (double)before < thr_q && thr_q <= above + (double)(before + qi)) s_cut = ci;
      atomicMax(&s_cmax, ci);
      atomicMin(&s_cmin, ci);
    }
  }
  __syncthreads();
  u64 cut = s_cut;
  if (cut == 0ull && n_all > 0 && n_all <= kTpCap) {
    // rounding at the window's edge left no candidate that crosses thr: the
    // first candidate when the mass above already reaches thr, else the last
    cut = above + (double)above_q >= thr_q ? s_cmax : s_cmin;
  }
  if (cut == 0ull) return;   // not reached: the window is kept whole
  if (sh == 64) {
    // every token of the window was gathered: drop those below the cut
    for (int i = threadIdx.x; i < n_all; i += kTpThreads)
      if (c_comp[i] < cut) TT::st1(out, c_pos[i], TT::kNegInf);
  } else {
    // the split narrowed the candidates: drop the window's tokens below the cut
    sh = 64;
    tp_row_groups<T>(in, V, P.vec, [&](int e0, const uint4 &r, int nv) {
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const uint32_t b = TT::get(r, k);
        u64 comp;
        if (k < nv && in_window(b, e0 + k, comp) && comp < cut) TT::st1(out, e0 + k, TT::kNegInf);
      }
    });
  }
}

// ---------------------------------------------------------------------------
// topp_bin_kernel: rows of at most kTbMaxV logits. The same set with exact
// per-bin masses, so that the write pass needs no weights.
//
// Pass 2 puts every logit in one of 8192 bins of 1/128 of a binade of weight
// (bin f: weights within 2^(+-1/256) of 2^(-f/128)) and adds, with two 32-bit
// shared atomics, 1 to the bin's count and q = round(2^22 v) - 2^22 to its
// offset sum, where v = w 2^(f/128) is the weight relative to the bin's
// nominal one (|q| <= 11373, so V <= kTbMaxV keeps the sum inside int32).
// v comes from one SFU exp2 of (x - m) c + f/128, at most 1/256 in
// magnitude and formed with fmas that round only that small sum (the
// product (x - m) c_hi is never rounded on its own), so the exponent's own
// error is below 2^-31 and v's is the SFU's.
// A bin's mass is then 2^(-f/128) (n_f + R_f 2^-22): each weight within
// 2^-23 of its quantised value and about 2e-7 of its exact one. The masses
// go to 2^-40 fixed point with a 64 x 64-bit product (2^(-j/128) in 2^-62
// fixed point from the host, an exact shift for the binade), so Z, the
// cumulative sums and the mass above the window are exact 64-bit integers
// and the kernel is deterministic. A block scan gives the window of bins
// where the running mass reaches ceil(top_p Z) (with a 1e-6 Z margin: one
// bin in nearly every row), and bisection over the logits' ordered bits
// gives the two logit thresholds of its edges (bins are non-increasing in the
// logit). Pass 3 then keeps x >= x_keep, with packed two-lane compares for
// 16-bit logits, and gathers the window's tokens (x_keep <= x < x_above) for
// the ranking, as the general kernel does.
constexpr int kTbBins = 8192;
constexpr int kTbPer = kTbBins / kTpThreads;     // bins per thread in the scan
constexpr int kTbMaxV = 188000;                  // 188000 * 11373 < 2^31
constexpr size_t kTbSmem = (size_t)kTbBins * 8 + (size_t)kTpCap * (8 + 8 + 4) + 256 * 8;
static_assert(kTbPer * kTpThreads == kTbBins, "bins per thread");

// (hi:lo) = a * b, then >> s (44 <= s < 128)
__device__ __forceinline__ u64 tb_mulshift(u64 a, u64 b, int s) {
  const u64 lo = a * b, hi = __umul64hi(a, b);
  if (s >= 64) return s >= 128 ? 0ull : hi >> (s - 64);
  return (hi << (64 - s)) | (lo >> s);
}

// value bits of a 16- or 32-bit logit from its ordered key (the inverse of
// the key map of tp_composite)
template <typename T>
__device__ __forceinline__ uint32_t tb_from_key(uint32_t k) {
  using TT = TpType<T>;
  return (k & TT::kSign) ? (k & ~TT::kSign) : (~k & TT::kKeyMask);
}
template <typename T>
__device__ __forceinline__ uint32_t tb_key(uint32_t b) {
  using TT = TpType<T>;
  return (b & TT::kSign) ? (~b & TT::kKeyMask) : (b | TT::kSign);
}

template <typename T>
__global__ void __launch_bounds__(kTpThreads, 2) topp_bin_kernel(const __grid_constant__ TpParams P) {
  using TT = TpType<T>;
  constexpr int G = TT::G;
  extern __shared__ __align__(16) uint8_t tb_smem[];
  unsigned *cnt = reinterpret_cast<unsigned *>(tb_smem);                 // [kTbBins]
  int *dsum = reinterpret_cast<int *>(tb_smem + (size_t)kTbBins * 4);    // [kTbBins]
  u64 *c_comp = reinterpret_cast<u64 *>(tb_smem + (size_t)kTbBins * 8);  // [kTpCap]
  u64 *c_q = c_comp + kTpCap;                                           // [kTpCap]
  u64 *rhist = c_q + kTpCap;                                            // [256]
  int *c_pos = reinterpret_cast<int *>(rhist + 256);                    // [kTpCap]
  __shared__ u64 s_warp64[kTpWarps];
  __shared__ float s_wmax[kTpWarps];
  __shared__ int s_wflag[kTpWarps];
  __shared__ int s_flo, s_fhi, s_sel;
  __shared__ u64 s_above, s_above_q, s_cut, s_cmax, s_cmin;
  __shared__ uint32_t s_xkeep, s_xabove;
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

  // ---- 1. row maximum (max ignores NaN; max.NaN propagates it, for the flag) ----
  uint32_t wmax = TT::kNegInfWord, wnan = TT::kNegInfWord;
  tp_row_groups<T, false, kTpUnroll1>(in, V, P.vec, [&](int, const uint4 &r, int) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      wmax = TT::pmax(wmax, (&r.x)[j]);
      wnan = TT::pmax_nan(wnan, (&r.x)[j]);
    }
  });
  for (int i = threadIdx.x; i < kTbBins; i += kTpThreads) {
    cnt[i] = 0u;
    dsum[i] = 0;
  }
  if (threadIdx.x == 0) {
    s_count = 0u; s_sel = -1; s_flo = 0; s_fhi = kTbBins - 2;
    s_above = 0ull; s_above_q = 0ull; s_cut = 0ull; s_cmax = 0ull; s_cmin = ~0ull;
  }
  {
    float mx = warp_max(TT::word_max(wmax));
    int flag = TT::word_nan(wnan) ? 1 : 0;
    flag = (int)__reduce_or_sync(0xffffffffu, (unsigned)flag);
    if (lane == 0) { s_wmax[warp] = mx; s_wflag[warp] = flag; }
  }
  __syncthreads();
  float m = -INFINITY;
  int flag = 0;
#pragma unroll
  for (int w = 0; w < kTpWarps; ++w) { m = fmaxf(m, s_wmax[w]); flag |= s_wflag[w]; }
  if ((flag || m == INFINITY) && threadIdx.x == 0) atomic_or_status(P.status, SV_DEV_NONFINITE);

  if (!(m > -INFINITY) || m == INFINITY) {
    // nothing to rank (no finite logit, or a +inf one): the row is passed
    // through unchanged and the sampling flags it
    if (out != in)
      tp_row_groups<T>(in, V, 0, [&](int e0, const uint4 &r, int nv) {
#pragma unroll
        for (int k = 0; k < G; ++k)
          if (k < nv) TT::st1(out, e0 + k, TT::get(r, k));
      });
    return;
  }

  // bin = round(-128 d c_hi), d = x - m, from one fma onto the integer grid
  // of [2^23, 2^24) (-128 c_hi is exact), capped at the last bin (which also
  // takes -inf and NaN); h = d c_hi rounded, for the weights of the window's
  // tokens
  const float c_hi = P.c_hi, c_lo = P.c_lo;
  const float nc128 = -128.f * c_hi;
  const float top = 8388608.f + (float)(kTbBins - 1);
  auto bin_of = [&](float x, float &d, float &h, float &y) {
    d = __fsub_rn(x, m);
    h = __fmul_rn(d, c_hi);
    y = fminf(fmaf(d, nc128, 8388608.f), top);
    return __float_as_int(y) - 0x4B000000;
  };
  // lo: the rounding of the exponent d c (fma for the product, two-sum for
  // x - m where it is not exact)
  auto lo_of = [&](float x, float d, float h) {
    float l = fmaf(d, c_hi, -h);
    l = fmaf(d, c_lo, l);
    if (!TT::kExactDiff) {
      const float bb = d - x;
      const float d_lo = (x - (d - bb)) + (-m - bb);
      l = fmaf(d_lo, c_hi, l);
    }
    return l;
  };
  auto weight_of = [&](float x, float d, float h) -> float {
    const float t = tp_ex2(h);
    return fmaf(t, lo_of(x, d, h) * 0.693147180559945309f, t);
  };

  // ---- 2. counts and quantised offsets per bin ----
  tp_row_groups<T, false, kTpUnroll1>(in, V, P.vec, [&](int, const uint4 &r, int) {
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const float x = TT::val(TT::get(r, k));
      float d, h, y;
      const int fb = bin_of(x, d, h, y);
      // the exponent against bin fb's nominal weight, (x - m) c + fb / 128,
      // in [-1/256, 1/256]: d c_hi + fb / 128 from one fma (the exact sum
      // rounded once, an error below 2^-32), then d c_lo and, where x - m
      // is not exact in fp32, the part of it that d dropped
      const float sf = fmaf(y, 0.0078125f, -65536.f);   // fb / 128, exact
      float rr = fmaf(d, c_hi, sf);
      rr = fmaf(d, c_lo, rr);
      if (!TT::kExactDiff) {
        const float bb = d - x;
        const float d_lo = (x - (d - bb)) + (-m - bb);
        rr = fmaf(d_lo, c_hi, rr);
      }
      const float v = tp_ex2(rr);
      // 2^22 v + 2^23 rounded to an integer in [2^23, 2^24) has the bits
      // 0x4B400000 + q: the bin sums those bits modulo 2^32, and the scan
      // takes n_f 0x4B400000 back off. The last bin (which also takes -inf
      // and NaN) collects whatever its logits give; the scan counts it as
      // empty
      atomicAdd(&cnt[fb], 1u);
      atomicAdd(reinterpret_cast<unsigned *>(&dsum[fb]), __float_as_uint(fmaf(v, 4194304.f, 8388608.f)));
    }
  });
  __syncthreads();
  u64 thr;
  {
    // bin masses in 2^-40 fixed point, their exact scan, Z, and the window
    u64 a[kTbPer];
    u64 part = 0;
#pragma unroll
    for (int j = 0; j < kTbPer; ++j) {
      const int f = threadIdx.x * kTbPer + j;
      const int sq = (int)((unsigned)dsum[f] - cnt[f] * 0x4B400000u);   // the offsets' sum (|.| < 2^31)
      const u64 N = f == kTbBins - 1 ? 0ull : (u64)((int64_t)cnt[f] * 4194304 + (int64_t)sq);
      a[j] = tb_mulshift(P.base[f & 127], N, 44 + (f >> 7));
      part += a[j];
    }
    u64 Z;
    u64 cum = tp_block_excl_scan(part, s_warp64, &Z);
    const double td = ceil(P.top_p * (double)Z);
    thr = td < 1.0 ? 1ull : (td >= (double)Z ? Z : (u64)td);
    const u64 marg = (u64)(1e-6 * (double)Z) + 1;
    const u64 lo_u = thr > marg ? thr - marg : 1ull, hi_u = thr + marg;
#pragma unroll
    for (int j = 0; j < kTbPer; ++j) {
      const int f = threadIdx.x * kTbPer + j;
      if (cum < lo_u && lo_u <= cum + a[j]) { s_flo = f; s_above = cum; }
      if (cum < hi_u && hi_u <= cum + a[j]) s_fhi = f;
      cum += a[j];
    }
  }
  __syncthreads();
  const int f_lo = s_flo, f_hi = max(s_flo, min(s_fhi, kTbBins - 2));
  const u64 above = s_above;   // exact mass of the bins above the window
  if (threadIdx.x < 2) {
    // bisection over the ordered keys between -inf (last bin) and m (bin 0):
    // the smallest key whose bin is at most F. x_keep: F = f_hi (x >= x_keep
    // <=> bin <= f_hi); x_above: F = f_lo - 1 (none when f_lo = 0)
    const int F = threadIdx.x == 0 ? f_hi : f_lo - 1;
    uint32_t res;
    if (F < 0) {
      res = TT::kInf;   // +inf: no logit lies above a window at the top
    } else {
      // m is one of the row's logits: its bits in the logit type
      uint32_t mb;
      if constexpr (sizeof(T) == 4) mb = __float_as_uint(m);
      else if constexpr (std::is_same<T, __nv_bfloat16>::value) mb = __float_as_uint(m) >> 16;
      else mb = (uint32_t)__half_as_ushort(__float2half(m));
      // invariant: bin(value of lo) > F (lo starts at -inf, the last bin),
      // bin(value of hi) <= F (hi starts at m, bin 0)
      uint32_t lo = tb_key<T>(TT::kNegInf), hi = tb_key<T>(mb);
      while (hi - lo > 1) {
        const uint32_t mid = lo + (hi - lo) / 2;
        float d, h, y;
        if (bin_of(TT::val(tb_from_key<T>(mid)), d, h, y) <= F) hi = mid;
        else lo = mid;
      }
      res = tb_from_key<T>(hi);
    }
    if (threadIdx.x == 0) s_xkeep = res;
    else s_xabove = res;
  }
  __syncthreads();
  const uint32_t xk_b = s_xkeep, xa_b = s_xabove;
  const float x_keep = TT::val(xk_b), x_above = TT::val(xa_b);

  // ---- 3. write the row: x >= x_keep stays, the window's tokens
  // (x_keep <= x < x_above) are gathered ----
  auto gather_one = [&](int e, uint32_t b, unsigned slot) {
    const float x = TT::val(b);
    float d, h, y;
    bin_of(x, d, h, y);
    c_comp[slot] = tp_composite<T>(b, e);
    c_q[slot] = __float2ull_rn(weight_of(x, d, h) * kTpQuant);
    c_pos[slot] = e;
  };
  // (the output is written with streaming stores and the row read evict-
  // first, so that neither displaces the rows other CTAs still re-read from L2)
  tp_row_groups<T, true>(in, V, P.vec, [&](int e0, const uint4 &r, int nv) {
    uint32_t ow[4];
    unsigned cm = 0;
    if constexpr (sizeof(T) == 4) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float x = __uint_as_float((&r.x)[k]);
        const bool keep = x >= x_keep;
        ow[k] = keep ? (&r.x)[k] : TT::kNegInf;
        cm |= (keep && !(x >= x_above) && k < nv) ? 1u << k : 0u;
      }
    } else {
      const uint32_t k2 = xk_b | (xk_b << 16), a2 = xa_b | (xa_b << 16);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t w = (&r.x)[j];
        uint32_t km, am;
        if constexpr (std::is_same<T, __nv_bfloat16>::value) {
          km = __hge2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&w), *reinterpret_cast<const __nv_bfloat162 *>(&k2));
          am = __hge2_mask(*reinterpret_cast<const __nv_bfloat162 *>(&w), *reinterpret_cast<const __nv_bfloat162 *>(&a2));
        } else {
          km = __hge2_mask(*reinterpret_cast<const __half2 *>(&w), *reinterpret_cast<const __half2 *>(&k2));
          am = __hge2_mask(*reinterpret_cast<const __half2 *>(&w), *reinterpret_cast<const __half2 *>(&a2));
        }
        ow[j] = (w & km) | (TT::kNegInfWord & ~km);
        const unsigned c2 = km & ~am;
        cm |= ((c2 & 0xffffu) ? 1u : 0u) << (2 * j);
        cm |= ((c2 >> 16) ? 1u : 0u) << (2 * j + 1);
      }
      cm &= (nv >= G) ? 0xffu : ((1u << nv) - 1u);
    }
    if (P.vec && nv == G) {
      __stcs(reinterpret_cast<uint4 *>(static_cast<T *>(out) + e0), make_uint4(ow[0], ow[1], ow[2], ow[3]));
    } else {
#pragma unroll
      for (int k = 0; k < G; ++k)
        if (k < nv) TT::st1(out, e0 + k, sizeof(T) == 4 ? ow[k % 4] : ((ow[k >> 1] >> ((k & 1) * 16)) & 0xffffu));
    }
    if (cm) {
      unsigned slot = atomicAdd(&s_count, (unsigned)__popc(cm));
#pragma unroll
      for (int k = 0; k < G; ++k) {
        if (((cm >> k) & 1u) && slot < (unsigned)kTpCap) gather_one(e0 + k, TT::get(r, k), slot);
        slot += (cm >> k) & 1u;
      }
    }
  });
  __syncthreads();

  // ---- the rare split: more than kTpCap tokens in the window. Histogram
  // them by the next 8 bits of the composite, keep the digit where the
  // running mass reaches thr, and gather again. Logits outside the window
  // were final after pass 3 and the window's are unchanged in `in` (also when
  // out == in), so the passes read `in`. ----
  int sh = 64;        // the composite's bits at and above sh equal pfx
  u64 pfx = 0ull;
  u64 above_q = 0ull; // exact mass of the window's tokens above the prefix
  int n_all = (int)s_count;
  auto in_window = [&](uint32_t b, int e, u64 &comp) {
    const float x = TT::val(b);
    if (!(x >= x_keep) || x >= x_above) return false;
    comp = tp_composite<T>(b, e);
    return sh >= 64 || (comp >> sh) == pfx;
  };
  while (n_all > kTpCap && sh > 0) {
    const int nsh = sh > 8 ? sh - 8 : 0;
    const int width = sh - nsh;
    __syncthreads();   // every thread has read s_count and s_sel before they are reset
    for (int i = threadIdx.x; i < 256; i += kTpThreads) rhist[i] = 0ull;
    if (threadIdx.x == 0) { s_count = 0u; s_sel = -1; }
    __syncthreads();
    tp_row_groups<T>(in, V, P.vec, [&](int e0, const uint4 &r, int nv) {
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const uint32_t b = TT::get(r, k);
        u64 comp;
        if (k < nv && in_window(b, e0 + k, comp)) {
          const float x = TT::val(b);
          float d, h, y;
          bin_of(x, d, h, y);
          atomicAdd(&rhist[(int)((comp >> nsh) & ((1ull << width) - 1ull))],
                    __float2ull_rn(weight_of(x, d, h) * kTpQuant));
        }
      }
    });
    __syncthreads();
    {
      // digits in descending order: entry i is digit 255 - i
      const int i = threadIdx.x;
      const u64 mine = i < 256 ? rhist[255 - i] : 0ull;
      u64 tot;
      const u64 cum = above + above_q + tp_block_excl_scan(mine, s_warp64, &tot);
      if (i < 256 && mine > 0ull && cum < thr && thr <= cum + mine) {
        s_sel = 255 - i;
        s_above_q = cum - above;
      }
      __syncthreads();
      const int sel0 = s_sel;
      __syncthreads();   // read by every thread before thread 0 may write it
      if (sel0 < 0) {
        if (threadIdx.x == 0) {
          // rounding left no digit that crosses: the first nonempty digit when
          // the mass above already reaches thr, else the last
          const bool before_all = above + above_q >= thr;
          u64 c = above_q;
          for (int dgt = 255; dgt >= 0; --dgt) {
            if (rhist[dgt] == 0ull) continue;
            if (before_all) { s_sel = dgt; s_above_q = c; break; }
            s_sel = dgt; s_above_q = c;
            c += rhist[dgt];
          }
        }
        __syncthreads();
      }
    }
    above_q = s_above_q;
    pfx = (sh >= 64 ? 0ull : (pfx << width)) | (u64)(s_sel < 0 ? 0 : s_sel);
    sh = nsh;
    tp_row_groups<T>(in, V, P.vec, [&](int e0, const uint4 &r, int nv) {
      unsigned cm = 0;
#pragma unroll
      for (int k = 0; k < G; ++k) {
        u64 comp;
        if (k < nv && in_window(TT::get(r, k), e0 + k, comp)) cm |= 1u << k;
      }
      if (cm) {
        unsigned slot = atomicAdd(&s_count, (unsigned)__popc(cm));
#pragma unroll
        for (int k = 0; k < G; ++k) {
          if (((cm >> k) & 1u) && slot < (unsigned)kTpCap) gather_one(e0 + k, TT::get(r, k), slot);
          slot += (cm >> k) & 1u;
        }
      }
    });
    __syncthreads();
    n_all = (int)s_count;
  }

  // ---- the cut: candidate i is the cut iff the mass before it (everything
  // above the window and the prefix, plus every candidate with a larger
  // composite) is below thr and reaches thr with it ----
  if (n_all <= kTpCap) {
    for (int i = threadIdx.x; i < n_all; i += kTpThreads) {
      const u64 ci = c_comp[i], qi = c_q[i];
      u64 before = above + above_q;
      for (int j = 0; j < n_all; ++j) before += (c_comp[j] > ci) ? c_q[j] : 0ull;
      if (before < thr && thr <= before + qi) s_cut = ci;
      atomicMax(&s_cmax, ci);
      atomicMin(&s_cmin, ci);
    }
  }
  __syncthreads();
  u64 cut = s_cut;
  if (cut == 0ull && n_all > 0 && n_all <= kTpCap) {
    // rounding at the window's edge left no candidate that crosses thr: the
    // first candidate when the mass above already reaches thr, else the last
    cut = above + above_q >= thr ? s_cmax : s_cmin;
  }
  if (cut == 0ull) return;   // not reached: the window is kept whole
  if (sh == 64) {
    for (int i = threadIdx.x; i < n_all; i += kTpThreads)
      if (c_comp[i] < cut) TT::st1(out, c_pos[i], TT::kNegInf);
  } else {
    sh = 64;
    tp_row_groups<T>(in, V, P.vec, [&](int e0, const uint4 &r, int nv) {
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const uint32_t b = TT::get(r, k);
        u64 comp;
        if (k < nv && in_window(b, e0 + k, comp) && comp < cut) TT::st1(out, e0 + k, TT::kNegInf);
      }
    });
  }
}

}  // namespace

// Launches the filter over rows0 rows of in0 -> out0 followed by rows1 rows of
// in1 -> out1 (all [rows][V] of one dtype). Host checks are the caller's.
// In place (out == in) is allowed: no CTA touches another row, and after a
// row's pass 3 every later read of it only asks whether a logit is in fbin,
// whose logits pass 3 leaves unchanged (and any other logit is in another bin
// both before and after its write), so a read that still sees the old value
// classifies it the same way.
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
  // the largest s (at most 22, so that w 2^(f/32 + s) + 2^23 rounds to an
  // integer) with V (2^(s + 1/64) + 1/2) < 2^32: no bin sum overflows
  int qb = 22;
  while (qb > 0 && (double)V * (std::ldexp(1.0111, qb) + 0.5) >= 4294967296.0) --qb;
  P.qbits = qb;
  P.win_eps = std::ldexp(1.0111, -(qb + 1)) + 4e-6;
  P.status = status;
  cudaError_t e = cudaSuccess;
  const dim3 grid(rows0 + rows1);
  if (V <= kTbMaxV) {
    // exact per-bin masses: rows up to kTbMaxV logits
    for (int j = 0; j < 128; ++j) P.base[j] = (unsigned long long)std::llround(std::ldexp(std::exp2(-j / 128.0), 62));
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [] {
      const cudaError_t e1 = cudaFuncSetAttribute(topp_bin_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTbSmem);
      const cudaError_t e2 = cudaFuncSetAttribute(topp_bin_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTbSmem);
      const cudaError_t e3 = cudaFuncSetAttribute(topp_bin_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTbSmem);
      attr = e1 != cudaSuccess ? e1 : (e2 != cudaSuccess ? e2 : e3);
    });
    if (attr != cudaSuccess) return fail(SV_ERR_CUDA, "top-p filter: cudaFuncSetAttribute: %s", cudaGetErrorString(attr));
    switch (dtype) {
      case SV_F32: e = launch_k(topp_bin_kernel<float>, grid, dim3(kTpThreads), kTbSmem, s, 1, P); break;
      case SV_BF16: e = launch_k(topp_bin_kernel<__nv_bfloat16>, grid, dim3(kTpThreads), kTbSmem, s, 1, P); break;
      case SV_F16: e = launch_k(topp_bin_kernel<__half>, grid, dim3(kTpThreads), kTbSmem, s, 1, P); break;
      default: return fail(SV_ERR_UNSUPPORTED, "top-p filter: logits must be f32, bf16 or f16");
    }
  } else {
    switch (dtype) {
      case SV_F32: e = launch_k(topp_row_kernel<float>, grid, dim3(kTpThreads), 0, s, 1, P); break;
      case SV_BF16: e = launch_k(topp_row_kernel<__nv_bfloat16>, grid, dim3(kTpThreads), 0, s, 1, P); break;
      case SV_F16: e = launch_k(topp_row_kernel<__half>, grid, dim3(kTpThreads), 0, s, 1, P); break;
      default: return fail(SV_ERR_UNSUPPORTED, "top-p filter: logits must be f32, bf16 or f16");
    }
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

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
// One cluster of up to 16 CTAs per row; each CTA keeps its slice of the row
// (at most 32 KB) in shared memory, so the row is read from memory once and
// written once. Steps:
//   1. row maximum (block, then cluster through distributed shared memory);
//   2. a 2048-bin histogram of the masses by -log2(weight) in steps of 1/32
//      (bins in descending logit order), summed over the cluster;
//   3. the bin where the cumulative mass reaches ceil(top_p * Z);
//   4. that bin's tokens are gathered into the cluster's first CTA (if more
//      than 512, the bin is first split by the composite's bits, 8 at a
//      time, until at most 512 remain) and each one's cumulative mass is
//      computed by direct comparison of composites, which gives the cut;
//   5. every element is written back, or -inf below the cut: bins above the
//      cut's bin stay, bins below go, the composite decides within it.
// Bins are one fma from the logit, so only the histogram pass and the
// gathered tokens compute the precise weights.

#include <cmath>
#include <mutex>

#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kTpThreads = 256;
constexpr int kTpVec = 8;        // 16-byte vectors per thread
constexpr int kTpBins = 2048;    // first-level bins: 1/32 of a binade of weight each
constexpr int kTpCap = 512;      // candidates ranked directly
constexpr float kTpQuant = 1099511627776.0f;  // 2^40

typedef unsigned long long u64;

struct TpParams {
  const void *in0;
  void *out0;
  int rows0;
  const void *in1;
  void *out1;
  int V;
  int slice;     // elements per CTA (a multiple of the elements per vector)
  int vec;       // rows are 16-byte aligned: vector loads and stores
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
  static __device__ __forceinline__ uint32_t get(const uint4 &r, int k) { return (&r.x)[k]; }
  static __device__ __forceinline__ float val(uint32_t b) { return __uint_as_float(b); }
};
template <>
struct TpType<__nv_bfloat16> {
  static constexpr int G = 8;
  static constexpr uint32_t kSign = 0x8000u, kMag = 0x7fffu, kInf = 0x7f80u;
  static constexpr uint32_t kNegInf = 0xff80u, kKeyMask = 0xffffu;
  static __device__ __forceinline__ uint32_t get(const uint4 &r, int k) {
    const uint32_t w = (&r.x)[k >> 1];
    return (k & 1) ? (w >> 16) : (w & 0xffffu);
  }
  static __device__ __forceinline__ float val(uint32_t b) { return __uint_as_float(b << 16); }
};
template <>
struct TpType<__half> {
  static constexpr int G = 8;
  static constexpr uint32_t kSign = 0x8000u, kMag = 0x7fffu, kInf = 0x7c00u;
  static constexpr uint32_t kNegInf = 0xfc00u, kKeyMask = 0xffffu;
  static __device__ __forceinline__ uint32_t get(const uint4 &r, int k) {
    const uint32_t w = (&r.x)[k >> 1];
    return (k & 1) ? (w >> 16) : (w & 0xffffu);
  }
  static __device__ __forceinline__ float val(uint32_t b) {
    return __half2float(__ushort_as_half((unsigned short)b));
  }
};

__device__ __forceinline__ float tp_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ u64 ld_dsmem_u64(uint32_t addr) {
  u64 v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void st_dsmem_u64(uint32_t addr, u64 v) {
  asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
}

__device__ __forceinline__ uint32_t tp_cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// One element: its bits with NaN made -inf and -0 made +0 (canonical), whether
// it was NaN, and its composite key.
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

// Exclusive block scan of one u64 per thread; *total gets the block sum.
__device__ __forceinline__ u64 block_excl_scan_u64(u64 v, u64 *s_warp, u64 *total) {
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
  for (int w = 0; w < kTpThreads / 32; ++w) {
    const u64 x = s_warp[w];
    if (w < warp) before += x;
    tot += x;
  }
  __syncthreads();
  *total = tot;
  return before + incl - v;
}

// Calls f(e, bits) for every element e < n of this CTA's slice in shared
// memory: full 16-byte groups round-robin over the threads, then the ragged
// last group on one thread.
template <typename T, typename F>
__device__ __forceinline__ void tp_for_each(const uint4 *sl, int n, F f) {
  constexpr int G = TpType<T>::G;
  const int nfull = n / G;
  for (int g = threadIdx.x; g < nfull; g += kTpThreads) {
    const uint4 r = sl[g];
#pragma unroll
    for (int k = 0; k < G; ++k) f(g * G + k, TpType<T>::get(r, k));
  }
  const int rem = n - nfull * G;
  if (rem > 0 && (int)threadIdx.x == nfull % kTpThreads) {
    const uint4 r = sl[nfull];
#pragma unroll
    for (int k = 0; k < G; ++k)
      if (k < rem) f(nfull * G + k, TpType<T>::get(r, k));
  }
}

__device__ __forceinline__ unsigned atom_add_dsmem_u32(uint32_t addr, unsigned v) {
  unsigned old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}

// In the histogram whose logical entries [threadIdx.x * PER, +PER) this
// thread holds in h, the logical entry where the running mass, starting from
// `above`, first reaches thr; the winner writes phys(entry) to *s_sel and the
// mass before it to *s_above. Returns the total of all entries.
template <int PER, typename Phys>
__device__ __forceinline__ u64 tp_find_cross(const u64 (&h)[PER], Phys phys, u64 above, u64 thr, u64 *s_warp,
                                             int *s_sel, u64 *s_above) {
  u64 mine = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) mine += h[j];
  u64 tot;
  u64 cum = above + block_excl_scan_u64(mine, s_warp, &tot);
#pragma unroll
  for (int j = 0; j < PER; ++j) {
    const u64 nx = cum + h[j];
    if (cum < thr && thr <= nx) {
      *s_sel = phys((int)threadIdx.x * PER + j);
      *s_above = cum;
    }
    cum = nx;
  }
  __syncthreads();
  return tot;
}

template <typename T>
__global__ void __launch_bounds__(kTpThreads) topp_filter_kernel(const __grid_constant__ TpParams P) {
  using TT = TpType<T>;
  constexpr int G = TT::G;
  extern __shared__ uint4 sl[];     // this CTA's slice of the row (dynamic)
  __shared__ u64 h_mass[kTpBins];   // this CTA's histogram (read by the whole cluster)
  __shared__ u64 h_red[kTpBins];    // this CTA's segment of the cluster's totals
  __shared__ u64 s_segtot;          // ... and its sum
  __shared__ int s_owner;           // the CTA whose segment holds the crossing
  __shared__ u64 c_comp[kTpCap];    // first CTA: gathered candidates
  __shared__ u64 c_q[kTpCap];
  __shared__ u64 s_warp64[kTpThreads / 32];
  __shared__ int s_warp32[kTpThreads / 32];
  __shared__ int s_wflag[kTpThreads / 32];
  __shared__ float s_max;
  __shared__ int s_flag;            // bit 0: a NaN, bit 1: +inf
  __shared__ int s_sel;
  __shared__ u64 s_above;
  __shared__ u64 s_cut;
  __shared__ unsigned s_gcount;     // first CTA: candidates gathered so far

  pdl_wait();
  pdl_trigger();
  const int rank = (int)cluster_ctarank();
  const int CS = (int)tp_cluster_nctarank();
  const int row = blockIdx.y;
  const T *in;
  T *out;
  if (row < P.rows0) {
    in = static_cast<const T *>(P.in0) + (int64_t)row * P.V;
    out = static_cast<T *>(P.out0) + (int64_t)row * P.V;
  } else {
    in = static_cast<const T *>(P.in1) + (int64_t)(row - P.rows0) * P.V;
    out = static_cast<T *>(P.out1) + (int64_t)(row - P.rows0) * P.V;
  }
  const int lo = rank * P.slice;
  const int n = max(0, min(P.slice, P.V - lo));
  in += lo;
  out += lo;
  const int ng = (n + G - 1) / G;

  // ---- load the slice, and its maximum (NaN counts as -inf and is flagged) ----
  float mx = -INFINITY;
  int flag = 0;
  for (int g = threadIdx.x; g < ng; g += kTpThreads) {
    uint4 r = make_uint4(0u, 0u, 0u, 0u);
    if (P.vec && (g + 1) * G <= n) {
      r = __ldg(reinterpret_cast<const uint4 *>(in) + g);
    } else {
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const int e = g * G + k;
        if (e < n) {
          if (sizeof(T) == 4) (&r.x)[k] = __float_as_uint(__ldg(reinterpret_cast<const float *>(in) + e));
          else (&r.x)[k >> 1] |= (uint32_t)__ldg(reinterpret_cast<const unsigned short *>(in) + e) << ((k & 1) * 16);
        }
      }
    }
    sl[g] = r;
#pragma unroll
    for (int k = 0; k < G; ++k) {
      if (g * G + k < n) {
        bool nan;
        const float x = TT::val(tp_canon<T>(TT::get(r, k), nan));
        flag |= nan ? 1 : 0;
        flag |= (x == INFINITY) ? 2 : 0;
        mx = fmaxf(mx, x);
      }
    }
  }
  mx = warp_max(mx);
  flag = (int)__reduce_or_sync(0xffffffffu, (unsigned)flag);
  if ((threadIdx.x & 31) == 0) {
    s_warp32[threadIdx.x >> 5] = __float_as_int(mx);
    s_wflag[threadIdx.x >> 5] = flag;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = -INFINITY;
    int f = 0;
    for (int w = 0; w < kTpThreads / 32; ++w) {
      b = fmaxf(b, __int_as_float(s_warp32[w]));
      f |= s_wflag[w];
    }
    s_max = b;
    s_flag = f;
  }
  __syncthreads();
  cluster_sync();
  float m = -INFINITY;
  int rflag = 0;
  for (int r = 0; r < CS; ++r) {
    m = fmaxf(m, ld_dsmem_f32(mapa(&s_max, r)));
    rflag |= ld_dsmem_s32(mapa(&s_flag, r));
  }
  cluster_sync();   // every CTA has read the others' maxima
  if (rflag && rank == 0 && threadIdx.x == 0) atomic_or_status(P.status, SV_DEV_NONFINITE);

  if (!(m > -INFINITY) || m == INFINITY) {
    // nothing to rank (an empty or all -inf row, or a +inf logit): the row is
    // passed through unchanged and the sampling flags it
    for (int g = threadIdx.x; g < ng; g += kTpThreads) {
      const uint4 r = sl[g];
      if (P.vec && (g + 1) * G <= n) {
        *(reinterpret_cast<uint4 *>(out) + g) = r;
      } else {
#pragma unroll
        for (int k = 0; k < G; ++k) {
          const int e = g * G + k;
          if (e < n) {
            if (sizeof(T) == 4) reinterpret_cast<uint32_t *>(out)[e] = TT::get(r, k);
            else reinterpret_cast<unsigned short *>(out)[e] = (unsigned short)TT::get(r, k);
          }
        }
      }
    }
    return;
  }

  // Bins: b(x) = floor(-32 (x c_hi - fl(m c_hi))), one fma from the logit,
  // non-increasing in x and computed the same way in every pass (bin 2047
  // also takes everything below 2^-64 of the maximum, and -inf).
  // Weights: 2^ex with ex = (x - m) c taken as hi + lo: x - m by two-sum
  // (exact), times c = c_hi + c_lo with an fma for the product's rounding.
  // 2^hi comes from the SFU (relative error below 1.5e-7 on [-30, 0]) and
  // 2^lo as the first-order factor 1 + lo ln 2 (|lo| is at most an ulp of
  // hi, so the neglected term is ~1e-12).
  const float c_hi = P.c_hi, c_lo = P.c_lo;
  const float mc = __fmul_rn(m, c_hi);
  auto bin_of = [&](float x) { return min(kTpBins - 1, (int)(-fmaf(x, c_hi, -mc) * 32.f)); };
  auto mass_of = [&](float x) -> u64 {
    if (!(x > -INFINITY)) return 0ull;
    const float d = x - m;
    const float bb = d - x;
    const float d_lo = (x - (d - bb)) + (-m - bb);
    const float h = d * c_hi;
    float l = fmaf(d, c_hi, -h);
    l = fmaf(d, c_lo, l);
    l = fmaf(d_lo, c_hi, l);
    const float t = tp_ex2(h);
    if (!(t > 0.f)) return 0ull;
    return __float2ull_rn(fmaf(t, l * 0.693147180559945309f, t) * kTpQuant);
  };
  const int lane = threadIdx.x & 31;

  // ---- first-level histogram of the quantised masses ----
  for (int i = threadIdx.x; i < kTpBins; i += kTpThreads) h_mass[i] = 0ull;
  if (threadIdx.x == 0) { s_gcount = 0u; s_sel = -1; s_above = 0ull; s_cut = 0ull; }
  __syncthreads();
  tp_for_each<T>(sl, n, [&](int, uint32_t b) {
    bool nan;
    const float x = TT::val(tp_canon<T>(b, nan));
    const int bn = bin_of(x);
    if (bn < kTpBins - 1) {
      const u64 q = mass_of(x);
      if (q) atomicAdd(&h_mass[bn], q);
    }
  });
  __syncthreads();
  cluster_sync();

  // ---- the bin where the running mass reaches ceil(top_p Z) ----
  // Reduce-scatter: CTA `rank` sums the bins [b0, b1) over the cluster
  // (coalesced reads of the others' shared memory), then only the segment
  // totals are exchanged; the CTA whose segment holds the crossing finds the
  // bin and publishes it.
  const int seg = (kTpBins + CS - 1) / CS;
  const int b0 = min(kTpBins, rank * seg), b1 = min(kTpBins, b0 + seg);
  for (int i = b0 + (int)threadIdx.x; i < b1; i += kTpThreads) {
    u64 t = 0;
    for (int r = 0; r < CS; ++r) t += ld_dsmem_u64(mapa(&h_mass[i], r));
    h_red[i - b0] = t;
  }
  __syncthreads();
  constexpr int kPer = kTpBins / kTpThreads;   // entries per thread in the scan (segments are at most kTpBins)
  u64 h8[kPer];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int i = (int)threadIdx.x * kPer + j;
    h8[j] = i < b1 - b0 ? h_red[i] : 0ull;
  }
  u64 seg_tot;
  {
    u64 mine = 0;
#pragma unroll
    for (int j = 0; j < kPer; ++j) mine += h8[j];
    (void)block_excl_scan_u64(mine, s_warp64, &seg_tot);
  }
  if (threadIdx.x == 0) s_segtot = seg_tot;
  cluster_sync();
  u64 Z = 0, before = 0;
  for (int r = 0; r < CS; ++r) {
    const u64 t = ld_dsmem_u64(mapa(&s_segtot, r));
    if (r < rank) before += t;
    Z += t;
  }
  u64 thr = (u64)ceil(P.top_p * (double)Z);
  thr = thr < 1ull ? 1ull : (thr > Z ? Z : thr);
  if (before < thr && thr <= before + seg_tot)
    (void)tp_find_cross<kPer>(h8, [b0](int i) { return b0 + i; }, before, thr, s_warp64, &s_sel, &s_above);
  if (threadIdx.x == 0) {
    // which CTA holds the crossing: the same arithmetic in every CTA
    u64 acc = 0;
    int owner = 0;
    for (int r = 0; r < CS; ++r) {
      const u64 t = ld_dsmem_u64(mapa(&s_segtot, r));
      if (acc < thr && thr <= acc + t) owner = r;
      acc += t;
    }
    s_owner = owner;
  }
  cluster_sync();
  const int bin = ld_dsmem_s32(mapa(&s_sel, s_owner));
  u64 above = ld_dsmem_u64(mapa(&s_above, s_owner));

  // ---- gather the bin's elements into the first CTA (warp-aggregated slots) ----
  const uint32_t gcount = mapa(&s_gcount, 0);
  auto gather = [&](int e, uint32_t cb, float x, bool cand) {
    const unsigned am = __activemask();
    const unsigned bal = __ballot_sync(am, cand);
    if (!bal) return;
    const int leader = __ffs(bal) - 1;
    unsigned base = 0;
    if (lane == leader) base = atom_add_dsmem_u32(gcount, (unsigned)__popc(bal));
    base = __shfl_sync(am, base, leader);
    if (cand) {
      const unsigned slot = base + (unsigned)__popc(bal & ((1u << lane) - 1u));
      if (slot < (unsigned)kTpCap) {
        st_dsmem_u64(mapa(&c_comp[slot], 0), tp_composite<T>(cb, lo + e));
        st_dsmem_u64(mapa(&c_q[slot], 0), mass_of(x));
      }
    }
  };
  tp_for_each<T>(sl, n, [&](int e, uint32_t b) {
    bool nan;
    const uint32_t cb = tp_canon<T>(b, nan);
    const float x = TT::val(cb);
    gather(e, cb, x, bin_of(x) == bin);
  });
  cluster_sync();
  int n_all = ld_dsmem_s32(gcount);

  if (n_all > kTpCap) {
    // Rare: more than kTpCap elements share the bin (many equal or nearly
    // equal logits). Split them by the composite's bits, 8 at a time from
    // the top, keeping the part where the running mass reaches thr, until at
    // most kTpCap remain (composites are distinct, so this ends).
    int sh = 64;
    u64 pfx = 0ull;
    auto is_cand = [&](int e, uint32_t cb, float x) {
      if (bin_of(x) != bin) return false;
      return sh >= 64 || (tp_composite<T>(cb, lo + e) >> sh) == pfx;
    };
    while (n_all > kTpCap && sh > 0) {
      const int nsh = sh > 8 ? sh - 8 : 0;
      const int width = sh - nsh;
      cluster_sync();   // every CTA is done reading the previous histogram and counter
      for (int i = threadIdx.x; i < 256; i += kTpThreads) h_mass[i] = 0ull;
      if (threadIdx.x == 0) { s_gcount = 0u; s_sel = -1; }
      __syncthreads();
      tp_for_each<T>(sl, n, [&](int e, uint32_t b) {
        bool nan;
        const uint32_t cb = tp_canon<T>(b, nan);
        const float x = TT::val(cb);
        if (is_cand(e, cb, x)) {
          const u64 q = mass_of(x);
          const int d = (int)((tp_composite<T>(cb, lo + e) >> nsh) & ((1ull << width) - 1ull));
          if (q) atomicAdd(&h_mass[d], q);
        }
      });
      __syncthreads();
      cluster_sync();
      u64 h1[1] = {0ull};
      for (int r = 0; r < CS; ++r) h1[0] += ld_dsmem_u64(mapa(&h_mass[255 - threadIdx.x], r));
      (void)tp_find_cross<1>(h1, [](int i) { return 255 - i; }, above, thr, s_warp64, &s_sel, &s_above);
      above = s_above;
      pfx = (sh >= 64 ? 0ull : (pfx << width)) | (u64)(s_sel < 0 ? 0 : s_sel);
      sh = nsh;
      cluster_sync();   // the first CTA's counter is zero everywhere it is read
      tp_for_each<T>(sl, n, [&](int e, uint32_t b) {
        bool nan;
        const uint32_t cb = tp_canon<T>(b, nan);
        const float x = TT::val(cb);
        gather(e, cb, x, is_cand(e, cb, x));
      });
      cluster_sync();
      n_all = ld_dsmem_s32(gcount);
    }
  }

  // ---- rank the gathered candidates in the first CTA ----
  if (rank == 0 && n_all <= kTpCap) {
    // candidate i is the cut iff the mass before it (the bins and radix parts
    // above, plus every candidate with a larger composite) is below thr and
    // reaches thr with it
    for (int i = threadIdx.x; i < n_all; i += kTpThreads) {
      const u64 ci = c_comp[i], qi = c_q[i];
      u64 before = 0;
      for (int j = 0; j < n_all; ++j) before += (c_comp[j] > ci) ? c_q[j] : 0ull;
      if (above + before < thr && thr <= above + before + qi) s_cut = ci;
    }
  }
  __syncthreads();
  cluster_sync();
  const u64 cut = ld_dsmem_u64(mapa(&s_cut, 0));   // 0: no cut found, keep the row
  cluster_sync();   // the first CTA stays until every CTA has read the cut

  // ---- write the filtered slice: bins above the cut's bin stay, bins below
  // go, and within the cut's bin the composite decides ----
  auto keep_of = [&](int e, uint32_t b) {
    bool nan;
    const uint32_t cb = tp_canon<T>(b, nan);
    if (nan) return false;
    if (cut == 0ull) return true;
    const int bn = bin_of(TT::val(cb));
    return bn < bin || (bn == bin && tp_composite<T>(cb, lo + e) >= cut);
  };
  for (int g = threadIdx.x; g < ng; g += kTpThreads) {
    const uint4 r = sl[g];
    const bool full = (g + 1) * G <= n;
    uint32_t ob[G];
#pragma unroll
    for (int k = 0; k < G; ++k) {
      const uint32_t b = TT::get(r, k);
      ob[k] = (full || g * G + k < n) && keep_of(g * G + k, b) ? b : TT::kNegInf;
    }
    if (P.vec && full) {
      uint4 o;
      if (sizeof(T) == 4) {
        o = make_uint4(ob[0], ob[1 % G], ob[2 % G], ob[3 % G]);
      } else {
#pragma unroll
        for (int k = 0; k < G; k += 2) (&o.x)[k >> 1] = ob[k] | (ob[(k + 1) % G] << 16);
      }
      *(reinterpret_cast<uint4 *>(out) + g) = o;
    } else {
#pragma unroll
      for (int k = 0; k < G; ++k) {
        const int e = g * G + k;
        if (e < n) {
          if (sizeof(T) == 4) reinterpret_cast<uint32_t *>(out)[e] = ob[k];
          else reinterpret_cast<unsigned short *>(out)[e] = (unsigned short)ob[k];
        }
      }
    }
  }
}

}  // namespace

// Launches the filter over rows0 rows of in0 -> out0 followed by rows1 rows of
// in1 -> out1 (all [rows][V] of one dtype). Host checks are the caller's.
sv_status launch_topp_filter(sv_dtype dtype, const void *in0, void *out0, int rows0, const void *in1, void *out1,
                             int rows1, int V, float temperature, float top_p, int32_t *status, cudaStream_t s) {
  const int es = dtype_bytes(dtype);
  const int G = 16 / es;
  const int per_cta = kTpVec * kTpThreads * G;
  const int cs = (V + per_cta - 1) / per_cta;
  if (cs > 16) return fail(SV_ERR_UNSUPPORTED, "top-p filter: V = %d above %d for this dtype", V, 16 * per_cta);
  if (rows0 + rows1 > 65535) return fail(SV_ERR_UNSUPPORTED, "top-p filter: more than 65535 rows");
  if (rows0 + rows1 == 0) return ok();
  TpParams P = {};
  P.in0 = in0; P.out0 = out0; P.rows0 = rows0;
  P.in1 = in1; P.out1 = out1;
  P.V = V;
  P.slice = ((V + cs - 1) / cs + G - 1) / G * G;
  P.vec = aligned(in0, 16) && aligned(out0, 16) && (rows1 == 0 || (aligned(in1, 16) && aligned(out1, 16))) &&
          ((size_t)V * es) % 16 == 0;
  const double cd = 1.4426950408889634074 / (double)temperature;
  P.c_hi = (float)cd;
  P.c_lo = (float)(cd - (double)P.c_hi);
  P.top_p = (double)top_p;
  P.status = status;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    const int dyn = kTpVec * kTpThreads * 16;   // the largest slice
    cudaError_t r[6] = {
        cudaFuncSetAttribute(topp_filter_kernel<float>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
        cudaFuncSetAttribute(topp_filter_kernel<__nv_bfloat16>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
        cudaFuncSetAttribute(topp_filter_kernel<__half>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1),
        cudaFuncSetAttribute(topp_filter_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn),
        cudaFuncSetAttribute(topp_filter_kernel<__nv_bfloat16>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn),
        cudaFuncSetAttribute(topp_filter_kernel<__half>, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn)};
    for (cudaError_t x : r)
      if (x != cudaSuccess && attr_err == cudaSuccess) attr_err = x;
  });
  if (attr_err != cudaSuccess) return fail(SV_ERR_CUDA, "top-p filter attributes: %s", cudaGetErrorString(attr_err));
  cudaError_t e = cudaSuccess;
  const dim3 grid(cs, rows0 + rows1);
  const size_t dyn = (size_t)P.slice * es;
  switch (dtype) {
    case SV_F32: e = launch_k(topp_filter_kernel<float>, grid, dim3(kTpThreads), dyn, s, cs, P); break;
    case SV_BF16: e = launch_k(topp_filter_kernel<__nv_bfloat16>, grid, dim3(kTpThreads), dyn, s, cs, P); break;
    case SV_F16: e = launch_k(topp_filter_kernel<__half>, grid, dim3(kTpThreads), dyn, s, cs, P); break;
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

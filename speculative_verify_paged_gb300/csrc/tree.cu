// Rejection sampling over a draft tree: one cluster per sequence walks the tree
// from the root. At node u the residual starts as r = p_u; u's children
// (drafted from q_u) are tried in BFS order, child c with token x accepted
// iff uniforms[c][0] * q_u(x) < r(x); a rejection replaces r by
// norm(max(0, r - q_u)); an accepted child becomes u; when every child of u
// is rejected, or u is a leaf, the token is drawn from r by the inverse CDF
// with v = uniforms[u][1] (the reading of "standard rejection sampling" over
// the BFS tree of "KV Cache + Speculative Decoding", Q14 and section 8.2,
// with the chain rule of quant67 "speculative decoding" section 3.1; for a
// chain it is that rule).
//
// The residuals never need to be stored: after k rejections at u,
//   r_k = max(0, p - c_k q) / D_k,  c_0 = 0, D_0 = 1,
//   c_{k+1} = c_k + D_k,  D_{k+1} = sum_x max(0, p(x) - c_{k+1} q(x)),
// (induction: max(0, r_k - q) = max(0, p - c_k q - D_k q) / D_k), so a
// rejection costs one row-wide sum and the draw one more pass. The rows'
// (max, sum, entropy) statistics come from a pre-pass over all rows in
// parallel.
//
// Optionally (typical != NULL) the accept test is typical acceptance, the
// Medusa rule the pages describe as an approximate alternative ("speculative
// decoding" survey section 9.1, "KV Cache + Speculative Decoding" Q18): child
// x of u is accepted iff p_u(x) > min(epsilon, delta exp(-H(p_u))), with no
// residual; when no child passes, the token is drawn from p_u.
//
// Arithmetic is fp32 in a fixed order (each thread owns a contiguous chunk of
// token ids, sums groups of 8, then a block tree), so the kernel is
// deterministic; its decisions agree with exact arithmetic unless a uniform
// lies within ~1e-6 (relative) of its boundary.

#include <climits>
#include <cmath>
#include <type_traits>

#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kTrThreads = 512;
constexpr int kTrCluster = 4;            // CTAs per sequence in the walk
constexpr int kTrWarps = kTrThreads / 32;
constexpr int kTrMaxNodes = 64;

struct TreeParams {
  const void *target;      // [B][n][V]
  const void *draft;       // [B][n][V] logits (T) or probabilities (f32)
  const int32_t *parent;   // [B][n]
  const int32_t *tokens;   // [B][n]
  const float *uniforms;   // [B][n][2]
  int32_t *out_tokens;     // [B][n]
  int32_t *num_acc;        // [B]
  int32_t *path;           // [B][n]
  int32_t *status;
  float4 *stats;           // [B][2n] (max, S = sum of 2^t, H in nats, 0), t = fl(l c) - fl(max c): target rows, then draft rows
  int typical;             // typical acceptance instead of rejection sampling
  float tau_eps, tau_delta;
  int B, n, V, slice, chunk;   // token ids per walk CTA and per thread (multiples of 8)
  int vec_t, vec_d;        // rows 16-byte aligned: vector loads
  float c;                 // log2(e) / T
};

__device__ __forceinline__ float tr_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float ld_f32(const float *p, int i) { return __ldg(p + i); }
__device__ __forceinline__ float ld_f32(const __nv_bfloat16 *p, int i) { return __bfloat162float(p[i]); }
__device__ __forceinline__ float ld_f32(const __half *p, int i) { return __half2float(p[i]); }

// Eight consecutive values starting at i (a multiple of 8) as floats.
template <typename T>
__device__ __forceinline__ void ld8(const T *row, int i, bool vec, float (&x)[8]) {
  if (vec) {
    if (sizeof(T) == 4) {
      const float4 a = __ldg(reinterpret_cast<const float4 *>(row + i));
      const float4 b = __ldg(reinterpret_cast<const float4 *>(row + i) + 1);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    } else {
      const uint4 v = __ldg(reinterpret_cast<const uint4 *>(row + i));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        if (std::is_same<T, __nv_bfloat16>::value) {
          x[2 * k] = __uint_as_float(w[k] << 16);
          x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        } else {
          const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&w[k]));
          x[2 * k] = f.x;
          x[2 * k + 1] = f.y;
        }
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < 8; ++k) x[k] = ld_f32(row, i + k);
  }
}

// Eight consecutive elements as loaded (16-bit types: one 16-byte vector;
// f32: two), decoded only when used, so that several loads can be in flight.
template <typename T>
struct Raw8 {
  uint4 a, b;
};

template <typename T>
__device__ __forceinline__ void ld_raw(const T *row, int i, Raw8<T> &r) {
  r.a = __ldg(reinterpret_cast<const uint4 *>(row + i));
  if (sizeof(T) == 4) r.b = __ldg(reinterpret_cast<const uint4 *>(row + i) + 1);
}

template <typename T>
__device__ __forceinline__ float raw_at(const Raw8<T> &r, int k) {
  if (sizeof(T) == 4) return __uint_as_float(k < 4 ? (&r.a.x)[k] : (&r.b.x)[k - 4]);
  const uint32_t w = (&r.a.x)[k >> 1];
  const uint32_t h = (k & 1) ? (w >> 16) : (w & 0xffffu);
  if (std::is_same<T, __nv_bfloat16>::value) return __uint_as_float(h << 16);
  return __half2float(__ushort_as_half((unsigned short)h));
}

// f(lp, lq, id) over the chunk [lo, hi) of two rows (p and q) in token
// order: nfull whole groups of eight from lo (two groups of 16-byte loads in
// flight when the rows are aligned), then the rest one element at a time;
// with use_q false the q row is not read and lq is 0.
template <typename T, typename TD, typename F>
__device__ __forceinline__ void tr_each2(const T *pr, bool vt, const TD *qr, bool vd, bool use_q, int lo, int nfull,
                                         int hi, F f) {
  constexpr int NB = 2;
  int g = 0;
  if (vt && (vd || !use_q)) {
    for (; g + NB <= nfull; g += NB) {
      Raw8<T> a[NB];
      Raw8<TD> d[NB];
#pragma unroll
      for (int u = 0; u < NB; ++u) {
        ld_raw(pr, lo + 8 * (g + u), a[u]);
        if (use_q) ld_raw(qr, lo + 8 * (g + u), d[u]);
      }
#pragma unroll
      for (int u = 0; u < NB; ++u)
#pragma unroll
        for (int k = 0; k < 8; ++k) f(raw_at(a[u], k), use_q ? raw_at(d[u], k) : 0.f, lo + 8 * (g + u) + k);
    }
  }
  for (; g < nfull; ++g) {
    float x[8], y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    ld8(pr, lo + 8 * g, vt, x);
    if (use_q) ld8(qr, lo + 8 * g, vd, y);
#pragma unroll
    for (int k = 0; k < 8; ++k) f(x[k], y[k], lo + 8 * g + k);
  }
  for (int i = lo + 8 * nfull; i < hi; ++i) f(ld_f32(pr, i), use_q ? ld_f32(qr, i) : 0.f, i);
}

__device__ __forceinline__ float tr_block_sum(float v, float *s_red) {
  v = warp_sum(v);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  float t = lane < kTrWarps ? s_red[lane] : 0.f;
  t = warp_sum(t);
  return t;   // every thread of warp 0..31 holds the total (all warps recompute it)
}

// Exclusive scan of one float per thread in thread order; *total the sum.
__device__ __forceinline__ float tr_block_excl_scan(float v, float *s_red, float *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  __syncthreads();
  if (lane == 31) s_red[warp] = incl;
  __syncthreads();
  float before = 0.f, tot = 0.f;
  for (int w = 0; w < kTrWarps; ++w) {
    const float x = s_red[w];
    if (w < warp) before += x;
    tot += x;
  }
  *total = tot;
  return before + incl - v;
}

// (max, sum) of every row the walk may need, one CTA per row, all rows of all
// sequences at once: grid (2n, B); row x < n is target row x, row n + u the
// draft row of node u (skipped for leaves and for draft probabilities). One
// online pass: each thread keeps (m, s) over its 16-byte groups (coalesced,
// round-robin), rescaling s when m grows; the block combines the pairs.
// The terms are 2^(fl(l c) - fl(m c)) with the final m, the reference the
// walk evaluates p(x) and q(x) against.
constexpr int kTsThreads = 512;

// (m, S, A) with S = sum 2^t and A = sum 2^t t, t = fl(l c) - fl(m c):
// moving the reference from m to m' > m (d = fl(m' c) - fl(m c)) scales S by
// 2^-d and turns A into 2^-d (A - d S).
__device__ __forceinline__ void tr_msa_combine(float &m, float &s, float &a, float m2, float s2, float a2, float c) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) { m = mn; s = 0.f; a = 0.f; return; }
  const float rc = __fmul_rn(mn, c);
  float s1 = 0.f, a1 = 0.f, s3 = 0.f, a3 = 0.f;
  if (m != -INFINITY) {
    const float d = rc - __fmul_rn(m, c), f = tr_ex2(-d);
    s1 = s * f;
    a1 = (a - d * s) * f;
  }
  if (m2 != -INFINITY) {
    const float d = rc - __fmul_rn(m2, c), f = tr_ex2(-d);
    s3 = s2 * f;
    a3 = (a2 - d * s2) * f;
  }
  s = s1 + s3;
  a = a1 + a3;
  m = mn;
}

template <typename T, int DK>
__global__ void __launch_bounds__(kTsThreads) tree_row_stats_kernel(const __grid_constant__ TreeParams P) {
  using TD = typename std::conditional<DK == 1, float, T>::type;
  __shared__ float s_m[kTsThreads / 32], s_s[kTsThreads / 32], s_a[kTsThreads / 32];
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.y, x = blockIdx.x, n = P.n, V = P.V;
  const bool draft_row = x >= n;
  const int node = draft_row ? x - n : x;
  if (draft_row) {
    if (DK == 1 || P.typical) return;
    bool has_child = false;
    for (int j = node + 1; j < n; ++j) has_child |= __ldg(P.parent + (int64_t)b * n + j) == node;
    if (!has_child) return;
  }
  const float c = P.c;
  float m = -INFINITY, sum = 0.f, ent = 0.f;   // ent: sum 2^t t
  auto add8 = [&](const float (&v)[8]) {
    float mx = v[0];
#pragma unroll
    for (int k = 1; k < 8; ++k) mx = fmaxf(mx, v[k]);
    if (mx > m) {
      if (m == -INFINITY) {
        sum = 0.f;
        ent = 0.f;
      } else {
        const float d = __fmul_rn(mx, c) - __fmul_rn(m, c), f = tr_ex2(-d);
        ent = (ent - d * sum) * f;
        sum *= f;
      }
      m = mx;
    }
    if (m == -INFINITY) return;
    const float mc = __fmul_rn(m, c);
    float g = 0.f, h = 0.f;
    if (P.typical) {   // the entropy term only matters to typical acceptance
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float t = fmaf(v[k], c, -mc), e = tr_ex2(t);
        g += e;
        h += t > -INFINITY ? e * t : 0.f;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) g += tr_ex2(fmaf(v[k], c, -mc));
    }
    sum += g;
    ent += h;
  };
  auto run = [&](const auto *row, bool vec) {
    const int ng = V / 8;
    for (int g = threadIdx.x; g < ng; g += kTsThreads) {
      float v[8];
      ld8(row, 8 * g, vec, v);
      add8(v);
    }
    if ((int)threadIdx.x == 0 && V % 8) {
      float v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = 8 * ng + k < V ? ld_f32(row, 8 * ng + k) : -INFINITY;
      add8(v);
    }
  };
  if (draft_row) run(static_cast<const TD *>(P.draft) + ((int64_t)b * n + node) * V, P.vec_d);
  else run(static_cast<const T *>(P.target) + ((int64_t)b * n + node) * V, P.vec_t);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, sum, o),
                a2 = __shfl_xor_sync(0xffffffffu, ent, o);
    tr_msa_combine(m, sum, ent, m2, s2, a2, c);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) { s_m[warp] = m; s_s[warp] = sum; s_a[warp] = ent; }
  __syncthreads();
  if (threadIdx.x == 0) {
    float mm = s_m[0], ss = s_s[0], aa = s_a[0];
    for (int w = 1; w < kTsThreads / 32; ++w) tr_msa_combine(mm, ss, aa, s_m[w], s_s[w], s_a[w], c);
    // H = -sum p ln p = ln S - ln 2 * A / S  (p = 2^t / S, ln p = t ln 2 - ln S)
    const float H = (ss > 0.f) ? logf(ss) - 0.693147180559945309f * aa / ss : 0.f;
    P.stats[(int64_t)b * 2 * n + x] = make_float4(mm, ss, H, 0.f);
  }
}

// The walk: one cluster of kTrCluster CTAs per sequence, CTA r owning the
// token slice [r slice, (r + 1) slice) and each of its threads a chunk of
// it. Every decision is computed identically in every CTA (point loads, and
// cluster sums read in rank order), so control flow is cluster-uniform.
template <typename T, int DK>
__global__ void __launch_bounds__(kTrThreads, 2) sample_tree_kernel(const __grid_constant__ TreeParams P) {
  using TD = typename std::conditional<DK == 1, float, T>::type;
  __shared__ int par[kTrMaxNodes];
  __shared__ int tok[kTrMaxNodes];
  __shared__ float s_red[kTrWarps];
  __shared__ float s_part[2];            // this CTA's block total, alternating per cluster exchange
  __shared__ int s_owner, s_y, s_first, s_last;

  pdl_wait();
  pdl_trigger();
  const int rank = (int)cluster_ctarank();
  const int CS = (int)gridDim.x;         // the cluster spans the grid's x dimension
  const int b = blockIdx.y, n = P.n, V = P.V;
  const int tid = threadIdx.x;
  if (tid < n) {
    par[tid] = __ldg(P.parent + (int64_t)b * n + tid);
    tok[tid] = __ldg(P.tokens + (int64_t)b * n + tid);
  }
  __syncthreads();
  int32_t *out = P.out_tokens + (int64_t)b * n;
  int32_t *path = P.path + (int64_t)b * n;
  if (rank == 0)
    for (int j = tid; j < n; j += kTrThreads) { out[j] = -1; path[j] = -1; }
  bool ok = par[0] == -1;
  for (int j = 1; j < n; ++j) ok &= par[j] >= 0 && par[j] < j;
  if (!ok) {
    if (rank == 0 && tid == 0) { atomic_or_status(P.status, SV_DEV_BAD_TREE); P.num_acc[b] = 0; }
    return;
  }

  const float c = P.c;
  const int s_lo = min(V, rank * P.slice), s_hi = min(V, s_lo + P.slice);
  const int lo = min(s_hi, s_lo + tid * P.chunk), hi = min(s_hi, lo + P.chunk);
  const int nfull = (hi - lo) / 8;       // whole groups of 8 in this thread's chunk
  const T *trow_base = static_cast<const T *>(P.target) + (int64_t)b * n * V;
  const TD *drow_base = static_cast<const TD *>(P.draft) + (int64_t)b * n * V;
  const bool vt = P.vec_t, vd = P.vec_d;
  int xchg = 0;
  // the per-CTA totals of every CTA, in rank order (one cluster barrier)
  auto cluster_parts = [&](float mine_cta, float (&parts)[kTrCluster]) {
    const int slot = xchg & 1;
    ++xchg;
    if (tid == 0) s_part[slot] = mine_cta;
    cluster_sync();
#pragma unroll
    for (int r = 0; r < kTrCluster; ++r) parts[r] = r < CS ? ld_dsmem_f32(mapa(&s_part[slot], r)) : 0.f;
  };

  int u = 0, depth = 0;
  for (;;) {
    const T *prow = trow_base + (int64_t)u * V;
    const TD *qrow = drow_base + (int64_t)u * V;
    float m_q = 0.f, S_q = 1.f;
    const float4 sp = P.stats[(int64_t)b * 2 * n + u];
    const float m_p = sp.x, S_p = sp.y;
    // typical acceptance: the threshold min(eps, delta exp(-H(p_u)))
    const float tau = P.typical ? fminf(P.tau_eps, P.tau_delta * expf(-sp.z)) : 0.f;
    const float mpc = __fmul_rn(m_p, c), inv_p = 1.f / S_p;
    bool has_child = false;
    for (int j = u + 1; j < n; ++j) has_child |= par[j] == u;
    if (has_child && DK == 0 && !P.typical) {
      const float4 sq = P.stats[(int64_t)b * 2 * n + n + u];
      m_q = sq.x;
      S_q = sq.y;
    }
    if (!(m_p > -INFINITY && m_p < INFINITY) ||
        (DK == 0 && has_child && !P.typical && !(m_q > -INFINITY && m_q < INFINITY))) {
      // a row without a finite maximum: flagged, the walk stops here
      if (rank == 0 && tid == 0) { atomic_or_status(P.status, SV_DEV_NONFINITE); P.num_acc[b] = depth; }
      cluster_sync();   // no CTA leaves while another may read its shared memory
      return;
    }
    const float mqc = __fmul_rn(m_q, c), inv_q = 1.f / S_q;
    auto p_of = [&](float l) { return tr_ex2(fmaf(l, c, -mpc)) * inv_p; };
    auto q_of = [&](float l) { return DK == 1 ? l : tr_ex2(fmaf(l, c, -mqc)) * inv_q; };

    float coef = 0.f, D = 1.f;   // the residual is max(0, p - coef q) / D
    int accepted = -1;
    for (int ch = u + 1; ch < n && accepted < 0; ++ch) {
      if (par[ch] != u) continue;
      const int x = tok[ch];
      if (x < 0 || x >= V) {   // flagged; such a child is never accepted and changes nothing
        if (rank == 0 && tid == 0) atomic_or_status(P.status, SV_DEV_BAD_TOKEN);
        continue;
      }
      if (P.typical) {   // no residual: the next child is tested against the same threshold
        if (p_of(ld_f32(prow, x)) > tau) {
          accepted = ch;
          break;
        }
        continue;
      }
      const float px = p_of(ld_f32(prow, x)), qx = q_of(ld_f32(qrow, x));
      const float rx = fmaxf(0.f, px - coef * qx) / D;
      const float uu = __ldg(P.uniforms + ((int64_t)b * n + ch) * 2);
      if (uu * qx < rx) {
        accepted = ch;
        break;
      }
      // rejected: the next residual
      coef += D;
      float acc = 0.f, grp = 0.f;
      int cnt = 0;
      tr_each2(prow, vt, qrow, vd, true, lo, nfull, hi, [&](float lp, float lq, int) {
        grp += fmaxf(0.f, p_of(lp) - coef * q_of(lq));
        if (++cnt == 8) { acc += grp; grp = 0.f; cnt = 0; }
      });
      float parts[kTrCluster];
      cluster_parts(tr_block_sum(acc + grp, s_red), parts);
      D = 0.f;
#pragma unroll
      for (int r = 0; r < kTrCluster; ++r) D += parts[r];
      if (!(D > 0.f)) { coef = 0.f; D = 1.f; }   // cannot happen in exact arithmetic: draw from p
    }
    if (accepted >= 0) {
      if (rank == 0 && tid == 0) { out[depth] = tok[accepted]; path[depth] = accepted; }
      ++depth;
      u = accepted;
      continue;
    }

    // ---- draw from max(0, p - coef q) (p itself when coef = 0) ----
    auto w_of = [&](float lp, float lq) { return coef == 0.f ? p_of(lp) : fmaxf(0.f, p_of(lp) - coef * q_of(lq)); };
    float mine = 0.f, grp = 0.f;
    int cnt = 0, first_pos = INT_MAX, last_pos = -1;
    tr_each2(prow, vt, qrow, vd, coef != 0.f, lo, nfull, hi, [&](float lp, float lq, int i) {
      const float w = w_of(lp, lq);
      grp += w;
      if (w > 0.f) { first_pos = min(first_pos, i); last_pos = i; }
      if (++cnt == 8) { mine += grp; grp = 0.f; cnt = 0; }
    });
    mine += grp;
    float Zc;
    const float before_cta = tr_block_excl_scan(mine, s_red, &Zc);
    float parts[kTrCluster];
    cluster_parts(Zc, parts);
    float Z = 0.f, off = 0.f;
#pragma unroll
    for (int r = 0; r < kTrCluster; ++r) {
      if (r < rank) off += parts[r];
      Z += parts[r];
    }
    const float target = __ldg(P.uniforms + ((int64_t)b * n + u) * 2 + 1) * Z;
    // the CTA, then the chunk, holding y = min{y : C(y) > v Z}: the last
    // whose running sum before it is <= v Z (the same sums in every CTA)
    int owner_rank = 0;
    {
      float o = 0.f;
#pragma unroll
      for (int r = 0; r < kTrCluster; ++r) {
        if (r < CS && o <= target) owner_rank = r;
        o += parts[r];
      }
    }
    const float before = off + before_cta;
    if (tid == 0) { s_owner = 0; s_y = -1; s_first = INT_MAX; s_last = -1; }
    __syncthreads();
    if (rank == owner_rank && before <= target) atomicMax(&s_owner, tid);
    __syncthreads();
    const int owner = s_owner;
    if (rank == owner_rank && (tid >> 5) == (owner >> 5)) {
      // the owner's warp rescans the owner's chunk: lane l takes per
      // consecutive tokens, a warp scan of their weights (from the owner's
      // running sum) finds the lane holding the first y with C(y) > v Z
      const int lane = tid & 31;
      const int olo = min(s_hi, s_lo + owner * P.chunk), ohi = min(s_hi, olo + P.chunk);
      const int per = (P.chunk + 31) / 32;
      const int a0 = min(ohi, olo + lane * per), a1 = min(ohi, a0 + per);
      float part = 0.f;
      for (int i = a0; i < a1; ++i) part += w_of(ld_f32(prow, i), coef != 0.f ? ld_f32(qrow, i) : 0.f);
      float incl = part;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float t = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += t;
      }
      const float obefore = __shfl_sync(0xffffffffu, before, owner & 31);
      const float start = obefore + incl - part;
      const bool here = a0 < a1 && start + part > target && start <= target;
      const unsigned hit = __ballot_sync(0xffffffffu, here);
      if (hit && lane == __ffs(hit) - 1) {
        float cum = start;
        for (int i = a0; i < a1; ++i) {
          cum += w_of(ld_f32(prow, i), coef != 0.f ? ld_f32(qrow, i) : 0.f);
          if (cum > target) { s_y = i; break; }
        }
      }
    }
    // rounding can leave v Z past the owner's chunk: then the next token with
    // weight, or the last one with weight when there is none after it
    if (rank > owner_rank || (rank == owner_rank && tid > owner)) atomicMin(&s_first, first_pos);
    atomicMax(&s_last, last_pos);
    __syncthreads();
    cluster_sync();
    if (rank == 0 && tid == 0) {
      int y = -1, first = INT_MAX, last = -1;
      for (int r = 0; r < CS; ++r) {
        if (r == owner_rank) y = ld_dsmem_s32(mapa(&s_y, r));
        first = min(first, ld_dsmem_s32(mapa(&s_first, r)));
        last = max(last, ld_dsmem_s32(mapa(&s_last, r)));
      }
      out[depth] = y >= 0 ? y : (first != INT_MAX ? first : last);
      P.num_acc[b] = depth;
    }
    cluster_sync();   // the first CTA has read every CTA's results
    return;
  }
}

}  // namespace
}  // namespace sv

extern "C" size_t spec_verify_sample_tree_workspace_size(int B, int n) {
  if (B < 0 || n < 1) return 0;
  return sv::align_up((size_t)B * 2 * n * sizeof(float4), 256);
}

extern "C" sv_status spec_verify_sample_tree(const void *target_logits, sv_dtype logit_dtype, const void *draft,
                                             sv_dtype draft_dtype, int draft_is_probs,
                                             const int32_t *tree_parent, const int32_t *tree_tokens,
                                             const float *uniforms, int B, int n, int V, float temperature,
                                             const sv_typical_acceptance *typical, int32_t *out_tokens,
                                             int32_t *num_accepted, int32_t *path_nodes, void *workspace,
                                             size_t workspace_bytes, int32_t *dev_status, sv_stream_t stream) {
  using namespace sv;
  if (B < 0 || n < 1 || V < 1)
    return fail(SV_ERR_INVALID_ARG, "spec_verify_sample_tree: bad sizes B=%d n=%d V=%d", B, n, V);
  if (n > kTrMaxNodes) return fail(SV_ERR_UNSUPPORTED, "spec_verify_sample_tree: at most 64 tree nodes");
  if (V > (1 << 28)) return fail(SV_ERR_UNSUPPORTED, "spec_verify_sample_tree: V above 2^28");
  if (!(temperature > 0.f) || !std::isfinite(temperature))
    return fail(SV_ERR_INVALID_ARG, "spec_verify_sample_tree: temperature must be finite and > 0");
  if (!target_logits || !tree_parent || !tree_tokens || !uniforms || !out_tokens || !num_accepted || !path_nodes ||
      (n > 1 && !draft && !typical))
    return fail(SV_ERR_INVALID_ARG, "spec_verify_sample_tree: null pointer argument");
  if (logit_dtype != SV_F32 && logit_dtype != SV_BF16 && logit_dtype != SV_F16)
    return fail(SV_ERR_UNSUPPORTED, "spec_verify_sample_tree: logits must be f32, bf16 or f16");
  if (n > 1 && draft) {
    if (draft_is_probs && draft_dtype != SV_F32)
      return fail(SV_ERR_UNSUPPORTED, "spec_verify_sample_tree: draft probabilities must be f32");
    if (!draft_is_probs && draft_dtype != logit_dtype)
      return fail(SV_ERR_UNSUPPORTED, "spec_verify_sample_tree: draft logits must have the target's dtype");
  }
  if (typical && !(typical->epsilon > 0.f && typical->delta > 0.f && std::isfinite(typical->epsilon) &&
                   std::isfinite(typical->delta)))
    return fail(SV_ERR_INVALID_ARG, "spec_verify_sample_tree: typical acceptance needs epsilon, delta > 0");
  const size_t need = align_up((size_t)B * 2 * n * sizeof(float4), 256);
  if (!workspace || workspace_bytes < need)
    return fail(SV_ERR_WORKSPACE, "spec_verify_sample_tree: workspace needs %zu bytes", need);
  if (!aligned(workspace, 256)) return fail(SV_ERR_WORKSPACE, "spec_verify_sample_tree: workspace not 256-byte aligned");
  if (B == 0) return ok();
  TreeParams P = {};
  P.stats = static_cast<float4 *>(workspace);
  P.typical = typical != nullptr;
  P.tau_eps = typical ? typical->epsilon : 0.f;
  P.tau_delta = typical ? typical->delta : 0.f;
  P.target = target_logits; P.draft = draft ? draft : target_logits;
  P.parent = tree_parent; P.tokens = tree_tokens; P.uniforms = uniforms;
  P.out_tokens = out_tokens; P.num_acc = num_accepted; P.path = path_nodes; P.status = dev_status;
  P.B = B; P.n = n; P.V = V;
  P.slice = ((V + kTrCluster - 1) / kTrCluster + 7) / 8 * 8;
  P.chunk = ((P.slice + kTrThreads - 1) / kTrThreads + 7) / 8 * 8;
  const int es_t = dtype_bytes(logit_dtype), es_d = draft_is_probs ? 4 : es_t;
  P.vec_t = aligned(target_logits, 16) && ((size_t)V * es_t) % 16 == 0;
  P.vec_d = aligned(P.draft, 16) && ((size_t)V * es_d) % 16 == 0;
  P.c = (float)(1.4426950408889634074 / (double)temperature);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  const bool probs = draft_is_probs && n > 1 && draft;
  const dim3 sgrid(2 * n, B);
  switch (logit_dtype) {
    case SV_F32:
      e = probs ? launch_k(tree_row_stats_kernel<float, 1>, sgrid, dim3(kTsThreads), 0, s, 1, P)
                : launch_k(tree_row_stats_kernel<float, 0>, sgrid, dim3(kTsThreads), 0, s, 1, P);
      break;
    case SV_BF16:
      e = probs ? launch_k(tree_row_stats_kernel<__nv_bfloat16, 1>, sgrid, dim3(kTsThreads), 0, s, 1, P)
                : launch_k(tree_row_stats_kernel<__nv_bfloat16, 0>, sgrid, dim3(kTsThreads), 0, s, 1, P);
      break;
    default:
      e = probs ? launch_k(tree_row_stats_kernel<__half, 1>, sgrid, dim3(kTsThreads), 0, s, 1, P)
                : launch_k(tree_row_stats_kernel<__half, 0>, sgrid, dim3(kTsThreads), 0, s, 1, P);
      break;
  }
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_sample_tree statistics launch: %s", cudaGetErrorString(e));
  switch (logit_dtype) {
    case SV_F32:
      e = probs ? launch_k(sample_tree_kernel<float, 1>, dim3(kTrCluster, B), dim3(kTrThreads), 0, s, kTrCluster, P)
                : launch_k(sample_tree_kernel<float, 0>, dim3(kTrCluster, B), dim3(kTrThreads), 0, s, kTrCluster, P);
      break;
    case SV_BF16:
      e = probs ? launch_k(sample_tree_kernel<__nv_bfloat16, 1>, dim3(kTrCluster, B), dim3(kTrThreads), 0, s, kTrCluster, P)
                : launch_k(sample_tree_kernel<__nv_bfloat16, 0>, dim3(kTrCluster, B), dim3(kTrThreads), 0, s, kTrCluster, P);
      break;
    default:
      e = probs ? launch_k(sample_tree_kernel<__half, 1>, dim3(kTrCluster, B), dim3(kTrThreads), 0, s, kTrCluster, P)
                : launch_k(sample_tree_kernel<__half, 0>, dim3(kTrCluster, B), dim3(kTrThreads), 0, s, kTrCluster, P);
      break;
  }
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_sample_tree launch: %s", cudaGetErrorString(e));
  return ok();
}

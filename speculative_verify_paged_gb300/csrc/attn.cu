// spec_verify_attn: paged GQA attention of the K+1 verify queries.
//
// What is computed ("KV Cache + Speculative Decoding" sections 5.2-5.3 and
// 6.3): for sequence b, kv head g and query row r = j*G + hh (query position
// j, head h = g*G + hh), out = softmax_t(scale * q . K_t) V_t over keys
// t <= L_b - n_new + j, K_t / V_t read through the block table.
//
// Design (flash-decoding style split-KV, CS336 lecture 10 section 9.2):
//   * work items are pieces of (sequence, kv head) pairs. By default
//     attn_order_kernel sorts splits of a fixed size longest first and each
//     CTA of attn_tc5_kernel takes one. On request (blocks_per_split = 0),
//     attn_part_kernel cuts the tiles of all sequences into equal ranges, one
//     per CTA slot and kv head, and each CTA of attn_tc5_bal_kernel walks its
//     range through one or more pairs, so every CTA streams the same number
//     of tiles whatever the lengths;
//   * attn_tc5_kernel on the fifth-generation tensor
//     cores: all (K+1)*G query rows of the GQA group share one M = 128 MMA
//     tile, so every K/V byte is read from HBM once per step; two producer
//     warps stream (block, head) K and V tiles with 4-D TMA tensor copies
//     (128-byte swizzle) through shared-memory rings guarded by mbarriers;
//     one thread issues tcgen05.mma with S, P and O in tensor memory; a
//     softmax warpgroup runs the online softmax in the log2 domain with a
//     lazy rescale, masking only the tiles that reach the diagonal or the
//     end of the split. bf16 caches feed the MMAs directly; fp8 e4m3 tiles
//     are widened exactly to f16 by two converter warps, with k_scale folded
//     into the score scale and v_scale into the output;
//   * a piece that does not cover its whole pair writes an unnormalised
//     partial (acc, m, l) and the merge kernels combine them with the
//     log-sum-exp rule
//     m = max m_s, l = sum l_s 2^(m_s - m), O = sum acc_s 2^(m_s - m) / l.
// A plain CUDA-core kernel covers fp32 caches and shapes outside the
// tensor-core path (any d_head <= 256, any block size).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <type_traits>

#include "sv_common.cuh"

namespace sv {
namespace {

// ------------------------------------------------------------ constants ---
constexpr int kD = 128;           // head dim of the tensor-core path
constexpr int kBS = 16;           // block size of the tensor-core path
constexpr int kGenThreads = 128;
constexpr int kGenKeys = 32;

// ------------------------------------------------------ PTX: tensor core ---
template <bool F16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (F16) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
  }
}

// maximum of a tile's N scores per row as a tree of depth log2 N (a chain
// of N - 1 dependent maxima otherwise sits on every tile's critical path)
template <int N>
__device__ __forceinline__ float t5_tile_max(const float (&x)[N]) {
  static_assert(N >= 2 && (N & (N - 1)) == 0, "power of two");
  float m[N / 2];
#pragma unroll
  for (int k = 0; k < N / 2; ++k) m[k] = fmaxf(x[k], x[k + N / 2]);
#pragma unroll
  for (int w = N / 4; w >= 1; w >>= 1)
#pragma unroll
    for (int k = 0; k < w; ++k) m[k] = fmaxf(m[k], m[k + w]);
  return m[0];
}

// 2^x on the SFU (results below 2^-126 flush to zero)
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// two fp32 values -> two e4m3 codes (x0 in the low byte), rounded to
// nearest even, saturating at +-448
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float x0, float x1) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(x1), "f"(x0));
  return r;
}

// two e4m3 codes (low byte first) -> f16x2
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t out;
  asm volatile("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(out) : "h"(v));
  return out;
}

// 4-D TMA tile copy into shared memory, completion on `bar`.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            int c3, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}


// ------------------------------------------------- tensor-core kernel -----
struct TcParams {   // 64-byte aligned through its CUtensorMap members
  CUtensorMap tmk;
  CUtensorMap tmv;
  const void *q;
  void *out;       // [B][n_new][H_q][kD] bf16, written directly when a sequence has one split
  const float *k_scale;
  const float *v_scale;
  const int32_t *block_table;
  const int32_t *seq_lens;
  float *ws_acc;   // [B][H_kv][S][R][kD]
  float *ws_ml;    // [B][H_kv][S][R][2]
  const int32_t *order;   // split mode: work items s + S (g + H_kv b), longest first (NULL: blockIdx.x)
  const int4 *work;       // balanced mode: per CTA (b, g, first tile, tiles) of its tile range
  int32_t *seq_pre_w;     // balanced mode: first tile of each sequence (written by the partition)
  int4 *split_w;          // balanced mode: (count, T), then the sequences split across CTAs
  int balanced;           // 1: CTA c takes tiles [c T / C, (c + 1) T / C) of all (b, g) pairs
  int ncta;               // balanced mode: C
  const uint64_t *anc;    // [B][n_new] ancestor masks of a draft tree (NULL: a chain)
  int32_t *status;
  int B, n_new, H_q, H_kv, G, R, max_blocks, num_blocks, bps, S;
  int tblk;           // paged blocks per tile of the kernel launched (balanced work counts)
  int role[3];        // tensor-map dims 1..3 hold (0 = slot, 1 = kv head, 2 = block)
  float scale_log2;   // softmax_scale * log2(e)
  uint64_t wait_ns;   // limit of each wait on another warp's signal
  unsigned withhold;  // test hook: SV_TEST_WITHHOLD_COPIES issues no K/V copies
};

// TMA coordinates {d, dim1, dim2, dim3} of tile (kv head g, physical block)
__device__ __forceinline__ void tile_coords(const TcParams &P, int g, int phys, int (&c)[3]) {
#pragma unroll
  for (int k = 0; k < 3; ++k) c[k] = P.role[k] == 0 ? 0 : (P.role[k] == 1 ? g : phys);
}

// ------------------------------------------- tcgen05 tensor-core kernel ---
// The same attention on the fifth-generation tensor cores: accumulators live
// in tensor memory (TMEM), one thread issues the MMAs, and the softmax warps
// read S and write P through TMEM, so no warp holds an accumulator in
// registers.
//
// CTA = its work items in order (one split, or a balanced range), 256
// threads (288 for fp8 caches):
//   warps 0-3  softmax warpgroup; thread w*32+l owns query row w*32+l
//              (TMEM lane w*32+l: warp w may only touch lanes 32w..32w+31)
//              and first writes that row of Q into shared memory (fp8
//              caches with at most 64 rows: warps 0-1; warps 2-3 widen V)
//   warps 4, 5 TMA producers (one lane each, in separate warps so that neither
//              waits behind the other's barrier): warp 4 streams K tiles,
//              warp 5 V stages, each into its own shared-memory ring (a K
//              stage is free again as soon as its Q K^T has run, a V stage
//              after its P V)
//   warp 6     TMEM owner; lane 0 issues the MMAs from a polling loop, so
//              Q K^T runs ahead whenever K data and an S buffer are ready.
//              It sits on the third scheduler (warp id % 4 = 2), away from
//              the softmax warps that own rows 0-63.
//   warp 7     idle (fp8 caches: it and warp 8 widen V stages to f16)
// A tile is Cfg::kBlk paged blocks (N = 16 kBlk keys). Per tile t, with
// buffer u = t % kT5SBuf:
//   S[u] = Q K^T           (M=128 padded query rows, N keys, K=128)
//   P[u] = 2^(S c - m)      bf16, written over the first N/2 columns of S[u]
//   O   += P V              (M=128, N=128 head dims, K=16 keys per MMA)
// Each buffer has its own "P V done" barrier, so every wait is at most one
// phase behind its barrier.
// Shared-memory operands use the 128-byte swizzle: Q and K are K-major (head
// dim contiguous), V is MN-major (head dim contiguous along N).
constexpr int kT5Blk = 2;                      // blocks of a 32-key unit (V stages, the order's work counts)
constexpr int kT5SBuf = 2;                     // S / P buffers in TMEM
constexpr int kT5MmaWarp = 6;
constexpr int kT5MaxR = 128;
// Tiles of 64 keys. The tile loop's rate is set by the number of Q K^T
// MMAs per key (an MMA of N = 64 keys costs about what one of N = 32 does),
// so a tile takes 64 keys; two 64-column S buffers and O then fill the CTA's
// 256 TMEM columns and Q is the shared-memory A operand (QR rows: for QR = 64
// the MMA's rows 64-127 read the shared memory after Q, and their rows of S,
// P and O are never used). K stages hold a tile, V streams in 32-key stages,
// two per tile.
// FP8: e4m3 caches. TMA lands the raw 16 x 128-byte tile of each block in
// rings of their own. Q K^T reads the raw K tiles directly (kind::f8f6f4):
// each query row, scaled by a power of two, is split into two e4m3 terms
// (hi + lo, about the precision of its bf16 values), and the two partial
// products accumulate in the S buffer. V is widened exactly to f16 (every
// e4m3 value is an f16 value) by converter warps into a second ring laid
// out as the 16-bit stages are, and P V runs on f16 operands. Four warps
// widen V when the group has at most 64 query rows (softmax warps 2 and 3
// hold no rows then), else two.
// The rings take what two CTAs per SM leave.
template <int QR, bool FP8> struct T5Cfg {
  static constexpr int kBlk = 4;                             // paged blocks per tile
  static constexpr int kN = 16 * kBlk;                       // keys per tile
  static constexpr int kVPT = kBlk / kT5Blk;                 // 32-key V stages per tile
  static constexpr int kQBytes = QR * 256;                   // bf16: two head-dim halves; fp8: hi and lo terms
  static constexpr int kKHalf = kBlk * 2048;                 // a head-dim half of a 16-bit K tile
  static constexpr int kKTile = 2 * kKHalf;
  static constexpr int kVHalf = kT5Blk * 2048;               // a head-dim half of a 16-bit V stage
  static constexpr int kVTile = 2 * kVHalf;
  static constexpr int kKS = 3;                              // K stages (raw for FP8)
  static constexpr int kVS = FP8 ? 4 : (QR == 64 ? 5 : 3);   // V stages (raw for FP8)
  static constexpr int kCVS = FP8 ? (QR == 64 ? 6 : 4) : 0;  // widened V stages
  static constexpr int kConvW = FP8 ? (QR == 64 ? 4 : 2) : 0;   // V converter warps
  static constexpr int kSoftW = FP8 && QR == 64 ? 2 : 4;     // warps in the softmax role
  static constexpr int kKRaw = FP8 ? kBlk * 2048 : kKTile;   // bytes of a K ring stage
  static constexpr int kVRaw = FP8 ? kT5Blk * 2048 : kVTile; // bytes of a V ring stage
  static constexpr int kThreads = FP8 ? 288 : 256;
  static constexpr int kSmem = 1024 + kQBytes + kKS * kKRaw + kVS * kVRaw + kCVS * kVTile;
  static constexpr uint32_t kOCol = kT5SBuf * kN;             // O after the S buffers
  static_assert(kOCol + 128 <= 256, "TMEM budget");
  static_assert(kVPT == 2, "V stages per tile");
  static_assert(kSmem <= 1024 + 106496, "two CTAs per SM");
};
constexpr uint32_t kT5Cols = 256;              // TMEM columns: S/P buffers, O

__device__ __forceinline__ uint64_t t5_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;   // descriptor version of the sm_100 family
  d |= (uint64_t)2 << 61;   // 128-byte swizzle
  return d;
}

__device__ __forceinline__ void t5_mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
               "r"(a), "l"(b), "r"(idesc), "r"(acc));
}

// A from shared memory (descriptor)
__device__ __forceinline__ void t5_mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
               "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

// kind::f8f6f4 (e4m3 A and B, 32 elements of K per MMA), A from shared memory
__device__ __forceinline__ void t5_mma_ss_f8(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
               "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void t5_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void t5_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void t5_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void t5_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void t5_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void t5_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void t5_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Non-blocking probe of a barrier phase.
__device__ __forceinline__ bool t5_test(uint64_t *bar, uint32_t phase) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(phase)
      : "memory");
  return done != 0;
}

// Bounded wait (limit_ns) that gives up at once after any earlier wait of the
// CTA gave up.
__device__ __forceinline__ bool t5_wait(uint64_t *bar, uint32_t phase, volatile int *abort_flag, uint64_t limit_ns) {
  if (*abort_flag) return false;
  if (mbar_wait(bar, phase, limit_ns)) return true;
  *abort_flag = 1;
  return false;
}

// The work items of a CTA of the balanced-mode kernel: blocks [blk0, blk1)
// of kv head g of sequence b. The sequence of tiles (P.tblk blocks each) of
// all sequences in order is cut into NR equal ranges, and CTA c runs range c / H_kv for kv
// head c % H_kv, so every CTA streams the same number of tiles; a range may
// end inside one sequence and go on through whole sequences into the next. A
// piece of a (b, g) pair that another CTA shares writes a partial: entry 2c
// for the CTA's first item, 2c + 1 for its last. Every role of the CTA walks
// the same items in the same order.
struct T5Item {
  int b, g, blk0, blk1, L, nblk;
  int64_t ent;   // partial entry
  bool whole;    // the item covers all of (b, g): written directly
};
struct T5Walk {
  int b, g, off, left, idx;
};

__device__ __forceinline__ bool t5_item(const TcParams &P, T5Walk &w, T5Item &it) {
  if (w.idx == 0) {
    const int4 wk = P.work[blockIdx.x / P.H_kv];   // written by the partition kernel
    w.b = wk.x; w.g = (int)(blockIdx.x % P.H_kv); w.off = wk.z; w.left = wk.w;
  }
  if (w.left <= 0) return false;
  int L = 0, nt = 0;
  for (;;) {   // sequences with invalid lengths hold no tiles
    if (w.b >= P.B) return false;
    L = P.seq_lens[w.b];
    nt = (L >= P.n_new && L <= P.max_blocks * kBS) ? ((L + kBS - 1) / kBS + P.tblk - 1) / P.tblk : 0;
    if (nt > 0) break;
    ++w.b;
  }
  const int take = min(nt - w.off, w.left);
  it.b = w.b; it.g = w.g; it.L = L;
  it.nblk = (L + kBS - 1) / kBS;
  it.blk0 = w.off * P.tblk;
  it.blk1 = min(it.nblk, (w.off + take) * P.tblk);
  it.whole = w.off == 0 && take == nt;
  it.ent = 2 * (int64_t)blockIdx.x + (w.idx > 0 ? 1 : 0);
  w.left -= take;
  w.off = 0;
  ++w.b;   // the range goes on with the next sequence, same kv head
  ++w.idx;
  return true;
}

// Longest-first order of the tcgen05 kernel's work items. A work item is
// split s of kv head g of sequence b; its work is its number of 32-key
// tiles. One CTA counting-sorts the (s, b) pairs by descending work (kv heads
// innermost; empty splits, and sequences with invalid lengths, last). The
// order within a bucket is that of the atomics: each item is still computed
// once, and its result does not depend on when.
// It reads only seq_lens and writes only its own part of the workspace, so
// it runs while the previous kernel of the stream is still running (that
// kernel passed its own wait, so everything before it has completed; the
// library's kernels never write seq_lens; an attention kernel of the
// previous call lets the next kernel start only once each of its CTAs has
// read its item from this order). It waits for that kernel at its end, so
// the attention kernel's wait on this one still covers, for example, the
// K/V rows the append kernel writes.
constexpr int kOrdThreads = 1024;
constexpr int kOrdMaxTiles = 1023;   // buckets 0..kOrdMaxTiles
constexpr int kOrdPairs = 4;         // (s, b) pairs a thread keeps in registers
__global__ void __launch_bounds__(kOrdThreads) attn_order_kernel(const int32_t *seq_lens, int B, int S, int H_kv,
                                                                 int bps, int n_new, int max_blocks, int32_t *order) {
  pdl_trigger();
  __shared__ int cur[kOrdMaxTiles + 1];
  const int tid = threadIdx.x, lane = tid & 31;
  const int T = min(kOrdMaxTiles, (bps + kT5Blk - 1) / kT5Blk);
  const int npairs = S * B;
  auto work = [&](int p) {
    const int sp = p % S, bp = p / S;
    const int L = seq_lens[bp];
    if (L < n_new || L > max_blocks * kBS) return 0;
    const int blk = min(bps, (L + kBS - 1) / kBS - sp * bps);
    return blk > 0 ? min(T, (blk + kT5Blk - 1) / kT5Blk) : 0;
  };
  for (int w = tid; w <= T; w += kOrdThreads) cur[w] = 0;
  // the first kOrdPairs pairs of this thread keep their work in registers
  int wk[kOrdPairs];
#pragma unroll
  for (int k = 0; k < kOrdPairs; ++k) {
    const int p = tid + k * kOrdThreads;
    wk[k] = p < npairs ? work(p) : 0;
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kOrdPairs; ++k)
    if (tid + k * kOrdThreads < npairs) atomicAdd(&cur[wk[k]], 1);
  for (int p = tid + kOrdPairs * kOrdThreads; p < npairs; p += kOrdThreads) atomicAdd(&cur[work(p)], 1);
  __syncthreads();
  if (tid < 32) {
    // bucket starts, the most work first: lane l takes buckets
    // [T - (l+1) per + 1, T - l per] in descending order
    const int per = (T + 1 + 31) / 32;
    const int hi = T - lane * per, lo = max(0, hi - per + 1);
    int sum = 0;
    for (int w = hi; w >= lo; --w) sum += cur[w];
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    int acc = incl - sum;
    for (int w = hi; w >= lo; --w) {
      const int c = cur[w];
      cur[w] = acc;
      acc += c;
    }
  }
  __syncthreads();
  auto place = [&](int p, int w) {
    const int pos = atomicAdd(&cur[w], 1);
    const int sp = p % S, bp = p / S;
    for (int gg = 0; gg < H_kv; ++gg) order[(int64_t)pos * H_kv + gg] = sp + S * (gg + H_kv * bp);
  };
#pragma unroll
  for (int k = 0; k < kOrdPairs; ++k)
    if (tid + k * kOrdThreads < npairs) place(tid + k * kOrdThreads, wk[k]);
  for (int p = tid + kOrdPairs * kOrdThreads; p < npairs; p += kOrdThreads) place(p, work(p));
  pdl_wait();
}

// Balanced partition for the tcgen05 kernel: one CTA. The global tile
// sequence holds, for every sequence b in order, the ceil(ceil(L_b / 16) /
// tblk) tiles of b (tblk blocks each, the tile of the kernel launched after
// it; none for an invalid length, which it flags). It is cut
// into NR equal ranges, range r = [r T / NR, (r + 1) T / NR), and CTAs
// r H_kv .. r H_kv + H_kv - 1 run range r for kv heads 0 .. H_kv - 1: the
// CTAs reading the heads of one block run side by side, as the heads of a
// block sit next to each other in the pool. work[r] = (b, 0, first tile
// within b, tile count); seq_pre[b] is the first tile of sequence b
// (seq_pre[B] = T), from which the merge finds a pair's pieces. Like the
// order kernel it overlaps the previous kernel of the stream and waits for it
// only before its first global write (the previous kernel may be a merge
// that still reads this workspace).
constexpr int kPartThreads = 1024;
constexpr int kPartSmemB = 4096;   // prefixes kept in shared memory up to this batch
__global__ void __launch_bounds__(kPartThreads) attn_part_kernel(const int32_t *seq_lens, int B, int n_new,
                                                                 int max_blocks, int tblk, int NR, int4 *work,
                                                                 int32_t *seq_pre, int4 *split, int32_t *status) {
  pdl_trigger();
  __shared__ int s_pre[kPartSmemB + 1];
  __shared__ int s_warp[kPartThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const bool big = B > kPartSmemB;
  if (big) pdl_wait();
  int carry = 0;
  for (int base = 0; base < B; base += kPartThreads) {
    const int b = base + tid;
    int v = 0;
    if (b < B) {
      const int L = seq_lens[b];
      if (L >= n_new && L <= max_blocks * kBS) v = ((L + kBS - 1) / kBS + tblk - 1) / tblk;
      else atomic_or_status(status, SV_DEV_BAD_SEQ_LEN);
    }
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int before = 0, tot = 0;
    for (int w = 0; w < kPartThreads / 32; ++w) {
      const int x = s_warp[w];
      before += w < warp ? x : 0;
      tot += x;
    }
    if (b < B) {
      const int ex = carry + before + incl - v;
      if (big) seq_pre[b] = ex;
      else s_pre[b] = ex;
    }
    carry += tot;
    __syncthreads();
  }
  const int T = carry;
  if (!big) {
    pdl_wait();
    for (int b = tid; b < B; b += kPartThreads) seq_pre[b] = s_pre[b];
    if (tid == 0) s_pre[B] = T;
  }
  if (tid == 0) seq_pre[B] = T;
  __syncthreads();
  const int32_t *pre = big ? seq_pre : s_pre;
  for (int r = tid; r < NR; r += kPartThreads) {
    const int t0 = (int)((int64_t)r * T / NR), t1 = (int)((int64_t)(r + 1) * T / NR);
    int4 wk = make_int4(0, 0, 0, 0);
    if (t1 > t0) {
      // the last sequence whose first tile is at or before t0 holds it
      int lo = 0, hi = B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= t0) lo = mid;
        else hi = mid - 1;
      }
      wk = make_int4(lo, 0, t0 - pre[lo], t1 - t0);
    }
    work[r] = wk;
  }
  // the sequences that more than one range holds (each meets a range
  // boundary, so there are at most NR - 1): split[1..n] = (b, first tile A,
  // tiles nt, first range r0), split[0] = (n, T)
  __shared__ int s_n;
  if (tid == 0) s_n = 0;
  __syncthreads();
  if (T > 0) {
    for (int b = tid; b < B; b += kPartThreads) {
      const int64_t A = pre[b], nt = pre[b + 1] - pre[b];
      const int64_t r0 = ((A + 1) * NR - 1) / T;
      if (nt > 0 && ((A + nt) * NR - 1) / T > r0)
        split[1 + atomicAdd(&s_n, 1)] = make_int4(b, (int)A, (int)nt, (int)r0);
    }
  }
  __syncthreads();
  if (tid == 0) split[0] = make_int4(s_n, T, 0, 0);
}

// One query row into shared memory as the K-major, 128-byte-swizzled A
// operand of Q K^T; a row past R (src null) is zeros.
// bf16: two head-dim halves of QR rows of 128 bytes, the 16-byte chunks of
// row r at chunk index ^ (r % 8).
// FP8: the row times 2^s, s chosen so that its largest |q| lies in
// [2^7, 2^8) (inside e4m3's range), as two e4m3 terms: hi = e4m3(y) and
// lo = e4m3(y - hi), each QR rows of 128 bytes (all 128 head dims), so that
// hi + lo carries the 8 significant bits of a bf16 value exactly for
// |y| >= 2^-2, i.e. down to 2^-9 of the row's largest element (smaller ones
// lose bits in e4m3's subnormals, an error below 2^-17 of the largest). k_scale 2^-s folds into the
// row's score scale, which is returned. Two passes over the row (the second
// from L1).
template <int QR, bool FP8>
__device__ __forceinline__ float t5_store_q(uint32_t q_smem, int row, const uint4 *src, float k_scale) {
  if constexpr (FP8) {
    float amax = 0.f;
    if (src) {
#pragma unroll 4
      for (int k = 0; k < 16; ++k) {
        const uint4 v = __ldg(src + k);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
          amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(w[e] << 16)), fabsf(__uint_as_float(w[e] & 0xffff0000u))));
      }
    }
    const int ex = amax > 0.f ? max(-100, (int)((__float_as_uint(amax) >> 23) & 0xff) - 127) : 0;
    const float up = __uint_as_float((uint32_t)(127 + 7 - ex) << 23);   // 2^s, s = 7 - ex
    const float fold = k_scale * __uint_as_float((uint32_t)(127 - 7 + ex) << 23);
#pragma unroll 2
    for (int j = 0; j < 8; ++j) {   // 16 head dims: one 16-byte chunk of each term
      const uint4 v0 = src ? __ldg(src + 2 * j) : make_uint4(0u, 0u, 0u, 0u);
      const uint4 v1 = src ? __ldg(src + 2 * j + 1) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
      uint32_t hi[4], lo[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        uint32_t hp[2], lp[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const uint32_t ww = w[2 * e + h];
          const float y0 = __uint_as_float(ww << 16) * up, y1 = __uint_as_float(ww & 0xffff0000u) * up;
          const uint32_t c = f32x2_to_e4m3x2(y0, y1);
          const uint32_t f = e4m3x2_to_f16x2((uint16_t)c);
          const float2 hv = __half22float2(*reinterpret_cast<const __half2 *>(&f));
          hp[h] = c;
          lp[h] = f32x2_to_e4m3x2(y0 - hv.x, y1 - hv.y);
        }
        hi[e] = hp[0] | (hp[1] << 16);
        lo[e] = lp[0] | (lp[1] << 16);
      }
      const uint32_t off = row * 128 + ((j ^ (row & 7)) << 4);
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(q_smem + off), "r"(hi[0]), "r"(hi[1]), "r"(hi[2]),
                   "r"(hi[3])
                   : "memory");
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(q_smem + QR * 128 + off), "r"(lo[0]), "r"(lo[1]),
                   "r"(lo[2]), "r"(lo[3])
                   : "memory");
    }
    // the tensor cores read it through the async proxy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    return fold;
  } else {
#pragma unroll
    for (int c = 0; c < 16; ++c) {
      const uint4 v = src ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
      const uint32_t qa = q_smem + (c >> 3) * (QR * 128) + row * 128 + (((c & 7) ^ (row & 7)) << 4);
      asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(qa), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
    }
    // the tensor cores read it through the async proxy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    return 1.f;
  }
}

template <int QR, bool FP8>
__global__ void __launch_bounds__(T5Cfg<QR, FP8>::kThreads, 2) attn_tc5_kernel(const __grid_constant__ TcParams P) {
  using Cfg = T5Cfg<QR, FP8>;
  constexpr int KS = Cfg::kKS, VS = Cfg::kVS;
  constexpr int CVS = Cfg::kCVS > 0 ? Cfg::kCVS : 1;
  constexpr int SW = Cfg::kSoftW, CW = Cfg::kConvW;
  constexpr int TB = Cfg::kBlk, TN = Cfg::kN, VPT = Cfg::kVPT;
  constexpr uint32_t OC = Cfg::kOCol;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t k_full[KS], k_empty[KS], v_full[VS], v_empty[VS];
  // FP8: widened V stages, filled by the converter warps, freed by the MMAs
  __shared__ __align__(8) uint64_t vc_full[CVS], vc_empty[CVS];
  __shared__ __align__(8) uint64_t s_full[kT5SBuf], p_full[kT5SBuf], o_done[kT5SBuf], mma_drain, q_full;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    // K stages are freed by the MMAs; raw V stages by the MMAs (bf16) or by
    // the CW converter warps (FP8), whose widened stages the MMAs free
    for (int k = 0; k < KS; ++k) {
      mbar_init(&k_full[k], 1);
      mbar_init(&k_empty[k], 1);
    }
    for (int k = 0; k < VS; ++k) {
      mbar_init(&v_full[k], 1);
      mbar_init(&v_empty[k], FP8 ? CW : 1);
    }
    if (FP8) {
      for (int k = 0; k < CVS; ++k) {
        mbar_init(&vc_full[k], CW);
        mbar_init(&vc_empty[k], 1);
      }
    }
    for (int k = 0; k < kT5SBuf; ++k) {
      mbar_init(&s_full[k], 1);
      mbar_init(&p_full[k], SW);
      mbar_init(&o_done[k], 1);
    }
    mbar_init(&mma_drain, 1);
    mbar_init(&q_full, SW);   // the softmax warps wrote their Q rows
    abort_flag = 0;
    fence_mbarrier_init();
  }
  // (the barriers live in shared memory: set up while the previous kernel
  // of the stream finishes)
  pdl_wait();
  // the work item: split s of kv head g of sequence b, in the longest-first
  // order the order kernel wrote (the CTAs launched first take the longest
  // splits, so the last wave is made of the shortest ones), or with no
  // order (a grid that fits the CTA slots at once) item = blockIdx.x
  // (a plain load: the order kernel may still have been writing the order
  // when this CTA started, so it is not read-only data for this kernel)
  const int item = P.order ? P.order[blockIdx.x] : (int)blockIdx.x;
  // the next kernel of the stream may start (and the next call's order
  // kernel overwrite the order) only once every CTA has read its item
  pdl_trigger();
  if (item < 0 || item >= (int)gridDim.x) {
    if (threadIdx.x == 0) atomic_or_status(P.status, SV_DEV_BAD_WORK);
    return;
  }
  const int s = item % P.S, g = (item / P.S) % P.H_kv, b = item / (P.S * P.H_kv);
  // the producers read the split's first 64 block-table entries alongside
  // the sequence length (the row is max_blocks entries long; entries past
  // the sequence are read but never used)
  int tab_cur = 0, tab_nxt = 0;
  if (warp == 4 || warp == 5) {
    const int avail = P.max_blocks - s * P.bps;
    const int32_t *row0 = P.block_table + (int64_t)b * P.max_blocks + (int64_t)s * P.bps;
    tab_cur = lane < avail ? __ldg(row0 + lane) : 0;
    tab_nxt = 32 + lane < avail ? __ldg(row0 + 32 + lane) : 0;
  }
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t q_smem = smem_u32(smem);   // Q, the A operand of Q K^T
  const uint32_t k_ring = q_smem + Cfg::kQBytes;
  const uint32_t v_ring = k_ring + KS * Cfg::kKRaw;
  // the V ring the MMAs read: the widened one for FP8, else the TMA ring
  const uint32_t vc_ring = FP8 ? v_ring + VS * Cfg::kVRaw : v_ring;

  const int L = P.seq_lens[b];
  if (L < P.n_new || L > P.max_blocks * kBS) {
    if (tid == 0 && g == 0 && s == 0) atomic_or_status(P.status, SV_DEV_BAD_SEQ_LEN);
    return;
  }
  const int nblk = (L + kBS - 1) / kBS;
  const int blk0 = s * P.bps;
  if (blk0 >= nblk) return;   // the merge never reads this split
  const int blk1 = min(nblk, blk0 + P.bps);
  const int nblocks = blk1 - blk0;
  const int n_tiles = (nblocks + TB - 1) / TB;
  const int R = P.R;

  __syncthreads();
  volatile int *abf = &abort_flag;

  if (warp == 4 || warp == 5) {
    // ------------------------------------------------------------ producers --
    // warp 4 streams K tiles, warp 5 V stages (VPT of 32 keys per tile; a
    // stage of a tile that ends before it completes with a plain arrival, so
    // the ring's phases stay one per stage)
    {
      // the whole warp walks the block table 32 entries at a time (the next
      // 32 prefetched); lane 0 waits for free stages and issues the copies
      const bool isv = warp == 5;
      const int NS = isv ? VS : KS;
      const int SB = isv ? kT5Blk : TB;                                // blocks per stage
      const uint32_t sbytes = isv ? Cfg::kVRaw : Cfg::kKRaw;
      const uint32_t half = isv ? Cfg::kVHalf : Cfg::kKHalf;           // 16-bit: second head-dim half
      uint64_t *fullb = isv ? v_full : k_full;
      uint64_t *emptyb = isv ? v_empty : k_empty;
      const uint32_t ring = isv ? v_ring : k_ring;
      const CUtensorMap *map = isv ? &P.tmv : &P.tmk;
      const int32_t *table = P.block_table + (int64_t)b * P.max_blocks + blk0;
      int cur = tab_cur;
      int nxt = tab_nxt;
      int chunk = 0;
      int issued = 0;
      // (test hook: with the copies withheld every wait on them runs out,
      // with nothing in flight)
      const int n_issue = (P.withhold & SV_TEST_WITHHOLD_COPIES) ? 0 : n_tiles * (isv ? VPT : 1);
      for (int i = 0; i < n_issue; ++i) {
        const int first = i * SB;   // stage i holds blocks first .. first + SB - 1
        if ((first >> 5) != chunk) {
          chunk = first >> 5;
          cur = nxt;
          const int rel = (chunk + 1) * 32 + lane;
          nxt = rel < nblocks ? table[rel] : 0;
        }
        int phys[TB];
#pragma unroll
        for (int kk = 0; kk < TB; ++kk) phys[kk] = __shfl_sync(0xffffffffu, cur, (first + kk) & 31);
        const int st = i % NS;
        bool go = true;
        if (lane == 0) {
          if (i >= NS && !t5_wait(&emptyb[st], ((i / NS) & 1) ^ 1, abf, P.wait_ns)) {
            go = false;
          } else {
            const int nvalid = max(0, min(SB, nblocks - first));
            if (nvalid == 0) {
              mbar_arrive(&fullb[st]);   // past the end of the split: nothing to copy
            } else {
              // a block is 2 KB of e4m3 (one 128-byte box row per slot) or two
              // 2 KB head-dim halves of bf16
              mbar_arrive_expect_tx(&fullb[st], (uint32_t)(nvalid * (FP8 ? 2048 : 2 * 2048)));
              const uint32_t base = ring + st * sbytes;
              for (int kk = 0; kk < nvalid; ++kk) {
                int ph = phys[kk];
                if (ph < 0 || ph >= P.num_blocks) {
                  if (!isv) atomic_or_status(P.status, SV_DEV_BAD_BLOCK);
                  ph = 0;   // stay in bounds; the output of this sequence is flagged
                }
                int c[3];
                tile_coords(P, g, ph, c);
                tma_load_4d(base + kk * 2048, map, 0, c[0], c[1], c[2], &fullb[st]);
                if (!FP8) tma_load_4d(base + half + kk * 2048, map, 64, c[0], c[1], c[2], &fullb[st]);
              }
            }
            issued = i + 1;
          }
        }
        if (!__shfl_sync(0xffffffffu, (int)go, 0)) break;
      }
      // the copies in flight land before the CTA may exit
      if (lane == 0) {
        for (int t = max(0, issued - NS); t < issued; ++t)
          if (!mbar_wait(&fullb[t % NS], (t / NS) & 1)) atomic_or_status(P.status, SV_DEV_TIMEOUT);
      }
    }
  } else if (warp < SW || warp == kT5MmaWarp) {
    // the softmax warps store Q (their rows) while the MMA warp allocates TMEM
    float q_fold = 1.f;
    if (warp < SW) {
      const int row = tid;
      const uint4 *src = nullptr;
      if (row < R) {
        const int j = row / P.G, hh = row % P.G;
        src = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(P.q) +
                                              (((int64_t)b * P.n_new + j) * P.H_q + (int64_t)g * P.G + hh) * kD);
      }
      if (row < QR) q_fold = t5_store_q<QR, FP8>(q_smem, row, src, FP8 ? P.k_scale[g] : 1.f);
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_full);
    }
    if (warp == kT5MmaWarp) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                   "r"(kT5Cols));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    t5_fence_before();
    named_bar_sync(1, 32 * (SW + 1));   // TMEM allocated
    t5_fence_after();
    const uint32_t tb = tmem_base;

    if (warp == kT5MmaWarp) {
      // ---------------------------------------------------------- MMA issuer --
      if (lane == 0) {
        // f32 accumulators; A and B bf16 (formats 1), or for FP8 e4m3 in Q K^T
        // (kind::f8f6f4, format 0) and f16 in P V (format 0)
        constexpr uint32_t ab = FP8 ? 0u : (1u << 7) | (1u << 10);
        const uint32_t idesc_qk = (1u << 4) | ab | ((uint32_t)(TN >> 3) << 17) | (8u << 24);
        const uint32_t idesc_pv = (1u << 4) | ab | (1u << 16) | (16u << 17) | (8u << 24);
        static_assert(TN % 16 == 0 && TN <= 256, "MMA N");
        int tq = 0, tp = 0;   // next tiles for Q K^T and for P V
        bool q_ready = false;
        uint64_t t_last = global_ns();
        while (tp < n_tiles) {
          bool progressed = false;
          if (!q_ready) q_ready = t5_test(&q_full, 0);
          if (q_ready && tq < n_tiles && tq - tp < kT5SBuf) {
            // K stage: the TMA ring (raw e4m3 codes for FP8)
            const int KR = KS;
            const int ks = tq % KR, sb = tq % kT5SBuf;
            uint64_t *kf = k_full;
            // S buffer sb is free once the P V of tile tq - kT5SBuf has run
            const bool sfree = tq < kT5SBuf || t5_test(&o_done[sb], ((tq / kT5SBuf) - 1) & 1);
            if (sfree && t5_test(&kf[ks], (tq / KR) & 1)) {
              t5_fence_after();
              const uint32_t kb = k_ring + ks * Cfg::kKRaw;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                // A = Q and B = K from shared memory. bf16: 16 head dims per step over
                // the two head-dim halves; FP8: 32 head dims per step, the hi term of Q
                // (kk < 4) then the lo term, against the raw codes
                const uint64_t ad = t5_desc(q_smem + (kk >> 2) * (QR * 128) + (kk & 3) * 32, 16, 1024);
                if constexpr (FP8)
                  t5_mma_ss_f8(tb + sb * TN, ad, t5_desc(kb + (kk & 3) * 32, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
                else
                  t5_mma_ss(tb + sb * TN, ad, t5_desc(kb + (kk >> 2) * Cfg::kKHalf + (kk & 3) * 32, 16, 1024), idesc_qk,
                            kk > 0 ? 1u : 0u);
              }
              t5_commit(&s_full[sb]);
              t5_commit(&k_empty[ks]);
              ++tq;
              progressed = true;
            }
          }
          if (tp < tq) {
            // the tile's V stages: the TMA ring (bf16) or the widened ring (FP8)
            const int VR = FP8 ? CVS : VS;
            const int sb = tp % kT5SBuf;
            uint64_t *vf = FP8 ? vc_full : v_full;
            bool ready = t5_test(&p_full[sb], (tp / kT5SBuf) & 1);
#pragma unroll
            for (int h = 0; h < VPT; ++h) ready = ready && t5_test(&vf[(tp * VPT + h) % VR], ((tp * VPT + h) / VR) & 1);
            if (ready) {
              t5_fence_after();
              // stages past the end of the split hold nothing to multiply
              const int nvs = min(VPT, (min(TB, nblocks - tp * TB) + kT5Blk - 1) / kT5Blk);
#pragma unroll
              for (int h = 0; h < VPT; ++h) {
                if (h < nvs) {
                  const uint32_t vb = vc_ring + ((tp * VPT + h) % VR) * Cfg::kVTile;
#pragma unroll
                  for (int j = 0; j < kT5Blk; ++j)   // 16 keys per MMA
                    t5_mma_ts(tb + OC, tb + sb * TN + 8 * (kT5Blk * h + j), t5_desc(vb + j * 2048, Cfg::kVHalf, 1024),
                              idesc_pv, (tp > 0 || h > 0 || j > 0) ? 1u : 0u);
                }
              }
#pragma unroll
              for (int h = 0; h < VPT; ++h) {
                const int vs = (tp * VPT + h) % VR;
                t5_commit(FP8 ? &vc_empty[vs] : &v_empty[vs]);
              }
              t5_commit(&o_done[sb]);
              ++tp;
              progressed = true;
            }
          }
          if (progressed) {
            t_last = global_ns();
          } else if (*abf || global_ns() - t_last > P.wait_ns) {
            *abf = 1;
            break;
          } else {
            __nanosleep(64);   // leave issue slots to the other warps of this scheduler
          }
        }
        // every MMA issued has completed before TMEM can be released
        t5_commit(&mma_drain);
        if (!mbar_wait(&mma_drain, 0)) atomic_or_status(P.status, SV_DEV_TIMEOUT);
      }
      __syncwarp();
    } else {
      // ------------------------------------------------------------ softmax ----
      const int row = tid;   // the softmax warps
      const bool warp_live = warp * 32 < R;
      const bool live = row < R;
      const uint32_t lane_base = tb + ((uint32_t)(warp * 32) << 16);
      const int lim = live ? L - P.n_new + row / P.G : -1;   // last visible key of this row
      // draft tree: of the new keys, only the row's ancestors are visible
      const uint64_t anc = (P.anc && live) ? P.anc[(int64_t)b * P.n_new + row / P.G] : ~0ull;
      const int end_key = min(L, blk1 * kBS);                 // first key this split does not own
      const float sl2 = P.scale_log2 * q_fold;
      float m_ref = -INFINITY, l = 0.f;
      bool ok = true;
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int sb = t % kT5SBuf;
        ok = __all_sync(0xffffffffu, t5_wait(&s_full[sb], (t / kT5SBuf) & 1, abf, P.wait_ns));
        if (!ok) break;
        t5_fence_after();
        const int key0 = (blk0 + t * TB) * kBS;
        if (warp_live) {
          float x[TN];
          {
            uint32_t r[TN];
#pragma unroll
            for (int c0 = 0; c0 < TN; c0 += 16)
              t5_ld16(lane_base + sb * TN + c0, *reinterpret_cast<uint32_t(*)[16]>(r + c0));
            t5_wait_ld();
#pragma unroll
            for (int k = 0; k < TN; ++k) x[k] = __uint_as_float(r[k]);   // unscaled scores
          }
          if (key0 + TN > end_key || key0 + TN - 1 > L - P.n_new) {   // reaches the diagonal or the end
#pragma unroll
            for (int k = 0; k < TN; ++k)
              if (key0 + k > lim || key0 + k >= end_key) x[k] = -INFINITY;
            if (P.anc) {   // draft tree: new keys off the row's ancestor path go too
#pragma unroll
              for (int k = 0; k < TN; ++k) {
                const int rel = key0 + k - (L - P.n_new);
                if (rel >= 0 && !((anc >> (rel & 63)) & 1ull)) x[k] = -INFINITY;
              }
            }
          }
          // maximum as a tree; the scale is positive, so scaling the maximum
          // gives the maximum of the scaled scores (rounding is monotone)
          float mx = t5_tile_max(x) * sl2;
          // rows past R hold whatever Q's unused rows produce: they must not
          // vote for a rescale of the warp
          if (!live) mx = -INFINITY;
          // the reference moves only when a tile exceeds it by more than 8
          const bool up = mx > m_ref + 8.f;
          float a = 1.f;
          if (up) {
            a = m_ref == -INFINITY ? 0.f : ex2f(m_ref - mx);
            m_ref = mx;
          }
          if (t > 0 && __any_sync(0xffffffffu, up)) {
            // rescale O: the previous P V must have landed first
            const int pb = (t - 1) % kT5SBuf;
            ok = __all_sync(0xffffffffu, t5_wait(&o_done[pb], ((t - 1) / kT5SBuf) & 1, abf, P.wait_ns));
            t5_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < 128; c0 += 16) {
              uint32_t r[16];
              t5_ld16(lane_base + OC + c0, r);
              t5_wait_ld();
#pragma unroll
              for (int k = 0; k < 16; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * a);
              t5_st16(lane_base + OC + c0, r);
            }
            t5_wait_st();
          }
          l *= a;
          const float base = m_ref == -INFINITY ? 0.f : m_ref;
          // exponent arguments x c - base two at a time (packed fma), sums
          // in four packed chains
          const float2 c2 = make_float2(sl2, sl2), nb2 = make_float2(-base, -base);
          float2 ps2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
          for (int c0 = 0; c0 < TN; c0 += 32) {
            uint32_t w[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const float2 y = __ffma2_rn(make_float2(x[c0 + 2 * k], x[c0 + 2 * k + 1]), c2, nb2);
              const float2 pp = make_float2(ex2f(y.x), ex2f(y.y));
              ps2[k & 1] = __fadd2_rn(ps2[k & 1], pp);
              w[k] = pack2<FP8>(pp.x, pp.y);
            }
            t5_st16(lane_base + sb * TN + c0 / 2, w);
          }
          t5_wait_st();
          const float2 pst = __fadd2_rn(ps2[0], ps2[1]);
          l += pst.x + pst.y;
        }
        if (!FP8 && key0 + TN > end_key && warp == 0) {
          // keys past the split or the sequence (not loaded, or stale): V rows
          // zeroed, once the V stage holding them has landed, so that
          // 0 * (anything) = 0 (stages wholly past the end are not multiplied;
          // FP8: the converter writes those rows as zeros)
          for (int h = 0; h < VPT; ++h) {
            const int k0 = key0 + 16 * kT5Blk * h;   // first key of the stage
            if (k0 >= end_key || k0 + 16 * kT5Blk <= end_key) continue;
            const int vi = t * VPT + h;
            if (!t5_wait(&v_full[vi % VS], (vi / VS) & 1, abf, P.wait_ns)) ok = false;
            const uint32_t vb = v_ring + (vi % VS) * Cfg::kVRaw;
            for (int k = end_key - k0 + lane; k < 16 * kT5Blk; k += 32) {
              const uint32_t off = (uint32_t)((k >> 4) * 2048 + (k & 15) * 128);
#pragma unroll
              for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                for (int c = 0; c < 8; ++c)
                  asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(vb + hh * Cfg::kVHalf + off + c * 16),
                               "r"(0u)
                               : "memory");
            }
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        t5_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[sb]);
        ok = __all_sync(0xffffffffu, ok);
      }
      // ---- epilogue: O of this row -------------------------------------------
      const int lb = (n_tiles - 1) % kT5SBuf;
      const bool have = __all_sync(0xffffffffu, ok && t5_wait(&o_done[lb], ((n_tiles - 1) / kT5SBuf) & 1, abf, P.wait_ns));
      t5_fence_after();
      if (have && warp_live) {
        const int nsplit = (nblk + P.bps - 1) / P.bps;
        const int64_t ent = ((int64_t)b * P.H_kv + g) * P.S + s;
        __nv_bfloat16 *out = nullptr;
        float *acc = nullptr;
        if (live) {
          const int j = row / P.G, hh = row % P.G;
          out = static_cast<__nv_bfloat16 *>(P.out) + (((int64_t)b * P.n_new + j) * P.H_q + (int64_t)g * P.G + hh) * kD;
          acc = P.ws_acc + (ent * P.R + row) * kD;
        }
        // FP8: the values are codes; v_scale makes them values again
        const float vsc = FP8 ? P.v_scale[g] : 1.f;
        const float il = (l > 0.f ? 1.f / l : 0.f) * vsc;
#pragma unroll 1
        for (int c0 = 0; c0 < 128; c0 += 64) {
          uint32_t r[64];
#pragma unroll
          for (int c = 0; c < 64; c += 16) t5_ld16(lane_base + OC + c0 + c, *reinterpret_cast<uint32_t(*)[16]>(r + c));
          t5_wait_ld();
          if (live) {
            if (nsplit == 1) {
#pragma unroll
              for (int c = 0; c < 64; c += 8) {
                uint32_t w[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  w[k] = pack2<false>(__uint_as_float(r[c + 2 * k]) * il, __uint_as_float(r[c + 2 * k + 1]) * il);
                *reinterpret_cast<uint4 *>(out + c0 + c) = make_uint4(w[0], w[1], w[2], w[3]);
              }
            } else {
#pragma unroll
              for (int c = 0; c < 64; c += 4)
                *reinterpret_cast<float4 *>(acc + c0 + c) =
                    make_float4(__uint_as_float(r[c]) * vsc, __uint_as_float(r[c + 1]) * vsc,
                                __uint_as_float(r[c + 2]) * vsc, __uint_as_float(r[c + 3]) * vsc);
            }
          }
        }
        if (live && nsplit > 1) {
          P.ws_ml[(ent * P.R + row) * 2] = m_ref;
          P.ws_ml[(ent * P.R + row) * 2 + 1] = l;
        }
      }
    }
  }
  if constexpr (FP8) {
    // -------------------------------------------------- V: e4m3 -> f16 ---
    // Converter warps 8 and 7 (and 3 and 2 when the softmax needs two warps)
    // widen the V stages. A raw stage is two blocks of 16 slots x 128 codes
    // (128-byte swizzle); the CW warps share its 16-byte chunks: chunk
    // q = 32 cw + lane + 32 CW j is key row q / 8, head dims 16 (q % 8) ..
    // + 15, and lands as two 16-byte chunks of one head-dim half of the f16
    // stage. Rows of keys past the split or the sequence are written as
    // zeros.
    const int cw = warp == 8 ? 0 : (warp == 7 ? 1 : (warp == 3 ? 2 : (warp == 2 ? 3 : CW)));
    if (cw < CW) {
      const int NS = VS, NC = CVS;
      const int sblk = kT5Blk;   // blocks per stage
      const uint32_t rbytes = Cfg::kVRaw, cbytes = Cfg::kVTile;
      const uint32_t chalf = Cfg::kVHalf;
      uint64_t *rfull = v_full;
      uint64_t *rempty = v_empty;
      uint64_t *cfull = vc_full;
      uint64_t *cempty = vc_empty;
      const uint32_t rring = v_ring;
      const uint32_t cring = vc_ring;
      const int end_key = min(L, blk1 * kBS);
      const int n_st = n_tiles * VPT;
      const int nch = sblk * 128;   // 16-byte chunks of a raw stage
      for (int i = 0; i < n_st; ++i) {
        const int rs = i % NS, cs = i % NC;
        bool ok = __all_sync(0xffffffffu, t5_wait(&rfull[rs], (i / NS) & 1, abf, P.wait_ns));
        if (ok && i >= NC) ok = __all_sync(0xffffffffu, t5_wait(&cempty[cs], ((i / NC) - 1) & 1, abf, P.wait_ns));
        if (!ok) break;
        const uint32_t src = rring + rs * rbytes, dst = cring + cs * cbytes;
        const int key0 = (blk0 + i * sblk) * kBS;
#pragma unroll 4
        for (int q = 32 * cw + lane; q < nch; q += 32 * CW) {
          const int row = q >> 3, ch = q & 7, blk = row >> 4, r16 = row & 15;
          uint32_t v0, v1, v2, v3;
          asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                       : "r"(src + blk * 2048 + r16 * 128 + ((ch ^ (r16 & 7)) << 4)));
          uint32_t h[8];
          if (key0 + row < end_key) {
            const uint32_t w[4] = {v0, v1, v2, v3};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              h[2 * e] = e4m3x2_to_f16x2((uint16_t)(w[e] & 0xffffu));
              h[2 * e + 1] = e4m3x2_to_f16x2((uint16_t)(w[e] >> 16));
            }
          } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) h[e] = 0u;
          }
          const uint32_t rowb = dst + (ch >> 2) * chalf + row * 128;
          const int c8 = 2 * (ch & 3);
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(rowb + ((c8 ^ (r16 & 7)) << 4)), "r"(h[0]),
                       "r"(h[1]), "r"(h[2]), "r"(h[3])
                       : "memory");
          asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(rowb + (((c8 + 1) ^ (r16 & 7)) << 4)),
                       "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7])
                       : "memory");
        }
        // the tensor cores read the widened stage through the async proxy
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&rempty[rs]);   // the raw stage may be refilled
          mbar_arrive(&cfull[cs]);    // the widened stage may be read
        }
      }
    }
  }
  if (tid == 0 && *abf) atomic_or_status(P.status, SV_DEV_TIMEOUT);
  t5_fence_before();
  __syncthreads();
  t5_fence_after();
  if (warp == kT5MmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kT5Cols));
}

// The balanced-mode kernel: the same roles, pipelines and per-tile work as
// attn_tc5_kernel, but a CTA runs a list of work items (see T5Walk): every
// role walks the same items, and ring stages, S buffers and barrier phases
// follow the CTA's running tile count, so the pipelines flow from one item
// into the next. (A single kernel for both modes measured 7 % slower in split
// mode: 6 % more instructions on the per-tile paths.)
template <int QR, bool FP8>
__global__ void __launch_bounds__(T5Cfg<QR, FP8>::kThreads, 2) attn_tc5_bal_kernel(const __grid_constant__ TcParams P) {
  pdl_wait();
  pdl_trigger();
  using Cfg = T5Cfg<QR, FP8>;
  constexpr int KS = Cfg::kKS, VS = Cfg::kVS;
  constexpr int CVS = Cfg::kCVS > 0 ? Cfg::kCVS : 1;
  constexpr int SW = Cfg::kSoftW, CW = Cfg::kConvW;
  constexpr int TB = Cfg::kBlk, TN = Cfg::kN, VPT = Cfg::kVPT;
  constexpr uint32_t OC = Cfg::kOCol;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t k_full[KS], k_empty[KS], v_full[VS], v_empty[VS];
  // FP8: widened V stages, filled by the converter warps, freed by the MMAs
  __shared__ __align__(8) uint64_t vc_full[CVS], vc_empty[CVS];
  __shared__ __align__(8) uint64_t s_full[kT5SBuf], p_full[kT5SBuf], o_done[kT5SBuf], mma_drain, q_full;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {
    // a CTA with no work leaves before it sets anything up
    T5Walk w0 = {};
    T5Item it0;
    if (!t5_item(P, w0, it0)) return;
  }
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t q_smem = smem_u32(smem);   // Q, the A operand of Q K^T
  const uint32_t k_ring = q_smem + Cfg::kQBytes;
  const uint32_t v_ring = k_ring + KS * Cfg::kKRaw;
  // the V ring the MMAs read: the widened one for FP8, else the TMA ring
  const uint32_t vc_ring = FP8 ? v_ring + VS * Cfg::kVRaw : v_ring;
  const int R = P.R;

  if (tid == 0) {
    // K stages are freed by the MMAs; raw V stages by the MMAs (bf16) or by
    // the CW converter warps (FP8), whose widened stages the MMAs free
    for (int k = 0; k < KS; ++k) {
      mbar_init(&k_full[k], 1);
      mbar_init(&k_empty[k], 1);
    }
    for (int k = 0; k < VS; ++k) {
      mbar_init(&v_full[k], 1);
      mbar_init(&v_empty[k], FP8 ? CW : 1);
    }
    if (FP8) {
      for (int k = 0; k < CVS; ++k) {
        mbar_init(&vc_full[k], CW);
        mbar_init(&vc_empty[k], 1);
      }
    }
    for (int k = 0; k < kT5SBuf; ++k) {
      mbar_init(&s_full[k], 1);
      mbar_init(&p_full[k], SW);
      mbar_init(&o_done[k], 1);
    }
    mbar_init(&mma_drain, 1);
    mbar_init(&q_full, SW);   // the softmax warps wrote their Q rows (one phase per item)
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  volatile int *abf = &abort_flag;
  // Every ring stage, S buffer and barrier phase below is indexed by the
  // CTA's running tile count u over all its items, so the pipelines flow from
  // one item into the next.

  if (warp == 4 || warp == 5) {
    // ------------------------------------------------------------ producers --
    // warp 4 streams K tiles, warp 5 V stages (VPT of 32 keys per tile; a
    // stage of a tile that ends before it completes with a plain arrival);
    // the whole warp walks the block table 32 entries at a time (the next 32
    // prefetched); lane 0 waits for free stages and issues the copies
    const bool isv = warp == 5;
    const int NS = isv ? VS : KS;
    const int SPT = isv ? VPT : 1;                                   // stages per tile
    const int SB = isv ? kT5Blk : TB;                                // blocks per stage
    const uint32_t sbytes = isv ? Cfg::kVRaw : Cfg::kKRaw;
    const uint32_t half = isv ? Cfg::kVHalf : Cfg::kKHalf;           // 16-bit: second head-dim half
    uint64_t *fullb = isv ? v_full : k_full;
    uint64_t *emptyb = isv ? v_empty : k_empty;
    const uint32_t ring = isv ? v_ring : k_ring;
    const CUtensorMap *map = isv ? &P.tmv : &P.tmk;
    T5Walk wk = {};
    T5Item it;
    int i = 0, issued = 0;   // the CTA's running stage count
    bool go = true;
    // (test hook: with the copies withheld every wait on them runs out,
    // with nothing in flight)
    const bool withhold = (P.withhold & SV_TEST_WITHHOLD_COPIES) != 0;
    while (go && !withhold && t5_item(P, wk, it)) {
      const int nblocks = it.blk1 - it.blk0;
      const int n_st = (nblocks + TB - 1) / TB * SPT;
      const int32_t *table = P.block_table + (int64_t)it.b * P.max_blocks + it.blk0;
      int cur = lane < nblocks ? table[lane] : 0;
      int nxt = 32 + lane < nblocks ? table[32 + lane] : 0;
      int chunk = 0;
      for (int q = 0; q < n_st; ++q, ++i) {
        const int first = q * SB;   // the item's stage q holds blocks first .. first + SB - 1
        if ((first >> 5) != chunk) {
          chunk = first >> 5;
          cur = nxt;
          const int rel = (chunk + 1) * 32 + lane;
          nxt = rel < nblocks ? table[rel] : 0;
        }
        int phys[TB];
#pragma unroll
        for (int kk = 0; kk < TB; ++kk) phys[kk] = __shfl_sync(0xffffffffu, cur, (first + kk) & 31);
        const int st = i % NS;
        if (lane == 0) {
          if (i >= NS && !t5_wait(&emptyb[st], ((i / NS) & 1) ^ 1, abf, P.wait_ns)) {
            go = false;
          } else {
            const int nvalid = max(0, min(SB, nblocks - first));
            if (nvalid == 0) {
              mbar_arrive(&fullb[st]);   // past the end of the item: nothing to copy
            } else {
              // a block is 2 KB of e4m3 (one 128-byte box row per slot) or two
              // 2 KB head-dim halves of bf16
              mbar_arrive_expect_tx(&fullb[st], (uint32_t)(nvalid * (FP8 ? 2048 : 2 * 2048)));
              const uint32_t base = ring + st * sbytes;
              for (int kk = 0; kk < nvalid; ++kk) {
                int ph = phys[kk];
                if (ph < 0 || ph >= P.num_blocks) {
                  if (!isv) atomic_or_status(P.status, SV_DEV_BAD_BLOCK);
                  ph = 0;   // stay in bounds; the output of this sequence is flagged
                }
                int c[3];
                tile_coords(P, it.g, ph, c);
                tma_load_4d(base + kk * 2048, map, 0, c[0], c[1], c[2], &fullb[st]);
                if (!FP8) tma_load_4d(base + half + kk * 2048, map, 64, c[0], c[1], c[2], &fullb[st]);
              }
            }
            issued = i + 1;
          }
        }
        go = __shfl_sync(0xffffffffu, (int)go, 0) != 0;
        if (!go) break;
      }
    }
    // the copies in flight land before the CTA may exit
    if (lane == 0) {
      for (int t = max(0, issued - NS); t < issued; ++t)
        if (!mbar_wait(&fullb[t % NS], (t / NS) & 1)) atomic_or_status(P.status, SV_DEV_TIMEOUT);
    }
  } else if (warp < SW || warp == kT5MmaWarp) {
    if (warp == kT5MmaWarp) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                   "r"(kT5Cols));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    t5_fence_before();
    named_bar_sync(1, 32 * (SW + 1));   // TMEM allocated
    t5_fence_after();
    const uint32_t tb = tmem_base;

    if (warp == kT5MmaWarp) {
      // ---------------------------------------------------------- MMA issuer --
      if (lane == 0) {
        // f32 accumulators; A and B bf16 (formats 1), or for FP8 e4m3 in Q K^T
        // (kind::f8f6f4, format 0) and f16 in P V (format 0)
        constexpr uint32_t ab = FP8 ? 0u : (1u << 7) | (1u << 10);
        const uint32_t idesc_qk = (1u << 4) | ab | ((uint32_t)(TN >> 3) << 17) | (8u << 24);
        const uint32_t idesc_pv = (1u << 4) | ab | (1u << 16) | (16u << 17) | (8u << 24);
        static_assert(TN % 16 == 0 && TN <= 256, "MMA N");
        // the items in order, each with the split kernel's loop; u0 is the
        // CTA's running tile count at the item's start. The next item's
        // Q K^T could not start earlier anyway: its Q is written after this
        // item's epilogue, which waits for the last P V.
        T5Walk wk = {};
        T5Item it;
        int u0 = 0, xq = 0;
        bool okm = true;
        while (okm && t5_item(P, wk, it)) {
          const int nblocks = it.blk1 - it.blk0;
          const int n_tiles = (nblocks + TB - 1) / TB;
          int tq = 0, tp = 0;   // next tiles for Q K^T and for P V
          bool q_ready = false;
          uint64_t t_last = global_ns();
          while (tp < n_tiles) {
            bool progressed = false;
            if (!q_ready) q_ready = t5_test(&q_full, xq & 1);
            if (q_ready && tq < n_tiles && tq - tp < kT5SBuf) {
              // K stage: the TMA ring (raw e4m3 codes for FP8)
              const int KR = KS;
              const int uq = u0 + tq;
              const int ks = uq % KR, sb = uq % kT5SBuf;
              uint64_t *kf = k_full;
              // S buffer sb is free once the P V of tile uq - kT5SBuf has run
              const bool sfree = uq < kT5SBuf || t5_test(&o_done[sb], ((uq / kT5SBuf) - 1) & 1);
              if (sfree && t5_test(&kf[ks], (uq / KR) & 1)) {
                t5_fence_after();
                const uint32_t kb = k_ring + ks * Cfg::kKRaw;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                  // A = Q and B = K from shared memory. bf16: 16 head dims per step over
                  // the two head-dim halves; FP8: 32 head dims per step, the hi term of Q
                  // (kk < 4) then the lo term, against the raw codes
                  const uint64_t ad = t5_desc(q_smem + (kk >> 2) * (QR * 128) + (kk & 3) * 32, 16, 1024);
                  if constexpr (FP8)
                    t5_mma_ss_f8(tb + sb * TN, ad, t5_desc(kb + (kk & 3) * 32, 16, 1024), idesc_qk, kk > 0 ? 1u : 0u);
                  else
                    t5_mma_ss(tb + sb * TN, ad, t5_desc(kb + (kk >> 2) * Cfg::kKHalf + (kk & 3) * 32, 16, 1024), idesc_qk,
                              kk > 0 ? 1u : 0u);
                }
                t5_commit(&s_full[sb]);
                t5_commit(&k_empty[ks]);
                ++tq;
                progressed = true;
              }
            }
            if (tp < tq) {
              // the tile's V stages: the TMA ring (bf16) or the widened ring (FP8)
              const int VR = FP8 ? CVS : VS;
              const int up = u0 + tp;
              const int sb = up % kT5SBuf;
              uint64_t *vf = FP8 ? vc_full : v_full;
              bool ready = t5_test(&p_full[sb], (up / kT5SBuf) & 1);
#pragma unroll
              for (int h = 0; h < VPT; ++h) ready = ready && t5_test(&vf[(up * VPT + h) % VR], ((up * VPT + h) / VR) & 1);
              if (ready) {
                t5_fence_after();
                // stages past the end of the item hold nothing to multiply
                const int nvs = min(VPT, (min(TB, nblocks - tp * TB) + kT5Blk - 1) / kT5Blk);
#pragma unroll
                for (int h = 0; h < VPT; ++h) {
                  if (h < nvs) {
                    const uint32_t vb = vc_ring + ((up * VPT + h) % VR) * Cfg::kVTile;
#pragma unroll
                    for (int j = 0; j < kT5Blk; ++j)   // an item's first P V starts O afresh
                      t5_mma_ts(tb + OC, tb + sb * TN + 8 * (kT5Blk * h + j),
                                t5_desc(vb + j * 2048, Cfg::kVHalf, 1024), idesc_pv,
                                (tp > 0 || h > 0 || j > 0) ? 1u : 0u);
                  }
                }
#pragma unroll
                for (int h = 0; h < VPT; ++h) {
                  const int vs = (up * VPT + h) % VR;
                  t5_commit(FP8 ? &vc_empty[vs] : &v_empty[vs]);
                }
                t5_commit(&o_done[sb]);
                ++tp;
                progressed = true;
              }
            }
            if (progressed) {
              t_last = global_ns();
            } else if (*abf || global_ns() - t_last > P.wait_ns) {
              *abf = 1;
              okm = false;
              break;
            } else {
              __nanosleep(64);   // leave issue slots to the other warps of this scheduler
            }
          }
          u0 += n_tiles;
          ++xq;
        }
        // every MMA issued has completed before TMEM can be released
        t5_commit(&mma_drain);
        if (!mbar_wait(&mma_drain, 0)) atomic_or_status(P.status, SV_DEV_TIMEOUT);
      }
      __syncwarp();
    } else {
      // ------------------------------------------------------------ softmax ----
      const int row = tid;   // the softmax warps
      const bool warp_live = warp * 32 < R;
      const bool live = row < R;
      const uint32_t lane_base = tb + ((uint32_t)(warp * 32) << 16);
      T5Walk wk = {};
      T5Item it;
      int u = 0;
      bool ok = true;
      while (ok && t5_item(P, wk, it)) {
        const int b = it.b, g = it.g, L = it.L;
        const int nblocks = it.blk1 - it.blk0;
        const int n_tiles = (nblocks + TB - 1) / TB;
        const int lim = live ? L - P.n_new + row / P.G : -1;   // last visible key of this row
        // draft tree: of the new keys, only the row's ancestors are visible
        const uint64_t anc = (P.anc && live) ? P.anc[(int64_t)b * P.n_new + row / P.G] : ~0ull;
        const int end_key = min(L, it.blk1 * kBS);             // first key this item does not own
        float sl2 = P.scale_log2;
        {
          // The previous item's Q K^T have all run: its epilogue waited for
          // its last P V.
          const uint4 *src = nullptr;
          if (live) {
            const int j = row / P.G, hh = row % P.G;
            src = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(P.q) +
                                                  (((int64_t)b * P.n_new + j) * P.H_q + (int64_t)g * P.G + hh) * kD);
          }
          if (row < QR) sl2 *= t5_store_q<QR, FP8>(q_smem, row, src, FP8 ? P.k_scale[g] : 1.f);
          t5_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&q_full);
        }
        float m_ref = -INFINITY, l = 0.f;
        for (int t = 0; t < n_tiles && ok; ++t, ++u) {
          const int sb = u % kT5SBuf;
          ok = __all_sync(0xffffffffu, t5_wait(&s_full[sb], (u / kT5SBuf) & 1, abf, P.wait_ns));
          if (!ok) break;
          t5_fence_after();
          const int key0 = (it.blk0 + t * TB) * kBS;
          if (warp_live) {
            float x[TN];
            {
              uint32_t r[TN];
#pragma unroll
              for (int c0 = 0; c0 < TN; c0 += 16)
                t5_ld16(lane_base + sb * TN + c0, *reinterpret_cast<uint32_t(*)[16]>(r + c0));
              t5_wait_ld();
#pragma unroll
              for (int k = 0; k < TN; ++k) x[k] = __uint_as_float(r[k]);   // unscaled scores
            }
            if (key0 + TN > end_key || key0 + TN - 1 > L - P.n_new) {   // reaches the diagonal or the end
#pragma unroll
              for (int k = 0; k < TN; ++k)
                if (key0 + k > lim || key0 + k >= end_key) x[k] = -INFINITY;
              if (P.anc) {   // draft tree: new keys off the row's ancestor path go too
#pragma unroll
                for (int k = 0; k < TN; ++k) {
                  const int rel = key0 + k - (L - P.n_new);
                  if (rel >= 0 && !((anc >> (rel & 63)) & 1ull)) x[k] = -INFINITY;
                }
              }
            }
            float mx = t5_tile_max(x) * sl2;   // the scale is positive
            // rows past R hold whatever Q's unused rows produce: they must not
            // vote for a rescale of the warp
            if (!live) mx = -INFINITY;
            // the reference moves only when a tile exceeds it by more than 8
            const bool upd = mx > m_ref + 8.f;
            float a = 1.f;
            if (upd) {
              a = m_ref == -INFINITY ? 0.f : ex2f(m_ref - mx);
              m_ref = mx;
            }
            if (t > 0 && __any_sync(0xffffffffu, upd)) {
              // rescale O: the previous P V must have landed first
              const int pb = (u - 1) % kT5SBuf;
              ok = __all_sync(0xffffffffu, t5_wait(&o_done[pb], ((u - 1) / kT5SBuf) & 1, abf, P.wait_ns));
              t5_fence_after();
#pragma unroll 1
              for (int c0 = 0; c0 < 128; c0 += 16) {
                uint32_t r[16];
                t5_ld16(lane_base + OC + c0, r);
                t5_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k) r[k] = __float_as_uint(__uint_as_float(r[k]) * a);
                t5_st16(lane_base + OC + c0, r);
              }
              t5_wait_st();
            }
            l *= a;
            const float base = m_ref == -INFINITY ? 0.f : m_ref;
            const float2 c2 = make_float2(sl2, sl2), nb2 = make_float2(-base, -base);
            float2 ps2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
            for (int c0 = 0; c0 < TN; c0 += 32) {
              uint32_t w[16];
#pragma unroll
              for (int k = 0; k < 16; ++k) {
                const float2 y = __ffma2_rn(make_float2(x[c0 + 2 * k], x[c0 + 2 * k + 1]), c2, nb2);
                const float2 pp = make_float2(ex2f(y.x), ex2f(y.y));
                ps2[k & 1] = __fadd2_rn(ps2[k & 1], pp);
                w[k] = pack2<FP8>(pp.x, pp.y);
              }
              t5_st16(lane_base + sb * TN + c0 / 2, w);
            }
            t5_wait_st();
            const float2 pst = __fadd2_rn(ps2[0], ps2[1]);
            l += pst.x + pst.y;
          }
          if (!FP8 && key0 + TN > end_key && warp == 0) {
            // keys past the item or the sequence (not loaded, or stale): V rows
            // zeroed, once the V stage holding them has landed, so that
            // 0 * (anything) = 0 (stages wholly past the end are not
            // multiplied; FP8: the converter writes those rows as zeros)
            for (int h = 0; h < VPT; ++h) {
              const int k0 = key0 + 16 * kT5Blk * h;   // first key of the stage
              if (k0 >= end_key || k0 + 16 * kT5Blk <= end_key) continue;
              const int vi = u * VPT + h;
              if (!t5_wait(&v_full[vi % VS], (vi / VS) & 1, abf, P.wait_ns)) ok = false;
              const uint32_t vb = v_ring + (vi % VS) * Cfg::kVRaw;
              for (int k = end_key - k0 + lane; k < 16 * kT5Blk; k += 32) {
                const uint32_t off = (uint32_t)((k >> 4) * 2048 + (k & 15) * 128);
#pragma unroll
                for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                  for (int c = 0; c < 8; ++c)
                    asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(vb + hh * Cfg::kVHalf + off + c * 16),
                                 "r"(0u)
                                 : "memory");
              }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          }
          t5_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&p_full[sb]);
          ok = __all_sync(0xffffffffu, ok);
        }
        if (!ok) break;
        // ---- epilogue: O of this row ------------------------------------------
        const int lu = u - 1;   // the item's last tile
        const bool have = __all_sync(0xffffffffu, t5_wait(&o_done[lu % kT5SBuf], (lu / kT5SBuf) & 1, abf, P.wait_ns));
        t5_fence_after();
        if (!have) {
          ok = false;
          break;
        }
        if (warp_live) {
          __nv_bfloat16 *out = nullptr;
          float *acc = nullptr;
          if (live) {
            const int j = row / P.G, hh = row % P.G;
            out = static_cast<__nv_bfloat16 *>(P.out) + (((int64_t)b * P.n_new + j) * P.H_q + (int64_t)g * P.G + hh) * kD;
            acc = P.ws_acc + (it.ent * P.R + row) * kD;
          }
          // FP8: the values are codes; v_scale makes them values again
          const float vsc = FP8 ? P.v_scale[g] : 1.f;
          const float il = (l > 0.f ? 1.f / l : 0.f) * vsc;
#pragma unroll 1
          for (int c0 = 0; c0 < 128; c0 += 64) {
            uint32_t r[64];
#pragma unroll
            for (int c = 0; c < 64; c += 16) t5_ld16(lane_base + OC + c0 + c, *reinterpret_cast<uint32_t(*)[16]>(r + c));
            t5_wait_ld();
            if (live) {
              if (it.whole) {
#pragma unroll
                for (int c = 0; c < 64; c += 8) {
                  uint32_t w[4];
#pragma unroll
                  for (int k = 0; k < 4; ++k)
                    w[k] = pack2<false>(__uint_as_float(r[c + 2 * k]) * il, __uint_as_float(r[c + 2 * k + 1]) * il);
                  *reinterpret_cast<uint4 *>(out + c0 + c) = make_uint4(w[0], w[1], w[2], w[3]);
                }
              } else {
#pragma unroll
                for (int c = 0; c < 64; c += 4)
                  *reinterpret_cast<float4 *>(acc + c0 + c) =
                      make_float4(__uint_as_float(r[c]) * vsc, __uint_as_float(r[c + 1]) * vsc,
                                  __uint_as_float(r[c + 2]) * vsc, __uint_as_float(r[c + 3]) * vsc);
              }
            }
          }
          if (live && !it.whole) {
            P.ws_ml[(it.ent * P.R + row) * 2] = m_ref;
            P.ws_ml[(it.ent * P.R + row) * 2 + 1] = l;
          }
        }
        // the epilogue's TMEM loads finish before the next item's first P V
        // (which waits for this warp's arrival on its P buffer) may overwrite O
      }
    }
  }
  if constexpr (FP8) {
    // -------------------------------------------------- V: e4m3 -> f16 ---
    // as in attn_tc5_kernel, over the CTA's items: the running stage count
    // indexes the rings, and rows of keys past the item or the sequence are
    // written as zeros
    const int cw = warp == 8 ? 0 : (warp == 7 ? 1 : (warp == 3 ? 2 : (warp == 2 ? 3 : CW)));
    if (cw < CW) {
      const int NS = VS, NC = CVS;
      const int sblk = kT5Blk;   // blocks per stage
      const uint32_t rbytes = Cfg::kVRaw, cbytes = Cfg::kVTile;
      const uint32_t chalf = Cfg::kVHalf;
      uint64_t *rfull = v_full;
      uint64_t *rempty = v_empty;
      uint64_t *cfull = vc_full;
      uint64_t *cempty = vc_empty;
      const uint32_t rring = v_ring;
      const uint32_t cring = vc_ring;
      const int nch = sblk * 128;   // 16-byte chunks of a raw stage
      T5Walk wk = {};
      T5Item it;
      int i = 0;   // the CTA's running stage count
      bool ok = true;
      while (ok && t5_item(P, wk, it)) {
        const int end_key = min(it.L, it.blk1 * kBS);
        const int n_st = (it.blk1 - it.blk0 + TB - 1) / TB * VPT;
        for (int q0 = 0; q0 < n_st; ++q0, ++i) {
          const int rs = i % NS, cs = i % NC;
          ok = __all_sync(0xffffffffu, t5_wait(&rfull[rs], (i / NS) & 1, abf, P.wait_ns));
          if (ok && i >= NC) ok = __all_sync(0xffffffffu, t5_wait(&cempty[cs], ((i / NC) - 1) & 1, abf, P.wait_ns));
          if (!ok) break;
          const uint32_t src = rring + rs * rbytes, dst = cring + cs * cbytes;
          const int key0 = (it.blk0 + q0 * sblk) * kBS;
#pragma unroll 4
          for (int q = 32 * cw + lane; q < nch; q += 32 * CW) {
            const int row = q >> 3, ch = q & 7, blk = row >> 4, r16 = row & 15;
            uint32_t v0, v1, v2, v3;
            asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(v0), "=r"(v1), "=r"(v2), "=r"(v3)
                         : "r"(src + blk * 2048 + r16 * 128 + ((ch ^ (r16 & 7)) << 4)));
            uint32_t h[8];
            if (key0 + row < end_key) {
              const uint32_t w[4] = {v0, v1, v2, v3};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                h[2 * e] = e4m3x2_to_f16x2((uint16_t)(w[e] & 0xffffu));
                h[2 * e + 1] = e4m3x2_to_f16x2((uint16_t)(w[e] >> 16));
              }
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) h[e] = 0u;
            }
            const uint32_t rowb = dst + (ch >> 2) * chalf + row * 128;
            const int c8 = 2 * (ch & 3);
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(rowb + ((c8 ^ (r16 & 7)) << 4)), "r"(h[0]),
                         "r"(h[1]), "r"(h[2]), "r"(h[3])
                         : "memory");
            asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(rowb + (((c8 + 1) ^ (r16 & 7)) << 4)),
                         "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7])
                         : "memory");
          }
          // the tensor cores read the widened stage through the async proxy
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&rempty[rs]);   // the raw stage may be refilled
            mbar_arrive(&cfull[cs]);    // the widened stage may be read
          }
        }
      }
    }
  }
  if (tid == 0 && *abf) atomic_or_status(P.status, SV_DEV_TIMEOUT);
  t5_fence_before();
  __syncthreads();
  t5_fence_after();
  if (warp == kT5MmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kT5Cols));
}

// ----------------------------------------------------- CUDA-core kernel ---
struct GenParams {
  const void *q;
  void *out;
  const void *k_cache;
  const void *v_cache;
  const float *k_scale;
  const float *v_scale;
  const int32_t *block_table;
  const int32_t *seq_lens;
  float *ws_acc;   // [B][H_kv][S][R][d]
  float *ws_ml;    // [B][H_kv][S][R][2]
  const uint64_t *anc;    // [B][n_new] ancestor masks of a draft tree (NULL: a chain)
  int32_t *status;
  int B, n_new, H_q, H_kv, G, R, d, bs, max_blocks, num_blocks, bps, S;
  int64_t block_stride, head_stride, slot_stride;
  float scale_log2;
};

template <typename T>
__device__ __forceinline__ float kv_value(const void *pool, int64_t off, float scale);
template <>
__device__ __forceinline__ float kv_value<float>(const void *pool, int64_t off, float) {
  return static_cast<const float *>(pool)[off];
}
template <>
__device__ __forceinline__ float kv_value<__nv_bfloat16>(const void *pool, int64_t off, float) {
  return __bfloat162float(static_cast<const __nv_bfloat16 *>(pool)[off]);
}
template <>
__device__ __forceinline__ float kv_value<uint8_t>(const void *pool, int64_t off, float scale) {
  const uint8_t code = static_cast<const uint8_t *>(pool)[off];
  const uint32_t h = e4m3x2_to_f16x2((uint16_t)code);
  return __half2float(__ushort_as_half((unsigned short)(h & 0xffff))) * scale;
}

template <typename TKV, typename TQ>
__global__ void __launch_bounds__(kGenThreads) attn_generic_kernel(const __grid_constant__ GenParams P) {
  pdl_wait();
  pdl_trigger();
  extern __shared__ float gsm[];
  const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int R = P.R, d = P.d;
  float *q_s = gsm;                       // [R][d]
  float *o_s = q_s + R * d;               // [R][d]
  float *k_s = o_s + R * d;               // [kGenKeys][d]
  float *v_s = k_s + kGenKeys * d;        // [kGenKeys][d]
  float *p_s = v_s + kGenKeys * d;        // [R][kGenKeys]
  float *m_s = p_s + R * kGenKeys;        // [R]
  float *l_s = m_s + R;                   // [R]
  float *c_s = l_s + R;                   // [R]

  const int L = P.seq_lens[b];
  if (L < P.n_new || L > P.max_blocks * P.bs) {
    if (tid == 0 && g == 0 && s == 0) atomic_or_status(P.status, SV_DEV_BAD_SEQ_LEN);
    return;
  }
  const int nblk = (L + P.bs - 1) / P.bs;
  const int blk0 = s * P.bps;
  if (blk0 >= nblk) return;
  const int t_begin = blk0 * P.bs, t_end = min(L, min(nblk, blk0 + P.bps) * P.bs);
  const float ks = std::is_same<TKV, uint8_t>::value ? P.k_scale[g] : 1.f;
  const float vsc = std::is_same<TKV, uint8_t>::value ? P.v_scale[g] : 1.f;

  for (int idx = tid; idx < R * d; idx += blockDim.x) {
    const int r = idx / d, c = idx % d;
    const int j = r / P.G, hh = r % P.G;
    const int64_t off = (((int64_t)b * P.n_new + j) * P.H_q + (int64_t)g * P.G + hh) * d + c;
    q_s[idx] = to_f32(static_cast<const TQ *>(P.q)[off]);
    o_s[idx] = 0.f;
  }
  for (int r = tid; r < R; r += blockDim.x) { m_s[r] = -INFINITY; l_s[r] = 0.f; }
  __syncthreads();
  const int32_t *table = P.block_table + (int64_t)b * P.max_blocks;

  for (int t0 = t_begin; t0 < t_end; t0 += kGenKeys) {
    for (int idx = tid; idx < kGenKeys * d; idx += blockDim.x) {
      const int kk = idx / d, c = idx % d;
      const int t = t0 + kk;
      float kv = 0.f, vv = 0.f;
      if (t < t_end) {
        int phys = table[t / P.bs];
        if (phys < 0 || phys >= P.num_blocks) {
          atomic_or_status(P.status, SV_DEV_BAD_BLOCK);
        } else {
          const int64_t off = (int64_t)phys * P.block_stride + (int64_t)g * P.head_stride +
                              (int64_t)(t % P.bs) * P.slot_stride + c;
          kv = kv_value<TKV>(P.k_cache, off, ks);
          vv = kv_value<TKV>(P.v_cache, off, vsc);
        }
      }
      k_s[idx] = kv;
      v_s[idx] = vv;
    }
    __syncthreads();
    for (int r = warp; r < R; r += blockDim.x / 32) {
      const int t = t0 + lane;
      const int lim = L - P.n_new + r / P.G;
      const int rel = t - (L - P.n_new);
      const bool in_tree = !P.anc || rel < 0 || ((P.anc[(int64_t)b * P.n_new + r / P.G] >> (rel & 63)) & 1ull);
      float sc = -INFINITY;
      if (t < t_end && t <= lim && in_tree) {
        float acc = 0.f;
        for (int c = 0; c < d; ++c) acc = fmaf(q_s[r * d + c], k_s[lane * d + c], acc);
        sc = acc * P.scale_log2;
      }
      const float mx = warp_max(sc);
      const float m_old = m_s[r];
      const float m_new = fmaxf(m_old, mx);
      const float base = m_new == -INFINITY ? 0.f : m_new;
      const float p = exp2f(sc - base);
      const float sum = warp_sum(p);
      p_s[r * kGenKeys + lane] = p;
      __syncwarp();
      if (lane == 0) {
        const float a = exp2f(m_old - base);
        c_s[r] = a;
        l_s[r] = l_s[r] * a + sum;
        m_s[r] = m_new;
      }
    }
    __syncthreads();
    for (int idx = tid; idx < R * d; idx += blockDim.x) {
      const int r = idx / d, c = idx % d;
      float acc = o_s[idx] * c_s[r];
      for (int kk = 0; kk < kGenKeys; ++kk) acc = fmaf(p_s[r * kGenKeys + kk], v_s[kk * d + c], acc);
      o_s[idx] = acc;
    }
    __syncthreads();
  }
  if ((nblk + P.bps - 1) / P.bps == 1) {   // single split: write the normalised output
    for (int idx = tid; idx < R * d; idx += blockDim.x) {
      const int r = idx / d, cc = idx % d;
      const int j = r / P.G, hh = r % P.G;
      const int64_t off = (((int64_t)b * P.n_new + j) * P.H_q + (int64_t)g * P.G + hh) * d + cc;
      const float v = l_s[r] > 0.f ? o_s[idx] / l_s[r] : 0.f;
      if (std::is_same<TQ, float>::value) static_cast<float *>(P.out)[off] = v;
      else static_cast<__nv_bfloat16 *>(P.out)[off] = __float2bfloat16_rn(v);
    }
    return;
  }
  const int64_t ent = ((int64_t)b * P.H_kv + g) * P.S + s;
  for (int idx = tid; idx < R * d; idx += blockDim.x) P.ws_acc[ent * R * d + idx] = o_s[idx];
  for (int r = tid; r < R; r += blockDim.x) {
    P.ws_ml[(ent * R + r) * 2] = m_s[r];
    P.ws_ml[(ent * R + r) * 2 + 1] = l_s[r];
  }
}

// ------------------------------------------------------------ LSE merge ---
struct MergeParams {
  const float *ws_acc;
  const float *ws_ml;
  const int32_t *seq_lens;
  const int32_t *seq_pre;   // balanced mode: first tile of each sequence, then T
  const int4 *split;        // balanced mode: (count, T), then (b, A, nt, r0) of each split sequence
  void *out;
  int B, n_new, H_q, H_kv, G, R, d, bs, max_blocks, bps, S, per_split;
  int C;                    // balanced mode: CTAs of the tcgen05 kernel (0: split mode)
};

// Split merge: WPR warps per output row (sequence, kv head, packed query row),
// each taking every WPR-th piece, kMB of them loaded at once (one round trip
// for up to WPR kMB splits) and folded into a running maximum (lanes own
// float4 column chunks); the warps' states are then combined through shared
// memory by the row's first warp.
template <typename TO, int WPR>
__global__ void __launch_bounds__(256) attn_merge_kernel(const __grid_constant__ MergeParams P) {
  pdl_wait();
  pdl_trigger();
  constexpr int kMaxChunks = 2;   // d <= 256
  __shared__ float4 xs_acc[8][kMaxChunks][32];
  __shared__ float xs_ml[8][2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wr = warp % WPR;                       // warp within the row group
  const int64_t rowid = (int64_t)blockIdx.x * (8 / WPR) + warp / WPR;
  const int R = P.R;
  const bool live = rowid < (int64_t)P.B * P.H_kv * R;

  int nsplit = 0, r = 0, g = 0, b = 0;
  int64_t bg = 0;
  if (live) {
    r = (int)(rowid % R);
    bg = rowid / R;
    g = (int)(bg % P.H_kv);
    b = (int)(bg / P.H_kv);
    const int L = P.seq_lens[b];
    if (L >= P.n_new && L <= P.max_blocks * P.bs) {
      const int nblk = (L + P.bs - 1) / P.bs;
      nsplit = (nblk + P.bps - 1) / P.bps;
    }
  }
  const int nc = P.d >> 2;   // float4 chunks per row
  float4 acc[kMaxChunks];
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  float m = -INFINITY, l = 0.f;
  if (nsplit > 1) {
    constexpr int kMB = 8;   // pieces a warp loads at once
    for (int e0 = wr; e0 < nsplit; e0 += WPR * kMB) {
      float me[kMB], le[kMB];
      float4 va[kMB][kMaxChunks];
#pragma unroll
      for (int u = 0; u < kMB; ++u) {
        const int e = e0 + u * WPR;
        me[u] = -INFINITY;
        le[u] = 0.f;
        if (e < nsplit) {
          const int64_t row = (bg * P.S + e) * R + r;
          me[u] = P.ws_ml[row * 2];
          le[u] = P.ws_ml[row * 2 + 1];
          const float4 *src = reinterpret_cast<const float4 *>(P.ws_acc + row * P.d);
#pragma unroll
          for (int k = 0; k < kMaxChunks; ++k)
            if (lane + 32 * k < nc) va[u][k] = src[lane + 32 * k];
        }
      }
      float mn = m;
#pragma unroll
      for (int u = 0; u < kMB; ++u) mn = fmaxf(mn, me[u]);
      const float base = mn == -INFINITY ? 0.f : mn;
      const float a = exp2f(m - base);
      l *= a;
#pragma unroll
      for (int k = 0; k < kMaxChunks; ++k) {
        acc[k].x *= a; acc[k].y *= a; acc[k].z *= a; acc[k].w *= a;
      }
#pragma unroll
      for (int u = 0; u < kMB; ++u) {
        if (e0 + u * WPR >= nsplit) continue;
        const float w = exp2f(me[u] - base);
        l += le[u] * w;
#pragma unroll
        for (int k = 0; k < kMaxChunks; ++k) {
          if (lane + 32 * k >= nc) continue;
          acc[k].x += va[u][k].x * w; acc[k].y += va[u][k].y * w;
          acc[k].z += va[u][k].z * w; acc[k].w += va[u][k].w * w;
        }
      }
      m = mn;
    }
  }
  if constexpr (WPR > 1) {
#pragma unroll
    for (int k = 0; k < kMaxChunks; ++k) xs_acc[warp][k][lane] = acc[k];
    if (lane == 0) { xs_ml[warp][0] = m; xs_ml[warp][1] = l; }
    __syncthreads();
    if (wr == 0) {
      for (int w2 = 1; w2 < WPR; ++w2) {
        const float me = xs_ml[warp + w2][0], le = xs_ml[warp + w2][1];
        const float mn = fmaxf(m, me);
        const float base = mn == -INFINITY ? 0.f : mn;
        const float a = exp2f(m - base), w = exp2f(me - base);
        l = l * a + le * w;
        m = mn;
#pragma unroll
        for (int k = 0; k < kMaxChunks; ++k) {
          const float4 v = xs_acc[warp + w2][k][lane];
          acc[k].x = acc[k].x * a + v.x * w;
          acc[k].y = acc[k].y * a + v.y * w;
          acc[k].z = acc[k].z * a + v.z * w;
          acc[k].w = acc[k].w * a + v.w * w;
        }
      }
    }
  }
  // nsplit == 1: written directly by the attention kernel
  if (!live || nsplit <= 1 || wr != 0) return;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  const int j = r / P.G, hh = r % P.G;
  const int64_t out_off = (((int64_t)b * P.n_new + j) * P.H_q + (int64_t)g * P.G + hh) * P.d;
#pragma unroll
  for (int k = 0; k < kMaxChunks; ++k) {
    const int cidx = lane + 32 * k;
    if (cidx < nc) {
      const float4 v = acc[k];
      if constexpr (std::is_same<TO, float>::value) {
        reinterpret_cast<float4 *>(static_cast<float *>(P.out) + out_off)[cidx] =
            make_float4(v.x * inv, v.y * inv, v.z * inv, v.w * inv);
      } else {
        __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(P.out) + out_off + 4 * cidx;
        *reinterpret_cast<__nv_bfloat162 *>(o) = __floats2bfloat162_rn(v.x * inv, v.y * inv);
        *reinterpret_cast<__nv_bfloat162 *>(o + 2) = __floats2bfloat162_rn(v.z * inv, v.w * inv);
      }
    }
  }
}

// Split merge for at most four splits: one CTA per (sequence, kv head). The
// length is read once and a sequence with a single split (written by the
// attention kernel) leaves at once; otherwise each warp merges a row (warp w
// takes rows w, w + warps, ...), its splits loaded together in one round
// trip.
template <typename TO>
__global__ void __launch_bounds__(1024) attn_merge_pair_kernel(const __grid_constant__ MergeParams P) {
  pdl_wait();
  pdl_trigger();
  constexpr int kMaxChunks = 2;   // d <= 256
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t bg = blockIdx.x;
  const int g = (int)(bg % P.H_kv), b = (int)(bg / P.H_kv);
  const int L = P.seq_lens[b];
  if (L < P.n_new || L > P.max_blocks * P.bs) return;
  const int nsplit = ((L + P.bs - 1) / P.bs + P.bps - 1) / P.bps;
  if (nsplit <= 1) return;
  const int R = P.R, nc = P.d >> 2;
  for (int r = warp; r < R; r += (int)(blockDim.x >> 5)) {
    float me[4], le[4];
    float4 va[4][kMaxChunks];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      me[e] = -INFINITY;
      le[e] = 0.f;
      if (e < nsplit) {
        const int64_t row = (bg * P.S + e) * R + r;
        me[e] = P.ws_ml[row * 2];
        le[e] = P.ws_ml[row * 2 + 1];
        const float4 *src = reinterpret_cast<const float4 *>(P.ws_acc + row * P.d);
#pragma unroll
        for (int k = 0; k < kMaxChunks; ++k)
          if (lane + 32 * k < nc) va[e][k] = src[lane + 32 * k];
      }
    }
    float m = -INFINITY;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (e < nsplit) m = fmaxf(m, me[e]);
    const float base = m == -INFINITY ? 0.f : m;
    float l = 0.f, w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      w[e] = e < nsplit ? exp2f(me[e] - base) : 0.f;
      l += e < nsplit ? le[e] * w[e] : 0.f;
    }
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int j = r / P.G, hh = r % P.G;
    const int64_t out_off = (((int64_t)b * P.n_new + j) * P.H_q + (int64_t)g * P.G + hh) * P.d;
#pragma unroll
    for (int k = 0; k < kMaxChunks; ++k) {
      const int cidx = lane + 32 * k;
      if (cidx >= nc) continue;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (e >= nsplit) continue;
        v.x += va[e][k].x * w[e]; v.y += va[e][k].y * w[e];
        v.z += va[e][k].z * w[e]; v.w += va[e][k].w * w[e];
      }
      if constexpr (std::is_same<TO, float>::value) {
        reinterpret_cast<float4 *>(static_cast<float *>(P.out) + out_off)[cidx] =
            make_float4(v.x * inv, v.y * inv, v.z * inv, v.w * inv);
      } else {
        __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(P.out) + out_off + 4 * cidx;
        *reinterpret_cast<__nv_bfloat162 *>(o) = __floats2bfloat162_rn(v.x * inv, v.y * inv);
        *reinterpret_cast<__nv_bfloat162 *>(o + 2) = __floats2bfloat162_rn(v.z * inv, v.w * inv);
      }
    }
  }
}

// Balanced-mode merge: only the sequences the partition listed as split
// (split[1..n] = (b, A, nt, r0)); row u of the work is (listed sequence
// u / (H_kv R), kv head, query row), WPR warps per row, rows taken
// grid-stride so that the launch does not depend on n. The pieces of (b, g)
// come from the ranges r0..r1 that meet b's tiles [A, A + nt) (range r holds
// [r T / NR, (r + 1) T / NR)), skipping empty ranges, each run for head g by
// CTA c = r H_kv + g; r0's piece is its CTA's last item (entry 2c + 1) unless
// r0 starts at A, every other one is its CTA's first (entry 2c). Warp wr of a
// row takes pieces wr, wr + WPR, ..., loading up to kMB of them at once (one
// round trip), and the WPR warps' states are combined through shared
// memory. d = 128 (the tcgen05 path): lane l owns float4 chunk l.
template <typename TO, int WPR>
__global__ void __launch_bounds__(256) attn_merge_bal_kernel(const __grid_constant__ MergeParams P) {
  pdl_wait();
  pdl_trigger();
  constexpr int kRows = 8 / WPR;  // rows per CTA and round
  constexpr int kMB = 8;          // pieces a warp loads at once
  __shared__ float4 xs_acc[8][32];
  __shared__ float xs_ml[8][2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wr = warp % WPR;
  const int R = P.R;
  const int4 hdr = P.split[0];
  const int64_t NR = P.C / P.H_kv, T = hdr.y;
  const int64_t nrows = (int64_t)hdr.x * P.H_kv * R;
  for (int64_t base = (int64_t)blockIdx.x * kRows; base < nrows; base += (int64_t)gridDim.x * kRows) {
    const int64_t u = base + warp / WPR;
    const bool live = u < nrows;
    int r = 0, g = 0, b = 0, npiece = 0;
    int64_t A = 0, r0 = 0;
    if (live) {
      r = (int)(u % R);
      g = (int)((u / R) % P.H_kv);
      const int4 sp = P.split[1 + (int)(u / ((int64_t)R * P.H_kv))];
      b = sp.x;
      A = sp.y;
      r0 = sp.w;
      npiece = (int)(((A + sp.z) * NR - 1) / T - r0) + 1;
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float m = -INFINITY, l = 0.f;
    for (int e0 = wr; e0 < npiece; e0 += kMB * WPR) {
      float me[kMB], le[kMB];
      float4 va[kMB];
#pragma unroll
      for (int k = 0; k < kMB; ++k) {
        const int e = e0 + k * WPR;
        const int64_t rg = r0 + e, t0 = rg * T / NR;
        me[k] = -INFINITY;
        le[k] = 0.f;
        va[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (e < npiece && (rg + 1) * T / NR > t0) {   // an empty range wrote nothing
          const int64_t row = (2 * (rg * P.H_kv + g) + ((e == 0 && t0 < A) ? 1 : 0)) * R + r;
          me[k] = P.ws_ml[row * 2];
          le[k] = P.ws_ml[row * 2 + 1];
          va[k] = reinterpret_cast<const float4 *>(P.ws_acc + row * P.d)[lane];
        }
      }
      float mn = m;
#pragma unroll
      for (int k = 0; k < kMB; ++k) mn = fmaxf(mn, me[k]);
      const float base_m = mn == -INFINITY ? 0.f : mn;
      const float a = exp2f(m - base_m);
      l *= a;
      acc.x *= a; acc.y *= a; acc.z *= a; acc.w *= a;
#pragma unroll
      for (int k = 0; k < kMB; ++k) {
        const float w = exp2f(me[k] - base_m);
        l += le[k] * w;
        acc.x += va[k].x * w; acc.y += va[k].y * w; acc.z += va[k].z * w; acc.w += va[k].w * w;
      }
      m = mn;
    }
    if constexpr (WPR > 1) {
      xs_acc[warp][lane] = acc;
      if (lane == 0) { xs_ml[warp][0] = m; xs_ml[warp][1] = l; }
      __syncthreads();
      if (wr == 0) {
        for (int w2 = 1; w2 < WPR; ++w2) {
          const float me = xs_ml[warp + w2][0], le = xs_ml[warp + w2][1];
          const float mn = fmaxf(m, me);
          const float base_m = mn == -INFINITY ? 0.f : mn;
          const float a = exp2f(m - base_m), w = exp2f(me - base_m);
          l = l * a + le * w;
          m = mn;
          const float4 v = xs_acc[warp + w2][lane];
          acc.x = acc.x * a + v.x * w;
          acc.y = acc.y * a + v.y * w;
          acc.z = acc.z * a + v.z * w;
          acc.w = acc.w * a + v.w * w;
        }
      }
      __syncthreads();   // xs_* are free for the next round
    }
    if (!live || wr != 0) continue;
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int j = r / P.G, hh = r % P.G;
    const int64_t out_off = (((int64_t)b * P.n_new + j) * P.H_q + (int64_t)g * P.G + hh) * P.d;
    if constexpr (std::is_same<TO, float>::value) {
      reinterpret_cast<float4 *>(static_cast<float *>(P.out) + out_off)[lane] =
          make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    } else {
      __nv_bfloat16 *o = static_cast<__nv_bfloat16 *>(P.out) + out_off + 4 * lane;
      *reinterpret_cast<__nv_bfloat162 *>(o) = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
      *reinterpret_cast<__nv_bfloat162 *>(o + 2) = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    }
  }
}

int num_sms();

template <typename TO>
void launch_merge(const MergeParams &M, int64_t rows, cudaStream_t st) {
  if (M.C > 0) {
    // a split sequence spans about NR / B + 2 ranges when the lengths are
    // equal; the grid covers every row that could need a merge (at most
    // NR - 1 split sequences) up to four CTAs per SM
    const int64_t NR = M.C / M.H_kv;
    const int64_t est = NR / std::max<int64_t>(1, M.B) + 2;
    const int wpr = est >= 48 ? 8 : (est >= 24 ? 4 : (est >= 12 ? 2 : 1));
    const int64_t maxrows = std::max<int64_t>(1, (NR - 1) * M.H_kv * M.R);
    const unsigned nb = (unsigned)std::max<int64_t>(1, std::min<int64_t>(4 * num_sms(), (maxrows * wpr + 7) / 8));
    switch (wpr) {
      case 8: launch_k(attn_merge_bal_kernel<TO, 8>, dim3(nb), dim3(256), 0, st, 1, M); break;
      case 4: launch_k(attn_merge_bal_kernel<TO, 4>, dim3(nb), dim3(256), 0, st, 1, M); break;
      case 2: launch_k(attn_merge_bal_kernel<TO, 2>, dim3(nb), dim3(256), 0, st, 1, M); break;
      default: launch_k(attn_merge_bal_kernel<TO, 1>, dim3(nb), dim3(256), 0, st, 1, M); break;
    }
    return;
  }
  if (M.S <= 4) {
    launch_k(attn_merge_pair_kernel<TO>, dim3((unsigned)(M.B * M.H_kv)), dim3(32 * std::min(32, M.R)), 0, st, 1, M);
    return;
  }
  // more warps per row when there are many splits (a warp loads up to 8
  // pieces in one round trip; at 38 splits 4 warps measured 91 us for the
  // 128K-context call against 92 and 97 us with 2 and 8)
  const int wpr = M.S >= 64 ? 8 : (M.S >= 16 ? 4 : (M.S >= 8 ? 2 : 1));
  const unsigned nb = (unsigned)((rows * wpr + 7) / 8);
  switch (wpr) {
    case 8: launch_k(attn_merge_kernel<TO, 8>, dim3(nb), dim3(256), 0, st, 1, M); break;
    case 4: launch_k(attn_merge_kernel<TO, 4>, dim3(nb), dim3(256), 0, st, 1, M); break;
    case 2: launch_k(attn_merge_kernel<TO, 2>, dim3(nb), dim3(256), 0, st, 1, M); break;
    default: launch_k(attn_merge_kernel<TO, 1>, dim3(nb), dim3(256), 0, st, 1, M); break;
  }
}

// ------------------------------------------------------------------ host ---

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

struct Plan {
  bool tc;
  int R, S, bps, per_split, d;
  int C;   // balanced mode (tcgen05 kernel, no explicit split size): CTAs; 0 otherwise
};

int num_sms() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 148;
  });
  return n;
}

int pow2_floor(int64_t x) {
  int p = 1;
  while ((int64_t)p * 2 <= x) p *= 2;
  return p;
}

// Split size (blocks per CTA): large enough that the fp32 partials a split
// writes stay within ~4 % of the KV bytes it reads, small enough that there
// are at least four waves of CTAs when the batch allows it.
Plan make_plan(int B, int n_new, int H_q, int H_kv, int d, int max_blocks, int bs, sv_dtype kv, sv_dtype qd,
               const sv_kv_layout *lay, int bps_req) {
  Plan p;
  p.R = n_new * (H_q / H_kv);
  p.d = d;
  const int es = dtype_bytes(kv);
  bool strides_ok = true;
  if (lay)
    strides_ok = (lay->block_stride * es) % 16 == 0 && (lay->head_stride * es) % 16 == 0 &&
                 (lay->slot_stride * es) % 16 == 0;
  p.tc = (kv == SV_BF16 || kv == SV_FP8_E4M3) && qd == SV_BF16 && d == kD && bs == kBS && p.R <= kT5MaxR &&
         strides_ok;
  p.C = 0;
  const int64_t pairs = (int64_t)B * H_kv, slots = 2 * num_sms();
  if (bps_req > 0) {
    p.bps = bps_req;
  } else if (bps_req < 0 && p.tc && (int64_t)std::max(B, 1) * ((max_blocks + kT5Blk - 1) / kT5Blk) < (1ll << 30)) {
    // balanced mode (asked for): ranges of tiles for all kv heads side by
    // side, about two CTAs per SM (what the shared memory and TMEM of one CTA
    // leave room for), each taking an equal share of all tiles
    const int64_t tiles = (int64_t)std::max(B, 1) * ((max_blocks + kT5Blk - 1) / kT5Blk);
    const int64_t nr = std::max<int64_t>(1, std::min<int64_t>(slots / H_kv, tiles));
    p.C = (int)(nr * H_kv);
    p.bps = 0;
    p.S = 1;
    p.per_split = 1;
    return p;
  } else if (p.tc) {
    // split mode on the tensor cores. With at least as many (sequence, kv
    // head) pairs as CTA slots (two per SM), one split per pair up to 512
    // blocks: the longest-first order balances the slots and no merge runs.
    // With fewer pairs, floor(slots / pairs) splits per pair, so the CTAs of
    // equal-length sequences fill the slots once (a block count that is a
    // multiple of 4 keeps the 64-key tiles whole).
    if (pairs >= slots) {
      p.bps = std::min(max_blocks, 512);
    } else {
      const int64_t per = std::max<int64_t>(1, slots / std::max<int64_t>(1, pairs));
      int bps = (int)((max_blocks + per - 1) / per);
      bps = std::min(512, (bps + 3) / 4 * 4);
      p.bps = std::max(4, bps);
    }
  } else {
    // fp32 caches are planned like bf16 ones so every dtype fits the same
    // workspace
    const double kv_per_block = 2.0 * bs * d * (kv == SV_FP8_E4M3 ? 1 : 2);
    const double partial = (double)p.R * (d + 2) * 4;
    const int min_bps = std::min(512, std::max(16, 2 * pow2_floor((int64_t)(partial / (0.04 * kv_per_block)))));
    const int max_bps = std::max(16, pow2_floor((int64_t)max_blocks * B * H_kv / (4 * num_sms())));
    p.bps = std::min(min_bps, max_bps);
  }
  p.S = (max_blocks + p.bps - 1) / p.bps;
  p.per_split = 1;
  return p;
}

// Partial entries: split mode one per split, balanced mode two per CTA.
size_t ws_entries(const Plan &p, int B, int H_kv) {
  return p.C > 0 ? (size_t)2 * p.C : (size_t)B * H_kv * p.S * p.per_split;
}

// partials (acc, then m and l), then the work order (split mode) or the
// per-CTA work and sequence prefixes (balanced mode)
size_t ws_bytes(const Plan &p, int B, int H_kv) {
  const size_t ent = ws_entries(p, B, H_kv) * p.R;
  const size_t tail = p.C > 0 ? align_up((size_t)p.C * sizeof(int4), 256) + align_up((size_t)(B + 1) * sizeof(int32_t), 256) +
                                   align_up((size_t)(p.C / H_kv + 1) * sizeof(int4), 256)
                              : align_up((size_t)B * H_kv * p.S * sizeof(int32_t), 256);
  return align_up(ent * p.d * sizeof(float), 256) + align_up(ent * 2 * sizeof(float), 256) + tail;
}

// Ancestor masks of the draft trees: bit i of anc[b][j] is set iff node i is
// node j or one of its ancestors ("KV Cache + Speculative Decoding", Q14 and
// section 8.2: tree nodes flattened in BFS order, mask M[j][i] = 1 iff i is
// in A(j), the ancestors of j including j). One CTA per sequence, one thread
// per node; parents are checked (node 0 the root with parent -1, else
// 0 <= parent[j] < j, which BFS order guarantees), and a node with a bad
// parent gets the chain mask of its position and sets SV_DEV_BAD_TREE.
__global__ void __launch_bounds__(64) attn_tree_kernel(const int32_t *parent, int n_new, uint64_t *anc,
                                                       int32_t *status) {
  pdl_wait();
  pdl_trigger();
  __shared__ int par[64];
  const int b = blockIdx.x, j = threadIdx.x;
  if (j < n_new) par[j] = __ldg(parent + (int64_t)b * n_new + j);
  __syncthreads();
  if (j >= n_new) return;
  bool ok = true;
  for (int i = 0; i <= j; ++i) ok &= (i == 0) ? par[0] == -1 : (par[i] >= 0 && par[i] < i);
  uint64_t m = 1ull << j;
  if (ok) {
    for (int p = par[j]; p >= 0; p = par[p]) m |= 1ull << p;   // strictly decreasing: at most j steps
  } else {
    m = (j == 63) ? ~0ull : ((1ull << (j + 1)) - 1ull);
    atomic_or_status(status, SV_DEV_BAD_TREE);
  }
  anc[(int64_t)b * n_new + j] = m;
}

template <int QR, bool FP8>
sv_status launch_tc5(const TcParams &P0, cudaStream_t st) {
  using Cfg = T5Cfg<QR, FP8>;
  TcParams P = P0;
  P.tblk = Cfg::kBlk;   // the partition counts this kernel's tiles
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_tc5_kernel<QR, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmem);
    if (attr_err == cudaSuccess)
      attr_err = cudaFuncSetAttribute(attn_tc5_bal_kernel<QR, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      Cfg::kSmem);
  });
  if (attr_err != cudaSuccess)
    return fail(SV_ERR_CUDA, "spec_verify_attn: cudaFuncSetAttribute: %s", cudaGetErrorString(attr_err));
  unsigned grid;
  if (P.balanced) {
    launch_k(attn_part_kernel, dim3(1), dim3(kPartThreads), 0, st, 1, P.seq_lens, P.B, P.n_new, P.max_blocks,
             P.tblk, P.ncta / P.H_kv, const_cast<int4 *>(P.work), P.seq_pre_w, P.split_w, P.status);
    grid = (unsigned)P.ncta;
  } else {
    grid = (unsigned)(P.S * P.H_kv * P.B);
    // Longest-first dispatch matters only when the CTAs take more than one
    // wave of the slots (two per SM); a grid that fits runs all its CTAs at
    // once, so it takes item = blockIdx.x and the order kernel (and its
    // latency before the first tile) is left out.
    if ((int64_t)grid <= 2 * (int64_t)num_sms()) {
      P.order = nullptr;
    } else {
      launch_k(attn_order_kernel, dim3(1), dim3(kOrdThreads), 0, st, 1, P.seq_lens, P.B, P.S, P.H_kv, P.bps, P.n_new,
               P.max_blocks, const_cast<int32_t *>(P.order));
    }
  }
  sv_status rc = check_launch("spec_verify_attn order launch");
  if (rc != SV_OK) return rc;
  if (P.balanced) launch_k(attn_tc5_bal_kernel<QR, FP8>, dim3(grid), dim3(Cfg::kThreads), Cfg::kSmem, st, 1, P);
  else launch_k(attn_tc5_kernel<QR, FP8>, dim3(grid), dim3(Cfg::kThreads), Cfg::kSmem, st, 1, P);
  return check_launch("spec_verify_attn tcgen05 launch");
}

template <typename TKV, typename TQ>
sv_status launch_gen(const GenParams &P, cudaStream_t st) {
  const size_t smem = sizeof(float) * ((size_t)2 * P.R * P.d + 2 * kGenKeys * P.d + (size_t)P.R * kGenKeys + 3 * P.R);
  if (smem > 200 * 1024) return fail(SV_ERR_UNSUPPORTED, "spec_verify_attn: (K+1)*G*d_head too large for the fp32 path");
  cudaError_t e = cudaFuncSetAttribute(attn_generic_kernel<TKV, TQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_attn: cudaFuncSetAttribute: %s", cudaGetErrorString(e));
  dim3 grid(P.S, P.H_kv, P.B);
  launch_k(attn_generic_kernel<TKV, TQ>, grid, dim3(kGenThreads), smem, st, 1, P);
  return check_launch("spec_verify_attn fp32 launch");
}

}  // namespace
}  // namespace sv

using namespace sv;

static sv_status attn_impl(const void *q, sv_dtype q_dtype, const void *k_cache, const void *v_cache,
                           sv_dtype kv_dtype, const sv_kv_layout *layout, const float *k_scale,
                           const float *v_scale, const int32_t *block_table, int max_blocks_per_seq,
                           const int32_t *seq_lens, int B, int n_new, int H_q, int H_kv, int d_head,
                           int block_size, int num_blocks, float softmax_scale, void *out, sv_dtype out_dtype,
                           void *workspace, size_t workspace_bytes, int32_t *dev_status, int bps_req,
                           const int32_t *tree_parent, sv_stream_t stream) {
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out)
    return fail(SV_ERR_INVALID_ARG, "spec_verify_attn: null pointer argument");
  if (tree_parent && n_new > 64)
    return fail(SV_ERR_UNSUPPORTED, "spec_verify_attn_tree: at most 64 tree nodes (n_new = %d)", n_new);
  if (B < 0 || n_new < 1 || H_q < 1 || H_kv < 1 || d_head < 1 || block_size < 1 || num_blocks < 1 ||
      max_blocks_per_seq < 1)
    return fail(SV_ERR_INVALID_ARG, "spec_verify_attn: bad sizes");
  if (H_q % H_kv != 0) return fail(SV_ERR_INVALID_ARG, "spec_verify_attn: H_q %% H_kv != 0");
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale))
    return fail(SV_ERR_INVALID_ARG, "spec_verify_attn: softmax_scale must be finite and > 0");
  if (q_dtype != out_dtype) return fail(SV_ERR_UNSUPPORTED, "spec_verify_attn: q and out dtypes must match");
  if (kv_dtype == SV_F32 && q_dtype != SV_F32)
    return fail(SV_ERR_UNSUPPORTED, "spec_verify_attn: fp32 caches take fp32 queries");
  if ((kv_dtype == SV_BF16 || kv_dtype == SV_FP8_E4M3) && q_dtype != SV_BF16)
    return fail(SV_ERR_UNSUPPORTED, "spec_verify_attn: bf16 / fp8 caches take bf16 queries");
  if (kv_dtype == SV_F16) return fail(SV_ERR_UNSUPPORTED, "spec_verify_attn: f16 caches are not supported");
  if (kv_dtype == SV_FP8_E4M3 && (!k_scale || !v_scale))
    return fail(SV_ERR_INVALID_ARG, "spec_verify_attn: fp8 caches need k_scale and v_scale");
  if (d_head > 256 || d_head % 4) return fail(SV_ERR_UNSUPPORTED, "spec_verify_attn: d_head must be a multiple of 4 and <= 256");
  if (B > 65535 || H_kv > 65535) return fail(SV_ERR_UNSUPPORTED, "spec_verify_attn: B or H_kv too large");
  if (layout && (layout->slot_stride < d_head || layout->head_stride < d_head || layout->block_stride < d_head))
    return fail(SV_ERR_INVALID_ARG, "spec_verify_attn: layout strides smaller than d_head");
  const Plan plan = make_plan(B, n_new, H_q, H_kv, d_head, max_blocks_per_seq, block_size, kv_dtype, q_dtype,
                              layout, bps_req);
  if (plan.R > 65535) return fail(SV_ERR_UNSUPPORTED, "spec_verify_attn: too many query rows per kv head");
  const size_t base_need = ws_bytes(plan, B, H_kv);
  const size_t need = base_need + (tree_parent ? align_up((size_t)B * n_new * sizeof(uint64_t), 256) : 0);
  if (!workspace || workspace_bytes < need)
    return fail(SV_ERR_WORKSPACE, "spec_verify_attn: workspace needs %zu bytes", need);
  if (!aligned(workspace, 256)) return fail(SV_ERR_WORKSPACE, "spec_verify_attn: workspace not 256-byte aligned");
  if (B == 0) return ok();

  const size_t ent = ws_entries(plan, B, H_kv) * plan.R;
  float *ws_acc = static_cast<float *>(workspace);
  float *ws_ml = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) +
                                           align_up(ent * d_head * sizeof(float), 256));
  const int G = H_q / H_kv;
  int64_t slot_stride = d_head, head_stride = (int64_t)block_size * d_head,
          block_stride = (int64_t)H_kv * block_size * d_head;
  if (layout) {
    slot_stride = layout->slot_stride;
    head_stride = layout->head_stride;
    block_stride = layout->block_stride;
  }
  const float scale_log2 = (float)((double)softmax_scale * 1.4426950408889634074);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  sv_status rc;
  uint64_t *anc = nullptr;
  if (tree_parent) {
    anc = reinterpret_cast<uint64_t *>(static_cast<uint8_t *>(workspace) + base_need);
    launch_k(attn_tree_kernel, dim3(B), dim3(64), 0, st, 1, tree_parent, n_new, anc, dev_status);
    rc = check_launch("spec_verify_attn_tree ancestor launch");
    if (rc != SV_OK) return rc;
  }
  if (plan.tc) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode();
    if (!enc) return fail(SV_ERR_CUDA, "spec_verify_attn: cuTensorMapEncodeTiled unavailable");
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16))
      return fail(SV_ERR_INVALID_ARG, "spec_verify_attn: cache pointers must be 16-byte aligned");
    TcParams P;
    memset(&P, 0, sizeof(P));
    const bool fp8 = kv_dtype == SV_FP8_E4M3;
    const int es = fp8 ? 1 : 2;
    // outer dims ordered by increasing stride; the box is 16 slots x 1 x 1,
    // so a tile always lands as 16 rows of d_head elements
    const int64_t st_of[3] = {slot_stride, head_stride, block_stride};
    const int64_t ext_of[3] = {block_size, H_kv, num_blocks};
    int order[3] = {0, 1, 2};
    std::sort(order, order + 3, [&](int x, int y) { return st_of[x] < st_of[y]; });
    cuuint64_t dims[4] = {(cuuint64_t)d_head, 0, 0, 0};
    cuuint64_t strides[3];
    cuuint32_t box[4] = {(cuuint32_t)(fp8 ? 128 : 64), 1, 1, 1};
    for (int k = 0; k < 3; ++k) {
      dims[k + 1] = (cuuint64_t)ext_of[order[k]];
      strides[k] = (cuuint64_t)(st_of[order[k]] * es);
      box[k + 1] = order[k] == 0 ? (cuuint32_t)block_size : 1u;
      P.role[k] = order[k];
    }
    cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    for (int w = 0; w < 2; ++w) {
      CUresult r = enc(w ? &P.tmv : &P.tmk, dt, 4, const_cast<void *>(w ? v_cache : k_cache), dims, strides, box,
                       estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
      if (r != CUDA_SUCCESS) return fail(SV_ERR_INVALID_ARG, "spec_verify_attn: cuTensorMapEncodeTiled failed (%d)", (int)r);
    }
    // the softmax warps read their Q rows with 16-byte loads
    if (!aligned(q, 16)) return fail(SV_ERR_INVALID_ARG, "spec_verify_attn: q must be 16-byte aligned");
    P.q = q; P.out = out; P.k_scale = k_scale; P.v_scale = v_scale; P.block_table = block_table; P.seq_lens = seq_lens;
    P.ws_acc = ws_acc; P.ws_ml = ws_ml; P.status = dev_status; P.anc = anc;
    uint8_t *tail = reinterpret_cast<uint8_t *>(ws_ml) + align_up(ent * 2 * sizeof(float), 256);
    P.order = reinterpret_cast<const int32_t *>(tail);
    if (plan.C > 0) {
      P.balanced = 1;
      P.ncta = plan.C;
      P.work = reinterpret_cast<const int4 *>(tail);
      P.seq_pre_w = reinterpret_cast<int32_t *>(tail + align_up((size_t)plan.C * sizeof(int4), 256));
      P.split_w = reinterpret_cast<int4 *>(reinterpret_cast<uint8_t *>(P.seq_pre_w) +
                                           align_up((size_t)(B + 1) * sizeof(int32_t), 256));
    }
    P.B = B; P.n_new = n_new; P.H_q = H_q; P.H_kv = H_kv; P.G = G; P.R = plan.R;
    P.max_blocks = max_blocks_per_seq; P.num_blocks = num_blocks; P.bps = plan.bps; P.S = plan.S;
    P.scale_log2 = scale_log2;
    P.wait_ns = wait_limit_ns();
    P.withhold = test_withhold();
    if (!fp8) rc = plan.R <= 64 ? launch_tc5<64, false>(P, st) : launch_tc5<128, false>(P, st);
    else rc = plan.R <= 64 ? launch_tc5<64, true>(P, st) : launch_tc5<128, true>(P, st);
  } else {
    GenParams P;
    P.q = q; P.out = out; P.k_cache = k_cache; P.v_cache = v_cache; P.k_scale = k_scale; P.v_scale = v_scale;
    P.block_table = block_table; P.seq_lens = seq_lens; P.ws_acc = ws_acc; P.ws_ml = ws_ml; P.status = dev_status;
    P.anc = anc;
    P.B = B; P.n_new = n_new; P.H_q = H_q; P.H_kv = H_kv; P.G = G; P.R = plan.R; P.d = d_head; P.bs = block_size;
    P.max_blocks = max_blocks_per_seq; P.num_blocks = num_blocks; P.bps = plan.bps; P.S = plan.S;
    P.block_stride = block_stride; P.head_stride = head_stride; P.slot_stride = slot_stride;
    P.scale_log2 = scale_log2;
    if (kv_dtype == SV_F32) rc = launch_gen<float, float>(P, st);
    else if (kv_dtype == SV_BF16) rc = launch_gen<__nv_bfloat16, __nv_bfloat16>(P, st);
    else rc = launch_gen<uint8_t, __nv_bfloat16>(P, st);
  }
  if (rc != SV_OK) return rc;
  // every sequence was written directly: one range, or one split
  if ((plan.C > 0 && plan.C / H_kv == 1) || (plan.C == 0 && plan.S == 1)) return ok();
  MergeParams M;
  memset(&M, 0, sizeof(M));
  if (plan.C > 0) {
    M.C = plan.C;
    M.seq_pre = reinterpret_cast<const int32_t *>(reinterpret_cast<uint8_t *>(ws_ml) +
                                                  align_up(ent * 2 * sizeof(float), 256) +
                                                  align_up((size_t)plan.C * sizeof(int4), 256));
    M.split = reinterpret_cast<const int4 *>(reinterpret_cast<const uint8_t *>(M.seq_pre) +
                                             align_up((size_t)(B + 1) * sizeof(int32_t), 256));
  }
  M.ws_acc = ws_acc; M.ws_ml = ws_ml; M.seq_lens = seq_lens; M.out = out;
  M.B = B; M.n_new = n_new; M.H_q = H_q; M.H_kv = H_kv; M.G = G; M.R = plan.R; M.d = d_head; M.bs = block_size;
  M.max_blocks = max_blocks_per_seq; M.bps = plan.bps; M.S = plan.S; M.per_split = plan.per_split;
  const int64_t rows = (int64_t)B * H_kv * plan.R;
  if (out_dtype == SV_F32) launch_merge<float>(M, rows, st);
  else launch_merge<__nv_bfloat16>(M, rows, st);
  return check_launch("spec_verify_attn merge launch");
}

// The plan depends on the cache dtype; size for the largest of them.
static size_t ws_bytes_any(int B, int n_new, int H_q, int H_kv, int d_head, int max_blocks_per_seq,
                           int block_size, int bps) {
  size_t best = 0;
  const sv_dtype kvs[3] = {SV_BF16, SV_FP8_E4M3, SV_F32};
  for (sv_dtype kv : kvs) {
    const sv_dtype qd = kv == SV_F32 ? SV_F32 : SV_BF16;
    Plan p = make_plan(B, n_new, H_q, H_kv, d_head, max_blocks_per_seq, block_size, kv, qd, nullptr, bps);
    best = std::max(best, ws_bytes(p, B, H_kv));
  }
  return best;
}

extern "C" size_t spec_verify_attn_workspace_size(int B, int n_new, int H_q, int H_kv, int d_head,
                                                  int max_blocks_per_seq, int block_size) {
  if (B < 0 || n_new < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv || d_head < 1 || max_blocks_per_seq < 1)
    return 0;
  return ws_bytes_any(B, n_new, H_q, H_kv, d_head, max_blocks_per_seq, block_size, 0);
}

extern "C" size_t spec_verify_attn_workspace_size_ex(int B, int n_new, int H_q, int H_kv, int d_head,
                                                     int max_blocks_per_seq, int block_size,
                                                     int blocks_per_split) {
  if (B < 0 || n_new < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv || d_head < 1 || max_blocks_per_seq < 1)
    return 0;
  if (blocks_per_split < 0) return 0;
  return ws_bytes_any(B, n_new, H_q, H_kv, d_head, max_blocks_per_seq, block_size,
                      blocks_per_split == 0 ? -1 : blocks_per_split);
}

extern "C" sv_status spec_verify_attn(const void *q, sv_dtype q_dtype, const void *k_cache, const void *v_cache,
                                      sv_dtype kv_dtype, const sv_kv_layout *layout, const float *k_scale,
                                      const float *v_scale, const int32_t *block_table, int max_blocks_per_seq,
                                      const int32_t *seq_lens, int B, int n_new, int H_q, int H_kv, int d_head,
                                      int block_size, int num_blocks, float softmax_scale, void *out,
                                      sv_dtype out_dtype, void *workspace, size_t workspace_bytes,
                                      int32_t *dev_status, sv_stream_t stream) {
  return attn_impl(q, q_dtype, k_cache, v_cache, kv_dtype, layout, k_scale, v_scale, block_table,
                   max_blocks_per_seq, seq_lens, B, n_new, H_q, H_kv, d_head, block_size, num_blocks,
                   softmax_scale, out, out_dtype, workspace, workspace_bytes, dev_status, 0, nullptr, stream);
}

extern "C" sv_status spec_verify_attn_ex(const void *q, sv_dtype q_dtype, const void *k_cache,
                                         const void *v_cache, sv_dtype kv_dtype, const sv_kv_layout *layout,
                                         const float *k_scale, const float *v_scale, const int32_t *block_table,
                                         int max_blocks_per_seq, const int32_t *seq_lens, int B, int n_new,
                                         int H_q, int H_kv, int d_head, int block_size, int num_blocks,
                                         float softmax_scale, void *out, sv_dtype out_dtype, void *workspace,
                                         size_t workspace_bytes, int32_t *dev_status, int blocks_per_split,
                                         sv_stream_t stream) {
  if (blocks_per_split < 0) return fail(SV_ERR_INVALID_ARG, "spec_verify_attn_ex: blocks_per_split < 0");
  return attn_impl(q, q_dtype, k_cache, v_cache, kv_dtype, layout, k_scale, v_scale, block_table,
                   max_blocks_per_seq, seq_lens, B, n_new, H_q, H_kv, d_head, block_size, num_blocks,
                   softmax_scale, out, out_dtype, workspace, workspace_bytes, dev_status,
                   blocks_per_split == 0 ? -1 : blocks_per_split, nullptr, stream);
}

extern "C" size_t spec_verify_attn_tree_workspace_size(int B, int n_new, int H_q, int H_kv, int d_head,
                                                       int max_blocks_per_seq, int block_size) {
  const size_t base = spec_verify_attn_workspace_size(B, n_new, H_q, H_kv, d_head, max_blocks_per_seq, block_size);
  if (base == 0 && B > 0) return 0;
  return base + align_up((size_t)B * n_new * sizeof(uint64_t), 256);
}

extern "C" sv_status spec_verify_attn_tree(const void *q, sv_dtype q_dtype, const void *k_cache, const void *v_cache,
                                           sv_dtype kv_dtype, const sv_kv_layout *layout, const float *k_scale,
                                           const float *v_scale, const int32_t *block_table,
                                           int max_blocks_per_seq, const int32_t *seq_lens,
                                           const int32_t *tree_parent, int B, int n_new, int H_q, int H_kv,
                                           int d_head, int block_size, int num_blocks, float softmax_scale,
                                           void *out, sv_dtype out_dtype, void *workspace,
                                           size_t workspace_bytes, int32_t *dev_status, sv_stream_t stream) {
  if (!tree_parent) return fail(SV_ERR_INVALID_ARG, "spec_verify_attn_tree: tree_parent is NULL");
  return attn_impl(q, q_dtype, k_cache, v_cache, kv_dtype, layout, k_scale, v_scale, block_table,
                   max_blocks_per_seq, seq_lens, B, n_new, H_q, H_kv, d_head, block_size, num_blocks,
                   softmax_scale, out, out_dtype, workspace, workspace_bytes, dev_status, 0, tree_parent, stream);
}

// Paged MLA verify attention in the absorbed form, and the latent append
// ("KV Cache + Speculative Decoding", sections 4.3-4.4 and 6.3). Each token
// caches one row [c ; k^R] of d_c + d_r = 512 + 64 bf16 values, shared by all
// heads. Query row (position j, head i) is q_lat = [W_UK[i]^T q^C ; q^R]. Its
// score against a cached row is q_lat . row * scale, under the verify causal
// mask. Its output is the latent sum_s w_s c_s (d_c = 512 values), which the
// caller multiplies by W_UV[i] or folds into the output projection.
//
// With 128 heads a sequence has (K+1) * 128 query rows against one shared
// row per token: about 1200 multiply-adds per cached byte, so the kernel is
// bound by the tensor cores, not by HBM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "sv_common.cuh"

namespace sv {
namespace {

constexpr int kLD = 576;                           // cached row: d_c + d_r
constexpr int kLC = 512;                           // d_c: the value part of a row
constexpr int kLR = kLD - kLC;                     // d_r
constexpr int kLChunks = kLD / 64;                 // 64-wide chunks (one 128-byte swizzle span each)
constexpr int kLHalf = kLC / 2;                    // output columns per CTA
constexpr int kLBS = 16;                           // block size
constexpr int kLQChunkBytes = 128 * 128;           // 128 query rows x 64 values
constexpr int kLThreads = 192;
constexpr int kLProdWarp = 4;
constexpr int kLMmaWarp = 5;
constexpr uint32_t kLCols = 512;                   // TMEM columns

// Tile geometry for NK keys per tile. TMEM holds two S/P buffers of NK
// columns, the 256-column output half and as many Q chunks (32 columns of
// bf16 pairs each) as fit; the other Q chunks and the ring of NK-key stages
// share the shared memory.
template <int NK> struct MlaCfg {
  static constexpr int kBlk = NK / kLBS;                      // blocks per tile
  static constexpr int kChunkBytes = NK * 128;                // one 64-wide chunk of a tile
  static constexpr int kTileBytes = kLChunks * kChunkBytes;
  static constexpr uint32_t kOCol = 2 * NK;
  static constexpr uint32_t kQCol = kOCol + kLHalf;
  static constexpr int kQTm = (int)(kLCols - kQCol) / 32;     // Q chunks in TMEM
  static constexpr int kQSm = kLChunks - kQTm;                // Q chunks in shared memory
  static constexpr int kStages = (227 * 1024 - 1024 - 256 - kQSm * kLQChunkBytes) / kTileBytes;
  static constexpr int kSmem = 1024 + kQSm * kLQChunkBytes + kStages * kTileBytes;
  static_assert(kQCol + 32 * kQTm <= kLCols, "TMEM budget");
  static_assert(kStages >= 2, "at least two stages");
  static_assert(NK % 16 == 0 && NK <= 256, "MMA N");
};
constexpr int kLNK = 64;                           // keys per tile of the launched kernel
constexpr int kLCtaTarget = 2 * 152;               // CTAs that fill the GPU twice over
constexpr int kLMinBlocksPerSplit = 16;

struct MlaParams {   // 64-byte aligned through its CUtensorMap members
  CUtensorMap tmc;   // cache [num_blocks][16][576] bf16: box 64 values x 16 slots x 1 block
  CUtensorMap tmq;   // q [B][R][576] bf16: box 64 values x q_box rows x 1
  const __nv_bfloat16 *q;
  __nv_bfloat16 *out;   // [B][R][512]
  float *ws_acc;        // [B][S][R][512] unnormalised partial outputs
  float *ws_ml;         // [B][S][R][2]   (reference max in log2 units, sum)
  const int32_t *block_table;
  const int32_t *seq_lens;
  const int32_t *order;   // sequences longest first (NULL: batch order)
  int32_t *status;
  int B, n_new, H, R, n_mt, max_blocks, num_blocks, bps, S, q_box;
  float scale_log2;
};

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1, int c2,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// shared-memory matrix descriptor, 128-byte swizzle, sm_100-family version
__device__ __forceinline__ uint64_t ml_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFF);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

__device__ __forceinline__ void ml_mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
               "l"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void ml_mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
               "r"(a), "l"(b), "r"(idesc), "r"(acc));
}

__device__ __forceinline__ void ml_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void ml_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void ml_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void ml_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}

__device__ __forceinline__ void ml_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void ml_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void ml_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ bool ml_test(uint64_t *bar, uint32_t phase) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(phase)
      : "memory");
  return done != 0;
}

// bounded wait that gives up at once after any earlier wait of the CTA gave up
__device__ __forceinline__ bool ml_wait(uint64_t *bar, uint32_t phase, volatile int *abort_flag) {
  if (*abort_flag) return false;
  if (mbar_wait(bar, phase)) return true;
  *abort_flag = 1;
  return false;
}

__device__ __forceinline__ float ml_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t ml_pack_bf16(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// CTA = (output half hv, row tile mt, split s) x sequence b; 192 threads.
// The numbers below are for the launched NK = 64 (two stages; Q chunks 0-3
// in TMEM, 4-8 in shared memory).
//   warps 0-3  softmax: thread t owns query row 128 mt + t (TMEM lane t);
//              they first write their rows' TMEM chunks of Q
//   warp 4     TMA producer: the shared-memory chunks of Q for the row tile,
//              then the ring of NK-key tiles (every chunk of every row: keys
//              and values are the same cached rows)
//   warp 5     TMEM owner; lane 0 issues the MMAs from a polling loop
// Per tile t, buffer u = t % 2:
//   S[u] = Q K^T        M=128 rows, N=NK keys, K=576 (36 MMAs of K=16)
//   P[u] = 2^(S c - m)  bf16 over the first NK/2 columns of S[u]
//   O   += P V          M=128, N=256 values of half hv, K=16 keys per MMA
// A ring stage is free again once the P V of its tile has run. Both output
// halves compute the same S: the 128 x 512 fp32 output and an S tile do not
// fit in one CTA's 512 TMEM columns.
template <int NK>
__global__ void __launch_bounds__(kLThreads, 1) attn_mla_kernel(const __grid_constant__ MlaParams P) {
  pdl_wait();
  pdl_trigger();
  using Cfg = MlaCfg<NK>;
  constexpr int kLN = NK, kLStages = Cfg::kStages, kLChunkBytes = Cfg::kChunkBytes, kLTileBytes = Cfg::kTileBytes;
  constexpr int kLQTm = Cfg::kQTm, kLQSm = Cfg::kQSm, kBlk = Cfg::kBlk;
  constexpr uint32_t kLOCol = Cfg::kOCol, kLQCol = Cfg::kQCol;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t kv_full[kLStages], kv_empty[kLStages];
  __shared__ __align__(8) uint64_t s_full[2], p_full[2], o_done[2], q_tm, q_sm, mma_drain;
  __shared__ uint32_t tmem_base;
  __shared__ int abort_flag;

  const int hv = blockIdx.x & 1;
  const int mt = (blockIdx.x >> 1) % P.n_mt;
  const int s = (blockIdx.x >> 1) / P.n_mt;
  const int b = P.order ? P.order[blockIdx.y] : (int)blockIdx.y;   // written by the order kernel
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t q_smem = smem_u32(smem);
  const uint32_t ring = q_smem + kLQSm * kLQChunkBytes;

  if (b < 0 || b >= (int)gridDim.y) {   // (both CTAs of a pair share blockIdx.y)
    if (tid == 0) atomic_or_status(P.status, SV_DEV_BAD_WORK);
    return;
  }
  const int L = P.seq_lens[b];
  if (L < P.n_new || L > P.max_blocks * kLBS) {
    if (tid == 0 && blockIdx.x == 0) atomic_or_status(P.status, SV_DEV_BAD_SEQ_LEN);
    return;
  }
  const int nblk = (L + kLBS - 1) / kLBS;
  const int blk0 = s * P.bps;
  if (blk0 >= nblk) return;   // the merge never reads this split
  const int blk1 = min(nblk, blk0 + P.bps);
  const int nblocks = blk1 - blk0;
  const int n_tiles = (nblocks + kBlk - 1) / kBlk;

  if (tid == 0) {
    for (int k = 0; k < kLStages; ++k) {
      mbar_init(&kv_full[k], 1);
      mbar_init(&kv_empty[k], 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&s_full[k], 1);
      mbar_init(&p_full[k], 4);
      mbar_init(&o_done[k], 1);
    }
    mbar_init(&q_tm, 4);
    mbar_init(&q_sm, 1);
    mbar_init(&mma_drain, 1);
    abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  volatile int *abf = &abort_flag;

  if (warp == kLProdWarp) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      mbar_arrive_expect_tx(&q_sm, (uint32_t)(kLQSm * P.q_box * 128));
      for (int c = 0; c < kLQSm; ++c)
        tma_load_3d(q_smem + c * kLQChunkBytes, &P.tmq, (kLQTm + c) * 64, mt * 128, b, &q_sm);
    }
    // the warp walks the block table 32 entries at a time (the next 32
    // prefetched); lane 0 waits for free stages and issues the copies
    const int32_t *table = P.block_table + (int64_t)b * P.max_blocks + blk0;
    int cur = lane < nblocks ? table[lane] : 0;
    int nxt = 32 + lane < nblocks ? table[32 + lane] : 0;
    int chunk = 0, issued = 0;
    for (int t = 0; t < n_tiles; ++t) {
      const int first = kBlk * t;
      if ((first >> 5) != chunk) {
        chunk = first >> 5;
        cur = nxt;
        const int rel = (chunk + 1) * 32 + lane;
        nxt = rel < nblocks ? table[rel] : 0;
      }
      int phys[kBlk];
#pragma unroll
      for (int kk = 0; kk < kBlk; ++kk) phys[kk] = __shfl_sync(0xffffffffu, cur, (first + kk) & 31);
      const int st = t % kLStages;
      bool go = true;
      if (lane == 0) {
        if (t >= kLStages && !ml_wait(&kv_empty[st], ((t / kLStages) & 1) ^ 1, abf)) {
          go = false;
        } else {
          const int nvalid = min(kBlk, nblocks - first);
          mbar_arrive_expect_tx(&kv_full[st], (uint32_t)(nvalid * kLChunks * 2048));
          const uint32_t base = ring + st * kLTileBytes;
          for (int kk = 0; kk < nvalid; ++kk) {
            int ph = phys[kk];
            if (ph < 0 || ph >= P.num_blocks) {
              atomic_or_status(P.status, SV_DEV_BAD_BLOCK);
              ph = 0;   // stay in bounds; the output of this sequence is flagged
            }
            for (int c = 0; c < kLChunks; ++c)
              tma_load_3d(base + c * kLChunkBytes + kk * 2048, &P.tmc, c * 64, 0, ph, &kv_full[st]);
          }
          issued = t + 1;
        }
      }
      if (!__shfl_sync(0xffffffffu, (int)go, 0)) break;
    }
    // the copies in flight land before the CTA may exit
    if (lane == 0) {
      if (!mbar_wait(&q_sm, 0)) atomic_or_status(P.status, SV_DEV_TIMEOUT);
      for (int t = max(0, issued - kLStages); t < issued; ++t)
        if (!mbar_wait(&kv_full[t % kLStages], (t / kLStages) & 1)) atomic_or_status(P.status, SV_DEV_TIMEOUT);
    }
  } else {
    if (warp == kLMmaWarp) {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)),
                   "r"(kLCols));
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    ml_fence_before();
    named_sync(1, 160);   // TMEM allocated
    ml_fence_after();
    const uint32_t tb = tmem_base;

    if (warp == kLMmaWarp) {
      // ---------------------------------------------------------- MMA issuer --
      if (lane == 0) {
        // f32 accumulate, bf16 A and B, N >> 3 at bit 17, M >> 4 at bit 24;
        // P V reads B (the values) MN-major
        const uint32_t idesc_qk = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(kLN >> 3) << 17) | (8u << 24);
        const uint32_t idesc_pv =
            (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((uint32_t)(kLHalf >> 3) << 17) | (8u << 24);
        int tq = 0, tp = 0;
        bool q_ready = false;
        uint64_t t_last = global_ns();
        while (tp < n_tiles) {
          bool progressed = false;
          if (!q_ready) q_ready = ml_test(&q_tm, 0) && ml_test(&q_sm, 0);
          if (q_ready && tq < n_tiles && tq - tp < 2) {
            const int st = tq % kLStages, sb = tq & 1;
            const bool sfree = tq < 2 || ml_test(&o_done[sb], ((tq >> 1) - 1) & 1);
            if (sfree && ml_test(&kv_full[st], (tq / kLStages) & 1)) {
              ml_fence_after();
              const uint32_t kb = ring + st * kLTileBytes;
              const uint32_t d = tb + sb * kLN;
#pragma unroll
              for (int c = 0; c < kLChunks; ++c) {
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                  const uint64_t bd = ml_desc(kb + c * kLChunkBytes + kk * 32, 16, 1024);
                  const uint32_t acc = (c | kk) ? 1u : 0u;
                  if (c < kLQTm)
                    ml_mma_ts(d, tb + kLQCol + 32 * c + 8 * kk, bd, idesc_qk, acc);
                  else
                    ml_mma_ss(d, ml_desc(q_smem + (c - kLQTm) * kLQChunkBytes + kk * 32, 16, 1024), bd, idesc_qk,
                              acc);
                }
              }
              ml_commit(&s_full[sb]);
              ++tq;
              progressed = true;
            }
          }
          if (tp < tq) {
            const int st = tp % kLStages, sb = tp & 1;
            if (ml_test(&p_full[sb], (tp >> 1) & 1)) {
              ml_fence_after();
              const uint32_t vb = ring + st * kLTileBytes + 4 * hv * kLChunkBytes;
#pragma unroll
              for (int j = 0; j < kBlk; ++j)
                ml_mma_ts(tb + kLOCol, tb + sb * kLN + 8 * j, ml_desc(vb + j * 2048, kLChunkBytes, 1024), idesc_pv,
                          (tp > 0 || j > 0) ? 1u : 0u);
              ml_commit(&kv_empty[st]);
              ml_commit(&o_done[sb]);
              ++tp;
              progressed = true;
            }
          }
          if (progressed) {
            t_last = global_ns();
          } else if (*abf || global_ns() - t_last > kWaitLimitNs) {
            *abf = 1;
            break;
          } else {
            __nanosleep(64);
          }
        }
        // every MMA issued has completed before TMEM can be released
        ml_commit(&mma_drain);
        if (!mbar_wait(&mma_drain, 0)) atomic_or_status(P.status, SV_DEV_TIMEOUT);
      }
      __syncwarp();
    } else {
      // ------------------------------------------------------------ softmax ----
      const int row = tid;
      const int r = mt * 128 + row;
      const bool live = r < P.R;
      const bool warp_live = mt * 128 + warp * 32 < P.R;
      const uint32_t lane_base = tb + ((uint32_t)(warp * 32) << 16);
      const int lim = live ? L - P.n_new + r / P.H : -1;   // last visible key of this row
      const int end_key = min(L, blk1 * kLBS);              // first key this split does not own
      const float sl2 = P.scale_log2;
      if (warp_live) {
        // Q chunks 0..5 of this row into TMEM, bf16 pairs in memory order
        const uint4 *src = reinterpret_cast<const uint4 *>(P.q + ((int64_t)b * P.R + r) * kLD);
#pragma unroll 1
        for (int c0 = 0; c0 < kLQTm * 2; ++c0) {
          uint32_t w[16];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 v = live ? __ldg(src + 4 * c0 + k) : make_uint4(0u, 0u, 0u, 0u);
            w[4 * k] = v.x; w[4 * k + 1] = v.y; w[4 * k + 2] = v.z; w[4 * k + 3] = v.w;
          }
          ml_st16(lane_base + kLQCol + 16 * c0, w);
        }
        ml_wait_st();
      }
      ml_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&q_tm);

      float m_ref = -INFINITY, l = 0.f;
      bool ok = true;
      for (int t = 0; t < n_tiles && ok; ++t) {
        const int sb = t & 1, st = t % kLStages;
        ok = __all_sync(0xffffffffu, ml_wait(&s_full[sb], (t >> 1) & 1, abf));
        if (!ok) break;
        ml_fence_after();
        const int key0 = (blk0 + kBlk * t) * kLBS;
        if (warp_live) {
          float x[kLN];
          {
            uint32_t rr[kLN];
#pragma unroll
            for (int c0 = 0; c0 < kLN; c0 += 16)
              ml_ld16(lane_base + sb * kLN + c0, *reinterpret_cast<uint32_t(*)[16]>(rr + c0));
            ml_wait_ld();
#pragma unroll
            for (int k = 0; k < kLN; ++k) x[k] = __uint_as_float(rr[k]) * sl2;
          }
          if (key0 + kLN > end_key || key0 + kLN - 1 > L - P.n_new) {   // reaches the diagonal or the end
#pragma unroll
            for (int k = 0; k < kLN; ++k)
              if (key0 + k > lim || key0 + k >= end_key) x[k] = -INFINITY;
          }
          float mx = -INFINITY;
#pragma unroll
          for (int k = 0; k < kLN; ++k) mx = fmaxf(mx, x[k]);
          if (!live) mx = -INFINITY;   // padding rows never vote for a rescale
          // the reference moves only when a tile exceeds it by more than 8
          const bool up = mx > m_ref + 8.f;
          float a = 1.f;
          if (up) {
            a = m_ref == -INFINITY ? 0.f : ml_ex2(m_ref - mx);
            m_ref = mx;
          }
          if (t > 0 && __any_sync(0xffffffffu, up)) {
            // rescale O: the previous P V must have landed first
            ok = __all_sync(0xffffffffu, ml_wait(&o_done[(t - 1) & 1], ((t - 1) >> 1) & 1, abf));
            ml_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < kLHalf; c0 += 16) {
              uint32_t rr[16];
              ml_ld16(lane_base + kLOCol + c0, rr);
              ml_wait_ld();
#pragma unroll
              for (int k = 0; k < 16; ++k) rr[k] = __float_as_uint(__uint_as_float(rr[k]) * a);
              ml_st16(lane_base + kLOCol + c0, rr);
            }
            ml_wait_st();
          }
          l *= a;
          const float base = m_ref == -INFINITY ? 0.f : m_ref;
          float ps = 0.f;
#pragma unroll
          for (int c0 = 0; c0 < kLN; c0 += 32) {
            uint32_t w[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const float p0 = ml_ex2(x[c0 + 2 * k] - base), p1 = ml_ex2(x[c0 + 2 * k + 1] - base);
              ps += p0 + p1;
              w[k] = ml_pack_bf16(p0, p1);
            }
            ml_st16(lane_base + sb * kLN + c0 / 2, w);
          }
          ml_wait_st();
          l += ps;
        }
        if (key0 + kLN > end_key && warp == 0) {
          // keys past the split or the sequence (not loaded, or rows of a
          // block past the sequence): their value rows of this half are
          // zeroed, so that 0 * (anything) = 0
          if (!ml_wait(&kv_full[st], (t / kLStages) & 1, abf)) ok = false;
          const uint32_t vb = ring + st * kLTileBytes + 4 * hv * kLChunkBytes;
          for (int k = max(0, end_key - key0) + lane; k < kLN; k += 32) {
            const uint32_t off = (uint32_t)((k >> 4) * 2048 + (k & 15) * 128);
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
              for (int q16 = 0; q16 < 8; ++q16)
                asm volatile("st.shared.v4.u32 [%0], {%1,%1,%1,%1};" ::"r"(vb + c * kLChunkBytes + off + q16 * 16),
                             "r"(0u)
                             : "memory");
          }
          fence_proxy_async_shared();
        }
        ml_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&p_full[sb]);
        ok = __all_sync(0xffffffffu, ok);
      }
      // ---- epilogue: this half of the row's output ----------------------------
      const int lb = (n_tiles - 1) & 1;
      const bool have = __all_sync(0xffffffffu, ok && ml_wait(&o_done[lb], ((n_tiles - 1) >> 1) & 1, abf));
      ml_fence_after();
      if (have && warp_live) {
        const int nsplit = (nblk + P.bps - 1) / P.bps;
        const int64_t ent = ((int64_t)b * P.S + s) * P.R + r;
        const float il = l > 0.f ? 1.f / l : 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < kLHalf; c0 += 64) {
          uint32_t rr[64];
#pragma unroll
          for (int c = 0; c < 64; c += 16) ml_ld16(lane_base + kLOCol + c0 + c, *reinterpret_cast<uint32_t(*)[16]>(rr + c));
          ml_wait_ld();
          if (live) {
            if (nsplit == 1) {
              __nv_bfloat16 *o = P.out + ((int64_t)b * P.R + r) * kLC + hv * kLHalf + c0;
#pragma unroll
              for (int c = 0; c < 64; c += 8) {
                uint32_t w[4];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                  w[k] = ml_pack_bf16(__uint_as_float(rr[c + 2 * k]) * il, __uint_as_float(rr[c + 2 * k + 1]) * il);
                *reinterpret_cast<uint4 *>(o + c) = make_uint4(w[0], w[1], w[2], w[3]);
              }
            } else {
              float *acc = P.ws_acc + ent * kLC + hv * kLHalf + c0;
#pragma unroll
              for (int c = 0; c < 64; c += 4)
                *reinterpret_cast<float4 *>(acc + c) = make_float4(__uint_as_float(rr[c]), __uint_as_float(rr[c + 1]),
                                                                   __uint_as_float(rr[c + 2]), __uint_as_float(rr[c + 3]));
            }
          }
        }
        if (live && nsplit > 1 && hv == 0) {
          P.ws_ml[ent * 2] = m_ref;
          P.ws_ml[ent * 2 + 1] = l;
        }
      }
    }
  }
  if (tid == 0 && *abf) atomic_or_status(P.status, SV_DEV_TIMEOUT);
  ml_fence_before();
  __syncthreads();
  ml_fence_after();
  if (warp == kLMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kLCols));
}

// Longest-first order of the sequences (ties by batch index): the CTAs of
// the longest contexts start first, so the last wave holds short ones. Rank
// of b = number of sequences that come before it; order[rank] = b. It reads
// only seq_lens (which no kernel of the library writes), so it runs while the
// previous kernel of the stream finishes, and waits for it at its end.
constexpr int kLMaxOrder = 4096;
__global__ void __launch_bounds__(1024) mla_order_kernel(const int32_t *seq_lens, int B, int32_t *order) {
  pdl_trigger();
  __shared__ int lens[kLMaxOrder];
  for (int b = threadIdx.x; b < B; b += blockDim.x) lens[b] = seq_lens[b];
  __syncthreads();
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const int L = lens[b];
    int rank = 0;
    for (int c = 0; c < B; ++c) rank += (lens[c] > L) || (lens[c] == L && c < b);
    order[rank] = b;
  }
  pdl_wait();
}

// Merge of the splits of one query row: weights 2^(m_s - M) on the partial
// sums and normalisers (the log-sum-exp combination of split-KV attention).
// CTA = (row r, sequence b), 128 threads x 4 values.
__global__ void __launch_bounds__(128) attn_mla_merge_kernel(const float *ws_acc, const float *ws_ml,
                                                             const int32_t *seq_lens, int S, int R, int bps,
                                                             int max_blocks, int n_new, __nv_bfloat16 *out) {
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x, b = blockIdx.y;
  const int L = seq_lens[b];
  if (L < n_new || L > max_blocks * kLBS) return;   // flagged by the attention kernel
  const int nsplit = ((L + kLBS - 1) / kLBS + bps - 1) / bps;
  if (nsplit <= 1) return;                          // written directly
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, ws_ml[(((int64_t)b * S + s) * R + r) * 2]);
  float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const int64_t ent = ((int64_t)b * S + s) * R + r;
    const float m = ws_ml[ent * 2];
    const float w = m == -INFINITY ? 0.f : ml_ex2(m - M);
    den += w * ws_ml[ent * 2 + 1];
    const float4 a = *reinterpret_cast<const float4 *>(ws_acc + ent * kLC + threadIdx.x * 4);
    num.x += w * a.x; num.y += w * a.y; num.z += w * a.z; num.w += w * a.w;
  }
  const float il = den > 0.f ? 1.f / den : 0.f;
  __nv_bfloat162 lo = __floats2bfloat162_rn(num.x * il, num.y * il), hi = __floats2bfloat162_rn(num.z * il, num.w * il);
  uint2 v;
  v.x = *reinterpret_cast<uint32_t *>(&lo);
  v.y = *reinterpret_cast<uint32_t *>(&hi);
  *reinterpret_cast<uint2 *>(out + ((int64_t)b * R + r) * kLC + threadIdx.x * 4) = v;
}

// Latent append: one CTA per (new position j, sequence b); thread t copies
// 16 bytes of the 1152-byte row into slot pos % 16 of block table[pos / 16].
__global__ void __launch_bounds__(96) latent_append_kernel(const uint4 *c_new, uint4 *cache, const int32_t *table,
                                                           int max_blocks, const int32_t *seq_lens, int n_new,
                                                           int num_blocks, int32_t *status) {
  pdl_trigger();
  constexpr int kRowVec = kLD * 2 / 16;
  const int j = blockIdx.x, b = blockIdx.y;
  const int L = seq_lens[b];
  const bool len_ok = L >= n_new && L <= max_blocks * kLBS;
  const int pos = L - n_new + j;
  const int blk = len_ok ? table[(int64_t)b * max_blocks + pos / kLBS] : -1;
  const bool blk_ok = blk >= 0 && blk < num_blocks;
  uint4 v = make_uint4(0u, 0u, 0u, 0u);
  if ((int)threadIdx.x < kRowVec) v = __ldg(c_new + ((int64_t)b * n_new + j) * kRowVec + threadIdx.x);
  pdl_wait();
  if (!len_ok || !blk_ok) {
    if (threadIdx.x == 0) atomic_or_status(status, len_ok ? SV_DEV_BAD_BLOCK : SV_DEV_BAD_SEQ_LEN);
    return;
  }
  if ((int)threadIdx.x < kRowVec) cache[((int64_t)blk * kLBS + pos % kLBS) * kRowVec + threadIdx.x] = v;
}

struct MlaPlan {
  int R, n_mt, S, bps;
};

MlaPlan mla_plan(int B, int n_new, int H, int max_blocks) {
  MlaPlan p;
  p.R = n_new * H;
  p.n_mt = (p.R + 127) / 128;
  const int per_split = 2 * p.n_mt * std::max(B, 1);
  int S = 1;
  if (per_split < kLCtaTarget)
    S = std::max(1, std::min((kLCtaTarget + per_split - 1) / per_split,
                             (max_blocks + kLMinBlocksPerSplit - 1) / kLMinBlocksPerSplit));
  constexpr int blk = MlaCfg<kLNK>::kBlk;
  int bps = (max_blocks + S - 1) / S;
  bps = (bps + blk - 1) / blk * blk;   // whole tiles
  p.bps = std::max(blk, bps);
  p.S = (max_blocks + p.bps - 1) / p.bps;
  return p;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

// workspace: [partial outputs, (m, l) pairs] of a split context, then the
// sequence order (batches of at most kLMaxOrder sequences)
size_t mla_split_bytes(int B, const MlaPlan &p) {
  if (p.S <= 1) return 0;
  const size_t ent = (size_t)B * p.S * p.R;
  return align256(ent * kLC * sizeof(float)) + align256(ent * 2 * sizeof(float));
}

size_t mla_ws_bytes(int B, const MlaPlan &p) {
  return mla_split_bytes(B, p) + (B <= kLMaxOrder ? align256((size_t)B * sizeof(int32_t)) : 0);
}

PFN_cuTensorMapEncodeTiled_v12000 mla_encode_fn() {
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

}  // namespace
}  // namespace sv

using namespace sv;

extern "C" size_t spec_verify_attn_mla_workspace_size(int B, int n_new, int H, int max_blocks_per_seq) {
  if (B < 0 || n_new < 1 || H < 1 || max_blocks_per_seq < 1) return 0;
  return mla_ws_bytes(B, mla_plan(B, n_new, H, max_blocks_per_seq));
}

extern "C" sv_status spec_verify_attn_mla(const void *q_lat, sv_dtype q_dtype, const void *cache, sv_dtype cache_dtype,
                                          const int32_t *block_table, int max_blocks_per_seq, const int32_t *seq_lens,
                                          int B, int n_new, int H, int d_c, int d_r, int block_size, int num_blocks,
                                          float softmax_scale, void *out, void *workspace, size_t workspace_bytes,
                                          int32_t *dev_status, sv_stream_t stream) {
  if (B < 0 || n_new < 1 || H < 1 || max_blocks_per_seq < 1 || num_blocks < 1)
    return fail(SV_ERR_INVALID_ARG, "spec_verify_attn_mla: bad sizes B=%d n_new=%d H=%d max_blocks=%d num_blocks=%d",
                B, n_new, H, max_blocks_per_seq, num_blocks);
  if (d_c != kLC || d_r != kLR)
    return fail(SV_ERR_UNSUPPORTED, "spec_verify_attn_mla: d_c=%d d_r=%d (the kernel takes d_c=512, d_r=64)", d_c, d_r);
  if (block_size != kLBS) return fail(SV_ERR_UNSUPPORTED, "spec_verify_attn_mla: block_size must be 16");
  if (q_dtype != SV_BF16 || cache_dtype != SV_BF16)
    return fail(SV_ERR_UNSUPPORTED, "spec_verify_attn_mla: q and the cache must be bf16");
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale))
    return fail(SV_ERR_INVALID_ARG, "spec_verify_attn_mla: softmax_scale must be finite and > 0");
  if (B > 65535) return fail(SV_ERR_UNSUPPORTED, "spec_verify_attn_mla: B must be <= 65535");
  if ((int64_t)n_new * H > (1 << 24) || (int64_t)max_blocks_per_seq * kLBS > (1 << 30))
    return fail(SV_ERR_UNSUPPORTED, "spec_verify_attn_mla: sizes too large");
  if (B == 0) return ok();
  if (!q_lat || !cache || !block_table || !seq_lens || !out)
    return fail(SV_ERR_INVALID_ARG, "spec_verify_attn_mla: null pointer argument");
  if (!aligned(q_lat, 16) || !aligned(cache, 16) || !aligned(out, 16))
    return fail(SV_ERR_INVALID_ARG, "spec_verify_attn_mla: q, cache and out must be 16-byte aligned");
  const MlaPlan plan = mla_plan(B, n_new, H, max_blocks_per_seq);
  if ((int64_t)2 * plan.n_mt * plan.S > 0x7fffffff)
    return fail(SV_ERR_UNSUPPORTED, "spec_verify_attn_mla: grid too large");
  const size_t need = mla_ws_bytes(B, plan);
  if (!workspace || workspace_bytes < need)
    return fail(SV_ERR_WORKSPACE, "spec_verify_attn_mla: workspace of %zu bytes, %zu needed", workspace_bytes, need);
  if (!aligned(workspace, 256))
    return fail(SV_ERR_WORKSPACE, "spec_verify_attn_mla: workspace must be 256-byte aligned");

  PFN_cuTensorMapEncodeTiled_v12000 enc = mla_encode_fn();
  if (!enc) return fail(SV_ERR_CUDA, "spec_verify_attn_mla: cuTensorMapEncodeTiled unavailable");
  MlaParams P;
  memset(&P, 0, sizeof(P));
  cuuint32_t estr[3] = {1, 1, 1};
  {
    cuuint64_t dims[3] = {(cuuint64_t)kLD, (cuuint64_t)kLBS, (cuuint64_t)num_blocks};
    cuuint64_t strides[2] = {(cuuint64_t)kLD * 2, (cuuint64_t)kLBS * kLD * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kLBS, 1};
    CUresult r = enc(&P.tmc, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(cache), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(SV_ERR_INVALID_ARG, "spec_verify_attn_mla: cache tensor map failed (%d)", (int)r);
  }
  {
    // rows of a tile past R read as zeros (a box may reach past the tensor);
    // with fewer than 128 rows in all the box is those rows
    P.q_box = std::min(128, plan.R);
    cuuint64_t dims[3] = {(cuuint64_t)kLD, (cuuint64_t)plan.R, (cuuint64_t)B};
    cuuint64_t strides[2] = {(cuuint64_t)kLD * 2, (cuuint64_t)plan.R * kLD * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)P.q_box, 1};
    CUresult r = enc(&P.tmq, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q_lat), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(SV_ERR_INVALID_ARG, "spec_verify_attn_mla: q tensor map failed (%d)", (int)r);
  }
  P.q = static_cast<const __nv_bfloat16 *>(q_lat);
  P.out = static_cast<__nv_bfloat16 *>(out);
  const size_t ent = (size_t)B * plan.S * plan.R;
  const size_t split_bytes = mla_split_bytes(B, plan);
  P.ws_acc = split_bytes ? static_cast<float *>(workspace) : nullptr;
  P.ws_ml = split_bytes
                ? reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + align256(ent * kLC * sizeof(float)))
                : nullptr;
  int32_t *order = B <= kLMaxOrder ? reinterpret_cast<int32_t *>(static_cast<uint8_t *>(workspace) + split_bytes)
                                   : nullptr;
  P.order = order;
  P.block_table = block_table;
  P.seq_lens = seq_lens;
  P.status = dev_status;
  P.B = B; P.n_new = n_new; P.H = H; P.R = plan.R; P.n_mt = plan.n_mt;
  P.max_blocks = max_blocks_per_seq; P.num_blocks = num_blocks; P.bps = plan.bps; P.S = plan.S;
  P.scale_log2 = (float)((double)softmax_scale * 1.4426950408889634074);

  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(attn_mla_kernel<kLNK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    MlaCfg<kLNK>::kSmem);
  });
  if (attr_err != cudaSuccess)
    return fail(SV_ERR_CUDA, "spec_verify_attn_mla: kernel attributes: %s", cudaGetErrorString(attr_err));
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (order) {
    e = launch_k(mla_order_kernel, dim3(1), dim3(1024), 0, st, 1, seq_lens, B, order);
    if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_attn_mla order launch: %s", cudaGetErrorString(e));
  }
  e = launch_k(attn_mla_kernel<kLNK>, dim3(2 * plan.n_mt * plan.S, B), dim3(kLThreads),
                           (size_t)MlaCfg<kLNK>::kSmem, st, 1, P);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_attn_mla launch: %s", cudaGetErrorString(e));
  if (plan.S > 1) {
    e = launch_k(attn_mla_merge_kernel, dim3(plan.R, B), dim3(128), 0, st, 1, (const float *)P.ws_acc,
                 (const float *)P.ws_ml, seq_lens, plan.S, plan.R, plan.bps, max_blocks_per_seq, n_new, P.out);
    if (e != cudaSuccess) return fail(SV_ERR_CUDA, "spec_verify_attn_mla merge launch: %s", cudaGetErrorString(e));
  }
  return ok();
}

extern "C" sv_status kv_block_append_latent(const void *c_new, sv_dtype dtype, void *cache,
                                            const int32_t *block_table, int max_blocks_per_seq,
                                            const int32_t *seq_lens, int B, int n_new, int d_latent, int block_size,
                                            int num_blocks, int32_t *dev_status, sv_stream_t stream) {
  if (B < 0 || n_new < 1 || max_blocks_per_seq < 1 || num_blocks < 1)
    return fail(SV_ERR_INVALID_ARG, "kv_block_append_latent: bad sizes");
  if (d_latent != kLD) return fail(SV_ERR_UNSUPPORTED, "kv_block_append_latent: d_latent must be 576");
  if (block_size != kLBS) return fail(SV_ERR_UNSUPPORTED, "kv_block_append_latent: block_size must be 16");
  if (dtype != SV_BF16) return fail(SV_ERR_UNSUPPORTED, "kv_block_append_latent: rows must be bf16");
  if (B > 65535 || n_new > 65535) return fail(SV_ERR_UNSUPPORTED, "kv_block_append_latent: B and n_new <= 65535");
  if (B == 0) return ok();
  if (!c_new || !cache || !block_table || !seq_lens)
    return fail(SV_ERR_INVALID_ARG, "kv_block_append_latent: null pointer argument");
  if (!aligned(c_new, 16) || !aligned(cache, 16))
    return fail(SV_ERR_INVALID_ARG, "kv_block_append_latent: rows and cache must be 16-byte aligned");
  cudaError_t e = launch_k(latent_append_kernel, dim3(n_new, B), dim3(96), 0, reinterpret_cast<cudaStream_t>(stream),
                           1, static_cast<const uint4 *>(c_new), static_cast<uint4 *>(cache), block_table,
                           max_blocks_per_seq, seq_lens, n_new, num_blocks, dev_status);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "kv_block_append_latent launch: %s", cudaGetErrorString(e));
  return ok();
}

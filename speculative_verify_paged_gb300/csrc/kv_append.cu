// kv_block_append: scatter the K+1 new K/V rows of each sequence into the
// paged pools ("KV Cache + Speculative Decoding", section 6.2, append_token:
// page pos / block_size, slot pos % block_size), converting to the pool dtype.
#include <cuda_fp8.h>
#include <algorithm>
#include <cstring>
#include <type_traits>

#include <mutex>

#include "sv_common.cuh"

namespace sv {
namespace {

struct AppendArgs {
  const void *k_new, *v_new;
  void *k_cache, *v_cache;
  const float *k_scale, *v_scale;
  const int32_t *block_table, *seq_lens;
  int max_blocks, n_new, H_kv, d, bs, num_blocks;
  int64_t block_stride, head_stride, slot_stride;
  int32_t *status;
  bool vec_in, vec_out;   // 16-byte input loads / 8- or 16-byte pool stores allowed
};

template <typename TIn, int KV>
__device__ __forceinline__ void store_elem(void *cache, int64_t off, TIn x_in, float scale) {
  float x = to_f32(x_in);
  if constexpr (KV == SV_F32) {
    static_cast<float *>(cache)[off] = x;
  } else if constexpr (KV == SV_BF16) {
    static_cast<__nv_bfloat16 *>(cache)[off] = __float2bfloat16_rn(x);
  } else {
    float q = __fdiv_rn(x, scale);
    static_cast<uint8_t *>(cache)[off] =
        static_cast<uint8_t>(__nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3));
  }
}

// eight consecutive input elements as floats (one or two 16-byte loads when
// the rows allow it)
template <typename TIn>
__device__ __forceinline__ void load8_in(const TIn *src, bool vec, float (&x)[8]) {
  if constexpr (std::is_same<TIn, float>::value) {
    if (vec) {
      const float4 a = __ldg(reinterpret_cast<const float4 *>(src));
      const float4 b = __ldg(reinterpret_cast<const float4 *>(src) + 1);
      x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
      return;
    }
  } else {
    if (vec) {
      const uint4 w = __ldg(reinterpret_cast<const uint4 *>(src));
      const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[2 * k] = __uint_as_float(u[k] << 16);
        x[2 * k + 1] = __uint_as_float(u[k] & 0xffff0000u);
      }
      return;
    }
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) x[k] = to_f32(src[k]);
}

// eight consecutive pool elements at element offset off (one 8- or 16-byte
// store, or two, when the layout allows it)
template <int KV>
__device__ __forceinline__ void store8_out(void *cache, int64_t off, const float (&x)[8], float scale, bool vec) {
  if constexpr (KV == SV_F32) {
    float *d = static_cast<float *>(cache) + off;
    if (vec) {
      reinterpret_cast<float4 *>(d)[0] = make_float4(x[0], x[1], x[2], x[3]);
      reinterpret_cast<float4 *>(d)[1] = make_float4(x[4], x[5], x[6], x[7]);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) d[k] = x[k];
    }
  } else if constexpr (KV == SV_BF16) {
    __nv_bfloat16 h[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) h[k] = __float2bfloat16_rn(x[k]);
    __nv_bfloat16 *d = static_cast<__nv_bfloat16 *>(cache) + off;
    if (vec) {
      uint4 w;
      memcpy(&w, h, sizeof(w));
      *reinterpret_cast<uint4 *>(d) = w;
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) d[k] = h[k];
    }
  } else {
    uint8_t q[8];
#pragma unroll
    for (int k = 0; k < 8; ++k)
      q[k] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(__fdiv_rn(x[k], scale), __NV_SATFINITE, __NV_E4M3));
    uint8_t *d = static_cast<uint8_t *>(cache) + off;
    if (vec) {
      uint2 w;
      memcpy(&w, q, sizeof(w));
      *reinterpret_cast<uint2 *>(d) = w;
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) d[k] = q[k];
    }
  }
}

// One CTA per (new position j, sequence b); a thread takes groups of eight
// consecutive elements of one head row (d % 8 == 0; element by element
// otherwise). Everything it reads (lengths, block table, the new rows) is
// loaded before the wait on the previous kernel (the library's kernels
// never write them); only the stores into the pools wait, since a previous
// kernel may still be reading the pools.
template <typename TIn, int KV>
__global__ void __launch_bounds__(256) kv_append_kernel(AppendArgs a) {
  pdl_trigger();
  const int j = blockIdx.x, b = blockIdx.y;
  const int L = a.seq_lens[b];
  const bool len_ok = L >= a.n_new && L <= a.max_blocks * a.bs;
  const int pos = L - a.n_new + j;
  const int blk = len_ok ? a.block_table[(int64_t)b * a.max_blocks + pos / a.bs] : -1;
  const bool blk_ok = blk >= 0 && blk < a.num_blocks;
  const int64_t src0 = ((int64_t)b * a.n_new + j) * a.H_kv * a.d;
  const TIn *kn = static_cast<const TIn *>(a.k_new) + src0;
  const TIn *vn = static_cast<const TIn *>(a.v_new) + src0;
  if (a.d % 8 == 0) {
    const int groups = a.H_kv * a.d / 8;
    float kx[8], vx[8];
    const int e0 = threadIdx.x * 8;
    if ((int)threadIdx.x < groups) {
      load8_in<TIn>(kn + e0, a.vec_in, kx);
      load8_in<TIn>(vn + e0, a.vec_in, vx);
    }
    pdl_wait();
    if (!len_ok || !blk_ok) {
      if (threadIdx.x == 0) atomic_or_status(a.status, len_ok ? SV_DEV_BAD_BLOCK : SV_DEV_BAD_SEQ_LEN);
      return;
    }
    const int64_t base = (int64_t)blk * a.block_stride + (int64_t)(pos % a.bs) * a.slot_stride;
    for (int gi = threadIdx.x; gi < groups; gi += blockDim.x) {
      const int e = gi * 8;
      if (gi != (int)threadIdx.x) {   // more groups than threads
        load8_in<TIn>(kn + e, a.vec_in, kx);
        load8_in<TIn>(vn + e, a.vec_in, vx);
      }
      const int g = e / a.d, c = e - g * a.d;
      const int64_t off = base + (int64_t)g * a.head_stride + c;
      float ks = 1.f, vs = 1.f;
      if constexpr (KV == SV_FP8_E4M3) {
        ks = a.k_scale[g];
        vs = a.v_scale[g];
      }
      store8_out<KV>(a.k_cache, off, kx, ks, a.vec_out);
      store8_out<KV>(a.v_cache, off, vx, vs, a.vec_out);
    }
    return;
  }
  pdl_wait();
  if (!len_ok || !blk_ok) {
    if (threadIdx.x == 0) atomic_or_status(a.status, len_ok ? SV_DEV_BAD_BLOCK : SV_DEV_BAD_SEQ_LEN);
    return;
  }
  const int64_t base = (int64_t)blk * a.block_stride + (int64_t)(pos % a.bs) * a.slot_stride;
  const int total = a.H_kv * a.d;
  for (int e = threadIdx.x; e < total; e += blockDim.x) {
    const int g = e / a.d, c = e - g * a.d;
    const int64_t off = base + (int64_t)g * a.head_stride + c;
    float ks = 1.f, vs = 1.f;
    if constexpr (KV == SV_FP8_E4M3) {
      ks = a.k_scale[g];
      vs = a.v_scale[g];
    }
    store_elem<TIn, KV>(a.k_cache, off, kn[e], ks);
    store_elem<TIn, KV>(a.v_cache, off, vn[e], vs);
  }
}

template <typename TIn>
sv_status launch_in(const AppendArgs &a, sv_dtype kv_dtype, int B, cudaStream_t s) {
  dim3 grid(a.n_new, B);
  // a thread per group of eight elements (up to 256 threads)
  const int groups = a.d % 8 == 0 ? a.H_kv * a.d / 8 : 256;
  const dim3 block(std::max(32, std::min(256, (groups + 31) / 32 * 32)));
  switch (kv_dtype) {
    case SV_F32: launch_k(kv_append_kernel<TIn, SV_F32>, grid, block, 0, s, 1, a); break;
    case SV_BF16: launch_k(kv_append_kernel<TIn, SV_BF16>, grid, block, 0, s, 1, a); break;
    case SV_FP8_E4M3: launch_k(kv_append_kernel<TIn, SV_FP8_E4M3>, grid, block, 0, s, 1, a); break;
    default: return fail(SV_ERR_UNSUPPORTED, "kv_block_append: unsupported kv_dtype %d", kv_dtype);
  }
  return check_launch("kv_block_append launch");
}

}  // namespace
// ------------------------------------------------------------ tree commit ---
// After a tree round ("KV Cache + Speculative Decoding", Q14 and section 8.2)
// the accepted path's rows move next to the root: position L - n_new + 1 + i
// takes node path[i]'s row (position L - n_new + path[i]), for every kv head
// of K and V, so that the cache again holds every token of the sequence but
// the last one (section 7's invariant) once the length is rolled back. A
// path node's row can be a later destination (path[i] >= i + 1), so a CTA
// reads all of a head's moved rows into shared memory before it writes any.

constexpr int kCmThreads = 256;
constexpr int kCmMaxRowBytes = 1024;   // d_head * element size

struct CommitArgs {
  uint8_t *cache[2];                    // K, V
  const int32_t *block_table, *seq_lens, *path, *nacc;
  int max_blocks, n_new, H_kv, row_bytes, bs, num_blocks, unit;   // unit: 16 or 1 byte
  int64_t block_stride, head_stride, slot_stride;                 // bytes
  int32_t *status;
};

// grid (B, 2): sequence b, K (0) or V (1)
__global__ void __launch_bounds__(kCmThreads) kv_tree_commit_kernel(const __grid_constant__ CommitArgs a) {
  extern __shared__ __align__(16) uint8_t cm_buf[];
  __shared__ int64_t src_off[64], dst_off[64];
  __shared__ int s_ok;
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x, tid = threadIdx.x;
  uint8_t *cache = a.cache[blockIdx.y];
  const int L = __ldg(a.seq_lens + b);
  const int nacc = a.nacc[b];   // may come from the sampling kernel just before
  if (L < a.n_new || L > a.max_blocks * a.bs || nacc < 0 || nacc > a.n_new - 1) {
    if (tid == 0 && blockIdx.y == 0) atomic_or_status(a.status, SV_DEV_BAD_SEQ_LEN);
    return;
  }
  if (tid == 0) s_ok = 1;
  __syncthreads();
  const int base = L - a.n_new;
  for (int i = tid; i < nacc; i += kCmThreads) {
    const int node = a.path[(int64_t)b * a.n_new + i];
    const int s = base + node, d = base + 1 + i;
    bool ok = node >= 1 && node < a.n_new;
    int sb = 0, db = 0;
    if (ok) {
      sb = __ldg(a.block_table + (int64_t)b * a.max_blocks + s / a.bs);
      db = __ldg(a.block_table + (int64_t)b * a.max_blocks + d / a.bs);
      ok = sb >= 0 && sb < a.num_blocks && db >= 0 && db < a.num_blocks;
    }
    if (!ok) {
      s_ok = 0;
      continue;
    }
    src_off[i] = (int64_t)sb * a.block_stride + (int64_t)(s % a.bs) * a.slot_stride;
    dst_off[i] = (int64_t)db * a.block_stride + (int64_t)(d % a.bs) * a.slot_stride;
  }
  __syncthreads();
  if (!s_ok) {
    if (tid == 0 && blockIdx.y == 0) atomic_or_status(a.status, SV_DEV_BAD_TREE | SV_DEV_BAD_BLOCK);
    return;
  }
  const int units = a.row_bytes / a.unit;
  for (int g = 0; g < a.H_kv; ++g) {
    const int64_t hoff = (int64_t)g * a.head_stride;
    for (int idx = tid; idx < nacc * units; idx += kCmThreads) {
      const int i = idx / units, v = idx % units;
      const uint8_t *src = cache + src_off[i] + hoff + (int64_t)v * a.unit;
      if (a.unit == 16) reinterpret_cast<uint4 *>(cm_buf)[idx] = *reinterpret_cast<const uint4 *>(src);
      else cm_buf[idx] = *src;
    }
    __syncthreads();
    for (int idx = tid; idx < nacc * units; idx += kCmThreads) {
      const int i = idx / units, v = idx % units;
      uint8_t *dst = cache + dst_off[i] + hoff + (int64_t)v * a.unit;
      if (a.unit == 16) *reinterpret_cast<uint4 *>(dst) = reinterpret_cast<const uint4 *>(cm_buf)[idx];
      else *dst = cm_buf[idx];
    }
    __syncthreads();
  }
}

}  // namespace sv

extern "C" sv_status kv_tree_commit(void *k_cache, void *v_cache, sv_dtype kv_dtype, const sv_kv_layout *layout,
                                    const int32_t *block_table, int max_blocks_per_seq, const int32_t *seq_lens,
                                    const int32_t *path_nodes, const int32_t *num_accepted, int B, int n_new,
                                    int H_kv, int d_head, int block_size, int num_blocks, int32_t *dev_status,
                                    sv_stream_t stream) {
  using namespace sv;
  if (!k_cache || !v_cache || !block_table || !seq_lens || !path_nodes || !num_accepted)
    return fail(SV_ERR_INVALID_ARG, "kv_tree_commit: null pointer argument");
  if (B < 0 || n_new < 1 || H_kv < 1 || d_head < 1 || block_size < 1 || num_blocks < 1 || max_blocks_per_seq < 1)
    return fail(SV_ERR_INVALID_ARG, "kv_tree_commit: bad sizes");
  if (n_new > 64) return fail(SV_ERR_UNSUPPORTED, "kv_tree_commit: at most 64 tree nodes");
  const int es = dtype_bytes(kv_dtype);
  if (es == 0 || kv_dtype == SV_F16) return fail(SV_ERR_UNSUPPORTED, "kv_tree_commit: pools must be f32, bf16 or fp8");
  if (d_head * es > kCmMaxRowBytes) return fail(SV_ERR_UNSUPPORTED, "kv_tree_commit: rows above 1024 bytes");
  if (B == 0) return ok();
  CommitArgs a = {};
  a.cache[0] = static_cast<uint8_t *>(k_cache);
  a.cache[1] = static_cast<uint8_t *>(v_cache);
  a.block_table = block_table; a.seq_lens = seq_lens; a.path = path_nodes; a.nacc = num_accepted;
  a.max_blocks = max_blocks_per_seq; a.n_new = n_new; a.H_kv = H_kv; a.row_bytes = d_head * es;
  a.bs = block_size; a.num_blocks = num_blocks; a.status = dev_status;
  int64_t bst, hst, sst;
  if (layout) {
    bst = layout->block_stride; hst = layout->head_stride; sst = layout->slot_stride;
    if (sst < d_head || hst < d_head || bst < d_head)
      return fail(SV_ERR_INVALID_ARG, "kv_tree_commit: layout strides smaller than d_head");
  } else {
    sst = d_head; hst = (int64_t)block_size * d_head; bst = (int64_t)H_kv * block_size * d_head;
  }
  a.block_stride = bst * es; a.head_stride = hst * es; a.slot_stride = sst * es;
  a.unit = (a.row_bytes % 16 == 0 && aligned(k_cache, 16) && aligned(v_cache, 16) && a.block_stride % 16 == 0 &&
            a.head_stride % 16 == 0 && a.slot_stride % 16 == 0) ? 16 : 1;
  const size_t smem = (size_t)(n_new - 1) * a.row_bytes + 16;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(kv_tree_commit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    63 * kCmMaxRowBytes + 16);
  });
  if (attr_err != cudaSuccess) return fail(SV_ERR_CUDA, "kv_tree_commit attributes: %s", cudaGetErrorString(attr_err));
  const cudaError_t e = launch_k(kv_tree_commit_kernel, dim3(B, 2), dim3(kCmThreads), smem,
                                 reinterpret_cast<cudaStream_t>(stream), 1, a);
  if (e != cudaSuccess) return fail(SV_ERR_CUDA, "kv_tree_commit launch: %s", cudaGetErrorString(e));
  return ok();
}

extern "C" sv_status kv_block_append(const void *k_new, const void *v_new, sv_dtype new_dtype,
                                     void *k_cache, void *v_cache, sv_dtype kv_dtype,
                                     const sv_kv_layout *layout, const float *k_scale,
                                     const float *v_scale, const int32_t *block_table,
                                     int max_blocks_per_seq, const int32_t *seq_lens, int B,
                                     int n_new, int H_kv, int d_head, int block_size,
                                     int num_blocks, int32_t *dev_status, sv_stream_t stream) {
  using namespace sv;
  if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !seq_lens)
    return fail(SV_ERR_INVALID_ARG, "kv_block_append: null pointer argument");
  if (B < 0 || n_new < 1 || H_kv < 1 || d_head < 1 || block_size < 1 || num_blocks < 1 ||
      max_blocks_per_seq < 1)
    return fail(SV_ERR_INVALID_ARG,
                "kv_block_append: bad sizes B=%d n_new=%d H_kv=%d d_head=%d block_size=%d "
                "num_blocks=%d max_blocks_per_seq=%d",
                B, n_new, H_kv, d_head, block_size, num_blocks, max_blocks_per_seq);
  if (n_new > 65535) return fail(SV_ERR_UNSUPPORTED, "kv_block_append: n_new > 65535");
  if (kv_dtype == SV_FP8_E4M3 && (!k_scale || !v_scale))
    return fail(SV_ERR_INVALID_ARG, "kv_block_append: fp8 pools need k_scale and v_scale");
  if (new_dtype != SV_F32 && new_dtype != SV_BF16)
    return fail(SV_ERR_UNSUPPORTED, "kv_block_append: new rows must be f32 or bf16");
  if (B == 0) return ok();
  AppendArgs a;
  a.k_new = k_new; a.v_new = v_new; a.k_cache = k_cache; a.v_cache = v_cache;
  a.k_scale = k_scale; a.v_scale = v_scale; a.block_table = block_table; a.seq_lens = seq_lens;
  a.max_blocks = max_blocks_per_seq; a.n_new = n_new; a.H_kv = H_kv; a.d = d_head;
  a.bs = block_size; a.num_blocks = num_blocks; a.status = dev_status;
  if (layout) {
    a.block_stride = layout->block_stride;
    a.head_stride = layout->head_stride;
    a.slot_stride = layout->slot_stride;
    if (a.slot_stride < d_head || a.head_stride < d_head || a.block_stride < d_head)
      return fail(SV_ERR_INVALID_ARG, "kv_block_append: layout strides smaller than d_head");
  } else {
    a.slot_stride = d_head;
    a.head_stride = (int64_t)block_size * d_head;
    a.block_stride = (int64_t)H_kv * block_size * d_head;
  }
  // vector paths: every group of eight starts on a 16-byte (input) or
  // 8 * element-size (pool) boundary
  const int es_in = new_dtype == SV_F32 ? 4 : 2;
  const int es_out = kv_dtype == SV_F32 ? 4 : (kv_dtype == SV_BF16 ? 2 : 1);
  a.vec_in = d_head % 8 == 0 && aligned(k_new, 16) && aligned(v_new, 16);
  a.vec_out = d_head % 8 == 0 && aligned(k_cache, 16) && aligned(v_cache, 16) &&
              (a.block_stride * es_out) % (8 * es_out) == 0 && (a.head_stride * es_out) % (8 * es_out) == 0 &&
              (a.slot_stride * es_out) % (8 * es_out) == 0;
  (void)es_in;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (new_dtype == SV_F32) return launch_in<float>(a, kv_dtype, B, s);
  return launch_in<__nv_bfloat16>(a, kv_dtype, B, s);
}

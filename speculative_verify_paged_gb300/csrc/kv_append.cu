// kv_block_append: scatter the K+1 new K/V rows of each sequence into the
// paged pools ("KV Cache + Speculative Decoding", section 6.2, append_token:
// page pos / block_size, slot pos % block_size), converting to the pool dtype.
#include <cuda_fp8.h>
#include <algorithm>
#include <cstring>
#include <type_traits>

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
}  // namespace sv

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

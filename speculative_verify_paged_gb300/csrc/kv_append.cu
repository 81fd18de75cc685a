// kv_block_append: scatter the K+1 new K/V rows of each sequence into the
// paged pools ("KV Cache + Speculative Decoding", section 6.2, append_token:
// page pos / block_size, slot pos % block_size), converting to the pool dtype.
#include <cuda_fp8.h>

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

// One CTA per (new position j, sequence b); threads stride over H_kv * d.
template <typename TIn, int KV>
__global__ void __launch_bounds__(256) kv_append_kernel(AppendArgs a) {
  pdl_wait();
  pdl_trigger();
  const int j = blockIdx.x, b = blockIdx.y;
  const int L = a.seq_lens[b];
  if (L < a.n_new || L > a.max_blocks * a.bs) {
    if (threadIdx.x == 0) atomic_or_status(a.status, SV_DEV_BAD_SEQ_LEN);
    return;
  }
  const int pos = L - a.n_new + j;
  const int blk = a.block_table[(int64_t)b * a.max_blocks + pos / a.bs];
  if (blk < 0 || blk >= a.num_blocks) {
    if (threadIdx.x == 0) atomic_or_status(a.status, SV_DEV_BAD_BLOCK);
    return;
  }
  const int slot = pos % a.bs;
  const int64_t base = (int64_t)blk * a.block_stride + (int64_t)slot * a.slot_stride;
  const int64_t src0 = ((int64_t)b * a.n_new + j) * a.H_kv * a.d;
  const TIn *kn = static_cast<const TIn *>(a.k_new) + src0;
  const TIn *vn = static_cast<const TIn *>(a.v_new) + src0;
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
  switch (kv_dtype) {
    case SV_F32: launch_k(kv_append_kernel<TIn, SV_F32>, grid, dim3(256), 0, s, 1, a); break;
    case SV_BF16: launch_k(kv_append_kernel<TIn, SV_BF16>, grid, dim3(256), 0, s, 1, a); break;
    case SV_FP8_E4M3: launch_k(kv_append_kernel<TIn, SV_FP8_E4M3>, grid, dim3(256), 0, s, 1, a); break;
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
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (new_dtype == SV_F32) return launch_in<float>(a, kv_dtype, B, s);
  return launch_in<__nv_bfloat16>(a, kv_dtype, B, s);
}

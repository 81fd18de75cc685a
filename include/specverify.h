/*
 * specverify.h -- C ABI of libspecverify.so: the target-model verification
 * step of speculative decoding on one GB300 (sm_103a).
 *
 * Three operations:
 *   kv_block_append     write the K+1 new K/V rows of every sequence into the
 *                       paged cache ("KV Cache + Speculative Decoding",
 *                       section 6.2, PagedKVCache.append_token: page pos/16,
 *                       slot pos%16);
 *   spec_verify_attn    paged GQA attention of the K+1 new query positions
 *                       over the whole cache with the offset causal mask
 *                       (same page, sections 5.2-5.3 and 6.3,
 *                       MQA_GQA_Attention.forward; walkerchi "KV Cache"
 *                       section 3.3; CS336 lecture 10 section 9.2 on
 *                       FlashDecoding-style split-KV);
 *   spec_verify_sample  the rejection-sampling pass: softmax of target and
 *                       draft logits, accept x_i with probability
 *                       min(1, p_i(x_i)/q_i(x_i)), resample at the first
 *                       rejection n from norm(max(0, p_n - q_n)), bonus token
 *                       from p_{K+1} when all K are accepted (quant67
 *                       "speculative decoding" section 3.1; "KV Cache +
 *                       Speculative Decoding" sections 7.1-7.3 and 7.6).
 *
 * Conventions shared by every call
 *   - All tensor arguments are DEVICE pointers, row-major, densely packed in
 *     the layout stated next to them. The caller owns every buffer, including
 *     workspaces; the library never allocates or frees memory and keeps no
 *     state between calls (apart from a per-thread error string and the
 *     static scratch array of spec_verify_sample_static).
 *   - Every call is asynchronous on `stream` (NULL = the legacy default
 *     stream). Outputs are valid once the stream has reached the call.
 *   - Argument errors are detected on the host before any launch: the call
 *     returns SV_ERR_INVALID_ARG / SV_ERR_UNSUPPORTED / SV_ERR_WORKSPACE,
 *     touches no memory and sets the message returned by
 *     sv_last_error_string(). A failed launch returns SV_ERR_CUDA.
 *   - Values that live on the device (seq_lens, block-table entries, draft
 *     tokens) are checked by the kernels. A bad value never causes an
 *     out-of-bounds access: the access is skipped and a bit of SV_DEV_* is
 *     OR-ed into *dev_status (a device int32 the caller zeroes; may be NULL).
 *     Outputs that depended on the bad value are unspecified.
 *   - No C++ exception crosses this interface.
 *
 * Paged KV cache
 *   K and V pools: [num_blocks][H_kv][block_size][d_head] by default
 *   (layout == NULL), i.e. one (block, kv-head) tile is block_size*d_head
 *   contiguous elements. A non-NULL sv_kv_layout gives other strides (in
 *   elements; d_head is always contiguous), e.g. a per-layer slice of a pool
 *   shaped [pages][page_size][layers][2][H_kv][d_head].
 *   block_table: int32 [B][max_blocks_per_seq]; entry t/block_size of row b
 *   is the physical block holding position t of sequence b.
 *   seq_lens: int32 [B]; seq_lens[b] counts every KV position of sequence b
 *   INCLUDING the n_new = K+1 new ones, so query j sits at absolute position
 *   seq_lens[b] - n_new + j and sees keys t <= seq_lens[b] - n_new + j.
 *   Rolling back after a rejection is the caller's job: the next round uses
 *   seq_lens[b] - n_new + num_accepted[b] + 1 (the resampled or bonus token
 *   is not yet in the cache).
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st *sv_stream_t;

typedef enum {
  SV_OK = 0,
  SV_ERR_INVALID_ARG = 1,   /* null pointer, bad size or shape            */
  SV_ERR_UNSUPPORTED = 2,   /* valid but not implemented (dtype, d_head)  */
  SV_ERR_WORKSPACE = 3,     /* workspace NULL or smaller than required    */
  SV_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed       */
  SV_ERR_TIMEOUT = 5        /* a bounded device wait ran out              */
} sv_status;

typedef enum { SV_F32 = 0, SV_BF16 = 1, SV_F16 = 2, SV_FP8_E4M3 = 3 } sv_dtype;

/* Bits OR-ed into *dev_status by the kernels. */
enum {
  SV_DEV_BAD_SEQ_LEN = 1,   /* seq_lens[b] < n_new or > max_blocks_per_seq*block_size */
  SV_DEV_BAD_BLOCK = 2,     /* block-table entry outside [0, num_blocks)             */
  SV_DEV_BAD_TOKEN = 4,     /* draft token outside [0, V)                             */
  SV_DEV_TIMEOUT = 8,       /* a bounded wait on an asynchronous copy ran out        */
  SV_DEV_NONFINITE = 16     /* a logit row's maximum is not finite                   */
};

/* Strides of the paged pools in elements (d_head is contiguous). Each must be
 * a multiple of 16 bytes for the bf16 / fp8 attention path. */
typedef struct {
  int64_t block_stride;
  int64_t head_stride;
  int64_t slot_stride;
} sv_kv_layout;

/* Message of the last error on the calling thread ("" after success). */
const char *sv_last_error_string(void);

/* Number of kernels this library has launched successfully in this process
 * (all threads, all devices). Host-side count, no device access; a caller
 * takes the difference around a region to count its launches. */
unsigned long long sv_kernel_launches(void);

/* ------------------------------------------------------------------------ *
 * kv_block_append
 *   Writes k_new[b][j][g][:] and v_new[b][j][g][:] (j = 0..n_new-1) to
 *   position pos = seq_lens[b] - n_new + j of sequence b: pool block
 *   block_table[b][pos / block_size], slot pos % block_size, kv head g.
 *   k_new, v_new: [B][n_new][H_kv][d_head] of new_dtype (SV_F32 or SV_BF16).
 *   kv_dtype SV_F32 stores the value, SV_BF16 its round-to-nearest-even
 *   bf16, SV_FP8_E4M3 the e4m3 code of x / scale[g] (fp32 division, round to
 *   nearest even, saturated to +-448); k_scale/v_scale: float [H_kv], fp8
 *   only (else ignored). Copy-on-write and block allocation stay with the
 *   caller: every table entry the positions need must already be valid.
 * ------------------------------------------------------------------------ */
sv_status kv_block_append(const void *k_new, const void *v_new, sv_dtype new_dtype,
                          void *k_cache, void *v_cache, sv_dtype kv_dtype,
                          const sv_kv_layout *layout,
                          const float *k_scale, const float *v_scale,
                          const int32_t *block_table, int max_blocks_per_seq,
                          const int32_t *seq_lens,
                          int B, int n_new, int H_kv, int d_head, int block_size,
                          int num_blocks, int32_t *dev_status, sv_stream_t stream);

/* ------------------------------------------------------------------------ *
 * spec_verify_attn
 *   out[b][j][h][:] = sum_t softmax_t(s_t) * V_b[t][g][:] with
 *   s_t = softmax_scale * q[b][j][h][:] . K_b[t][g][:], g = h / (H_q/H_kv),
 *   over keys t <= seq_lens[b] - n_new + j (the offset causal mask).
 *   q: [B][n_new][H_q][d_head] of q_dtype; out: same shape, out_dtype.
 *   Supported: kv_dtype SV_F32 with q/out SV_F32, or kv_dtype SV_BF16 /
 *   SV_FP8_E4M3 with q/out SV_BF16; d_head a multiple of 4 and <= 256; any
 *   block_size. The tensor-core kernel takes bf16 / fp8 caches with
 *   d_head 128, block_size 16, (H_q/H_kv) * n_new <= 64 and pool strides
 *   that are multiples of 16 bytes; every other supported shape runs on a
 *   CUDA-core kernel with fp32 arithmetic.
 *   fp8 pools hold e4m3 codes; the key / value is code * k_scale[g] /
 *   code * v_scale[g] (k_scale, v_scale: float [H_kv] on the device).
 *   workspace: at least spec_verify_attn_workspace_size(...) bytes of device
 *   memory, 256-byte aligned; its contents need no initialisation.
 * ------------------------------------------------------------------------ */
size_t spec_verify_attn_workspace_size(int B, int n_new, int H_q, int H_kv, int d_head,
                                       int max_blocks_per_seq, int block_size);

sv_status spec_verify_attn(const void *q, sv_dtype q_dtype,
                           const void *k_cache, const void *v_cache, sv_dtype kv_dtype,
                           const sv_kv_layout *layout,
                           const float *k_scale, const float *v_scale,
                           const int32_t *block_table, int max_blocks_per_seq,
                           const int32_t *seq_lens,
                           int B, int n_new, int H_q, int H_kv, int d_head,
                           int block_size, int num_blocks, float softmax_scale,
                           void *out, sv_dtype out_dtype,
                           void *workspace, size_t workspace_bytes,
                           int32_t *dev_status, sv_stream_t stream);

/* Same as spec_verify_attn with an explicit split size: the keys of each
 * sequence are cut into chunks of blocks_per_split blocks that run in
 * parallel and are merged by log-sum-exp. The result does not depend on the
 * split size up to rounding; the workspace must hold
 * spec_verify_attn_workspace_size_ex(..., blocks_per_split) bytes. */
size_t spec_verify_attn_workspace_size_ex(int B, int n_new, int H_q, int H_kv, int d_head,
                                          int max_blocks_per_seq, int block_size,
                                          int blocks_per_split);

sv_status spec_verify_attn_ex(const void *q, sv_dtype q_dtype,
                              const void *k_cache, const void *v_cache, sv_dtype kv_dtype,
                              const sv_kv_layout *layout,
                              const float *k_scale, const float *v_scale,
                              const int32_t *block_table, int max_blocks_per_seq,
                              const int32_t *seq_lens,
                              int B, int n_new, int H_q, int H_kv, int d_head,
                              int block_size, int num_blocks, float softmax_scale,
                              void *out, sv_dtype out_dtype,
                              void *workspace, size_t workspace_bytes,
                              int32_t *dev_status, int blocks_per_split, sv_stream_t stream);

/* ------------------------------------------------------------------------ *
 * spec_verify_sample
 *   p_i = softmax(target_logits[b][i][:] / T), i = 0..K (row K is p_{K+1}).
 *   q_i = softmax(draft[b][i][:] / T) (draft_is_probs == 0, draft logits of
 *   draft_dtype) or draft[b][i][:] as given (draft_is_probs == 1, SV_F32).
 *   For i = 0..K-1 draft x_i = draft_tokens[b][i] is accepted iff
 *   u_i * q_i(x_i) < p_i(x_i), u_i = uniforms[b][i][0]. At the first
 *   rejection n the token y = min{y : C(y) > v_n * C(V-1)} is drawn, C the
 *   running sum in ascending token id of max(0, p_n - q_n), v_n =
 *   uniforms[b][n][1]; if all K are accepted y is drawn the same way from
 *   p_K with v_K = uniforms[b][K][1].
 *   target_logits: [B][K+1][V] (SV_F32, SV_BF16 or SV_F16);
 *   draft: [B][K][V]; draft_tokens: int32 [B][K]; uniforms: float
 *   [B][K+1][2] in [0, 1).
 *   Outputs: out_tokens int32 [B][K+1] = x_0 .. x_{n-1}, y, then -1;
 *   num_accepted int32 [B] = n in [0, K] (emitted = n + 1);
 *   p_at_draft / q_at_draft: float [B][K] = p_i(x_i), q_i(x_i) (optional,
 *   may be NULL).
 *   Decisions are those of exact arithmetic: the fp32 result of a row is used
 *   only when a rounding bound certifies it; otherwise the row is
 *   re-evaluated in float-float arithmetic (about 1e-9 relative error per
 *   term).
 *   temperature > 0. V >= 1, K >= 0.
 *   workspace: at least spec_verify_sample_workspace_size(B, K, V) bytes of
 *   device memory, 256-byte aligned; its contents need no initialisation.
 * ------------------------------------------------------------------------ */
size_t spec_verify_sample_workspace_size(int B, int K, int V);

sv_status spec_verify_sample(const void *target_logits, sv_dtype logit_dtype,
                             const void *draft, sv_dtype draft_dtype, int draft_is_probs,
                             const int32_t *draft_tokens, const float *uniforms,
                             int B, int K, int V, float temperature,
                             int32_t *out_tokens, int32_t *num_accepted,
                             float *p_at_draft, float *q_at_draft,
                             void *workspace, size_t workspace_bytes,
                             int32_t *dev_status, sv_stream_t stream);

/* Same as spec_verify_sample with option bits:
 *   SV_SAMPLE_FORCE_EXACT  resolve every sequence with the extended-precision
 *                          pass instead of only the rows rounding could
 *                          affect (used by tests to exercise that pass). */
enum { SV_SAMPLE_FORCE_EXACT = 1 };

sv_status spec_verify_sample_ex(const void *target_logits, sv_dtype logit_dtype,
                                const void *draft, sv_dtype draft_dtype, int draft_is_probs,
                                const int32_t *draft_tokens, const float *uniforms,
                                int B, int K, int V, float temperature,
                                int32_t *out_tokens, int32_t *num_accepted,
                                float *p_at_draft, float *q_at_draft,
                                void *workspace, size_t workspace_bytes,
                                int32_t *dev_status, unsigned flags, sv_stream_t stream);

/* ------------------------------------------------------------------------ *
 * spec_verify_sample_static
 *   The pages have no counterpart to this call; it exists for callers that
 *   cannot allocate device memory when they verify a round (an engine that
 *   reserves all GPU memory for its KV pool at start-up and forbids later
 *   allocations, or a caller whose fixed interface cannot pass a workspace).
 *   Same as spec_verify_sample without the workspace arguments: the
 *   workspace (spec_verify_sample_workspace_size(B, K, V) bytes: a 48-byte
 *   record and 16 * ceil(V / 8192) bytes of chunk statistics per (sequence,
 *   position), 8 bytes per sequence, plus 140.25 KB of scratch for the
 *   float-float pass) goes to a 1 MiB static device array inside the
 *   library, which every GPU that loads the library holds until the process
 *   exits. For V = 128256 and K = 4 that is B <= 592; larger sizes return
 *   SV_ERR_UNSUPPORTED with a message.
 *   Allocates nothing (no cudaMalloc / cudaFree or allocating library call).
 *   The first call on a device looks up the array's device address (with
 *   that device current); make that first call before any stream capture.
 *   Every call on a device shares the one array and leaves its contents
 *   behind; no call needs it zeroed. Calls that overlap on the GPU (other
 *   streams, other host threads) race on the array: serialise them.
 * ------------------------------------------------------------------------ */
sv_status spec_verify_sample_static(const void *target_logits, sv_dtype logit_dtype,
                                    const void *draft, sv_dtype draft_dtype, int draft_is_probs,
                                    const int32_t *draft_tokens, const float *uniforms,
                                    int B, int K, int V, float temperature,
                                    int32_t *out_tokens, int32_t *num_accepted,
                                    float *p_at_draft, float *q_at_draft,
                                    int32_t *dev_status, sv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */

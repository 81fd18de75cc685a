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
 *   - Kernels are launched with programmatic stream serialization: a call
 *     may start while the previous kernel of the stream drains, and
 *     kv_block_append reads its inputs (new rows, table, lengths) before
 *     it waits for that kernel. A kernel of the caller that produces those
 *     inputs must therefore not release its dependents early
 *     (griddepcontrol.launch_dependents before its last write); kernels that
 *     never do (the default) and copies are safe.
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
  SV_ERR_TIMEOUT = 5,       /* a bounded device wait ran out              */
  SV_ERR_OUT_OF_BLOCKS = 6  /* the block manager has too few free pages   */
} sv_status;

typedef enum { SV_F32 = 0, SV_BF16 = 1, SV_F16 = 2, SV_FP8_E4M3 = 3 } sv_dtype;

/* Bits OR-ed into *dev_status by the kernels. */
enum {
  SV_DEV_BAD_SEQ_LEN = 1,   /* seq_lens[b] < n_new or > max_blocks_per_seq*block_size */
  SV_DEV_BAD_BLOCK = 2,     /* block-table entry outside [0, num_blocks)             */
  SV_DEV_BAD_TOKEN = 4,     /* draft token outside [0, V)                             */
  SV_DEV_TIMEOUT = 8,       /* a bounded wait on an asynchronous copy ran out        */
  SV_DEV_NONFINITE = 16,    /* a logit row's maximum is not finite                   */
  SV_DEV_BAD_TREE = 32,     /* a draft-tree parent index is not a valid BFS parent   */
  SV_DEV_BAD_WORK = 64      /* a work-list entry the library wrote is out of range   */
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

/* Test hooks for the bounded waits (no counterpart in the pages; they exist
 * so that a test can make a wait run out without faulting anything).
 *   wait_limit_ns: the limit every later launch gives each of its device
 *     waits (0 restores the default of one second);
 *   withhold: signals later launches leave unsent, so that a wait on them
 *     runs out:
 *       SV_TEST_WITHHOLD_COPIES   spec_verify_attn's tensor-core kernel
 *         issues no K/V copies (nothing is in flight when its waits give up);
 *       SV_TEST_WITHHOLD_ARRIVALS  CTA 0 of spec_verify_sample's
 *         float-float pass does not arrive at its grid barriers, so every
 *         CTA's wait there runs out (the pass runs when a decision is not
 *         certified, or always with SV_SAMPLE_FORCE_EXACT).
 * A wait that runs out sets SV_DEV_TIMEOUT in the call's device status and
 * the kernel returns (outputs of that call are not valid); the next call
 * with the hooks cleared is unaffected. Process-wide; not for production
 * use. */
enum { SV_TEST_WITHHOLD_COPIES = 1, SV_TEST_WITHHOLD_ARRIVALS = 2 };
void sv_test_hooks(unsigned long long wait_limit_ns, unsigned withhold);

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
 * kv_tree_commit
 *   After a tree round (spec_verify_attn_tree + spec_verify_sample_tree) the
 *   n_new node rows of sequence b sit at positions L - n_new + j (node j,
 *   L = seq_lens[b]). This moves the accepted path next to the root:
 *   position L - n_new + 1 + i takes the row of node path_nodes[b][i] for
 *   i < num_accepted[b], every kv head, K and V (every row read before any
 *   is written). Rolling the length back to L - n_new + num_accepted[b] + 1
 *   (sv_bm_commit_verify) then leaves the prefix, the root and the path in
 *   order ("KV Cache + Speculative Decoding", section 7's invariant).
 *   path_nodes int32 [B][n_new] and num_accepted int32 [B]: device, as
 *   spec_verify_sample_tree writes them (num_accepted in [0, n_new - 1],
 *   path entries in [1, n_new)); a bad value sets SV_DEV_* bits and leaves
 *   that sequence unchanged. Pools as for kv_block_append (SV_F32, SV_BF16
 *   or SV_FP8_E4M3 codes, any sv_kv_layout); n_new <= 64, d_head * element
 *   size <= 1024.
 * ------------------------------------------------------------------------ */
sv_status kv_tree_commit(void *k_cache, void *v_cache, sv_dtype kv_dtype, const sv_kv_layout *layout,
                         const int32_t *block_table, int max_blocks_per_seq, const int32_t *seq_lens,
                         const int32_t *path_nodes, const int32_t *num_accepted,
                         int B, int n_new, int H_kv, int d_head, int block_size, int num_blocks,
                         int32_t *dev_status, sv_stream_t stream);

/* ------------------------------------------------------------------------ *
 * spec_verify_attn
 *   out[b][j][h][:] = sum_t softmax_t(s_t) * V_b[t][g][:] with
 *   s_t = softmax_scale * q[b][j][h][:] . K_b[t][g][:], g = h / (H_q/H_kv),
 *   over keys t <= seq_lens[b] - n_new + j (the offset causal mask).
 *   q: [B][n_new][H_q][d_head] of q_dtype; out: same shape, out_dtype.
 *   Supported: kv_dtype SV_F32 with q/out SV_F32, or kv_dtype SV_BF16 /
 *   SV_FP8_E4M3 with q/out SV_BF16; d_head a multiple of 4 and <= 256; any
 *   block_size. The tensor-core kernel takes bf16 / fp8 caches with
 *   d_head 128, block_size 16, (H_q/H_kv) * n_new <= 128 and pool strides
 *   that are multiples of 16 bytes (q must then be 16-byte aligned, else
 *   SV_ERR_INVALID_ARG); every other supported shape runs on a CUDA-core
 *   kernel with fp32 arithmetic.
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
 * parallel and are merged by log-sum-exp. blocks_per_split = 0 asks for
 * balanced ranges instead (tensor-core path; other paths take their default
 * split): the 64-key tiles of all sequences, end to end, are cut into equal
 * ranges, one per CTA slot (two per SM) and kv head, whatever the lengths;
 * this suits small batches of very uneven lengths. The result does not
 * depend on the split size up to rounding; the workspace must hold
 * spec_verify_attn_workspace_size_ex(..., blocks_per_split) bytes
 * (SV_ERR_INVALID_ARG for blocks_per_split < 0; the size query returns 0). */
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
 * spec_verify_attn_tree
 *   Tree verification ("KV Cache + Speculative Decoding", Q14 and section
 *   8.2): the n_new new positions of sequence b are the nodes of a draft
 *   tree flattened in BFS order, node 0 the root (the last accepted token).
 *   Query j sees every cached key before the new positions and, of the new
 *   positions, exactly its ancestors A(j) (j itself included): key
 *   seq_lens[b] - n_new + i is visible to query j iff i is in A(j). A chain
 *   (tree_parent[b][j] = j - 1) gives spec_verify_attn's causal mask.
 *   tree_parent: int32 [B][n_new] device; tree_parent[b][0] = -1 and
 *   0 <= tree_parent[b][j] < j for j >= 1; a node with another parent sets
 *   SV_DEV_BAD_TREE and is given the chain mask. n_new <= 64. Other
 *   arguments, layouts and support as for spec_verify_attn; the workspace
 *   is spec_verify_attn_tree_workspace_size(...) bytes (spec_verify_attn's
 *   plus 8 bytes per node for the ancestor masks).
 * ------------------------------------------------------------------------ */
size_t spec_verify_attn_tree_workspace_size(int B, int n_new, int H_q, int H_kv, int d_head,
                                            int max_blocks_per_seq, int block_size);

sv_status spec_verify_attn_tree(const void *q, sv_dtype q_dtype,
                                const void *k_cache, const void *v_cache, sv_dtype kv_dtype,
                                const sv_kv_layout *layout,
                                const float *k_scale, const float *v_scale,
                                const int32_t *block_table, int max_blocks_per_seq,
                                const int32_t *seq_lens, const int32_t *tree_parent,
                                int B, int n_new, int H_q, int H_kv, int d_head, int block_size,
                                int num_blocks, float softmax_scale,
                                void *out, sv_dtype out_dtype,
                                void *workspace, size_t workspace_bytes,
                                int32_t *dev_status, sv_stream_t stream);

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
 * Top-p ("KV Cache + Speculative Decoding", section 7.5 and Q21: the target
 * distribution becomes p truncated to its own top-p set and renormalised;
 * the draft distribution q is whatever the draft sampled from, and the
 * rejection rule stays exact with both).
 *
 * The top-p set of a row of softmax(logits / T): order the tokens by logit,
 * largest first, equal logits by ascending token id; the set is the shortest
 * prefix of that order whose probability reaches top_p. The masses are
 * taken in fixed point (weights of the row relative to its maximum, rounded
 * to multiples of 2^-40, summed exactly), so the set is deterministic and
 * matches exact arithmetic unless top_p lies within 5e-7 (as a fraction of
 * the row mass) of a cumulative mass.
 *
 * spec_topp_filter
 *   out[r][x] = logits[r][x] for x in the top-p set of row r, -inf elsewhere;
 *   softmax(out[r] / T) is then the truncated, renormalised distribution.
 *   logits, out: [rows][V] of dtype (SV_F32, SV_BF16 or SV_F16); out may
 *   equal logits. 0 < top_p <= 1 (1 copies the rows); temperature > 0.
 *   V <= 2^28. A row with a NaN
 *   logit has it removed from the set and sets SV_DEV_NONFINITE; a row
 *   with a +inf logit or no finite logit is copied unchanged (the sampling
 *   flags it).
 *
 * spec_verify_sample_topp
 *   spec_verify_sample with every target row replaced by its top-p filtered
 *   row (p -> p-tilde, including the bonus row) and, when draft_topp is 1,
 *   every draft logit row filtered the same way (the draft sampled from its
 *   own top-p distribution); draft_topp needs draft logits. top_p = 1 is
 *   plain spec_verify_sample. The filtered rows live at the front of the
 *   workspace: spec_verify_sample_topp_workspace_size(...) bytes, 256-byte
 *   aligned.
 * ------------------------------------------------------------------------ */
sv_status spec_topp_filter(const void *logits, sv_dtype dtype, int rows, int V, float temperature, float top_p,
                           void *out, int32_t *dev_status, sv_stream_t stream);

size_t spec_verify_sample_topp_workspace_size(int B, int K, int V, sv_dtype logit_dtype, int draft_topp);

sv_status spec_verify_sample_topp(const void *target_logits, sv_dtype logit_dtype,
                                  const void *draft, sv_dtype draft_dtype, int draft_is_probs,
                                  const int32_t *draft_tokens, const float *uniforms,
                                  int B, int K, int V, float temperature, float top_p, int draft_topp,
                                  int32_t *out_tokens, int32_t *num_accepted,
                                  float *p_at_draft, float *q_at_draft,
                                  void *workspace, size_t workspace_bytes,
                                  int32_t *dev_status, sv_stream_t stream);

/* ------------------------------------------------------------------------ *
 * spec_verify_sample_tree
 *   Rejection sampling over a draft tree (the BFS tree of
 *   spec_verify_attn_tree; "KV Cache + Speculative Decoding", Q14 and
 *   section 8.2, exact rejection of quant67 "speculative decoding" section
 *   3.1). Per sequence, from the root u = 0: the residual starts as r = p_u;
 *   u's children, drafted from q_u, are tried in BFS order, child c with
 *   token x = tree_tokens[b][c] accepted iff uniforms[b][c][0] * q_u(x) <
 *   r(x); a rejection replaces r by norm(max(0, r - q_u)); an accepted child
 *   becomes u; when every child of u is rejected, or u is a leaf, the token
 *   y = min{y : C(y) > v C(V-1)} is drawn from r (C the running sum in token
 *   order, v = uniforms[b][u][1]). A chain is spec_verify_sample's rule.
 *   target_logits: [B][n][V] (SV_F32, SV_BF16 or SV_F16), row j the target
 *   distribution after node j; draft: [B][n][V] logits of the same dtype
 *   (draft_is_probs == 0, softmax at T) or f32 probabilities, row u the
 *   distribution u's children were drawn from (rows of leaves unused);
 *   tree_parent: int32 [B][n] as for spec_verify_attn_tree; tree_tokens:
 *   int32 [B][n] (entry 0 unused); uniforms: float [B][n][2] in [0, 1).
 *   Outputs: out_tokens int32 [B][n] = the accepted tokens, the drawn one,
 *   then -1; num_accepted int32 [B]; path_nodes int32 [B][n] = the accepted
 *   nodes in order, then -1 (the caller keeps their K/V rows).
 *   n <= 64, V <= 2^28, temperature > 0. A bad tree sets SV_DEV_BAD_TREE,
 *   a token outside [0, V) SV_DEV_BAD_TOKEN (that child is never accepted),
 *   a row without a finite maximum SV_DEV_NONFINITE.
 *   fp32 arithmetic in a fixed order: deterministic, and equal to exact
 *   arithmetic unless a uniform lies within ~1e-6 of its boundary.
 *   typical: NULL for the exact rule above, else typical acceptance (below).
 *   workspace: spec_verify_sample_tree_workspace_size(B, n) bytes (each
 *   row's (max, sum, entropy), 32 bytes per node), 256-byte aligned, no
 *   initialisation needed.
 * ------------------------------------------------------------------------ */
/* Typical acceptance (opt-in, not exact): a draft x at node u is accepted
 * iff p_u(x) > min(epsilon, delta * exp(-H(p_u))), H the entropy of p_u in
 * nats; the first child in BFS order that passes is taken, and when none
 * does the token is drawn from p_u itself (no residual). The draft rows are
 * not read (draft may be NULL). "speculative decoding" survey section 9.1,
 * "KV Cache + Speculative Decoding" section 8.2 and Q18. */
typedef struct {
  float epsilon;
  float delta;
} sv_typical_acceptance;

size_t spec_verify_sample_tree_workspace_size(int B, int n);

sv_status spec_verify_sample_tree(const void *target_logits, sv_dtype logit_dtype,
                                  const void *draft, sv_dtype draft_dtype, int draft_is_probs,
                                  const int32_t *tree_parent, const int32_t *tree_tokens,
                                  const float *uniforms, int B, int n, int V, float temperature,
                                  const sv_typical_acceptance *typical,
                                  int32_t *out_tokens, int32_t *num_accepted, int32_t *path_nodes,
                                  void *workspace, size_t workspace_bytes,
                                  int32_t *dev_status, sv_stream_t stream);

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
 *   The address is kept per device together with the id of the context it
 *   was found in; a call in a new context of the device (after the old one
 *   was destroyed, e.g. by cudaDeviceReset) looks it up again.
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

/* ------------------------------------------------------------------------ *
 * Host block manager of the paged cache ("KV Cache + Speculative Decoding",
 * section 6.2, PagedKVCache: a free list used as a stack, one reference count
 * per physical page, one block table per sequence, copy-on-write on a write
 * to a shared page, share_prefix over whole pages; "KV Cache" section 3.3,
 * PagedAttention.fork). Pure host code: no call touches the GPU, allocates
 * device memory or needs CUDA. One manager per paged pool; a manager is not
 * thread-safe (serialise the calls on one manager).
 *
 * Sequences are named by caller-chosen int64 ids and record their length in
 * tokens; a sequence of length L owns exactly ceil(L / page_size) pages.
 * Free pages are handed out from the end of the free list and released pages
 * go back on its end (sv_bm_free_list lists it bottom to top). A call that
 * fails (SV_ERR_INVALID_ARG for a bad id or size, SV_ERR_OUT_OF_BLOCKS when
 * the pool is too small) changes nothing, also for a batch of sequences.
 *
 * A verify round with the kernels above:
 *   1. sv_bm_extend(ids, n_new = K+1): pages for the K+1 new rows; run the
 *      returned copy-on-write pairs with sv_copy_blocks over every pool
 *      (every layer's K and V) before anything writes those pages;
 *   2. sv_bm_block_table(ids) -> block_table / seq_lens for kv_block_append,
 *      spec_verify_attn (seq_lens then count the K+1 new rows);
 *   3. after spec_verify_sample, sv_bm_commit_verify(ids, K+1, num_accepted)
 *      with num_accepted copied to the host: each length becomes
 *      L - (K+1) + num_accepted + 1 (every token of the sequence but the
 *      resampled or bonus one, which enters the cache as the first new row
 *      of the next round), and pages past the new length are released.
 * ------------------------------------------------------------------------ */
typedef struct sv_block_manager sv_block_manager;

/* A manager of pages 0 .. num_blocks-1 (all free, free list in ascending
 * order) of page_size tokens; *out = NULL on failure. */
sv_status sv_bm_create(int num_blocks, int page_size, sv_block_manager **out);
void sv_bm_destroy(sv_block_manager *bm);                  /* NULL is a no-op */
int sv_bm_num_free(const sv_block_manager *bm);            /* -1 if bm NULL   */
int sv_bm_ref_count(const sv_block_manager *bm, int block); /* -1 out of range */
/* Copies the free list, bottom to top, to out[0 .. *n-1]; *n is set even when
 * cap is too small (then SV_ERR_INVALID_ARG). */
sv_status sv_bm_free_list(const sv_block_manager *bm, int32_t *out, int cap, int *n);

/* A new sequence of n_tokens tokens on ceil(n_tokens / page_size) fresh
 * pages (count 1); its first page is the last entry of the free list. */
sv_status sv_bm_allocate(sv_block_manager *bm, int64_t seq_id, int64_t n_tokens);
/* Drops the sequence; its pages lose one reference each, in table order, and
 * a page whose count reaches 0 goes back on the free list. */
sv_status sv_bm_free(sv_block_manager *bm, int64_t seq_id);
/* dst (a new id) shares every page of src and takes its length. */
sv_status sv_bm_fork(sv_block_manager *bm, int64_t src, int64_t dst);
/* dst (a new id) shares the first n_tokens / page_size (rounded down) pages
 * of src and has length (n_tokens / page_size) * page_size;
 * 0 <= n_tokens <= len(src). */
sv_status sv_bm_share_prefix(sv_block_manager *bm, int64_t src, int64_t dst, int64_t n_tokens);

/* Makes positions len .. len+n_new-1 of each listed sequence writable and
 * adds n_new to each length, sequence by sequence in list order: a position
 * past the table opens a fresh page; the first position written on a page
 * whose count is above 1 moves this sequence's reference to a fresh page
 * and records the pair (old, fresh) in cow_src[i], cow_dst[i]. The caller
 * copies each old page onto its fresh page (sv_copy_blocks) before any
 * write to the fresh page. At most one pair per sequence, so cow_src and
 * cow_dst (host int32 arrays) need cow_cap >= n_seqs entries; *n_cow is the
 * number written. No fresh page is the old page of another pair.
 * seq_ids: host int64 [n_seqs], distinct. */
sv_status sv_bm_extend(sv_block_manager *bm, const int64_t *seq_ids, int n_seqs, int n_new,
                       int32_t *cow_src, int32_t *cow_dst, int cow_cap, int *n_cow);
/* Rollback: the length becomes new_len (0 <= new_len <= len); pages past
 * ceil(new_len / page_size) are released in table order as by sv_bm_free. */
sv_status sv_bm_truncate(sv_block_manager *bm, int64_t seq_id, int64_t new_len);
/* After a verify round that appended n_new = K+1 rows: truncates sequence i
 * to len - n_new + num_accepted[i] + 1. num_accepted: host int32 [n_seqs],
 * each in [0, n_new - 1]; every length must be >= n_new. */
sv_status sv_bm_commit_verify(sv_block_manager *bm, const int64_t *seq_ids, int n_seqs, int n_new,
                              const int32_t *num_accepted);
sv_status sv_bm_seq_len(const sv_block_manager *bm, int64_t seq_id, int64_t *len);
/* Writes the listed sequences' tables, row i = seq_ids[i], into the host
 * int32 array table[n_seqs][max_blocks_per_seq] (entries past a sequence's
 * pages = -1) and their lengths into the host int32 array seq_lens[n_seqs].
 * SV_ERR_INVALID_ARG if a sequence holds more than max_blocks_per_seq pages
 * or is longer than INT32_MAX. */
sv_status sv_bm_block_table(const sv_block_manager *bm, const int64_t *seq_ids, int n_seqs,
                            int max_blocks_per_seq, int32_t *table, int32_t *seq_lens);

/* ------------------------------------------------------------------------ *
 * sv_copy_blocks
 *   The device half of copy-on-write: for every pool p and pair i, copies
 *   block_bytes bytes from pools[p] + src[i] * block_stride_bytes to
 *   pools[p] + dst[i] * block_stride_bytes. pools: HOST array of n_pools
 *   device pointers (16-byte aligned), e.g. every layer's K and V pool with
 *   block_bytes = H_kv * block_size * d_head * element size for the default
 *   layout, or one pool of [pages][page_size][layers][2][H_kv][d_head] with
 *   block_bytes = its page size in bytes. block_bytes and block_stride_bytes:
 *   multiples of 16, stride >= bytes. src, dst: DEVICE int32 [n_pairs]; a
 *   pair with an entry outside [0, num_blocks) is skipped and sets
 *   SV_DEV_BAD_BLOCK in *dev_status. Pairs must not chain (no dst is also a
 *   src), which holds for the pairs of one sv_bm_extend call. The copy waits
 *   for the previous kernel of the stream (its pages may be the source).
 * ------------------------------------------------------------------------ */
sv_status sv_copy_blocks(void *const *pools, int n_pools, int64_t block_stride_bytes, int64_t block_bytes,
                         const int32_t *src, const int32_t *dst, int n_pairs, int num_blocks,
                         int32_t *dev_status, sv_stream_t stream);

/* ------------------------------------------------------------------------ *
 * Multi-head latent attention (MLA), absorbed form
 *   ("KV Cache + Speculative Decoding", sections 4.3-4.4: the cache holds,
 *   per token and layer, one row [c ; k^R] of d_c + d_r values shared by all
 *   heads; section 4.3.3 and Q22: the up-projection W_UK of head i is
 *   absorbed into its query and W_UV into the output projection.)
 *
 * kv_block_append_latent
 *   Writes c_new[b][j][:] (bf16 [B][n_new][d_latent]) into the paged pool
 *   cache (bf16 [num_blocks][block_size][d_latent]) at position
 *   seq_lens[b] - n_new + j: block block_table[b][pos / block_size], slot
 *   pos % block_size. d_latent = 576, block_size = 16 (SV_ERR_UNSUPPORTED
 *   otherwise). Pointers 16-byte aligned. A length outside
 *   [n_new, max_blocks_per_seq * 16] sets SV_DEV_BAD_SEQ_LEN, a block
 *   outside [0, num_blocks) SV_DEV_BAD_BLOCK; that row is not written.
 *   Waits for the previous kernel of the stream before its stores.
 *   dev_status may be NULL (device errors then go unreported).
 *
 * spec_verify_attn_mla
 *   q_lat: bf16 [B][n_new][H][d_c + d_r], the absorbed query of position j,
 *   head i: [W_UK[i]^T q^C ; q^R] (q^R already rotated). cache: bf16
 *   [num_blocks][block_size][d_c + d_r] (k^R already rotated). For every
 *   (b, j, i): score_t = q_lat . cache_row(t) * softmax_scale for keys
 *   t <= seq_lens[b] - n_new + j, w = softmax(score), and
 *   out[b][j][i][:] = sum_t w_t cache_row(t)[0 .. d_c) (bf16
 *   [B][n_new][H][d_c]). The caller multiplies by W_UV[i] (or folds it into
 *   W_O). softmax_scale: 1 / sqrt(d_head + d_r) in MLAAttention (section 6.3).
 *   d_c = 512, d_r = 64, block_size = 16, bf16 only (SV_ERR_UNSUPPORTED
 *   otherwise). workspace: spec_verify_attn_mla_workspace_size(...) bytes,
 *   256-byte aligned: the partial outputs of a split context (only when the
 *   batch is too small to fill the GPU) and the longest-first order of the
 *   sequences (batches of up to 4096). Device errors as for
 *   spec_verify_attn. Waits for
 *   the previous kernel of the stream before it reads anything.
 * ------------------------------------------------------------------------ */
sv_status kv_block_append_latent(const void *c_new, sv_dtype dtype, void *cache,
                                 const int32_t *block_table, int max_blocks_per_seq,
                                 const int32_t *seq_lens, int B, int n_new, int d_latent,
                                 int block_size, int num_blocks, int32_t *dev_status,
                                 sv_stream_t stream);

size_t spec_verify_attn_mla_workspace_size(int B, int n_new, int H, int max_blocks_per_seq);

sv_status spec_verify_attn_mla(const void *q_lat, sv_dtype q_dtype, const void *cache,
                               sv_dtype cache_dtype, const int32_t *block_table,
                               int max_blocks_per_seq, const int32_t *seq_lens, int B, int n_new,
                               int H, int d_c, int d_r, int block_size, int num_blocks,
                               float softmax_scale, void *out, void *workspace,
                               size_t workspace_bytes, int32_t *dev_status, sv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */

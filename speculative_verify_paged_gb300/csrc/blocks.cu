// Host block manager of the paged KV cache and the device copy of pages for
// copy-on-write.
//
// The manager follows the PagedKVCache sketch of "KV Cache + Speculative
// Decoding" section 6.2: the free pages form a stack (allocation pops from
// the end, release pushes on the end), every physical page has a reference
// count, and every sequence owns a block table; a write to a page whose count
// is above one first moves that reference to a fresh copy. fork follows
// "KV Cache" section 3.3 (PagedAttention): the new sequence shares every page
// of its source. Rollback after verification edits only the table and the
// length (section 7 of the first page: the cache ends each round holding
// every token but the last one).
//
// Each sequence also records its length; its table always holds exactly
// ceil(len / page_size) pages. Calls that change several sequences check
// everything first (ids, capacities, free pages) and change nothing when a
// check fails.

#include <algorithm>
#include <unordered_map>
#include <unordered_set>
#include <vector>
#include <new>

#include "sv_common.cuh"

struct sv_block_manager {
  struct Seq {
    std::vector<int32_t> pages;
    int64_t len = 0;
  };
  int num_blocks = 0;
  int page_size = 0;
  std::vector<int32_t> free_list;  // a stack: back() is the next page handed out
  std::vector<int32_t> ref;
  std::unordered_map<int64_t, Seq> seqs;

  int64_t pages_for(int64_t n_tokens) const { return (n_tokens + page_size - 1) / page_size; }

  void release(int32_t pid) {
    if (--ref[pid] == 0) free_list.push_back(pid);
  }
  int32_t pop() {
    const int32_t pid = free_list.back();
    free_list.pop_back();
    return pid;
  }
};

namespace {

using BM = sv_block_manager;
using sv::fail;
using sv::ok;

sv_status no_seq(int64_t id) { return fail(SV_ERR_INVALID_ARG, "no sequence with id %lld", (long long)id); }

// Checks a batch of distinct, existing sequence ids.
sv_status check_batch(const BM *bm, const int64_t *ids, int n) {
  if (n < 0 || (n > 0 && !ids)) return fail(SV_ERR_INVALID_ARG, "bad sequence list");
  std::unordered_set<int64_t> seen;
  seen.reserve((size_t)n * 2);
  for (int i = 0; i < n; ++i) {
    if (!bm->seqs.count(ids[i])) return no_seq(ids[i]);
    if (!seen.insert(ids[i]).second)
      return fail(SV_ERR_INVALID_ARG, "sequence %lld appears twice", (long long)ids[i]);
  }
  return SV_OK;
}

// Free pages an extend of this batch pops: one per page opened past a table's
// end, one per shared page written (counted against the counts as the earlier
// sequences of the batch leave them, so two sharers copy once).
int64_t pages_needed(const BM *bm, const int64_t *ids, int n, int n_new) {
  std::unordered_map<int32_t, int> drop;
  int64_t need = 0;
  for (int i = 0; i < n; ++i) {
    const BM::Seq &s = bm->seqs.at(ids[i]);
    if (n_new == 0) continue;
    const int64_t first = s.len / bm->page_size;
    const int64_t last = (s.len + n_new - 1) / bm->page_size;
    for (int64_t idx = first; idx <= last; ++idx) {
      if (idx >= (int64_t)s.pages.size()) {
        ++need;
        continue;
      }
      const int32_t pid = s.pages[idx];
      auto it = drop.find(pid);
      const int d = it == drop.end() ? 0 : it->second;
      if (bm->ref[pid] - d > 1) {
        ++need;
        drop[pid] = d + 1;
      }
    }
  }
  return need;
}

void truncate_seq(BM *bm, BM::Seq &s, int64_t new_len) {
  const size_t keep = (size_t)bm->pages_for(new_len);
  for (size_t i = keep; i < s.pages.size(); ++i) bm->release(s.pages[i]);
  s.pages.resize(keep);
  s.len = new_len;
}

}  // namespace

#define SV_BM_TRY(body)                                                   \
  try {                                                                   \
    body                                                                  \
  } catch (const std::bad_alloc &) {                                      \
    return fail(SV_ERR_INVALID_ARG, "host memory exhausted");             \
  } catch (...) {                                                         \
    return fail(SV_ERR_INVALID_ARG, "unexpected host exception");         \
  }

extern "C" sv_status sv_bm_create(int num_blocks, int page_size, sv_block_manager **out) {
  if (!out) return fail(SV_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (num_blocks < 1 || page_size < 1)
    return fail(SV_ERR_INVALID_ARG, "num_blocks (%d) and page_size (%d) must be positive", num_blocks,
                page_size);
  SV_BM_TRY({
    BM *bm = new BM();
    bm->num_blocks = num_blocks;
    bm->page_size = page_size;
    bm->free_list.resize(num_blocks);
    for (int i = 0; i < num_blocks; ++i) bm->free_list[i] = i;
    bm->ref.assign(num_blocks, 0);
    *out = bm;
    return ok();
  })
}

extern "C" void sv_bm_destroy(sv_block_manager *bm) { delete bm; }

extern "C" int sv_bm_num_free(const sv_block_manager *bm) { return bm ? (int)bm->free_list.size() : -1; }

extern "C" int sv_bm_ref_count(const sv_block_manager *bm, int block) {
  if (!bm || block < 0 || block >= bm->num_blocks) return -1;
  return bm->ref[block];
}

extern "C" sv_status sv_bm_free_list(const sv_block_manager *bm, int32_t *out, int cap, int *n) {
  if (!bm || !n || cap < 0 || (cap > 0 && !out)) return fail(SV_ERR_INVALID_ARG, "bad arguments");
  *n = (int)bm->free_list.size();
  if (cap < *n) return fail(SV_ERR_INVALID_ARG, "cap %d < %d free pages", cap, *n);
  for (int i = 0; i < *n; ++i) out[i] = bm->free_list[i];
  return ok();
}

extern "C" sv_status sv_bm_allocate(sv_block_manager *bm, int64_t seq_id, int64_t n_tokens) {
  if (!bm) return fail(SV_ERR_INVALID_ARG, "manager is NULL");
  if (bm->seqs.count(seq_id)) return fail(SV_ERR_INVALID_ARG, "sequence %lld exists", (long long)seq_id);
  if (n_tokens < 0) return fail(SV_ERR_INVALID_ARG, "n_tokens < 0");
  const int64_t n = bm->pages_for(n_tokens);
  if (n > (int64_t)bm->free_list.size())
    return fail(SV_ERR_OUT_OF_BLOCKS, "%lld pages needed, %zu free", (long long)n, bm->free_list.size());
  SV_BM_TRY({
    BM::Seq s;
    s.pages.reserve((size_t)n);
    s.len = n_tokens;
    for (int64_t i = 0; i < n; ++i) s.pages.push_back(bm->free_list[bm->free_list.size() - 1 - i]);
    bm->seqs.emplace(seq_id, std::move(s));
    bm->free_list.resize(bm->free_list.size() - (size_t)n);
    for (int32_t pid : bm->seqs[seq_id].pages) bm->ref[pid] = 1;
    return ok();
  })
}

extern "C" sv_status sv_bm_free(sv_block_manager *bm, int64_t seq_id) {
  if (!bm) return fail(SV_ERR_INVALID_ARG, "manager is NULL");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return no_seq(seq_id);
  for (int32_t pid : it->second.pages) bm->release(pid);
  bm->seqs.erase(it);
  return ok();
}

static sv_status share(sv_block_manager *bm, int64_t src, int64_t dst, int64_t n_pages, int64_t len) {
  SV_BM_TRY({
    const BM::Seq &s = bm->seqs.at(src);
    BM::Seq d;
    d.pages.assign(s.pages.begin(), s.pages.begin() + n_pages);
    d.len = len;
    auto placed = bm->seqs.emplace(dst, std::move(d));
    for (int32_t pid : placed.first->second.pages) ++bm->ref[pid];
    return ok();
  })
}

extern "C" sv_status sv_bm_fork(sv_block_manager *bm, int64_t src, int64_t dst) {
  if (!bm) return fail(SV_ERR_INVALID_ARG, "manager is NULL");
  auto it = bm->seqs.find(src);
  if (it == bm->seqs.end()) return no_seq(src);
  if (bm->seqs.count(dst)) return fail(SV_ERR_INVALID_ARG, "sequence %lld exists", (long long)dst);
  return share(bm, src, dst, (int64_t)it->second.pages.size(), it->second.len);
}

extern "C" sv_status sv_bm_share_prefix(sv_block_manager *bm, int64_t src, int64_t dst, int64_t n_tokens) {
  if (!bm) return fail(SV_ERR_INVALID_ARG, "manager is NULL");
  auto it = bm->seqs.find(src);
  if (it == bm->seqs.end()) return no_seq(src);
  if (bm->seqs.count(dst)) return fail(SV_ERR_INVALID_ARG, "sequence %lld exists", (long long)dst);
  if (n_tokens < 0 || n_tokens > it->second.len)
    return fail(SV_ERR_INVALID_ARG, "n_tokens %lld outside [0, %lld]", (long long)n_tokens,
                (long long)it->second.len);
  const int64_t n = n_tokens / bm->page_size;
  return share(bm, src, dst, n, n * bm->page_size);
}

extern "C" sv_status sv_bm_extend(sv_block_manager *bm, const int64_t *seq_ids, int n_seqs, int n_new,
                                  int32_t *cow_src, int32_t *cow_dst, int cow_cap, int *n_cow) {
  if (!bm || !n_cow) return fail(SV_ERR_INVALID_ARG, "manager or n_cow is NULL");
  *n_cow = 0;
  if (n_new < 0) return fail(SV_ERR_INVALID_ARG, "n_new < 0");
  sv_status st = check_batch(bm, seq_ids, n_seqs);
  if (st != SV_OK) return st;
  if (cow_cap < n_seqs || (n_seqs > 0 && (!cow_src || !cow_dst)))
    return fail(SV_ERR_INVALID_ARG, "copy-on-write arrays must hold n_seqs (%d) pairs", n_seqs);
  const int64_t need = pages_needed(bm, seq_ids, n_seqs, n_new);
  if (need > (int64_t)bm->free_list.size())
    return fail(SV_ERR_OUT_OF_BLOCKS, "%lld pages needed, %zu free", (long long)need, bm->free_list.size());
  SV_BM_TRY({
    // reserve first so that no push_back below can throw half-way
    for (int i = 0; i < n_seqs; ++i) {
      BM::Seq &s = bm->seqs.at(seq_ids[i]);
      s.pages.reserve((size_t)bm->pages_for(s.len + n_new));
    }
    int nc = 0;
    for (int i = 0; i < n_seqs; ++i) {
      BM::Seq &s = bm->seqs.at(seq_ids[i]);
      if (n_new == 0) continue;
      const int64_t first = s.len / bm->page_size;
      const int64_t last = (s.len + n_new - 1) / bm->page_size;
      for (int64_t idx = first; idx <= last; ++idx) {
        if (idx >= (int64_t)s.pages.size()) {
          const int32_t pid = bm->pop();
          bm->ref[pid] = 1;
          s.pages.push_back(pid);
          continue;
        }
        const int32_t pid = s.pages[idx];
        if (bm->ref[pid] > 1) {
          const int32_t fresh = bm->pop();
          cow_src[nc] = pid;
          cow_dst[nc] = fresh;
          ++nc;
          --bm->ref[pid];
          bm->ref[fresh] = 1;
          s.pages[idx] = fresh;
        }
      }
      s.len += n_new;
    }
    *n_cow = nc;
    return ok();
  })
}

extern "C" sv_status sv_bm_truncate(sv_block_manager *bm, int64_t seq_id, int64_t new_len) {
  if (!bm) return fail(SV_ERR_INVALID_ARG, "manager is NULL");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return no_seq(seq_id);
  if (new_len < 0 || new_len > it->second.len)
    return fail(SV_ERR_INVALID_ARG, "new_len %lld outside [0, %lld]", (long long)new_len,
                (long long)it->second.len);
  truncate_seq(bm, it->second, new_len);
  return ok();
}

extern "C" sv_status sv_bm_commit_verify(sv_block_manager *bm, const int64_t *seq_ids, int n_seqs, int n_new,
                                         const int32_t *num_accepted) {
  if (!bm) return fail(SV_ERR_INVALID_ARG, "manager is NULL");
  if (n_new < 1) return fail(SV_ERR_INVALID_ARG, "n_new < 1");
  sv_status st = check_batch(bm, seq_ids, n_seqs);
  if (st != SV_OK) return st;
  if (n_seqs > 0 && !num_accepted) return fail(SV_ERR_INVALID_ARG, "num_accepted is NULL");
  for (int i = 0; i < n_seqs; ++i) {
    const int32_t a = num_accepted[i];
    if (a < 0 || a > n_new - 1)
      return fail(SV_ERR_INVALID_ARG, "num_accepted[%d] = %d outside [0, %d]", i, a, n_new - 1);
    if (bm->seqs.at(seq_ids[i]).len < n_new)
      return fail(SV_ERR_INVALID_ARG, "sequence %lld is shorter than n_new", (long long)seq_ids[i]);
  }
  for (int i = 0; i < n_seqs; ++i) {
    BM::Seq &s = bm->seqs.at(seq_ids[i]);
    truncate_seq(bm, s, s.len - n_new + num_accepted[i] + 1);
  }
  return ok();
}

extern "C" sv_status sv_bm_seq_len(const sv_block_manager *bm, int64_t seq_id, int64_t *len) {
  if (!bm || !len) return fail(SV_ERR_INVALID_ARG, "manager or len is NULL");
  auto it = bm->seqs.find(seq_id);
  if (it == bm->seqs.end()) return no_seq(seq_id);
  *len = it->second.len;
  return ok();
}

extern "C" sv_status sv_bm_block_table(const sv_block_manager *bm, const int64_t *seq_ids, int n_seqs,
                                       int max_blocks_per_seq, int32_t *table, int32_t *seq_lens) {
  if (!bm) return fail(SV_ERR_INVALID_ARG, "manager is NULL");
  if (max_blocks_per_seq < 1) return fail(SV_ERR_INVALID_ARG, "max_blocks_per_seq < 1");
  if (n_seqs < 0 || (n_seqs > 0 && (!seq_ids || !table || !seq_lens)))
    return fail(SV_ERR_INVALID_ARG, "bad arrays");
  for (int i = 0; i < n_seqs; ++i) {
    auto it = bm->seqs.find(seq_ids[i]);
    if (it == bm->seqs.end()) return no_seq(seq_ids[i]);
    if ((int64_t)it->second.pages.size() > max_blocks_per_seq)
      return fail(SV_ERR_INVALID_ARG, "sequence %lld holds %zu pages > max_blocks_per_seq %d",
                  (long long)seq_ids[i], it->second.pages.size(), max_blocks_per_seq);
    if (it->second.len > INT32_MAX) return fail(SV_ERR_INVALID_ARG, "length above INT32_MAX");
  }
  for (int i = 0; i < n_seqs; ++i) {
    const BM::Seq &s = bm->seqs.at(seq_ids[i]);
    int32_t *row = table + (int64_t)i * max_blocks_per_seq;
    const int np = (int)s.pages.size();
    for (int j = 0; j < np; ++j) row[j] = s.pages[j];
    for (int j = np; j < max_blocks_per_seq; ++j) row[j] = -1;
    seq_lens[i] = (int32_t)s.len;
  }
  return ok();
}

// ------------------------------------------------------------ page copy ---

namespace sv {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyVecPerCta = kCopyThreads * 8;  // 16-byte vectors one CTA moves (32 KB)
constexpr int kCopyPools = 32;                     // pool pointers per launch

struct CopyPools {
  char *p[kCopyPools];
};

// grid (n_pairs, pools in this launch, slices of a page); each CTA copies one
// 32 KB slice of one page of one pool. The source pages may have been written
// by the previous kernel in the stream, so the copy waits for it first.
__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(CopyPools pools, int64_t stride_vec,
                                                                   int64_t page_vec, const int32_t *src,
                                                                   const int32_t *dst, int num_blocks,
                                                                   int32_t *status) {
  pdl_wait();
  pdl_trigger();
  const int s = __ldg(src + blockIdx.x);
  const int d = __ldg(dst + blockIdx.x);
  if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) atomic_or_status(status, SV_DEV_BAD_BLOCK);
    return;
  }
  const uint4 *from = reinterpret_cast<const uint4 *>(pools.p[blockIdx.y]) + (int64_t)s * stride_vec;
  uint4 *to = reinterpret_cast<uint4 *>(pools.p[blockIdx.y]) + (int64_t)d * stride_vec;
  constexpr int kU = kCopyVecPerCta / kCopyThreads;
  for (int64_t v = (int64_t)blockIdx.z * kCopyVecPerCta + threadIdx.x; v < page_vec;
       v += (int64_t)gridDim.z * kCopyVecPerCta) {
    uint4 r[kU];
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (v + u * kCopyThreads < page_vec) r[u] = from[v + u * kCopyThreads];
#pragma unroll
    for (int u = 0; u < kU; ++u)
      if (v + u * kCopyThreads < page_vec) to[v + u * kCopyThreads] = r[u];
  }
}

}  // namespace
}  // namespace sv

extern "C" sv_status sv_copy_blocks(void *const *pools, int n_pools, int64_t block_stride_bytes,
                                    int64_t block_bytes, const int32_t *src, const int32_t *dst, int n_pairs,
                                    int num_blocks, int32_t *dev_status, sv_stream_t stream) {
  using namespace sv;
  if (n_pairs < 0 || n_pools < 0 || num_blocks < 1) return fail(SV_ERR_INVALID_ARG, "bad sizes");
  if (n_pairs == 0 || n_pools == 0) return ok();
  if (!pools || !src || !dst) return fail(SV_ERR_INVALID_ARG, "NULL pointer");
  if (block_bytes <= 0 || block_bytes % 16 || block_stride_bytes % 16 || block_stride_bytes < block_bytes)
    return fail(SV_ERR_INVALID_ARG,
                "block_bytes (%lld) and block_stride_bytes (%lld) must be positive multiples of 16 "
                "with stride >= bytes",
                (long long)block_bytes, (long long)block_stride_bytes);
  for (int i = 0; i < n_pools; ++i)
    if (!pools[i] || !aligned(pools[i], 16)) return fail(SV_ERR_INVALID_ARG, "pool %d NULL or not 16-byte aligned", i);
  const int64_t page_vec = block_bytes / 16;
  const unsigned slices = (unsigned)std::min<int64_t>((page_vec + kCopyVecPerCta - 1) / kCopyVecPerCta, 65535);
  for (int base = 0; base < n_pools; base += kCopyPools) {
    CopyPools cp = {};
    const int np = std::min(kCopyPools, n_pools - base);
    for (int i = 0; i < np; ++i) cp.p[i] = static_cast<char *>(pools[base + i]);
    const cudaError_t e = launch_k(copy_blocks_kernel, dim3((unsigned)n_pairs, (unsigned)np, slices),
                                   dim3(kCopyThreads), 0, (cudaStream_t)stream, 1, cp,
                                   block_stride_bytes / 16, page_vec, src, dst, num_blocks, dev_status);
    if (e != cudaSuccess) return fail(SV_ERR_CUDA, "copy_blocks launch: %s", cudaGetErrorString(e));
  }
  return ok();
}

"""Oracle for the paged KV append of the K+1 new positions.

Follows "KV Cache + Speculative Decoding" section 6.2 (PagedKVCache.append_token:
page index pos // page_size, slot pos % page_size, write k/v of every kv head
into that slot) with the paged pool layout [num_blocks, H_kv, block_size, d].
The new rows of sequence b go to positions L_b - n_new + j, j = 0..n_new-1,
where L_b = seq_lens[b] already counts them. Copy-on-write and page
allocation are the caller's job (the block table is given).

Storage conversion: f32 pools store the fp32 value, bf16 pools the
round-to-nearest-even bf16 value, fp8 pools the e4m3 code of x / scale[g]
(see fp8.py for the rounding reading).
"""
import numpy as np
import torch

from . import fp8 as _fp8


def kv_block_append(k_cache, v_cache, k_new, v_new, block_table, seq_lens,
                    block_size=16, kv_dtype="bf16", k_scale=None, v_scale=None):
    """Return new (k_cache, v_cache) CPU tensors with the rows written."""
    kc = k_cache.detach().cpu().clone()
    vc = v_cache.detach().cpu().clone()
    kn = k_new.detach().cpu().to(torch.float32)
    vn = v_new.detach().cpu().to(torch.float32)
    table = block_table.detach().cpu().numpy()
    lens = seq_lens.detach().cpu().numpy()
    B, n_new, H_kv, _ = kn.shape
    for b in range(B):
        for j in range(n_new):
            pos = int(lens[b]) - n_new + j
            blk = int(table[b, pos // block_size])
            slot = pos % block_size
            for g in range(H_kv):
                for cache, new, scale in ((kc, kn, k_scale), (vc, vn, v_scale)):
                    row = new[b, j, g]
                    if kv_dtype == "fp8_e4m3":
                        s = np.float32(scale[g].item())
                        code = _fp8.quantize(row.numpy(), s)
                        cache[blk, g, slot] = torch.from_numpy(code)
                    else:
                        cache[blk, g, slot] = row.to(cache.dtype)
    return kc, vc


def kv_tree_commit(k_cache, v_cache, block_table, seq_lens, n_new, path_nodes, num_accepted,
                   block_size=16):
    """Return new (k_cache, v_cache) with each sequence's accepted tree path
    moved next to the root.

    After a tree round ("KV Cache + Speculative Decoding", Q14 and section
    8.2) the n_new node rows sit at positions L - n_new + j (node j). The
    cache must then hold the prefix, the root and the accepted path, in
    order (the generation-loop invariant of section 7: every token of the
    sequence but the last one is cached): position L - n_new + 1 + i takes
    the row of node path_nodes[b][i], i < num_accepted[b], for every kv head
    of K and V. Other positions are left as they are (the rollback drops
    them).
    """
    kc = k_cache.detach().cpu().clone()
    vc = v_cache.detach().cpu().clone()
    src_k = k_cache.detach().cpu()
    src_v = v_cache.detach().cpu()
    table = block_table.detach().cpu().numpy()
    lens = seq_lens.detach().cpu().numpy()
    path = path_nodes.detach().cpu().numpy()
    nacc = num_accepted.detach().cpu().numpy()
    for b in range(table.shape[0]):
        base = int(lens[b]) - n_new
        for i in range(int(nacc[b])):
            s, d = base + int(path[b, i]), base + 1 + i
            sb, ss = int(table[b, s // block_size]), s % block_size
            db, ds = int(table[b, d // block_size]), d % block_size
            kc[db, :, ds] = src_k[sb, :, ss]
            vc[db, :, ds] = src_v[sb, :, ss]
    return kc, vc

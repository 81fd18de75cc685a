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

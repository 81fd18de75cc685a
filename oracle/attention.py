"""Oracle for paged GQA verify attention (fp64).

Follows "KV Cache + Speculative Decoding":
  * section 5.2 / 5.3: a per-sequence block table maps logical block
    t // block_size to a physical block; slot t % block_size inside it
    (PagedKVCache.append_token addressing in section 6.2);
  * section 6.3 MQA_GQA_Attention.forward: kv head g serves query heads
    g*G .. g*G+G-1 (repeat_interleave by the group size G = H_q / H_kv),
    scores q.k / sqrt(d_head), a causal mask tril(ones(L_new, L_total),
    diagonal = L_total - L_new), softmax over keys, weights @ V.

Step 1 (dense gather) rebuilds a contiguous per-sequence cache from the pool;
step 2 is textbook attention on it. No tiling, no online softmax, no splits.

Pool layout: [num_blocks, H_kv, block_size, d_head]. seq_lens[b] counts all
KV positions of sequence b including the n_new new ones, so query j sits at
absolute position L_b - n_new + j and sees keys t <= L_b - n_new + j.
fp8 pools hold e4m3 codes; the value is decode(code) * scale[g] (fp64).

Draft trees ("KV Cache + Speculative Decoding", Q14 and section 8.2): the
n_new new positions are tree nodes flattened in BFS order, node 0 the root;
the mask is M[j][i] = 1 iff i is an ancestor of j (j included), so query j
sees the keys before the new positions and the new positions of its
ancestors. A chain (parent j - 1) is the causal mask above.
"""
import numpy as np

from . import fp8 as _fp8


def _to_f64(x):
    import torch
    if isinstance(x, torch.Tensor):
        if x.dtype == torch.uint8:
            return x.cpu().numpy()
        return x.detach().cpu().to(torch.float64).numpy()
    return np.asarray(x)


def gather_dense(pool, block_table_row, L, block_size, scale=None, is_fp8=False):
    """Contiguous [L, H_kv, d] fp64 cache of one sequence from the paged pool."""
    pool = _to_f64(pool)
    table = np.asarray(block_table_row)
    t = np.arange(L)
    blk = table[t // block_size].astype(np.int64)     # physical block of position t
    slot = t % block_size                              # slot inside that block
    rows = pool[blk, :, slot, :]                       # [L, H_kv, d]
    if is_fp8:
        return _fp8.decode(rows) * np.asarray(scale, dtype=np.float64)[None, :, None]
    return rows.astype(np.float64)


def ancestors(parent, j):
    """A(j): node j and every node on its path to the root."""
    out = []
    while j >= 0:
        out.append(j)
        j = parent[j]
    return out


def tree_visibility(parent, L):
    """[n_new, L] bool: key t visible to query j (the Q14 mask over the new
    positions, every earlier key visible)."""
    n_new = len(parent)
    vis = np.zeros((n_new, L), dtype=bool)
    vis[:, : L - n_new] = True
    for j in range(n_new):
        for i in ancestors(parent, j):
            vis[j, L - n_new + i] = True
    return vis


def dense_attention(q, Kd, Vd, n_new, softmax_scale, parent=None):
    """Textbook GQA attention of the n_new queries of one sequence.

    q: [n_new, H_q, d]; Kd, Vd: [L, H_kv, d] (fp64). Returns [n_new, H_q, d].
    parent: the draft tree's parent indices (None: the causal chain).
    """
    q = np.asarray(q, dtype=np.float64)
    L = Kd.shape[0]
    H_q, H_kv = q.shape[1], Kd.shape[1]
    G = H_q // H_kv
    out = np.empty_like(q)
    if parent is None:
        visible = np.tril(np.ones((n_new, L), dtype=bool), k=L - n_new)
    else:
        visible = tree_visibility(parent, L)
    for h in range(H_q):
        g = h // G
        scores = (q[:, h, :] @ Kd[:, g, :].T) * softmax_scale          # [n_new, L]
        scores = np.where(visible, scores, -np.inf)
        scores = scores - scores.max(axis=1, keepdims=True)
        w = np.exp(scores)
        w = w / w.sum(axis=1, keepdims=True)
        out[:, h, :] = w @ Vd[:, g, :]
    return out


def verify_attention(q, k_cache, v_cache, block_table, seq_lens, softmax_scale,
                     block_size=16, kv_dtype="bf16", k_scale=None, v_scale=None,
                     batch_indices=None, tree_parent=None):
    """Attention output [B, n_new, H_q, d] in fp64 (rows of unlisted b are NaN)."""
    q = _to_f64(q)
    B, n_new = q.shape[0], q.shape[1]
    table = _to_f64(block_table).astype(np.int64)
    lens = _to_f64(seq_lens).astype(np.int64)
    is_fp8 = kv_dtype == "fp8_e4m3"
    ks = None if k_scale is None else _to_f64(k_scale)
    vs = None if v_scale is None else _to_f64(v_scale)
    kc, vc = _to_f64(k_cache), _to_f64(v_cache)
    out = np.full(q.shape, np.nan, dtype=np.float64)
    for b in (range(B) if batch_indices is None else batch_indices):
        L = int(lens[b])
        Kd = gather_dense(kc, table[b], L, block_size, ks, is_fp8)
        Vd = gather_dense(vc, table[b], L, block_size, vs, is_fp8)
        par = None if tree_parent is None else [int(x) for x in _to_f64(tree_parent)[b]]
        out[b] = dense_attention(q[b], Kd, Vd, n_new, softmax_scale, par)
    return out

"""Oracle for paged MLA verify attention (fp64). Test infrastructure: only
tests, the smoke check and the benchmark's CPU baseline use it.

Follows "KV Cache + Speculative Decoding":
  * section 4.3.1: only the latent c_t (d_c wide) is cached; head i rebuilds
    its key and value as W_UK[i] c_t and W_UV[i] c_t (d_head x d_c each);
  * section 4.4.2: decoupled RoPE: a rotated d_r-wide key k^R_t, shared by
    all heads, is cached beside the latent; the score of head i is
    q^C_i . k^C_i + q^R_i . k^R;
  * section 4.4.3: the cache holds d_c + d_r numbers per token and layer;
  * section 4.3.3 and Q22 (absorb): q^C_i . (W_UK[i] c) = (W_UK[i]^T q^C_i) . c
    and out_i = W_UV[i] (sum_s w_s c_s), so attention runs on the latent;
  * section 6.3, MLAAttention.forward: scores divided by sqrt(d_head + d_r),
    the causal mask tril(ones(L_new, L_tot), diagonal = L_tot - L_new),
    softmax over keys, weights times values; _rope rotates consecutive pairs
    (x[2k], x[2k+1]) by pos * base^(-2k/D).

The absorbed problem (the one the GPU path solves): per sequence, query row
(position j, head i) q_lat = [W_UK[i]^T q^C ; q^R] of width d_c + d_r; cache
row per token [c ; k^R]; score = q_lat . row * scale; output latent
o = sum_s w_s row_s[:d_c] (width d_c), which the caller multiplies by W_UV[i]
(or folds into the output projection).

Pool layout: [num_blocks, block_size, d_c + d_r] (one latent row per token,
no head axis). Block table and seq_lens as in the GQA oracle: seq_lens[b]
counts every position including the n_new new ones, query j sits at
L - n_new + j and sees keys t <= L - n_new + j.
"""
import math

import numpy as np


def _f64(x):
    import torch
    if isinstance(x, torch.Tensor):
        return x.detach().cpu().to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def rope(x, positions, base=10000.0):
    """Rotate consecutive pairs of the last axis of x [..., L, D] by pos * theta_k,
    theta_k = base^(-2k/D) (section 6.3, _rope); positions [L]."""
    x = _f64(x)
    D = x.shape[-1]
    assert D % 2 == 0
    k = np.arange(D // 2, dtype=np.float64)
    theta = base ** (-2.0 * k / D)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * theta[None, :]   # [L, D/2]
    c, s = np.cos(ang), np.sin(ang)
    re, im = x[..., 0::2], x[..., 1::2]
    out = np.empty_like(x)
    out[..., 0::2] = re * c - im * s
    out[..., 1::2] = re * s + im * c
    return out


def naive_heads_attention(q_c, q_r, c_kv, k_r, W_UK, W_UV, scale):
    """The un-absorbed form of one sequence (section 6.3): q_c [n, H, d_head],
    q_r [n, H, d_r] (rotated), c_kv [L, d_c], k_r [L, d_r] (rotated),
    W_UK, W_UV [H, d_head, d_c]. Keys and values are rebuilt per head.
    Returns [n, H, d_head]."""
    q_c, q_r, c_kv, k_r = _f64(q_c), _f64(q_r), _f64(c_kv), _f64(k_r)
    W_UK, W_UV = _f64(W_UK), _f64(W_UV)
    n, H, _ = q_c.shape
    L = c_kv.shape[0]
    k_c = np.einsum("hdc,lc->hld", W_UK, c_kv)           # [H, L, d_head]
    v = np.einsum("hdc,lc->hld", W_UV, c_kv)
    scores = np.einsum("nhd,hld->hnl", q_c, k_c) + np.einsum("nhr,lr->hnl", q_r, k_r)
    scores = scores * scale
    visible = np.tril(np.ones((n, L), dtype=bool), k=L - n)
    scores = np.where(visible[None], scores, -np.inf)
    scores -= scores.max(axis=-1, keepdims=True)
    w = np.exp(scores)
    w /= w.sum(axis=-1, keepdims=True)
    return np.einsum("hnl,hld->nhd", w, v)


def absorb_queries(q_c, q_r, W_UK):
    """q_lat [n, H, d_c + d_r] = [W_UK[i]^T q^C_i ; q^R_i] (section 4.3.3)."""
    q_c, q_r, W_UK = _f64(q_c), _f64(q_r), _f64(W_UK)
    return np.concatenate([np.einsum("hdc,nhd->nhc", W_UK, q_c), q_r], axis=-1)


def latent_attention(q_lat, rows, scale, d_c):
    """Absorbed attention of one sequence: q_lat [n, H, D], rows [L, D]
    (D = d_c + d_r). Returns the latent outputs [n, H, d_c]."""
    q_lat, rows = _f64(q_lat), _f64(rows)
    n = q_lat.shape[0]
    L = rows.shape[0]
    scores = np.einsum("nhc,lc->hnl", q_lat, rows) * scale
    visible = np.tril(np.ones((n, L), dtype=bool), k=L - n)
    scores = np.where(visible[None], scores, -np.inf)
    scores -= scores.max(axis=-1, keepdims=True)
    w = np.exp(scores)
    w /= w.sum(axis=-1, keepdims=True)
    return np.einsum("hnl,lc->nhc", w, rows[:, :d_c])


def gather_latent(pool, table_row, L, block_size):
    """Rows 0..L-1 of one sequence from the pool [num_blocks, bs, D]."""
    pool = _f64(pool)
    t = np.arange(L)
    blocks = np.asarray(table_row)[t // block_size]
    return pool[blocks, t % block_size]


def paged_mla_attention(q_lat, pool, block_table, seq_lens, scale, d_c, block_size=16):
    """q_lat [B, n, H, D]; pool [num_blocks, bs, D]. Returns [B, n, H, d_c]."""
    q_lat = _f64(q_lat)
    table = np.asarray(_f64(block_table), dtype=np.int64)
    lens = np.asarray(_f64(seq_lens), dtype=np.int64)
    out = np.empty(q_lat.shape[:3] + (d_c,))
    for b in range(q_lat.shape[0]):
        rows = gather_latent(pool, table[b], int(lens[b]), block_size)
        out[b] = latent_attention(q_lat[b], rows, scale, d_c)
    return out


def latent_append(pool, c_new, block_table, seq_lens, block_size=16):
    """Write c_new [B, n, D] at positions L - n .. L - 1 (section 6.2 addressing:
    block pos // bs, slot pos % bs). Returns a new fp64 pool."""
    pool = _f64(pool).copy()
    c_new = _f64(c_new)
    table = np.asarray(_f64(block_table), dtype=np.int64)
    lens = np.asarray(_f64(seq_lens), dtype=np.int64)
    B, n, _ = c_new.shape
    for b in range(B):
        for j in range(n):
            pos = int(lens[b]) - n + j
            pool[table[b, pos // block_size], pos % block_size] = c_new[b, j]
    return pool


def cache_bytes(n_layers, L_ctx, d_c, d_r, bytes_per_elem=2):
    """MLA cache of one sample (section 4.4.3 / 9.1): layers * L * (d_c + d_r) * bytes."""
    return n_layers * L_ctx * (d_c + d_r) * bytes_per_elem


def default_scale(d_head, d_r):
    """The scale MLAAttention uses: 1 / sqrt(d_head + d_r) (section 6.3)."""
    return 1.0 / math.sqrt(d_head + d_r)

"""Pins of the MLA oracle ("KV Cache + Speculative Decoding", sections 4.3-4.4,
6.3, 9.1 and Q22), none of which re-types the oracle's own formula:

- brute force: the un-absorbed form against a scalar loop with math.exp;
- the absorb identity: W_UV[i] times the latent output equals the output of
  the form that rebuilds every head's keys and values;
- paged equals dense for any permutation of physical blocks;
- closed forms: zero queries give the mean of the visible latents; a single
  visible key gives that key's latent;
- causality: rows after a query's position do not move it, its own row does;
- RoPE: shifting every position by the same offset leaves the output unchanged
  (R_t^T R_s depends on s - t only), and the rotation keeps norms;
- the pages' cache figures (tests/golden/pages_numbers.json): 1152 bytes per
  token and layer, ~0.27 GB for 60 layers x 4096 tokens in fp16, ~57x / 64x
  against 128-head MHA, ~1/3.5 of the 70B GQA cache and ~1/28 of same-scale
  MHA;
- the latent append writes the right slots and nothing else.
"""
import math

import numpy as np

from oracle import mla


def rand_heads(rng, n, H, L, d_head=8, d_c=12, d_r=4):
    return dict(q_c=rng.normal(size=(n, H, d_head)), q_r=rng.normal(size=(n, H, d_r)),
                c_kv=rng.normal(size=(L, d_c)), k_r=rng.normal(size=(L, d_r)),
                W_UK=rng.normal(size=(H, d_head, d_c)) / 3, W_UV=rng.normal(size=(H, d_head, d_c)) / 3)


def test_naive_form_against_scalar_loop():
    rng = np.random.default_rng(0)
    n, H, L = 3, 2, 7
    x = rand_heads(rng, n, H, L)
    scale = 0.37
    got = mla.naive_heads_attention(scale=scale, **x)
    for j in range(n):
        for i in range(H):
            k = [[sum(x["W_UK"][i, d, c] * x["c_kv"][t, c] for c in range(12)) for d in range(8)] for t in range(L)]
            v = [[sum(x["W_UV"][i, d, c] * x["c_kv"][t, c] for c in range(12)) for d in range(8)] for t in range(L)]
            vis = L - n + j + 1
            s = []
            for t in range(vis):
                dot = sum(x["q_c"][j, i, d] * k[t][d] for d in range(8))
                dot += sum(x["q_r"][j, i, r] * x["k_r"][t, r] for r in range(4))
                s.append(dot * scale)
            m = max(s)
            e = [math.exp(a - m) for a in s]
            z = sum(e)
            for d in range(8):
                ref = sum(e[t] * v[t][d] for t in range(vis)) / z
                assert abs(got[j, i, d] - ref) < 1e-12


def test_absorb_identity():
    rng = np.random.default_rng(1)
    for n, H, L in [(1, 1, 1), (5, 4, 40), (8, 3, 9)]:
        x = rand_heads(rng, n, H, L)
        scale = mla.default_scale(8, 4)
        naive = mla.naive_heads_attention(scale=scale, **x)
        q_lat = mla.absorb_queries(x["q_c"], x["q_r"], x["W_UK"])
        rows = np.concatenate([x["c_kv"], x["k_r"]], axis=1)
        lat = mla.latent_attention(q_lat, rows, scale, 12)
        up = np.einsum("hdc,nhc->nhd", x["W_UV"], lat)
        assert np.abs(up - naive).max() < 1e-12


def make_paged(rng, lens, bs, D, spare=3):
    nblk = [(L + bs - 1) // bs for L in lens]
    nb = sum(nblk) + spare
    perm = rng.permutation(nb)
    table = -np.ones((len(lens), max(nblk)), dtype=np.int64)
    off = 0
    for b, k in enumerate(nblk):
        table[b, :k] = perm[off:off + k]
        off += k
    pool = rng.normal(size=(nb, bs, D))
    return pool, table


def test_paged_equals_dense_any_permutation():
    rng = np.random.default_rng(2)
    D, d_c, n, H = 10, 8, 4, 3
    for bs in (1, 4, 16):
        lens = [n, 17, 50]
        pool, table = make_paged(rng, lens, bs, D)
        q = rng.normal(size=(len(lens), n, H, D))
        got = mla.paged_mla_attention(q, pool, table, lens, 0.5, d_c, bs)
        for b, L in enumerate(lens):
            rows = np.stack([pool[table[b, t // bs], t % bs] for t in range(L)])
            assert np.abs(got[b] - mla.latent_attention(q[b], rows, 0.5, d_c)).max() < 1e-13


def test_closed_forms():
    rng = np.random.default_rng(3)
    L, n, H, D, d_c = 20, 4, 2, 6, 5
    rows = rng.normal(size=(L, D))
    out = mla.latent_attention(np.zeros((n, H, D)), rows, 1.0, d_c)
    for j in range(n):
        assert np.allclose(out[j], rows[: L - n + j + 1, :d_c].mean(axis=0)[None], atol=1e-14)
    one = mla.latent_attention(rng.normal(size=(1, H, D)), rows[:1], 1.0, d_c)
    assert np.allclose(one[0], rows[0, :d_c][None], atol=1e-15)


def test_causality():
    rng = np.random.default_rng(4)
    L, n, H, D, d_c = 30, 5, 2, 6, 4
    rows = rng.normal(size=(L, D))
    q = rng.normal(size=(n, H, D))
    base = mla.latent_attention(q, rows, 0.7, d_c)
    for j in range(n):
        pos = L - n + j
        later = rows.copy()
        later[pos + 1:] = rng.normal(size=later[pos + 1:].shape)
        assert np.abs(mla.latent_attention(q, later, 0.7, d_c)[j] - base[j]).max() == 0
        own = rows.copy()
        own[pos] += 1.0
        assert np.abs(mla.latent_attention(q, own, 0.7, d_c)[j] - base[j]).max() > 1e-6


def test_rope_relative_positions():
    rng = np.random.default_rng(5)
    n, H, L, d_r = 3, 2, 11, 8
    x = rand_heads(rng, n, H, L, d_r=d_r)
    qr_raw, kr_raw = x.pop("q_r"), x.pop("k_r")
    pos_k = np.arange(L)
    pos_q = pos_k[L - n:]
    outs = []
    for shift in (0, 37, 1000):
        q_r = mla.rope(qr_raw.transpose(1, 0, 2), pos_q + shift).transpose(1, 0, 2)
        k_r = mla.rope(kr_raw, pos_k + shift)
        assert np.allclose(np.linalg.norm(k_r, axis=-1), np.linalg.norm(kr_raw, axis=-1), atol=1e-12)
        outs.append(mla.naive_heads_attention(q_r=q_r, k_r=k_r, scale=0.3, **x))
    assert np.abs(outs[1] - outs[0]).max() < 1e-10 and np.abs(outs[2] - outs[0]).max() < 1e-10
    # and a rotation that ignored the position would not be invariant under a relative change
    q_r = mla.rope(qr_raw.transpose(1, 0, 2), pos_q + 5).transpose(1, 0, 2)
    k_r = mla.rope(kr_raw, pos_k)
    assert np.abs(mla.naive_heads_attention(q_r=q_r, k_r=k_r, scale=0.3, **x) - outs[0]).max() > 1e-6


def test_cache_figures_of_the_pages():
    # section 9.1: 2 bytes x (512 + 64) per token and layer
    assert mla.cache_bytes(1, 1, 512, 64) == 1152
    # section 2.2: DeepSeek-V2, 60 layers, 4096 tokens, fp16: about 0.27 GB
    gb = mla.cache_bytes(60, 4096, 512, 64) / 2 ** 30
    assert abs(gb - 0.27) < 0.01
    # against the 70B GQA shape (2 * 8 * 128 = 2048 elements per token): 1/3.5 (section 4.4.3)
    assert abs(2048 / 576 - 3.5) < 0.1


def test_latent_append_slots():
    rng = np.random.default_rng(6)
    bs, D, n = 4, 6, 3
    lens = [5, 9]
    pool, table = make_paged(rng, lens, bs, D)
    new = rng.normal(size=(2, n, D))
    out = mla.latent_append(pool, new, table, lens, bs)
    for b, L in enumerate(lens):
        rows = mla.gather_latent(out, table[b], L, bs)
        old = mla.gather_latent(pool, table[b], L, bs)
        assert np.array_equal(rows[L - n:], new[b]) and np.array_equal(rows[:L - n], old[:L - n])
    touched = {(table[b, (L - n + j) // bs], (L - n + j) % bs) for b, L in enumerate(lens) for j in range(n)}
    for blk in range(pool.shape[0]):
        for s in range(bs):
            if (blk, s) not in touched:
                assert np.array_equal(out[blk, s], pool[blk, s])


def test_golden_mla_cache_numbers():
    import json
    import os
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")))["mla_cache"]
    per_tok, sample, ratios, vs = g
    assert mla.cache_bytes(1, 1, per_tok["d_c"], per_tok["d_r"], per_tok["bytes"]) == per_tok["printed_bytes_per_token_layer"]
    gib = mla.cache_bytes(sample["n_layers"], sample["L"], sample["d_c"], sample["d_r"], sample["bytes"]) / 2 ** 30
    assert abs(gib - sample["printed_gib_approx"]) < 0.01
    mha = 2 * ratios["H"] * ratios["d_head"]
    assert round(mha / (ratios["d_c"] + ratios["d_r"])) == ratios["printed_ratio_full"]
    assert round(mha / ratios["d_c"]) == ratios["printed_ratio_latent_only"]
    assert vs["mla_elems"] == mla.cache_bytes(1, 1, 512, 64, 1)
    assert abs(vs["gqa_elems"] / vs["mla_elems"] - vs["printed_gqa_ratio"]) < 0.1   # 3.56, printed as about 3.5
    assert round(vs["mha_elems"] / vs["mla_elems"]) == vs["printed_mha_ratio"]

"""Pins for the attention oracle.

  * dense attention equals torch's scaled_dot_product_attention (fp64, CPU)
    with K/V repeated per group and the offset causal mask of
    "KV Cache + Speculative Decoding" section 6.3 (a library routine on the
    special case of a contiguous cache);
  * paged = dense for any permutation of the physical blocks, for block sizes
    16 and 1, and whatever the unused blocks hold (section 5.2);
  * K = 0 gives the mean of the visible V rows (closed form);
  * a key past a query's causal limit never changes that query's output;
  * n_new = 1 is plain decode over all L keys; G = 1 (MHA) and H_kv = 1 (MQA);
  * fp8 pools decode as code value * per-head scale.
"""
import numpy as np
import pytest
import torch

from oracle import attention, fp8


def sdpa_reference(q, Kd, Vd, scale):
    """q [n, H_q, d]; Kd, Vd [L, H_kv, d] (fp64) -> [n, H_q, d] via torch SDPA."""
    n, H_q, d = q.shape
    L, H_kv, _ = Kd.shape
    G = H_q // H_kv
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]                    # [1, H, n, d]
    kt = torch.from_numpy(Kd).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    vt = torch.from_numpy(Vd).permute(1, 0, 2).repeat_interleave(G, dim=0)[None]
    mask = torch.tril(torch.ones(n, L, dtype=torch.bool), diagonal=L - n)
    out = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    return out[0].permute(1, 0, 2).numpy()


def build_pool(Kd_list, H_kv, d, block_size, rng, spare=3, garbage=1.0):
    """Scatter dense per-sequence caches into a permuted paged pool."""
    nblk = [(K.shape[0] + block_size - 1) // block_size for K in Kd_list]
    num_blocks = sum(nblk) + spare
    perm = rng.permutation(num_blocks)
    pool = rng.normal(0, garbage, size=(num_blocks, H_kv, block_size, d))
    table = np.full((len(Kd_list), max(nblk)), -1, dtype=np.int64)
    off = 0
    for b, K in enumerate(Kd_list):
        for i in range(nblk[b]):
            phys = perm[off + i]
            table[b, i] = phys
            rows = K[i * block_size:(i + 1) * block_size]
            pool[phys, :, :rows.shape[0], :] = rows.transpose(1, 0, 2)
        off += nblk[b]
    return pool, table


@pytest.mark.parametrize("H_q,H_kv,n_new,L", [(4, 2, 5, 40), (8, 8, 3, 33), (8, 1, 6, 17),
                                             (6, 3, 1, 50), (4, 4, 16, 16)])
def test_dense_matches_sdpa(H_q, H_kv, n_new, L):
    rng = np.random.default_rng(H_q * 100 + L)
    d = 16
    q = rng.normal(size=(n_new, H_q, d))
    Kd = rng.normal(size=(L, H_kv, d))
    Vd = rng.normal(size=(L, H_kv, d))
    scale = 1 / np.sqrt(d)
    got = attention.dense_attention(q, Kd, Vd, n_new, scale)
    ref = sdpa_reference(q, Kd, Vd, scale)
    assert np.allclose(got, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("block_size", [16, 1, 5])
def test_paged_equals_dense_any_permutation(block_size):
    rng = np.random.default_rng(block_size)
    B, H_q, H_kv, d, n_new = 3, 4, 2, 8, 4
    lens = [37, 16, 5]
    Kd = [rng.normal(size=(L, H_kv, d)) for L in lens]
    Vd = [rng.normal(size=(L, H_kv, d)) for L in lens]
    q = rng.normal(size=(B, n_new, H_q, d))
    scale = 0.3
    dense = np.stack([attention.dense_attention(q[b], Kd[b], Vd[b], n_new, scale) for b in range(B)])
    for trial in range(3):
        kp, table = build_pool(Kd, H_kv, d, block_size, np.random.default_rng(trial))
        vp, table_v = build_pool(Vd, H_kv, d, block_size, np.random.default_rng(trial))
        assert (table == table_v).all()
        got = attention.verify_attention(q, kp, vp, table, np.array(lens), scale,
                                         block_size=block_size, kv_dtype="f64")
        assert np.array_equal(got, dense)
        # garbage in unused blocks / slots changes nothing
        kp2, _ = build_pool(Kd, H_kv, d, block_size, np.random.default_rng(trial), garbage=1e3)
        got2 = attention.verify_attention(q, kp2, vp, table, np.array(lens), scale,
                                          block_size=block_size, kv_dtype="f64")
        assert np.array_equal(got2, dense)


def test_zero_keys_give_mean_of_visible_values():
    rng = np.random.default_rng(0)
    L, n_new, H_q, H_kv, d = 20, 4, 4, 2, 8
    q = rng.normal(size=(n_new, H_q, d))
    Kd = np.zeros((L, H_kv, d))
    Vd = rng.normal(size=(L, H_kv, d))
    out = attention.dense_attention(q, Kd, Vd, n_new, 0.5)
    for j in range(n_new):
        vis = L - n_new + j + 1
        for h in range(H_q):
            assert np.allclose(out[j, h], Vd[:vis, h // 2].mean(axis=0), atol=1e-14)


def test_keys_past_causal_limit_do_not_matter():
    rng = np.random.default_rng(1)
    L, n_new, H_q, H_kv, d = 30, 5, 4, 2, 8
    q = rng.normal(size=(n_new, H_q, d))
    Kd = rng.normal(size=(L, H_kv, d))
    Vd = rng.normal(size=(L, H_kv, d))
    base = attention.dense_attention(q, Kd, Vd, n_new, 0.4)
    for t in range(L - n_new + 1, L):
        K2, V2 = Kd.copy(), Vd.copy()
        K2[t] += 100.0
        V2[t] -= 50.0
        out = attention.dense_attention(q, K2, V2, n_new, 0.4)
        first_seeing = t - (L - n_new)       # query j sees t iff t <= L - n_new + j
        assert np.array_equal(out[:first_seeing], base[:first_seeing])
        assert not np.allclose(out[first_seeing:], base[first_seeing:])


def test_single_query_is_plain_decode():
    rng = np.random.default_rng(2)
    L, H_q, H_kv, d = 50, 4, 2, 8
    q = rng.normal(size=(1, H_q, d))
    Kd = rng.normal(size=(L, H_kv, d))
    Vd = rng.normal(size=(L, H_kv, d))
    out = attention.dense_attention(q, Kd, Vd, 1, 0.25)
    for h in range(H_q):
        s = Kd[:, h // 2] @ q[0, h] * 0.25
        w = np.exp(s - s.max())
        w /= w.sum()
        assert np.allclose(out[0, h], w @ Vd[:, h // 2], atol=1e-14)


def test_fp8_gather_decodes_with_per_head_scale():
    rng = np.random.default_rng(3)
    num_blocks, H_kv, bs, d = 4, 2, 16, 8
    codes = rng.integers(0, 256, size=(num_blocks, H_kv, bs, d)).astype(np.uint8)
    codes[(codes & 0x7F) == 0x7F] = 0x11
    scale = np.array([0.5, 0.125])
    table = np.array([2, 0, 3])
    L = 40
    dense = attention.gather_dense(torch.from_numpy(codes), table, L, bs, scale, is_fp8=True)
    table_vals = fp8.code_values()
    for t in range(L):
        for g in range(H_kv):
            exp = table_vals[codes[table[t // bs], g, t % bs]] * scale[g]
            assert np.array_equal(dense[t, g], exp)


def test_verify_attention_with_generated_tiny_config():
    import workloads
    cfg = workloads.CONFIGS["tiny"]
    inp = workloads.make_attention_inputs(cfg, seed=0)
    out = attention.verify_attention(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_table"],
                                     inp["seq_lens"], 1 / np.sqrt(cfg.d_head), kv_dtype=cfg.kv_dtype)
    # against SDPA on the dense caches the oracle gathers
    for b in range(cfg.B):
        L = int(inp["seq_lens"][b])
        Kd = attention.gather_dense(inp["k_cache"], inp["block_table"][b].numpy(), L, 16)
        Vd = attention.gather_dense(inp["v_cache"], inp["block_table"][b].numpy(), L, 16)
        ref = sdpa_reference(inp["q"][b].double().numpy(), Kd, Vd, 1 / np.sqrt(cfg.d_head))
        assert np.allclose(out[b], ref, atol=1e-12)

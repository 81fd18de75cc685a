"""Pins of the draft-tree attention oracle ("KV Cache + Speculative
Decoding", Q14 and section 8.2: BFS-flattened tree, query j sees its
ancestors among the new positions).

- Path equivalence: node j's output equals the causal (chain) attention of
  the last query of a shorter sequence whose new positions are only the
  nodes on j's root path, in order. The chain side is the plain tril mask,
  so this checks the ancestor mask against an independent construction.
- A chain (parent j - 1) reproduces the causal result exactly.
- A star (every parent the root) sees prefix, root and itself, checked by
  building that key set by hand.
- The paged oracle with a tree equals the dense one on the gathered cache.
"""
import numpy as np
import pytest

from oracle import attention as oatt


def random_tree(rng, n):
    parent = [-1]
    for j in range(1, n):
        parent.append(int(rng.integers(0, j)))
    return parent


def make(rng, L, n_new, H_q=4, H_kv=2, d=8):
    q = rng.normal(size=(n_new, H_q, d))
    K = rng.normal(size=(L, H_kv, d))
    V = rng.normal(size=(L, H_kv, d))
    return q, K, V


@pytest.mark.parametrize("seed", range(8))
def test_path_equivalence(seed):
    rng = np.random.default_rng(seed)
    n_new = int(rng.integers(2, 12))
    L = n_new + int(rng.integers(0, 20))
    q, K, V = make(rng, L, n_new)
    parent = random_tree(rng, n_new)
    scale = 0.3
    out = oatt.dense_attention(q, K, V, n_new, scale, parent)
    prefix = L - n_new
    for j in range(n_new):
        path = sorted(oatt.ancestors(parent, j))
        Kp = np.concatenate([K[:prefix], K[[prefix + i for i in path]]])
        Vp = np.concatenate([V[:prefix], V[[prefix + i for i in path]]])
        chain = oatt.dense_attention(q[path], Kp, Vp, len(path), scale)
        assert np.allclose(out[j], chain[-1], rtol=1e-12, atol=1e-12), (seed, j, path)


def test_chain_is_causal():
    rng = np.random.default_rng(1)
    q, K, V = make(rng, 30, 7)
    chain = [-1] + list(range(6))
    assert np.array_equal(oatt.dense_attention(q, K, V, 7, 0.5, chain), oatt.dense_attention(q, K, V, 7, 0.5))


def test_star_by_hand():
    rng = np.random.default_rng(2)
    L, n_new = 12, 5
    q, K, V = make(rng, L, n_new, H_q=2, H_kv=1)
    out = oatt.dense_attention(q, K, V, n_new, 1.0, [-1, 0, 0, 0, 0])
    for j in range(n_new):
        keys = list(range(L - n_new)) + sorted({L - n_new, L - n_new + j})
        for h in range(2):
            s = K[keys, 0] @ q[j, h]
            w = np.exp(s - s.max())
            w /= w.sum()
            assert np.allclose(out[j, h], w @ V[keys, 0], rtol=1e-12, atol=1e-12)


def test_visibility_of_a_small_tree_by_hand():
    # root 0; 1, 2 children of 0; 3 child of 1; 4 child of 2  (prefix of 3 keys)
    vis = oatt.tree_visibility([-1, 0, 0, 1, 2], 8)
    expect = np.array([
        [1, 1, 1, 1, 0, 0, 0, 0],
        [1, 1, 1, 1, 1, 0, 0, 0],
        [1, 1, 1, 1, 0, 1, 0, 0],
        [1, 1, 1, 1, 1, 0, 1, 0],
        [1, 1, 1, 1, 0, 1, 0, 1],
    ], dtype=bool)
    assert np.array_equal(vis, expect)


def test_paged_tree_equals_dense():
    import torch
    rng = np.random.default_rng(3)
    B, n_new, H_q, H_kv, d, bs = 2, 6, 4, 2, 8, 4
    lens = [9, 14]
    nb = 16
    kc = torch.from_numpy(rng.normal(size=(nb, H_kv, bs, d)))
    vc = torch.from_numpy(rng.normal(size=(nb, H_kv, bs, d)))
    perm = rng.permutation(nb)
    table = np.full((B, 4), -1, dtype=np.int32)
    table[0, :3] = perm[:3]
    table[1, :4] = perm[3:7]
    q = torch.from_numpy(rng.normal(size=(B, n_new, H_q, d)))
    parents = np.array([random_tree(rng, n_new) for _ in range(B)], dtype=np.int32)
    out = oatt.verify_attention(q, kc, vc, torch.from_numpy(table), torch.tensor(lens), 0.35, bs, "f32",
                                tree_parent=torch.from_numpy(parents))
    for b in range(B):
        Kd = oatt.gather_dense(kc.numpy(), table[b], lens[b], bs)
        Vd = oatt.gather_dense(vc.numpy(), table[b], lens[b], bs)
        ref = oatt.dense_attention(q[b].numpy(), Kd, Vd, n_new, 0.35, list(parents[b]))
        assert np.allclose(out[b], ref, rtol=1e-12, atol=1e-12)

"""Pins of the tree-commit oracle (moving the accepted path next to the root).

- A chain path (nodes 1, 2, ..., n) moves nothing.
- A hand-worked case where a source row is a later destination: node 2 goes
  to the first free position and node 4 to the second, which was node 2's
  old position... (every row read before any is written).
- A dense model over random trees: the cached prefix read back through the
  table after the commit equals prefix + root + the path's rows.
"""
import numpy as np
import torch

from oracle import kv_append as oapp


def paged(rng, L, bs, H, d, nb):
    table = torch.from_numpy(rng.permutation(nb)[: (L + bs - 1) // bs].astype(np.int32))[None]
    kc = torch.from_numpy(rng.normal(size=(nb, H, bs, d)))
    vc = torch.from_numpy(rng.normal(size=(nb, H, bs, d)))
    return table, kc, vc


def rows(cache, table, L, bs):
    t = np.arange(L)
    return cache[table[0, t // bs].long(), :, t % bs]


def test_chain_path_moves_nothing():
    rng = np.random.default_rng(0)
    table, kc, vc = paged(rng, 21, 4, 2, 8, 12)
    k2, v2 = oapp.kv_tree_commit(kc, vc, table, torch.tensor([21]), 5, torch.tensor([[1, 2, 3, -1, -1]]),
                                 torch.tensor([3]), block_size=4)
    assert torch.equal(k2, kc) and torch.equal(v2, vc)


def test_hand_worked_aliasing():
    # L = 10, n_new = 5: nodes 0..4 at positions 5..9; path (2, 4): position 6
    # takes node 2 (position 7), position 7 takes node 4 (position 9)
    bs, H, d, L = 4, 1, 2, 10
    table = torch.tensor([[2, 0, 1]], dtype=torch.int32)
    kc = torch.zeros(3, H, bs, d)
    for t in range(L):
        kc[table[0, t // bs], 0, t % bs] = float(t)
    vc = -kc
    k2, v2 = oapp.kv_tree_commit(kc, vc, table, torch.tensor([L]), 5, torch.tensor([[2, 4, -1, -1, -1]]),
                                 torch.tensor([2]), block_size=bs)
    got = rows(k2, table, L, bs)[:, 0, 0].tolist()
    assert got == [0, 1, 2, 3, 4, 5, 7, 9, 8, 9]
    assert torch.equal(rows(v2, table, L, bs), -rows(k2, table, L, bs))


def test_dense_model_random_trees():
    rng = np.random.default_rng(3)
    for _ in range(20):
        n = int(rng.integers(2, 9))
        L = n + int(rng.integers(0, 30))
        bs = int(rng.choice([1, 4, 16]))
        table, kc, vc = paged(rng, L, bs, 2, 4, (L + bs - 1) // bs + 3)
        parent = [-1] + [int(rng.integers(0, j)) for j in range(1, n)]
        leaf = int(rng.integers(0, n))
        path = []
        while leaf > 0:
            path.append(leaf)
            leaf = parent[leaf]
        path = path[::-1]
        nacc = len(path)
        pad = path + [-1] * (n - nacc)
        before = rows(kc, table, L, bs)
        k2, _ = oapp.kv_tree_commit(kc, vc, table, torch.tensor([L]), n, torch.tensor([pad]),
                                    torch.tensor([nacc]), block_size=bs)
        after = rows(k2, table, L, bs)
        base = L - n
        expect = torch.cat([before[: base + 1]] + [before[base + p][None] for p in path])
        assert torch.equal(after[: base + 1 + nacc], expect)

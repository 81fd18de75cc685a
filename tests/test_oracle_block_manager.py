"""Pins of the block-manager oracle against things other than itself.

- A dense model: every sequence is a plain Python list of token values
  (fork copies the list, share_prefix copies its whole-page prefix, extend
  appends, truncate cuts). Random programs run on the oracle with a page
  store that the test fills itself (it performs the copy-on-write copies
  the oracle asks for and writes each new position through the table);
  every sequence read back through its table must equal the dense list.
  A write that lands on a shared page, a missing copy or a wrong count
  breaks that equality or one of the invariants below.
- Invariants of the counts: ref_count[p] equals the number of table entries
  naming p; the free list holds exactly the pages with count 0, once each;
  a table holds ceil(len / page_size) pages.
- Values worked out by hand from the stack discipline of the section 6.2
  sketch of "KV Cache + Speculative Decoding".
- The rollback length: after a simulated speculative round the cache holds
  every token of the sequence but the last (the invariant the first page
  states for its generation loop).
"""
import random

import pytest

from oracle.block_manager import OutOfBlocks, PagedBlockManager


def check_invariants(bm, num_blocks):
    counts = [0] * num_blocks
    for s, pages in bm.block_table.items():
        assert len(pages) == -(-bm.length[s] // bm.page_size)
        assert len(set(pages)) == len(pages)
        for p in pages:
            counts[p] += 1
    assert counts == bm.ref_count
    assert sorted(bm.free_list) == [p for p in range(num_blocks) if counts[p] == 0]


class PageStore:
    """Physical page contents, kept by the test (the caller's side)."""

    def __init__(self, num_blocks, page_size):
        self.pages = [[None] * page_size for _ in range(num_blocks)]
        self.ps = page_size

    def copy(self, src, dst):
        self.pages[dst] = list(self.pages[src])

    def write(self, bm, s, pos, value):
        self.pages[bm.block_table[s][pos // self.ps]][pos % self.ps] = value

    def read(self, bm, s):
        return [self.pages[bm.block_table[s][t // self.ps]][t % self.ps]
                for t in range(bm.length[s])]


def run_program(seed, num_blocks=48, page_size=4, steps=400):
    rng = random.Random(seed)
    bm = PagedBlockManager(num_blocks, page_size)
    store = PageStore(num_blocks, page_size)
    dense = {}
    counter = [0]
    next_id = [0]

    def fresh():
        counter[0] += 1
        return counter[0]

    def new_id():
        next_id[0] += 1
        return next_id[0]

    n_cow = 0
    for _ in range(steps):
        op = rng.choice(["alloc", "alloc", "fork", "share", "extend", "extend", "extend",
                         "truncate", "commit", "free"])
        live = sorted(dense)
        if op == "alloc" or not live:
            s, n = new_id(), rng.randrange(0, 3 * page_size + 2)
            try:
                bm.allocate(s, n)
            except OutOfBlocks:
                continue
            dense[s] = [fresh() for _ in range(n)]
            for t, v in enumerate(dense[s]):
                store.write(bm, s, t, v)
        elif op == "fork":
            src, dst = rng.choice(live), new_id()
            bm.fork(src, dst)
            dense[dst] = list(dense[src])
        elif op == "share":
            src, dst = rng.choice(live), new_id()
            n = rng.randrange(0, len(dense[src]) + 1)
            bm.share_prefix(src, dst, n)
            dense[dst] = dense[src][: (n // page_size) * page_size]
        elif op == "extend":
            ids = rng.sample(live, rng.randrange(1, min(4, len(live)) + 1))
            n_new = rng.randrange(0, 2 * page_size + 2)
            before = {s: bm.length[s] for s in ids}
            free_before = len(bm.free_list)
            need = bm._pages_needed(ids, n_new)
            try:
                pairs = bm.extend(ids, n_new)
            except OutOfBlocks:
                assert need > free_before
                assert len(bm.free_list) == free_before
                assert all(bm.length[s] == before[s] for s in ids)
                continue
            assert free_before - len(bm.free_list) == need
            n_cow += len(pairs)
            for src, dst in pairs:
                store.copy(src, dst)
            for s in ids:
                for pos in range(before[s], before[s] + n_new):
                    v = fresh()
                    dense[s].append(v)
                    store.write(bm, s, pos, v)
        elif op == "truncate":
            s = rng.choice(live)
            n = rng.randrange(0, len(dense[s]) + 1)
            bm.truncate(s, n)
            del dense[s][n:]
        elif op == "commit":
            ids = [s for s in live if len(dense[s]) >= 3]
            if not ids:
                continue
            n_new = 3
            acc = [rng.randrange(0, n_new) for _ in ids]
            bm.commit_verify(ids, n_new, acc)
            for s, a in zip(ids, acc):
                del dense[s][len(dense[s]) - n_new + a + 1:]
        else:
            s = rng.choice(live)
            bm.free(s)
            del dense[s]
        check_invariants(bm, num_blocks)
        for s in dense:
            assert store.read(bm, s) == dense[s], (seed, op, s)
    return n_cow


@pytest.mark.parametrize("seed", range(12))
def test_random_programs_match_dense_model(seed):
    n_cow = run_program(seed)
    assert n_cow > 0, "program made no copy-on-write pair; pick another seed"


def test_stack_order_by_hand():
    # pool of 5 pages, free list [0 1 2 3 4]; pops come from the end
    bm = PagedBlockManager(5, page_size=16)
    bm.allocate("a", 40)                 # 3 pages
    assert bm.block_table["a"] == [4, 3, 2]
    assert bm.free_list == [0, 1]
    bm.fork("a", "b")
    assert bm.ref_count == [0, 0, 2, 2, 2]
    # b writes position 40 (page 2, slot 8): page 2 is shared -> copy to page 1
    assert bm.extend(["b"], 1) == [(2, 1)]
    assert bm.block_table["b"] == [4, 3, 1]
    assert bm.ref_count == [0, 1, 1, 2, 2]
    # a writes 40..48: page 2 is now a's alone (no copy); 48 opens page 0
    assert bm.extend(["a"], 9) == []
    assert bm.block_table["a"] == [4, 3, 2, 0]
    assert bm.free_list == []
    with pytest.raises(OutOfBlocks):
        bm.extend(["b"], 8)              # b: 41..48 would need a fifth page
    bm.free("a")                         # releases 4 3 2 0 in table order
    assert bm.free_list == [2, 0]
    assert bm.ref_count == [0, 1, 0, 1, 1]
    bm.truncate("b", 20)                 # keep ceil(20/16) = 2 pages, release page 1
    assert bm.block_table["b"] == [4, 3]
    assert bm.free_list == [2, 0, 1]
    bm.share_prefix("b", "c", 20)        # one whole page
    assert bm.block_table["c"] == [4] and bm.length["c"] == 16
    assert bm.ref_count == [0, 0, 0, 1, 2]


def test_two_sharers_copy_once():
    # both sequences extend into the same shared page in one batch: the first
    # takes a copy, the second then owns the page alone and writes in place
    bm = PagedBlockManager(4, page_size=4)
    bm.allocate(1, 3)
    bm.fork(1, 2)
    assert bm._pages_needed([1, 2], 1) == 1
    assert bm.extend([1, 2], 1) == [(3, 2)]
    assert bm.block_table == {1: [2], 2: [3]}
    assert bm.ref_count == [0, 0, 1, 1]


def test_batch_is_all_or_nothing():
    bm = PagedBlockManager(3, page_size=2)
    bm.allocate(1, 2)
    bm.allocate(2, 2)
    state = (list(bm.free_list), list(bm.ref_count), {k: list(v) for k, v in bm.block_table.items()})
    with pytest.raises(OutOfBlocks):
        bm.extend([1, 2], 1)             # two fresh pages, one free
    assert state == (bm.free_list, bm.ref_count, bm.block_table)
    assert bm.length == {1: 2, 2: 2}


@pytest.mark.parametrize("K", [1, 4, 7])
def test_rollback_keeps_all_but_last_token(K):
    rng = random.Random(K)
    ps = 4
    bm = PagedBlockManager(64, page_size=ps)
    seq = [rng.randrange(1000) for _ in range(9)]
    bm.allocate(0, len(seq) - 1)         # the cache holds all but the last token
    cache = list(seq[:-1])
    for _ in range(20):
        drafts = [rng.randrange(1000) for _ in range(K)]
        bm.extend([0], K + 1)            # rows for [last token, d_1 .. d_K]
        cache += [seq[-1]] + drafts
        n = rng.randrange(0, K + 1)
        y = rng.randrange(1000)
        seq += drafts[:n] + [y]
        bm.commit_verify([0], K + 1, [n])
        del cache[bm.length[0]:]
        assert bm.length[0] == len(seq) - 1
        assert cache == seq[:-1]


def test_argument_errors():
    bm = PagedBlockManager(4, page_size=4)
    bm.allocate(1, 5)
    with pytest.raises(KeyError):
        bm.allocate(1, 1)
    with pytest.raises(KeyError):
        bm.extend([9], 1)
    with pytest.raises(ValueError):
        bm.extend([1, 1], 1)
    with pytest.raises(ValueError):
        bm.truncate(1, 6)
    with pytest.raises(ValueError):
        bm.share_prefix(1, 2, 6)
    with pytest.raises(ValueError):
        bm.commit_verify([1], 3, [3])
    with pytest.raises(ValueError):
        bm.table([1], 1)

"""The library's block manager (C++ behind sv_bm_*) against the oracle.

Host code only, so these run without a GPU through the C ABI: the same random
programs drive both, and after every call the free list (in order), every
reference count, every block table, every length and the copy-on-write pairs
must be identical (integer work: bit-exact). Failing calls must fail on both
sides and leave both unchanged.
"""
import random

import pytest

from oracle.block_manager import OutOfBlocks as OracleOOB
from oracle.block_manager import PagedBlockManager


@pytest.fixture(scope="module")
def sv():
    import speculative_verify_paged_gb300 as sv
    sv.build()
    sv.load_library()
    return sv


def same_state(bm, ref, ids, max_blocks):
    assert bm.free_list() == ref.free_list
    assert bm.ref_counts() == ref.ref_count
    assert bm.num_free == len(ref.free_list)
    if ids:
        table, lens = bm.block_table(ids, max_blocks)
        rows, rlens = ref.table(ids, max_blocks)
        assert table.tolist() == rows
        assert lens.tolist() == rlens
    for s in ids:
        assert bm.seq_len(s) == ref.length[s]


def both(fn_lib, fn_ref, sv):
    """Run one call on both sides; both succeed (same result) or both fail."""
    err_lib = err_ref = None
    out_lib = out_ref = None
    try:
        out_lib = fn_lib()
    except sv.OutOfBlocks:
        err_lib = "oob"
    except sv.SpecVerifyError:
        err_lib = "arg"
    try:
        out_ref = fn_ref()
    except OracleOOB:
        err_ref = "oob"
    except (KeyError, ValueError):
        err_ref = "arg"
    assert err_lib == err_ref
    assert out_lib == out_ref
    return err_lib is None


def run_program(sv, seed, page_size):
    rng = random.Random(1000 * seed + page_size)
    nb = rng.choice([8, 40, 200])
    bm = sv.BlockManager(nb, page_size)
    ref = PagedBlockManager(nb, page_size)
    max_blocks = nb + 1
    next_id = 0
    n_cow = 0
    for _ in range(300):
        live = sorted(ref.block_table)
        op = rng.choice(["alloc", "alloc", "fork", "share", "extend", "extend", "extend",
                         "truncate", "commit", "free", "bad"])
        if op == "alloc" or not live:
            next_id += 1
            n = rng.randrange(0, 4 * page_size + 3)
            both(lambda: bm.allocate(next_id, n), lambda: ref.allocate(next_id, n), sv)
        elif op == "fork":
            next_id += 1
            src = rng.choice(live)
            both(lambda: bm.fork(src, next_id), lambda: ref.fork(src, next_id), sv)
        elif op == "share":
            next_id += 1
            src = rng.choice(live)
            n = rng.randrange(0, ref.length[src] + 1)
            both(lambda: bm.share_prefix(src, next_id, n), lambda: ref.share_prefix(src, next_id, n), sv)
        elif op == "extend":
            ids = rng.sample(live, rng.randrange(1, min(6, len(live)) + 1))
            n_new = rng.randrange(0, 3 * page_size + 2)
            out = []
            if both(lambda: out.append(bm.extend(ids, n_new)) or out[-1],
                    lambda: ref.extend(ids, n_new), sv):
                n_cow += len(out[-1])
        elif op == "truncate":
            s = rng.choice(live)
            n = rng.randrange(0, ref.length[s] + 1)
            both(lambda: bm.truncate(s, n), lambda: ref.truncate(s, n), sv)
        elif op == "commit":
            n_new = rng.choice([1, 2, 5])
            ids = rng.sample(live, rng.randrange(1, len(live) + 1))
            acc = [rng.randrange(0, n_new) for _ in ids]
            both(lambda: bm.commit_verify(ids, n_new, acc), lambda: ref.commit_verify(ids, n_new, acc), sv)
        elif op == "free":
            s = rng.choice(live)
            both(lambda: bm.free(s), lambda: ref.free(s), sv)
        else:
            # argument errors: unknown id, duplicate in a batch, out-of-range sizes
            s = rng.choice(live)
            bad = rng.choice(["unknown", "dup", "trunc", "share", "commit", "exists"])
            if bad == "unknown":
                both(lambda: bm.extend([s, 10**9], 1), lambda: ref.extend([s, 10**9], 1), sv)
            elif bad == "dup":
                both(lambda: bm.extend([s, s], 1), lambda: ref.extend([s, s], 1), sv)
            elif bad == "trunc":
                n = ref.length[s] + 1
                both(lambda: bm.truncate(s, n), lambda: ref.truncate(s, n), sv)
            elif bad == "share":
                n = ref.length[s] + 1
                both(lambda: bm.share_prefix(s, 10**9, n), lambda: ref.share_prefix(s, 10**9, n), sv)
            elif bad == "commit":
                both(lambda: bm.commit_verify([s], 2, [2]), lambda: ref.commit_verify([s], 2, [2]), sv)
            else:
                both(lambda: bm.allocate(s, 1), lambda: ref.allocate(s, 1), sv)
        same_state(bm, ref, sorted(ref.block_table), max_blocks)
    return n_cow


@pytest.mark.parametrize("seed", range(10))
@pytest.mark.parametrize("page_size", [1, 4, 16])
def test_random_programs_match_oracle(sv, seed, page_size):
    run_program(sv, seed, page_size)


def test_random_programs_make_copies(sv):
    # the programs do reach copy-on-write (not every one of them does)
    assert sum(run_program(sv, seed, 4) for seed in range(4)) > 0


def test_out_of_blocks_and_errors(sv):
    bm = sv.BlockManager(3, 2)
    bm.allocate(1, 2)
    bm.allocate(2, 2)
    with pytest.raises(sv.OutOfBlocks):
        bm.extend([1, 2], 1)
    assert bm.free_list() == [0] and bm.seq_len(1) == 2
    with pytest.raises(sv.OutOfBlocks):
        bm.allocate(3, 5)
    with pytest.raises(sv.SpecVerifyError):
        bm.block_table([1], 0)
    with pytest.raises(sv.SpecVerifyError):
        bm.seq_len(7)
    with pytest.raises(sv.SpecVerifyError):
        sv.BlockManager(0, 16)
    table, lens = bm.block_table([2, 1], 3)
    assert table.tolist() == [[1, -1, -1], [2, -1, -1]] and lens.tolist() == [2, 2]
    assert bm.ref_count(-1) == -1 and bm.ref_count(3) == -1


def test_verify_rounds_at_serving_scale(sv):
    # 64 sequences of 1024..8192 tokens, 16-token pages, K = 4: eight rounds
    # of extend(K+1) + commit, with a fork of every eighth sequence first
    rng = random.Random(5)
    K, ps = 4, 16
    nb = 64 * 8192 // ps + 512
    bm = sv.BlockManager(nb, ps)
    ref = PagedBlockManager(nb, ps)
    ids = list(range(64))
    for s in ids:
        n = rng.randrange(1024, 8193)
        bm.allocate(s, n)
        ref.allocate(s, n)
    for s in ids[::8]:
        bm.fork(s, 100 + s)
        ref.fork(s, 100 + s)
    ids = ids + [100 + s for s in ids[::8]]
    for _ in range(8):
        assert bm.extend(ids, K + 1) == ref.extend(ids, K + 1)
        acc = [rng.randrange(0, K + 1) for _ in ids]
        bm.commit_verify(ids, K + 1, acc)
        ref.commit_verify(ids, K + 1, acc)
    same_state(bm, ref, ids, 8192 // ps + 8)

"""Paged verify rounds driven by the library's block manager, on the GPU.

The manager (host C++) hands out pages, the copy kernel performs its
copy-on-write pairs, the append kernel writes the K+1 new rows through the
manager's tables, the attention kernel reads them, and commit_verify rolls
the lengths back. A dense model (every sequence's K and V rows as plain
tensors, appended and cut like the sequence) is the independent check: the
rows read back through each table must equal it bit for bit, and the
attention must match the fp64 oracle within the bf16 tolerance.
"""
import math
import random

import numpy as np
import pytest
import torch

from oracle import attention as oatt
from parity_utils import attn_tolerance

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sv():
    import speculative_verify_paged_gb300 as sv
    sv.load_library()
    return sv


def gather(pool, row, L, bs):
    pos = torch.arange(L)
    return pool[row[pos // bs].long(), :, pos % bs]          # [L, H_kv, d]


def rand_bf16(gen, *shape):
    return torch.randn(*shape, generator=gen).to(torch.bfloat16)


def test_rounds_with_fork_share_and_rollback(sv):
    gen = torch.Generator().manual_seed(11)
    rng = random.Random(11)
    nb, bs, H_kv, d, H_q, K, n_layers = 320, 16, 2, 128, 8, 3, 2
    pools_cpu = [rand_bf16(gen, nb, H_kv, bs, d) for _ in range(2 * n_layers)]   # K0 V0 K1 V1
    pools = [p.to(DEV) for p in pools_cpu]
    bm = sv.BlockManager(nb, bs)
    ids = list(range(6))
    dense = {}
    for s in ids:
        L = rng.randrange(20, 400)
        bm.allocate(s, L)
        table, _ = bm.block_table([s], 64)
        dense[s] = [gather(p, table[0], L, bs) for p in pools_cpu]
    # shared pages: two forks (shared partial last pages) and a prefix share
    partial = [s for s in ids if bm.seq_len(s) % bs][:2]
    assert len(partial) == 2
    for src in partial:
        bm.fork(src, 10 + src)
        dense[10 + src] = [x.clone() for x in dense[src]]
    sh = next(s for s in ids if s not in partial)
    n_share = bm.seq_len(sh) - 5
    bm.share_prefix(sh, 20, n_share)
    keep = (n_share // bs) * bs
    dense[20] = [x[:keep].clone() for x in dense[sh]]
    ids += [10 + s for s in partial] + [20]
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    n_cow = 0
    for rnd in range(4):
        pairs = bm.extend(ids, K + 1)
        n_cow += len(pairs)
        sv.copy_blocks(pools, pairs, nb, status=status)
        table, lens = bm.block_table(ids, 64, device=DEV)
        for layer in range(n_layers):
            k_new = rand_bf16(gen, len(ids), K + 1, H_kv, d)
            v_new = rand_bf16(gen, len(ids), K + 1, H_kv, d)
            sv.kv_block_append(k_new.to(DEV), v_new.to(DEV), pools[2 * layer], pools[2 * layer + 1],
                               table, lens, block_size=bs, status=status)
            for i, s in enumerate(ids):
                dense[s][2 * layer] = torch.cat([dense[s][2 * layer], k_new[i]])
                dense[s][2 * layer + 1] = torch.cat([dense[s][2 * layer + 1], v_new[i]])
        q = rand_bf16(gen, len(ids), K + 1, H_q, d)
        out = sv.spec_verify_attn(q.to(DEV), pools[0], pools[1], table, lens, block_size=bs,
                                  status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        host = [p.cpu() for p in pools]
        t_cpu, l_cpu = table.cpu(), lens.cpu()
        for i, s in enumerate(ids):
            L = int(l_cpu[i])
            assert L == dense[s][0].shape[0]
            for j in range(2 * n_layers):
                assert torch.equal(gather(host[j], t_cpu[i], L, bs), dense[s][j]), (rnd, s, j)
        ref = oatt.verify_attention(q, host[0], host[1], t_cpu, l_cpu, 1 / math.sqrt(d), bs)
        err = np.abs(out.float().cpu().numpy() - ref).max()
        assert err <= attn_tolerance("bf16"), err
        acc = [rng.randrange(0, K + 1) for _ in ids]
        bm.commit_verify(ids, K + 1, torch.tensor(acc, dtype=torch.int32, device=DEV))
        for s, a in zip(ids, acc):
            n = dense[s][0].shape[0] - (K + 1) + a + 1
            dense[s] = [x[:n] for x in dense[s]]
            assert bm.seq_len(s) == n
    assert n_cow >= 2     # the two forks' shared partial pages were copied


def test_copy_blocks_whole_page_layout(sv):
    # one pool of [pages][page_size][layers][2][H_kv][d]: a page is 5 MB, so
    # one pair spans many CTAs; a pair with an entry out of range is skipped
    gen = torch.Generator().manual_seed(3)
    pool_cpu = rand_bf16(gen, 8, 16, 80, 2, 8, 128)
    pool = pool_cpu.to(DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sv.copy_blocks([pool], [(0, 5), (3, 7), (-1, 2), (1, 8)], 8, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 2          # SV_DEV_BAD_BLOCK
    exp = pool_cpu.clone()
    exp[5] = pool_cpu[0]
    exp[7] = pool_cpu[3]
    assert torch.equal(pool.cpu(), exp)


def test_copy_blocks_partial_page_and_many_pools(sv):
    # block_bytes below the stride copies the head of each page only; 40 pools
    # take two launches of at most 32 pool pointers
    gen = torch.Generator().manual_seed(4)
    pools_cpu = [rand_bf16(gen, 6, 2, 16, 64) for _ in range(40)]
    pools = [p.to(DEV) for p in pools_cpu]
    stride = 2 * 16 * 64 * 2
    before = sv.kernel_launches()
    sv.copy_blocks(pools, [(1, 4), (2, 0)], 6, block_bytes=stride // 2)
    torch.cuda.synchronize()
    assert sv.kernel_launches() - before == 2
    for p_cpu, p in zip(pools_cpu, pools):
        exp = p_cpu.clone()
        exp[4, 0] = p_cpu[1, 0]             # first half of a page = kv head 0
        exp[0, 0] = p_cpu[2, 0]
        assert torch.equal(p.cpu(), exp)


def test_copy_blocks_rejects_misaligned_sizes(sv):
    pool = torch.zeros(4, 24, dtype=torch.uint8, device=DEV)
    with pytest.raises(sv.SpecVerifyError):
        sv.copy_blocks([pool], [(0, 1)], 4)             # 24-byte pages

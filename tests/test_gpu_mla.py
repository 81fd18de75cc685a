"""Paged MLA verify attention and the latent append on the GPU against the
oracle (C ABI).

Inputs: absorbed queries and latent rows ~ N(0, 1) in bf16, scale
1/sqrt(128 + 64) (d_head + d_r of the pages' DeepSeek-V2 shape), block
tables of randomly permuted physical blocks, lengths ragged and not
multiples of 16. Cases cover one and several 128-row tiles (H = 128 gives
(K+1) * 128 rows), a tile smaller than 128 rows, odd row counts, a split
context (one sequence, long) merged across splits, and lengths equal to
n_new. Bar: max abs error 2e-2 against the fp64 oracle (bf16 output).
"""
import math

import numpy as np
import pytest
import torch

from oracle import mla as omla

pytestmark = pytest.mark.gpu
DEV = "cuda"
D, DC, BS = 576, 512, 16
SCALE = 1.0 / math.sqrt(128 + 64)


@pytest.fixture(scope="module")
def sv():
    import speculative_verify_paged_gb300 as sv
    sv.load_library()
    return sv


def make(B, n_new, H, lens, seed, spare=5):
    g = torch.Generator().manual_seed(seed)
    nblk = [(L + BS - 1) // BS for L in lens]
    nb = sum(nblk) + spare
    perm = torch.randperm(nb, generator=g).to(torch.int32)
    table = torch.full((B, max(nblk) + 1), -1, dtype=torch.int32)
    off = 0
    for b, k in enumerate(nblk):
        table[b, :k] = perm[off:off + k]
        off += k
    cache = torch.randn(nb, BS, D, generator=g).to(torch.bfloat16)
    q = torch.randn(B, n_new, H, D, generator=g).to(torch.bfloat16)
    return q, cache, table, torch.tensor(lens, dtype=torch.int32)


def run(sv, q, cache, table, lens):
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = sv.spec_verify_attn_mla(q.to(DEV), cache.to(DEV), table.to(DEV), lens.to(DEV), SCALE, status=st)
    torch.cuda.synchronize()
    return out, int(st.item())


CASES = [
    # B, n_new, H, lens
    (2, 5, 16, [40, 300]),              # 80 rows: one partial tile
    (3, 5, 128, [1000, 77, 2049]),      # 640 rows: five full tiles
    (2, 4, 7, [4, 33]),                 # 28 rows, a length equal to n_new
    (1, 8, 16, [6000]),                 # split context with a merge
    (4, 1, 128, [17, 16, 15, 129]),     # one new position (plain decode)
    (2, 6, 50, [500, 1234]),            # 300 rows: tiles of 128, 128, 44
]


@pytest.mark.parametrize("B,n_new,H,lens", CASES, ids=["B%d-n%d-H%d" % c[:3] for c in CASES])
def test_mla_attention_matches_oracle(sv, B, n_new, H, lens):
    q, cache, table, L = make(B, n_new, H, lens, seed=B * 100 + n_new * 10 + H)
    out, st = run(sv, q, cache, table, L)
    assert st == 0
    ref = omla.paged_mla_attention(q, cache, table, L, SCALE, DC, BS)
    err = np.abs(out.float().cpu().numpy() - ref).max()
    assert err <= 2e-2, err


@pytest.mark.parametrize("lens", [[771], [771, 2051]], ids=["one", "two"])
def test_mla_last_split_fully_masked_for_early_rows(sv, lens):
    # lengths of 3 past a split boundary: the first n_new - 3 query rows see
    # no key of the last split, whose (m, l) then reach the merge as
    # (-inf, 0) with P = 0 against that split's V rows
    B, n_new, H = len(lens), 8, 16
    q, cache, table, L = make(B, n_new, H, lens, seed=55 + B)
    R = n_new * H
    ws = sv.mla_workspace_size(B, n_new, H, table.shape[1])
    # the workspace holds fp32 partials (512) and (m, l) per (sequence,
    # split, row), then the order: S from its size, the split size from the
    # plan's rounding to whole 64-key tiles
    per_split = B * R * (512 + 2) * 4
    S = (ws - 256) // per_split
    assert S >= 2 and ws == S * per_split + 256
    bps = -(-table.shape[1] // S)
    bps = -(-bps // 4) * 4
    for Lb in lens:
        assert 0 < Lb % (16 * bps) < n_new, (Lb, bps)
    out, st = run(sv, q, cache, table, L)
    assert st == 0
    ref = omla.paged_mla_attention(q, cache, table, L, SCALE, DC, BS)
    assert np.isfinite(out.float().cpu().numpy()).all()
    err = np.abs(out.float().cpu().numpy() - ref).max()
    assert err <= 2e-2, err


def test_mla_split_plan_is_used(sv):
    # one sequence of 6000 tokens leaves most of the GPU idle without splits
    assert sv.mla_workspace_size(1, 8, 16, 376) > 0
    assert sv.mla_workspace_size(64, 5, 128, 512) == 256   # only the sequence order


def test_latent_append_then_attention(sv):
    B, n_new, H, lens = 3, 5, 32, [64, 100, 5]
    q, cache, table, L = make(B, n_new, H, lens, seed=7)
    g = torch.Generator().manual_seed(8)
    new = torch.randn(B, n_new, D, generator=g).to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    dc = cache.to(DEV)
    sv.kv_block_append_latent(new.to(DEV), dc, table.to(DEV), L.to(DEV), status=st)
    out = sv.spec_verify_attn_mla(q.to(DEV), dc, table.to(DEV), L.to(DEV), SCALE, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref_pool = omla.latent_append(cache, new, table, L, BS)
    assert np.array_equal(dc.double().cpu().numpy(), ref_pool)
    ref = omla.paged_mla_attention(q, ref_pool, table, L, SCALE, DC, BS)
    assert np.abs(out.float().cpu().numpy() - ref).max() <= 2e-2


def test_mla_bad_inputs_are_flagged(sv):
    q, cache, table, L = make(2, 5, 16, [40, 300], seed=3)
    L[0] = 3                           # shorter than n_new
    table[1, 2] = cache.shape[0] + 7   # outside the pool
    out, st = run(sv, q, cache, table, L)
    assert st & 2 and st & 1           # SV_DEV_BAD_BLOCK | SV_DEV_BAD_SEQ_LEN
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_attn_mla(q.to(DEV), cache.to(DEV), table.to(DEV), L.to(DEV), SCALE, d_c=256)


def test_mla_full_size_sampled_sequences(sv):
    # the bench's DeepSeek-V2 shape, inputs and launch (64 sequences of
    # 1024-8192 tokens, 128 heads, no splits, longest-first order); the oracle
    # checks the shortest, the longest and a middle sequence
    B, n_new, H = 64, 5, 128
    g = torch.Generator(device="cpu").manual_seed(0)
    lens = torch.randint(1024, 8193, (B,), generator=g).tolist()
    nblk = [(L + BS - 1) // BS for L in lens]
    nb = sum(nblk) + 8
    perm = torch.randperm(nb, generator=g).to(torch.int32)
    table = torch.full((B, max(nblk)), -1, dtype=torch.int32)
    off = 0
    for b, k in enumerate(nblk):
        table[b, :k] = perm[off:off + k]
        off += k
    gd = torch.Generator(device=DEV).manual_seed(0)
    cache = torch.randn((nb, BS, D), generator=gd, device=DEV).to(torch.bfloat16)
    q = torch.randn((B, n_new, H, D), generator=gd, device=DEV).to(torch.bfloat16)
    assert sv.mla_workspace_size(B, n_new, H, table.shape[1]) == 256   # one split per sequence
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = sv.spec_verify_attn_mla(q, cache, table.to(DEV), torch.tensor(lens, dtype=torch.int32, device=DEV),
                                  SCALE, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    order = np.argsort(lens)
    for b in (int(order[0]), int(order[-1]), int(order[B // 2])):
        rows = cache[table[b, :nblk[b]].long().to(DEV)].reshape(-1, D)[: lens[b]].cpu()
        ref = omla.latent_attention(q[b].cpu(), rows, SCALE, DC)
        err = np.abs(out[b].float().cpu().numpy() - ref).max()
        assert err <= 2e-2, (b, lens[b], err)

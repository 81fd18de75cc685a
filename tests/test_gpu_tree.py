"""Draft-tree verify attention on the GPU against the oracle (C ABI).

Every cache dtype path (the tcgen05 bf16 kernel, the fp8 mma.sync kernel,
the fp32 kernel) runs random BFS trees of 2 to 64 nodes against the fp64
oracle at the attention tolerances; a chain given as a tree must reproduce
the causal call bit for bit; a bad parent must be flagged; the 70B layer
shape runs with a five-node tree on sampled sequences; and a whole tree
round (append, tree attention, tree sampling, kv_tree_commit) leaves the
pools equal to the oracle's commit bit for bit.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oatt
from parity_utils import attn_tolerance

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def sv():
    import speculative_verify_paged_gb300 as sv
    sv.load_library()
    return sv


def random_trees(B, n, seed):
    rng = np.random.default_rng(seed)
    out = np.empty((B, n), dtype=np.int32)
    for b in range(B):
        out[b, 0] = -1
        for j in range(1, n):
            # mostly shallow, bushy trees (the shape speculative trees take),
            # sometimes a long branch
            out[b, j] = rng.integers(max(0, j - 3), j) if rng.random() < 0.3 else rng.integers(0, max(1, j // 2 + 1))
    return out


def run(sv, cfg, a, parents, status=None):
    st = torch.zeros(1, dtype=torch.int32, device=DEV) if status is None else status
    out = sv.spec_verify_attn(a["q"], a["k_cache"], a["v_cache"], a["block_table"], a["seq_lens"],
                              1 / math.sqrt(cfg.d_head), a["k_scale"], a["v_scale"], block_size=cfg.block_size,
                              status=st, tree_parent=parents)
    torch.cuda.synchronize()
    return out, int(st.item())


CASES = [
    ("f32", {}, 6),
    ("bf16", {"kv_dtype": "bf16", "q_dtype": "bf16", "d_head": 128}, 8),
    ("bf16_g8_n16", {"kv_dtype": "bf16", "q_dtype": "bf16", "d_head": 128, "H_q": 16, "H_kv": 2,
                     "ctx": ("fixed", (40, 700))}, 16),
    ("bf16_n64", {"kv_dtype": "bf16", "q_dtype": "bf16", "d_head": 128, "H_q": 2, "H_kv": 1,
                  "ctx": ("fixed", (64, 300))}, 64),
    ("fp8", {"kv_dtype": "fp8_e4m3", "q_dtype": "bf16", "d_head": 128, "H_q": 8, "H_kv": 2}, 8),
    ("fp8_n32", {"kv_dtype": "fp8_e4m3", "q_dtype": "bf16", "d_head": 128, "H_q": 4, "H_kv": 2,
                 "ctx": ("fixed", (100, 33))}, 32),
]


@pytest.mark.parametrize("name,over,n_new", CASES, ids=[c[0] for c in CASES])
def test_tree_matches_oracle(sv, name, over, n_new):
    cfg = workloads.CONFIGS["tiny"].with_(K=n_new - 1, **over)
    a = workloads.make_attention_inputs(cfg, seed=n_new)
    parents = random_trees(cfg.B, n_new, seed=n_new)
    g = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v) for k, v in a.items()}
    out, st = run(sv, cfg, g, torch.from_numpy(parents).to(DEV))
    assert st == 0
    ref = oatt.verify_attention(a["q"], a["k_cache"], a["v_cache"], a["block_table"], a["seq_lens"],
                                1 / math.sqrt(cfg.d_head), cfg.block_size, cfg.kv_dtype, a["k_scale"],
                                a["v_scale"], tree_parent=torch.from_numpy(parents))
    err = np.abs(out.float().cpu().numpy() - ref).max()
    assert err <= attn_tolerance(cfg.kv_dtype), "max abs error %.3g" % err


@pytest.mark.parametrize("name,over,n_new", CASES[:2] + CASES[4:5], ids=[c[0] for c in CASES[:2] + CASES[4:5]])
def test_chain_tree_is_the_causal_call(sv, name, over, n_new):
    cfg = workloads.CONFIGS["tiny"].with_(K=n_new - 1, **over)
    a = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v)
         for k, v in workloads.make_attention_inputs(cfg, seed=3).items()}
    chain = torch.arange(-1, n_new - 1, dtype=torch.int32).repeat(cfg.B, 1).to(DEV)
    out_t, st = run(sv, cfg, a, chain)
    out_c = sv.spec_verify_attn(a["q"], a["k_cache"], a["v_cache"], a["block_table"], a["seq_lens"],
                                1 / math.sqrt(cfg.d_head), a["k_scale"], a["v_scale"], block_size=cfg.block_size)
    torch.cuda.synchronize()
    assert st == 0
    assert torch.equal(out_t, out_c)


def test_bad_parent_is_flagged(sv):
    cfg = workloads.CONFIGS["tiny"].with_(K=4, kv_dtype="bf16", q_dtype="bf16", d_head=128)
    a = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v)
         for k, v in workloads.make_attention_inputs(cfg, seed=5).items()}
    parents = torch.tensor([[-1, 0, 0, 3, 1], [-1, 0, 1, 2, 3]], dtype=torch.int32, device=DEV)  # 3 -> 3
    _, st = run(sv, cfg, a, parents)
    assert st & 32


def test_tree_full_size_70b(sv):
    # the 70B layer shape with a five-node tree: root, two children, one
    # grandchild under each (K + 1 = 5 positions as in the chain workload)
    cfg = workloads.CONFIGS["llama3_70b"]
    a = workloads.make_attention_inputs(cfg, seed=0, device=DEV)
    parents = torch.tensor([-1, 0, 0, 1, 2], dtype=torch.int32).repeat(cfg.B, 1)
    out, st = run(sv, cfg, a, parents.to(DEV))
    assert st == 0
    idx = [0, 17, 40, 63]
    cpu = {k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in a.items()}
    ref = oatt.verify_attention(cpu["q"], cpu["k_cache"], cpu["v_cache"], cpu["block_table"], cpu["seq_lens"],
                                1 / math.sqrt(cfg.d_head), cfg.block_size, cfg.kv_dtype, cpu["k_scale"],
                                cpu["v_scale"], batch_indices=idx, tree_parent=parents)
    err = np.abs(out.float().cpu().numpy()[idx] - ref[idx]).max()
    assert err <= attn_tolerance(cfg.kv_dtype), "max abs error %.3g" % err


@pytest.mark.parametrize("kv", ["bf16", "fp8_e4m3", "f32"])
def test_tree_round_commit(sv, kv):
    # a full tree round: append the n node rows, tree attention, tree
    # sampling, then move the accepted paths next to the root; the pools must
    # equal the oracle's commit bit for bit
    from oracle import kv_append as oapp
    from oracle import sampling as osamp
    over = {"f32": {}, "bf16": {"kv_dtype": "bf16", "q_dtype": "bf16", "d_head": 128},
            "fp8_e4m3": {"kv_dtype": "fp8_e4m3", "q_dtype": "bf16", "d_head": 128}}[kv]
    n = 8
    cfg = workloads.CONFIGS["tiny"].with_(K=n - 1, B=4, ctx=("fixed", (40, 64, 100, 9)), V=500, **over)
    a = {k: (v.to(DEV) if isinstance(v, torch.Tensor) else v)
         for k, v in workloads.make_attention_inputs(cfg, seed=21).items()}
    new = {k: v.to(DEV) for k, v in workloads.make_append_inputs(cfg, seed=21).items()}
    sv.kv_block_append(new["k_new"], new["v_new"], a["k_cache"], a["v_cache"], a["block_table"], a["seq_lens"],
                       a["k_scale"], a["v_scale"], block_size=cfg.block_size)
    parents = torch.from_numpy(random_trees(cfg.B, n, seed=21)).to(DEV)
    out, st = run(sv, cfg, a, parents)
    assert st == 0
    g = torch.Generator().manual_seed(21)
    tl = (torch.randn(cfg.B, n, cfg.V, generator=g) * 3).to(torch.bfloat16)
    dl = (tl.float() + torch.randn(cfg.B, n, cfg.V, generator=g)).to(torch.bfloat16)
    q = torch.softmax(dl.double(), -1)
    par_h = parents.cpu()
    tok = torch.zeros(cfg.B, n, dtype=torch.int32)
    for b in range(cfg.B):
        for c in range(1, n):
            tok[b, c] = int(torch.multinomial(q[b, par_h[b, c]], 1, generator=g))
    uv = torch.rand(cfg.B, n, 2, generator=g)
    toks, nacc, path = sv.spec_verify_sample_tree(tl.to(DEV), dl.to(DEV), parents, tok.to(DEV), uv.to(DEV))
    before_k, before_v = a["k_cache"].cpu(), a["v_cache"].cpu()
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    sv.kv_tree_commit(a["k_cache"], a["v_cache"], a["block_table"], a["seq_lens"], path, nacc,
                      block_size=cfg.block_size, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ek, ev = oapp.kv_tree_commit(before_k, before_v, a["block_table"], a["seq_lens"], n, path.cpu(), nacc.cpu(),
                                 cfg.block_size)
    view = (lambda t: t.view(torch.uint8)) if kv == "fp8_e4m3" else (lambda t: t)
    assert torch.equal(view(a["k_cache"].cpu()), view(ek)) and torch.equal(view(a["v_cache"].cpu()), view(ev))
    ref = osamp.tree_rejection_sample(tl, dl, par_h, tok, uv)
    clear = ref["margin"] > 1e-5
    assert np.array_equal(nacc.cpu().numpy()[clear], ref["num_accepted"][clear])


def test_tree_verify_step_and_block_manager(sv):
    # tree_verify_step through the binding, then the manager's rollback: the
    # rows read back through the manager's table are prefix, root and path
    from oracle import kv_append as oapp
    n, bs, H_kv, d = 6, 16, 2, 128
    cfg = workloads.CONFIGS["tiny"].with_(K=n - 1, B=3, ctx=("fixed", (50, 90, 33)), V=400, kv_dtype="bf16",
                                          q_dtype="bf16", d_head=d)
    bm = sv.BlockManager(64, bs)
    for b, L in enumerate((50 - n, 90 - n, 33 - n)):
        bm.allocate(b, L)
    ids = [0, 1, 2]
    assert bm.extend(ids, n) == []
    table, lens = bm.block_table(ids, 16, device=DEV)
    assert lens.tolist() == [50, 90, 33]
    g = torch.Generator().manual_seed(8)
    kc = torch.randn(64, H_kv, bs, d, generator=g).to(torch.bfloat16).to(DEV)
    vc = torch.randn(64, H_kv, bs, d, generator=g).to(torch.bfloat16).to(DEV)
    q = torch.randn(3, n, 4, d, generator=g).to(torch.bfloat16).to(DEV)
    kn = torch.randn(3, n, H_kv, d, generator=g).to(torch.bfloat16).to(DEV)
    vn = torch.randn(3, n, H_kv, d, generator=g).to(torch.bfloat16).to(DEV)
    parents = torch.tensor([[-1, 0, 0, 1, 1, 2]] * 3, dtype=torch.int32, device=DEV)
    tl = torch.randn(3, n, cfg.V, generator=g).to(torch.bfloat16).to(DEV)
    tok = torch.randint(0, cfg.V, (3, n), generator=g, dtype=torch.int32).to(DEV)
    uv = torch.rand(3, n, 2, generator=g).to(DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    kc0 = kc.clone()
    _, toks, nacc, path = sv.tree_verify_step(q, kn, vn, kc, vc, table, lens, parents, tl, tl, tok, uv, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # the expected pools: append by the oracle, then the oracle's commit
    ka, _ = oapp.kv_block_append(kc0.cpu(), kc0.cpu(), kn.cpu(), vn.cpu(), table.cpu(), lens.cpu(), bs, "bf16")
    ek, _ = oapp.kv_tree_commit(ka, ka, table.cpu(), lens.cpu(), n, path.cpu(), nacc.cpu(), bs)
    assert torch.equal(kc.cpu(), ek)
    bm.commit_verify(ids, n, nacc)
    table2, lens2 = bm.block_table(ids, 16)
    for b in range(3):
        assert lens2[b] == lens[b].item() - n + int(nacc[b]) + 1

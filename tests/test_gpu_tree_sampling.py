"""Tree rejection sampling on the GPU against the oracle (C ABI).

Inputs follow the sampling workloads: target logits N(0, 3^2), draft logits
target + N(0, sigma^2), random BFS trees, and every child's token drawn from
its parent's draft row (siblings i.i.d., as the exactness of the sibling rule
assumes). Tokens, accepted lengths and accepted paths must equal the
oracle's. The only excuse is a sequence whose first differing decision (in
the walk's order) has its uniform within 1e-5 of that decision's boundary;
such sequences are counted against 0.01 % of the decisions compared, which
at these batch sizes allows none.
"""
import numpy as np
import pytest
import torch

from oracle import sampling as osamp
from parity_utils import MAX_EXCUSED_FRACTION, compare_tree_sampling, first_tree_difference

pytestmark = pytest.mark.gpu
DEV = "cuda"
TDT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}


@pytest.fixture(scope="module")
def sv():
    import speculative_verify_paged_gb300 as sv
    sv.load_library()
    return sv


def random_parents(rng, B, n):
    par = np.empty((B, n), dtype=np.int32)
    for b in range(B):
        par[b, 0] = -1
        for j in range(1, n):
            par[b, j] = rng.integers(0, max(1, (j + 1) // 2)) if rng.random() < 0.7 else rng.integers(0, j)
    return par


def make_inputs(B, n, V, dt, seed, sigma=1.5, T=1.0, parents=None, probs=False):
    rng = np.random.default_rng(seed)
    g = torch.Generator().manual_seed(seed)
    tl = torch.randn(B, n, V, generator=g) * 3.0
    dl = tl + torch.randn(B, n, V, generator=g) * sigma
    tl, dl = tl.to(TDT[dt]), dl.to(TDT[dt])
    par = random_parents(rng, B, n) if parents is None else np.tile(np.asarray(parents, dtype=np.int32), (B, 1))
    q = torch.softmax(dl.double() / T, dim=-1)
    tok = np.zeros((B, n), dtype=np.int32)
    for b in range(B):
        for c in range(1, n):
            tok[b, c] = int(torch.multinomial(q[b, par[b, c]], 1, generator=g))
    uv = torch.rand(B, n, 2, generator=g)
    draft = q.float() if probs else dl
    return tl, draft, torch.from_numpy(par), torch.from_numpy(tok), uv


def check(sv, tl, draft, par, tok, uv, T=1.0, probs=False, typical=None):
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    out, nacc, path = sv.spec_verify_sample_tree(tl.to(DEV), draft.to(DEV), par.to(DEV), tok.to(DEV), uv.to(DEV),
                                                 draft_is_probs=probs, temperature=T, status=st, typical=typical)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = osamp.tree_rejection_sample(tl, draft, par, tok, uv, draft_is_probs=probs, temperature=T,
                                      typical=typical)
    compare_tree_sampling(out.cpu().numpy(), nacc.cpu().numpy(), path.cpu().numpy(), ref)
    return ref


CASES = [("bf16", 1000, 8, 1.0, False), ("f32", 5000, 16, 1.0, False), ("bf16", 32000, 5, 0.7, False),
         ("f16", 777, 6, 1.3, False), ("f32", 4099, 12, 1.0, True), ("bf16", 50, 64, 1.0, False),
         ("bf16", 300, 1, 1.0, False)]


@pytest.mark.parametrize("dt,V,n,T,probs", CASES, ids=["%s-V%d-n%d" % c[:3] for c in CASES])
def test_tree_sampling_matches_oracle(sv, dt, V, n, T, probs):
    inputs = make_inputs(32, n, V, dt, seed=V + n, T=T, probs=probs)
    ref = check(sv, *inputs, T=T, probs=probs)
    if n > 1:
        assert ref["num_accepted"].max() >= 1    # some paths go below the root


def test_chain_tree_agrees_with_the_oracle_chain(sv):
    n = 5
    tl, dl, par, tok, uv = make_inputs(48, n, 3000, "bf16", seed=9, parents=[-1, 0, 1, 2, 3])
    ref = check(sv, tl, dl, par, tok, uv)
    chain = osamp.rejection_sample(tl, dl[:, :n - 1], tok[:, 1:], _chain_uniforms(uv))
    # the two oracles walk the same chain in fp64 (the tree one renormalises
    # the residual before its draw): they may part only at a decision within
    # rounding of its boundary, and no more often than the parity bar allows
    excused, n_dec = 0, 0
    for b in range(tl.shape[0]):
        n_dec += len(ref["decisions"][b])
        if (chain["num_accepted"][b] == ref["num_accepted"][b]
                and np.array_equal(chain["out_tokens"][b], ref["out_tokens"][b])):
            continue
        path = np.full(n, -1)
        path[:chain["num_accepted"][b]] = np.arange(1, chain["num_accepted"][b] + 1)
        k, m = first_tree_difference(path, chain["out_tokens"][b], int(chain["num_accepted"][b]),
                                     ref["decisions"][b])
        assert m < 1e-12, "sequence %d: the chain and tree oracles differ at decision %d (margin %.3g)" % (b, k, m)
        excused += 1
    assert excused <= MAX_EXCUSED_FRACTION * n_dec


def _chain_uniforms(uv):
    # tree node j + 1 carries chain draft j's accept uniform; node j the draw of row j
    B, n, _ = uv.shape
    out = torch.empty(B, n, 2)
    out[:, :n - 1, 0] = uv[:, 1:, 0]
    out[:, n - 1, 0] = 0.5
    out[:, :, 1] = uv[:, :, 1]
    return out


def test_tree_sampling_full_vocab(sv):
    # the 70B batch shape: 64 sequences, 128256 bf16 logits, a five-node tree
    tl, dl, par, tok, uv = make_inputs(64, 5, 128256, "bf16", seed=0, parents=[-1, 0, 0, 1, 2])
    check(sv, tl, dl, par, tok, uv)


def test_bad_tree_and_token_are_flagged(sv):
    tl, dl, par, tok, uv = make_inputs(2, 4, 100, "bf16", seed=1, parents=[-1, 0, 0, 1])
    par[1, 2] = 2
    tok[0, 1] = 100
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    sv.spec_verify_sample_tree(tl.to(DEV), dl.to(DEV), par.to(DEV), tok.to(DEV), uv.to(DEV), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & 32 and int(st.item()) & 4


@pytest.mark.parametrize("dt,V,n,T,eps,delta", [("bf16", 2000, 8, 1.0, 0.09, 0.3), ("f32", 5000, 16, 1.6, 0.05, 0.5),
                                                ("bf16", 128256, 5, 1.0, 0.09, 0.3)])
def test_typical_acceptance_matches_oracle(sv, dt, V, n, T, eps, delta):
    inputs = make_inputs(32 if V < 100000 else 16, n, V, dt, seed=V + 7, T=T)
    ref = check(sv, *inputs, T=T, typical=(eps, delta))
    assert ref["num_accepted"].max() >= 1 and (ref["num_accepted"] < n - 1).any()

"""The comparison rules themselves, on the CPU: planted differences between an
oracle result and a copy of it must be found at the right decision."""
import numpy as np
import pytest

from oracle import sampling
from parity_utils import compare_sampling, compare_tree_sampling, first_tree_difference


def _tree_case(seed, B=8, n=6, V=40):
    rng = np.random.default_rng(seed)
    tl = rng.normal(0, 2, (B, n, V))
    dl = tl + rng.normal(0, 1, (B, n, V))
    par = np.zeros((B, n), dtype=np.int64)
    par[:, 0] = -1
    for b in range(B):
        for j in range(1, n):
            par[b, j] = rng.integers(0, j)
    q = sampling.softmax(dl)
    tok = np.zeros((B, n), dtype=np.int64)
    for b in range(B):
        for j in range(1, n):
            tok[b, j] = rng.choice(V, p=q[b, par[b, j]])
    uv = rng.uniform(0, 1, (B, n, 2))
    return sampling.tree_rejection_sample(tl, dl, par, tok, uv)


def test_identical_results_agree():
    ref = _tree_case(0)
    for b in range(ref["out_tokens"].shape[0]):
        assert first_tree_difference(ref["path_nodes"][b], ref["out_tokens"][b], int(ref["num_accepted"][b]),
                                     ref["decisions"][b]) is None
    assert compare_tree_sampling(ref["out_tokens"], ref["num_accepted"], ref["path_nodes"], ref)[0] == 0


def test_a_different_draw_is_the_last_decision():
    ref = _tree_case(1)
    b = 0
    na = int(ref["num_accepted"][b])
    out = ref["out_tokens"][b].copy()
    out[na] = (out[na] + 1) % 40
    k, m = first_tree_difference(ref["path_nodes"][b], out, na, ref["decisions"][b])
    assert k == len(ref["decisions"][b]) - 1 and m == ref["decisions"][b][-1][2]


def test_a_rejected_child_taken_is_found_at_its_test():
    for seed in range(20):
        ref = _tree_case(seed)
        for b in range(ref["out_tokens"].shape[0]):
            dec = ref["decisions"][b]
            # the first rejected test: pretend the GPU accepted that child
            rej = [k for k, d in enumerate(dec) if d[1] >= 0 and not d[3]]
            if not rej:
                continue
            k0 = rej[0]
            depth = sum(1 for d in dec[:k0] if d[1] >= 0 and d[3])
            path = ref["path_nodes"][b].copy()
            path[depth] = dec[k0][1]
            path[depth + 1:] = -1
            out = ref["out_tokens"][b].copy()
            assert first_tree_difference(path, out, depth + 1, dec)[0] == k0
            return
    pytest.fail("no sequence with a rejected test")


def test_a_real_mismatch_fails_the_comparison():
    ref = _tree_case(2)
    out = ref["out_tokens"].copy()
    b = int(np.argmax(np.array([d[-1][2] for d in ref["decisions"]])))   # a draw far from its boundary
    na = int(ref["num_accepted"][b])
    out[b, na] = (out[b, na] + 1) % 40
    with pytest.raises(AssertionError, match="differs at decision"):
        compare_tree_sampling(out, ref["num_accepted"], ref["path_nodes"], ref)


def test_chain_mismatch_outside_the_margin_fails():
    rng = np.random.default_rng(3)
    B, K, V = 6, 3, 30
    tl = rng.normal(0, 2, (B, K + 1, V))
    dl = tl[:, :K] + rng.normal(0, 1, (B, K, V))
    q = sampling.softmax(dl)
    tok = np.array([[rng.choice(V, p=q[b, i]) for i in range(K)] for b in range(B)])
    uv = rng.uniform(0, 1, (B, K + 1, 2))
    ref = sampling.rejection_sample(tl, dl, tok, uv)
    assert compare_sampling(ref["out_tokens"], ref["num_accepted"], ref)[0] == 0
    bad = ref["out_tokens"].copy()
    b = int(np.argmax(ref["cdf_margin"]))
    bad[b, ref["num_accepted"][b]] = (bad[b, ref["num_accepted"][b]] + 1) % V
    with pytest.raises(AssertionError, match="drawn token differs"):
        compare_sampling(bad, ref["num_accepted"], ref)

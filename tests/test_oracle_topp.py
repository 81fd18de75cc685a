"""Pins of the top-p part of the sampling oracle.

- Sets worked out by hand on dyadic distributions (logits = log p, far from
  any boundary), including equal logits, which the reading orders by token id.
- An independent formulation: sort ascending, accumulate from the small end,
  and drop every token whose tail mass is <= 1 - top_p. In exact arithmetic
  it keeps the same set; it shares no code with the oracle's prefix search.
- Defining properties on random rows: the set reaches top_p, the set minus
  its last member does not, nothing outside outranks anything inside.
- Special cases: top_p = 1 keeps everything; a tiny top_p keeps the argmax
  (the lowest id among equal maxima); temperature changes the masses but not
  the order.
- Composition: the rejection sampler on the filtered logits gives the same
  result as on explicit renormalised p-tilde probabilities.
"""
import numpy as np
import pytest

from oracle import sampling


def nucleus_from_tail(row, top_p, T=1.0):
    """Keep tokens whose mass counted from the least likely end exceeds 1 - top_p."""
    V = len(row)
    p = sampling.softmax(np.asarray(row, dtype=np.float64), T)
    asc = sorted(range(V), key=lambda i: (row[i], -i))        # least likely first
    keep = np.zeros(V, dtype=bool)
    tail = 0.0
    Z = p.sum()
    for i in asc:
        tail += p[i]
        keep[i] = tail > (1.0 - top_p) * Z
    return keep


def as_set(mask):
    return set(np.flatnonzero(mask).tolist())


@pytest.mark.parametrize("probs,top_p,expected", [
    ([0.5, 0.25, 0.125, 0.125], 0.7, {0, 1}),
    ([0.5, 0.25, 0.125, 0.125], 0.8, {0, 1, 2}),          # equal tail: lower id first
    ([0.5, 0.25, 0.125, 0.125], 0.9, {0, 1, 2, 3}),
    ([0.25, 0.25, 0.25, 0.25], 0.6, {0, 1, 2}),
    ([0.125, 0.5, 0.125, 0.25], 0.8, {1, 3, 0}),
    ([0.125, 0.5, 0.125, 0.25], 0.3, {1}),
    ([0.0625, 0.0625, 0.875], 0.9, {2, 0}),
])
def test_sets_by_hand(probs, top_p, expected):
    logits = np.log(np.asarray(probs))
    mask, margin = sampling.top_p_nucleus(logits, top_p)
    assert as_set(mask) == expected
    assert margin > 1e-3


@pytest.mark.parametrize("seed", range(20))
def test_matches_tail_formulation_and_properties(seed):
    rng = np.random.default_rng(seed)
    V = int(rng.integers(2, 300))
    row = rng.normal(0, 3, V)
    if seed % 3 == 0:
        row = np.round(row * 2) / 2                          # many equal logits
    if seed % 4 == 1:
        row[rng.integers(0, V, V // 5)] = -np.inf
    top_p = float(rng.uniform(0.05, 0.99))
    T = float(rng.choice([0.5, 1.0, 1.7]))
    mask, margin = sampling.top_p_nucleus(row, top_p, T)
    if margin < 1e-12:
        pytest.skip("boundary case: both formulations are within rounding")
    assert as_set(mask) == as_set(nucleus_from_tail(row, top_p, T))
    p = sampling.softmax(row, T)
    inside = np.flatnonzero(mask)
    assert p[inside].sum() >= top_p * p.sum()
    order = sorted(inside.tolist(), key=lambda i: (-row[i], i))
    last = order[-1]
    assert p[inside].sum() - p[last] < top_p * p.sum()
    for o in np.flatnonzero(~mask):
        assert row[o] < row[last] or (row[o] == row[last] and o > last)


def test_special_cases():
    row = np.array([1.0, 3.0, 3.0, -2.0, -np.inf])
    assert sampling.top_p_nucleus(row, 1.0)[0].all()
    assert as_set(sampling.top_p_nucleus(row, 1e-6)[0]) == {1}
    # temperature keeps the order, changes the masses: at T = 0.25 the two
    # maxima hold almost all the mass, at T = 8 the set grows
    assert as_set(sampling.top_p_nucleus(row, 0.9, 0.25)[0]) == {1, 2}
    assert as_set(sampling.top_p_nucleus(row, 0.9, 8.0)[0]) == {0, 1, 2, 3}


def test_filtered_logits_give_renormalised_p():
    rng = np.random.default_rng(7)
    B, K, V = 3, 2, 50
    tl = rng.normal(0, 2, (B, K + 1, V))
    dl = tl[:, :K] + rng.normal(0, 1, (B, K, V))
    tok = rng.integers(0, V, (B, K))
    uv = rng.uniform(0, 1, (B, K + 1, 2))
    got = sampling.rejection_sample(tl, dl, tok, uv, top_p=0.8)
    mask, _ = sampling.top_p_nucleus(tl, 0.8)
    p = np.where(mask, sampling.softmax(tl), 0.0)
    p /= p.sum(axis=-1, keepdims=True)
    exp = sampling.verify_from_probs(p, sampling.softmax(dl), tok, uv)
    assert np.array_equal(got["out_tokens"], exp["out_tokens"])
    assert np.allclose(got["p_at_draft"], exp["p_at_draft"], rtol=1e-12, atol=0)

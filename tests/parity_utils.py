"""Comparison rules shared by the GPU parity tests.

Tolerances (fixed for the verify step):
  * attention output: max abs error <= 2e-2 (bf16 KV) / 6e-2 (fp8 KV) against
    the fp64 oracle; the fp32 cache path uses 1e-4 (fp32 accumulation over
    <= 2^17 keys, errors ~1e-6);
  * p_i(x_i), q_i(x_i): within 1e-5 relative;
  * accept / reject decisions, accepted lengths, emitted tokens: identical,
    except a sequence whose first differing decision has the uniform within
    MARGIN = 1e-5 of the acceptance ratio (accept test) or of a CDF boundary
    (the draw); such excused sequences are counted and must stay below 0.01 %
    of all decisions compared.
"""
import os

import numpy as np

MARGIN = 1e-5
MAX_EXCUSED_FRACTION = 1e-4

# (test, excused sequences, decisions compared) of every sampling comparison
# of this session; conftest prints the totals in the terminal summary
EXCUSALS = []


def _record(excused, n_dec):
    EXCUSALS.append((os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0], int(excused), int(n_dec)))


def compare_sampling(out_tokens, num_accepted, ref, p_at=None, q_at=None):
    """Returns (n_excused, n_decisions); raises AssertionError on a real mismatch."""
    tok = np.asarray(out_tokens)
    nac = np.asarray(num_accepted)
    B, K1 = tok.shape
    K = K1 - 1
    excused = 0
    for b in range(B):
        if nac[b] == ref["num_accepted"][b] and np.array_equal(tok[b], ref["out_tokens"][b]):
            continue
        n_o, n_g = int(ref["num_accepted"][b]), int(nac[b])
        if n_o != n_g:
            i = min(n_o, n_g)
            m = float(ref["accept_margin"][b, i])
            assert m < MARGIN, ("sequence %d: accept decision at position %d differs "
                                "(gpu n=%d, oracle n=%d, margin %.3g)" % (b, i, n_g, n_o, m))
        else:
            m = float(ref["cdf_margin"][b])
            assert m < MARGIN, ("sequence %d: drawn token differs (gpu %s, oracle %s, CDF margin %.3g)"
                                % (b, tok[b].tolist(), ref["out_tokens"][b].tolist(), m))
        excused += 1
    n_dec = B * K1
    _record(excused, n_dec)
    assert excused <= MAX_EXCUSED_FRACTION * n_dec, "%d excused of %d decisions" % (excused, n_dec)
    if p_at is not None and K > 0:
        p = np.asarray(p_at, dtype=np.float64)
        q = np.asarray(q_at, dtype=np.float64)
        assert np.allclose(p, ref["p_at_draft"], rtol=1e-5, atol=1e-30), \
            "p_at_draft max rel err %.3g" % np.max(np.abs(p - ref["p_at_draft"]) / np.maximum(ref["p_at_draft"], 1e-300))
        assert np.allclose(q, ref["q_at_draft"], rtol=1e-5, atol=1e-30), \
            "q_at_draft max rel err %.3g" % np.max(np.abs(q - ref["q_at_draft"]) / np.maximum(ref["q_at_draft"], 1e-300))
    return excused, n_dec


def attn_tolerance(kv_dtype):
    return {"f32": 1e-4, "bf16": 2e-2, "fp8_e4m3": 6e-2}[kv_dtype]


def first_tree_difference(path, out, nacc, decisions):
    """The first decision of the oracle's tree walk that the GPU's result
    contradicts, as (index, margin), or None when the two agree.

    decisions: the oracle's (node u, child c, margin, outcome) in walk order
    (c = -1 for the final draw, whose outcome is the drawn token). The GPU
    tests u's children in the same BFS order, so it accepted child c at depth
    d iff path[d] == c; if every test agrees, both walks end at the same node
    and only the drawn token can differ."""
    depth = 0
    for k, (u, c, m, outcome) in enumerate(decisions):
        if c >= 0:
            g_acc = depth < nacc and int(path[depth]) == c
            if g_acc != bool(outcome):
                return k, m
            if outcome:
                depth += 1
        else:
            if nacc != depth or int(out[depth]) != int(outcome):
                return k, m
    return None


def compare_tree_sampling(out_tokens, num_accepted, path_nodes, ref):
    """Tree walks against the oracle: identical, except a sequence whose first
    differing decision lies within MARGIN of its boundary; such sequences are
    counted against MAX_EXCUSED_FRACTION of all decisions compared. Returns
    (n_excused, n_decisions); raises AssertionError on a real mismatch."""
    out = np.asarray(out_tokens)
    nac = np.asarray(num_accepted)
    path = np.asarray(path_nodes)
    excused, n_dec = 0, 0
    for b in range(out.shape[0]):
        dec = ref["decisions"][b]
        n_dec += len(dec)
        same = (nac[b] == ref["num_accepted"][b] and np.array_equal(out[b], ref["out_tokens"][b])
                and np.array_equal(path[b], ref["path_nodes"][b]))
        if same:
            continue
        diff = first_tree_difference(path[b], out[b], int(nac[b]), dec)
        assert diff is not None, "sequence %d: outputs differ but every decision agrees" % b
        k, m = diff
        assert m < MARGIN, ("sequence %d differs at decision %d %s (margin %.3g): gpu %s / %s, oracle %s / %s"
                            % (b, k, dec[k][:2], m, out[b].tolist(), path[b].tolist(),
                               ref["out_tokens"][b].tolist(), ref["path_nodes"][b].tolist()))
        excused += 1
    _record(excused, n_dec)
    assert excused <= MAX_EXCUSED_FRACTION * n_dec, "%d excused of %d decisions" % (excused, n_dec)
    return excused, n_dec

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
import numpy as np

MARGIN = 1e-5
MAX_EXCUSED_FRACTION = 1e-4


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

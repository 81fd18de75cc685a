"""Closed forms the pages state for speculative decoding and KV sizing.

  * acceptance rate alpha = sum_x min(p(x), q(x)) = 1 - 0.5 * ||p - q||_1
    ("KV Cache + Speculative Decoding" section 7.2; quant67 section 4.1)
  * rejection mass = sum_x max(0, p(x) - q(x)) = 1 - alpha, the normaliser of
    the residual distribution (quant67 section 3.2)
  * E[tokens per round] = (1 - alpha^(K+1)) / (1 - alpha) under i.i.d.
    acceptance, also written as the series sum_{j<K} alpha^j (1-alpha)(j+1)
    + alpha^K (K+1) ("KV Cache + Speculative Decoding" section 7.4;
    quant67 section 4.1, Theorem 3.5)
  * speedup = E[tokens] / (1 + K c) (quant67 section 4.2, Theorem 3.8)
  * KV bytes = 2 * L * N_layers * H_kv * d_head * bytes per element (times the
    batch) ("KV Cache + Speculative Decoding" section 2.1); MLA keeps
    N_layers * L * (d_c + d_r) * bytes (same page, section 2.2)
"""
import numpy as np


def alpha(p, q):
    return float(np.minimum(p, q).sum())


def alpha_from_l1(p, q):
    return 1.0 - 0.5 * float(np.abs(np.asarray(p) - np.asarray(q)).sum())


def residual_mass(p, q):
    return float(np.maximum(0.0, np.asarray(p) - np.asarray(q)).sum())


def expected_tokens(a, K):
    if a == 1.0:
        return float(K + 1)
    return (1.0 - a ** (K + 1)) / (1.0 - a)


def expected_tokens_series(a, K):
    return sum(a ** j * (1 - a) * (j + 1) for j in range(K)) + a ** K * (K + 1)


def speedup(a, K, c):
    return expected_tokens(a, K) / (1.0 + K * c)


def accepted_length_pmf(alphas):
    """P(number of accepted drafts = j), j = 0..K, for per-position acceptance
    probabilities alphas[0..K-1] (independent positions): a truncated
    geometric law."""
    K = len(alphas)
    pmf = []
    run = 1.0
    for j in range(K):
        pmf.append(run * (1.0 - alphas[j]))
        run *= alphas[j]
    pmf.append(run)
    return pmf


def kv_cache_bytes(L, n_layers, H_kv, d_head, bytes_per_elem, batch=1):
    return 2 * L * n_layers * H_kv * d_head * bytes_per_elem * batch


def mla_cache_bytes(L, n_layers, d_c, d_r, bytes_per_elem, batch=1):
    return n_layers * L * (d_c + d_r) * bytes_per_elem * batch

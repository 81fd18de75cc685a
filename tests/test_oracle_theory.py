"""Closed forms of the oracle pinned to the numbers the pages print."""
import json
import os

import numpy as np
import pytest

from oracle import theory

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "pages_numbers.json")))
GIB = 2 ** 30


@pytest.mark.parametrize("row", GOLDEN["kv_bytes_per_sample"], ids=lambda r: r["cite"][-30:])
def test_kv_bytes_per_sample(row):
    got = theory.kv_cache_bytes(row["L"], row["n_layers"], row["H_kv"], row["d_head"], row["bytes"])
    assert got / GIB == pytest.approx(row["printed_gib"], rel=0, abs=1e-12)


def test_kv_bytes_70b_exact_integer():
    # 1.25 GiB exactly for the 70B GQA shape at 4K fp16
    assert theory.kv_cache_bytes(4096, 80, 8, 128, 2) == 1_342_177_280


@pytest.mark.parametrize("row", GOLDEN["kv_bytes_per_token"], ids=lambda r: str(r["printed"]))
def test_kv_bytes_per_token(row):
    assert theory.kv_cache_bytes(1, row["n_layers"], row["H_kv"], row["d_head"], row["bytes"]) == row["printed"]


@pytest.mark.parametrize("row", GOLDEN["kv_bytes_batch_decimal_gb"], ids=lambda r: str(r["printed_gb"]))
def test_kv_bytes_batch(row):
    got = theory.kv_cache_bytes(row["L"], row["n_layers"], row["H_kv"], row["d_head"], row["bytes"],
                                batch=row["batch"])
    assert round(got / 1e9) == row["printed_gb"]


def test_mla_bytes():
    r = GOLDEN["mla_bytes_per_sample"]
    got = theory.mla_cache_bytes(r["L"], r["n_layers"], r["d_c"], r["d_r"], r["bytes"])
    assert got == 60 * 4096 * 576 * 2
    assert got / GIB == pytest.approx(r["printed_gib_approx"], rel=r["rel_tol"])


@pytest.mark.parametrize("row", GOLDEN["expected_tokens"], ids=lambda r: r["cite"][:20])
def test_expected_tokens_worked_numbers(row):
    t = theory.expected_tokens(row["alpha"], row["K"])
    assert t == pytest.approx(row["tokens"], abs=row["tol"])
    if "speedup" in row:
        assert 1 + row["K"] * row["c"] == pytest.approx(row["cost"])
        assert theory.speedup(row["alpha"], row["K"], row["c"]) == pytest.approx(row["speedup"], abs=5e-3)


def test_expected_tokens_page_garbled_value_uses_formula():
    r = GOLDEN["expected_tokens_page_garbled"]
    t = theory.expected_tokens(r["alpha"], r["K"])
    assert t == pytest.approx(r["closed_form_tokens"], abs=5e-5)
    # the printed 1.659 is off by more than rounding: the pin is the formula
    assert abs(t - r["printed_tokens"]) > 5e-3


@pytest.mark.parametrize("a", [0.0, 0.1, 0.4, 0.7, 0.95, 1.0])
@pytest.mark.parametrize("K", [0, 1, 4, 8])
def test_expected_tokens_series_equals_closed_form(a, K):
    assert theory.expected_tokens(a, K) == pytest.approx(theory.expected_tokens_series(a, K), rel=1e-12)


def test_expected_tokens_limits():
    # alpha -> 1: K+1 tokens; alpha -> 0: one token ("KV Cache + Speculative
    # Decoding" section 7.4, limit analysis)
    assert theory.expected_tokens(1 - 1e-9, 5) == pytest.approx(6.0, rel=1e-6)
    assert theory.expected_tokens(0.0, 5) == 1.0


def test_alpha_identities_random():
    rng = np.random.default_rng(1)
    for _ in range(50):
        p = rng.dirichlet(np.ones(7))
        q = rng.dirichlet(np.ones(7))
        a = theory.alpha(p, q)
        assert a == pytest.approx(theory.alpha_from_l1(p, q), abs=1e-12)
        assert theory.residual_mass(p, q) == pytest.approx(1 - a, abs=1e-12)


def test_accepted_length_pmf_sums_to_one_and_mean():
    al = [0.7] * 4
    pmf = theory.accepted_length_pmf(al)
    assert sum(pmf) == pytest.approx(1.0)
    # emitted = accepted + 1
    mean_emitted = sum((j + 1) * pj for j, pj in enumerate(pmf))
    assert mean_emitted == pytest.approx(theory.expected_tokens(0.7, 4))

"""Top-p on the GPU against the oracle (through the C ABI).

The kernel takes the top-p decision on weights within about 2.2e-7 of their
exact values, so a cumulative mass (as a fraction of the row mass) is within
TOPP_TOL = 1e-6 of exact with room to spare. The check per row: the
kernel's set must be exactly a prefix of the oracle's order (logit
descending, ties by ascending id), and that prefix must lie between the
oracle's sets for top_p - TOPP_TOL and top_p + TOPP_TOL; when no cumulative
mass lies in that band the set is the oracle's exactly. Kept logits must be
bit-identical to the input; every other entry is -inf.

Rows are built to reach every path of the kernels: ordinary rows, rows with
many equal logits, rows whose crossing bin holds more than the 512 tokens
ranked directly (all logits equal; a dense f32 cluster), NaN and -inf
entries, logits around 3e5, a vocabulary of one, the full 128256-token
vocabulary, and rows above 188000 logits (the general kernel).
"""
import numpy as np
import pytest
import torch

import workloads
from oracle import sampling as osamp
from parity_utils import compare_sampling

pytestmark = pytest.mark.gpu
DEV = "cuda"
TDT = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}
TOPP_TOL = 1e-6


@pytest.fixture(scope="module")
def sv():
    import speculative_verify_paged_gb300 as sv
    sv.load_library()
    return sv


def band(row, top_p, T):
    """Oracle order of a row and the allowed range [k_lo, k_hi] of set sizes."""
    V = row.shape[0]
    order = np.lexsort((np.arange(V), -row))
    c = np.cumsum(osamp.softmax(row, T)[order])
    Z = c[-1]
    lo_thr, hi_thr = (top_p - TOPP_TOL) * Z, min(top_p + TOPP_TOL, 1.0) * Z
    k_lo = min(int(np.searchsorted(c, lo_thr, side="left")), V - 1) + 1
    k_hi = min(int(np.searchsorted(c, hi_thr, side="left")), V - 1) + 1
    return order, k_lo, k_hi


def check_rows(out, x, top_p, T):
    """out, x: CPU tensors [rows, V] (x as given to the kernel)."""
    xd = x.double().numpy()
    keep = ~torch.isneginf(out).numpy()
    for r in range(x.shape[0]):
        order, k_lo, k_hi = band(xd[r], top_p, T)
        k = int(keep[r].sum())
        assert k_lo <= k <= k_hi, "row %d: %d tokens kept, oracle band [%d, %d]" % (r, k, k_lo, k_hi)
        assert keep[r][order[:k]].all(), "row %d: the kept set is not a prefix of the oracle order" % r
    kept = torch.from_numpy(keep)
    xv = x.view(torch.int16 if x.element_size() == 2 else torch.int32)
    ov = out.view(torch.int16 if x.element_size() == 2 else torch.int32)
    assert torch.equal(ov[kept], xv[kept]), "kept logits must be copied bit for bit"


def rows_for(kind, rows, V, dt, seed):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, V, generator=g) * 3.0
    if kind == "ties":
        x = torch.round(x * 2) / 2
    elif kind == "equal":
        x = torch.zeros(rows, V)
    elif kind == "dense":                    # thousands of distinct values in one bin
        x = torch.rand(rows, V, generator=g) * 0.01
    elif kind == "neginf":
        x[:, ::3] = float("-inf")
    elif kind == "huge":                     # |max logit / T| above 2^18
        x = 3.0e5 + torch.randn(rows, V, generator=g) * 3.0
    elif kind == "sharp":                    # a few dominant tokens and a long tail
        x = torch.randn(rows, V, generator=g) * 1.0
        x[:, :5] += 12.0
    return x.to(dt)


CASES = [("normal", "bf16", 1000), ("normal", "f32", 1000), ("normal", "f16", 4099), ("ties", "bf16", 5000),
         ("equal", "bf16", 4096), ("equal", "f32", 3000), ("dense", "f32", 50000), ("neginf", "bf16", 777),
         ("sharp", "bf16", 32000), ("normal", "bf16", 1), ("normal", "bf16", 17), ("normal", "bf16", 128256),
         ("normal", "f32", 128256), ("huge", "f32", 5000),
         # rows above 188000 logits take the general kernel (approximate bin
         # sums to find the window, compensated sums for the cut)
         ("normal", "bf16", 200003), ("ties", "f32", 190001),
         # the largest row of the exact-bin kernel, and the first of the general one
         ("dense", "f16", 188000), ("equal", "bf16", 188001)]


@pytest.mark.parametrize("kind,dt,V", CASES, ids=["%s-%s-%d" % c for c in CASES])
@pytest.mark.parametrize("top_p,T", [(0.9, 1.0), (0.5, 0.7), (0.99, 1.6), (0.05, 1.0)])
def test_filter_matches_oracle(sv, kind, dt, V, top_p, T):
    rows = 4 if V > 50000 else 12
    x = rows_for(kind, rows, V, TDT[dt], seed=V + int(top_p * 100))
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = sv.topp_filter(x.to(DEV), top_p, T, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    check_rows(out.cpu(), x, top_p, T)


def test_filter_in_place_unaligned_and_top_p_one(sv):
    x = rows_for("normal", 6, 1001, torch.bfloat16, seed=3)     # 2002-byte rows: scalar path
    d = x.to(DEV)
    sv.topp_filter(d, 0.8, 1.0, out=d)
    torch.cuda.synchronize()
    check_rows(d.cpu(), x, 0.8, 1.0)
    y = sv.topp_filter(x.to(DEV), 1.0)
    assert torch.equal(y.cpu().view(torch.int16), x.view(torch.int16))


def test_filter_nan_is_dropped_and_flagged(sv):
    x = rows_for("normal", 3, 2000, torch.float32, seed=5)
    x[1, 7] = float("nan")
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = sv.topp_filter(x.to(DEV), 0.9, status=status).cpu()
    torch.cuda.synchronize()
    assert int(status.item()) & 16
    assert torch.isneginf(out[1, 7])
    x[1, 7] = float("-inf")
    check_rows(out, x, 0.9, 1.0)


def test_filter_is_deterministic(sv):
    x = rows_for("ties", 8, 128256, torch.bfloat16, seed=9).to(DEV)
    a = sv.topp_filter(x, 0.9)
    b = sv.topp_filter(x, 0.9)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def clear_sequences(s, top_p, T, draft_top_p, idx):
    """Sequences none of whose filtered rows has a cumulative mass within
    TOPP_TOL of top_p (their sets are the oracle's exactly)."""
    tm = osamp.top_p_nucleus(s["target_logits"][idx].cpu().double().numpy(), top_p, T)[1]
    ok = (tm > TOPP_TOL).all(axis=1)
    if draft_top_p:
        dm = osamp.top_p_nucleus(s["draft_logits"][idx].cpu().double().numpy(), top_p, T)[1]
        ok &= (dm > TOPP_TOL).all(axis=1)
    return [b for b, o in zip(idx, ok) if o]


def compare_topp_sampling(s, tok, nac, p, q, top_p, T, draft_top_p, idx, min_clear):
    # sequences with a row inside the band are left out: the oracle's set is
    # exact there and the kernel's may be its neighbour (check_rows covers
    # the filtered rows themselves)
    clear = clear_sequences(s, top_p, T, draft_top_p, idx)
    assert len(clear) >= min_clear, "%d of %d sequences clear of the top-p band" % (len(clear), len(idx))
    sub = {k: v[clear].cpu() for k, v in s.items()}
    ref = osamp.rejection_sample(sub["target_logits"], sub["draft_logits"], sub["draft_tokens"],
                                 sub["uniforms"], temperature=T, top_p=top_p, draft_top_p=draft_top_p)
    compare_sampling(tok.cpu().numpy()[clear], nac.cpu().numpy()[clear], ref, p.cpu().numpy()[clear],
                     q.cpu().numpy()[clear])


@pytest.mark.parametrize("draft_top_p", [False, True])
@pytest.mark.parametrize("dt,V,top_p,T", [("bf16", 5000, 0.9, 1.0), ("f32", 3001, 0.7, 0.8),
                                            ("bf16", 32000, 0.8, 0.6)])
def test_sampling_topp_matches_oracle(sv, dt, V, top_p, T, draft_top_p):
    cfg = workloads.CONFIGS["tiny"].with_(B=24, ctx=("fixed", (64,) * 24), V=V, K=3, logit_dtype=dt)
    s = workloads.make_sampling_inputs(cfg, seed=V)
    g = {k: v.to(DEV) for k, v in s.items()}
    tok, nac, p, q = sv.spec_verify_sample(g["target_logits"], g["draft_logits"], g["draft_tokens"],
                                           g["uniforms"], temperature=T, top_p=top_p,
                                           draft_top_p=draft_top_p)
    torch.cuda.synchronize()
    compare_topp_sampling(s, tok, nac, p, q, top_p, T, draft_top_p, list(range(cfg.B)), min_clear=8)


def test_sampling_topp_full_vocab(sv):
    # the 70B-shaped batch (B = 64, K = 4, V = 128256 bf16) at top_p = 0.9
    cfg = workloads.CONFIGS["llama3_70b"]
    s = workloads.make_sampling_inputs(cfg, seed=0, device=DEV)
    tok, nac, p, q = sv.spec_verify_sample(s["target_logits"], s["draft_logits"], s["draft_tokens"],
                                           s["uniforms"], top_p=0.9, draft_top_p=True)
    torch.cuda.synchronize()
    compare_topp_sampling(s, tok, nac, p, q, 0.9, 1.0, True, list(range(cfg.B)), min_clear=16)
    # the filtered rows themselves, for two sequences
    out = sv.topp_filter(s["target_logits"][:2].reshape(-1, cfg.V), 0.9)
    torch.cuda.synchronize()
    check_rows(out.cpu(), s["target_logits"][:2].reshape(-1, cfg.V).cpu(), 0.9, 1.0)


def test_sampling_topp_argument_errors(sv):
    cfg = workloads.CONFIGS["tiny"].with_(B=2, ctx=("fixed", (64,) * 2), V=100)
    s = {k: v.to(DEV) for k, v in workloads.make_sampling_inputs(cfg, seed=1).items()}
    for bad in (0.0, 1.5, float("nan")):
        with pytest.raises(sv.SpecVerifyError):
            sv.spec_verify_sample(s["target_logits"], s["draft_logits"], s["draft_tokens"], s["uniforms"],
                                  top_p=bad)
    probs = torch.softmax(s["draft_logits"].float(), -1)
    with pytest.raises(sv.SpecVerifyError):
        sv.spec_verify_sample(s["target_logits"], probs, s["draft_tokens"], s["uniforms"], draft_is_probs=True,
                              top_p=0.9, draft_top_p=True)

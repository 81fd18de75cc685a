"""Host-side helpers of bench.py that need no GPU: the MLA leg's oracle
timing (median-length sequence, scaled by visible keys) and the CLI."""
import sys

import torch

import bench


def test_mla_oracle_time_scales_by_visible_keys():
    B, n_new, H = 3, 5, 4
    lens = [40, 100, 700]
    nblk = [(L + 15) // 16 for L in lens]
    nb = sum(nblk)
    table = torch.full((B, max(nblk)), -1, dtype=torch.int32)
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(0)).to(torch.int32)
    off = 0
    for b, k in enumerate(nblk):
        table[b, :k] = perm[off:off + k]
        off += k
    g = torch.Generator().manual_seed(1)
    cache = torch.randn(nb, 16, 576, generator=g).to(torch.bfloat16)
    q = torch.randn(B, n_new, H, 576, generator=g).to(torch.bfloat16)
    r = bench.mla_oracle_time(q, cache, table, lens, nblk, 0.07)
    assert r["kind"] == "oracle" and r["unit"] == "us per call" and r["cores"] >= 1
    assert "sequence 1 (100 tokens)" in r["sample"]   # the median length
    keys = lambda L: sum(L - n_new + j + 1 for j in range(n_new))
    timed_s = float(r["sample"].split(", ")[1].split(" s")[0])
    assert r["value"] > 0 and r["value"] >= 1e6 * timed_s * sum(keys(L) for L in lens) / keys(100) * 0.5


def test_cli_defaults(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    a = bench.parse()
    assert a.gpus == 1 and a.impl == "ours" and not a.mla_only and a.mla_batch == 64


def test_gpus_must_match_the_launched_world(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py", "--gpus", "8"])
    a = bench.parse()
    import pytest
    with pytest.raises(SystemExit, match="WORLD_SIZE is 1"):
        bench.check_world(a, 1)
    bench.check_world(a, 8)


def test_percentiles_and_summary():
    xs = [float(i) for i in range(11)]   # 0..10 ms
    assert bench.pct(xs, 50) == 5.0 and bench.pct(xs, 10) == 1.0 and bench.pct(xs, 90) == 9.0
    assert bench.pct([3.0, 1.0], 50) == 2.0
    d = bench.dist_summary([0.1, 0.2, 0.3])
    assert abs(d["median_us"] - 200.0) < 1e-9 and d["p10_us"] < d["median_us"] < d["p90_us"]


def test_other_configs_cover_every_workload_and_the_sigma_sweep():
    got = bench.other_configs("llama3_70b", 1.5)
    names = [n for n, _ in got]
    assert {"llama3_8b", "long", "fp8"} <= set(names)
    assert sorted(sg for n, sg in got if n == "llama3_70b") == [0.5, 3.0]
    assert "tiny" not in names
